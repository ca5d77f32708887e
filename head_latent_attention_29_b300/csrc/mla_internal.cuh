// Declarations shared by the translation units of libmla (host launchers and the
// device error word).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/mla.h"

namespace mla {

// Device error word: low byte = mla_status, bits 8.. = the site that set it.
// First writer wins (atomicCAS from 0); mla_get_device_error() reads and clears.
// libmla is built as one translation unit (libmla.cu), which defines it once.
__device__ unsigned int g_device_error = 0;

enum ErrorSite : unsigned int {
  kSiteAppendIndex = 1,
  kSiteDecodeLength = 2,
  kSiteDecodeWait = 3,
  kSiteDecodeTmem = 4,
  kSitePageIndex = 5,
};

__device__ __forceinline__ void record_error(mla_status st, unsigned int site) {
  atomicCAS(&g_device_error, 0u, static_cast<unsigned int>(st) | (site << 8));
}

// Element load/store in fp32 arithmetic for the two storage types.
__device__ __forceinline__ float ld_elem(const float* p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

constexpr int kPageRows = MLA_PAGE_ROWS;  // rows per page of a paged cache

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// RoPE frequencies as turns per position, u_i = theta_i / (2 pi) with theta_i =
// base^(-2i/d_r) for i < d_r/2 (d_r <= 128): computed once on the host in double,
// held as an unevaluated fp32 sum u_hi + u_lo (about 48 bits) and passed by value
// to the kernels.
struct RopeTable {
  float u_hi[64];
  float u_lo[64];
};

inline RopeTable rope_table(int d_r, double base) {
  RopeTable t = {};
  const double two_pi = 6.283185307179586476925;
  for (int i = 0; i < d_r / 2 && i < 64; ++i) {
    const double u = pow(base, -2.0 * i / d_r) / two_pi;
    t.u_hi[i] = static_cast<float>(u);
    t.u_lo[i] = static_cast<float>(u - static_cast<double>(t.u_hi[i]));
  }
  return t;
}

// Copy the first `half` entries of the table into shared memory: reading a kernel
// parameter at a per-thread index serialises on the constant cache, a shared-memory
// read does not.  Every thread of the block calls it (it ends in __syncthreads).
__device__ __forceinline__ void rope_table_to_smem(const RopeTable& t, int half, float* s_hi, float* s_lo) {
  for (int i = threadIdx.x; i < half && i < 64; i += blockDim.x) {
    s_hi[i] = t.u_hi[i];
    s_lo[i] = t.u_lo[i];
  }
  __syncthreads();
}

// sin/cos of the rotation angle pos * theta, all in fp32: the number of turns
// pos * u is formed exactly enough with FMA-based two-product (Dekker's exact
// product, here hi = p u_hi rounded and err = fma(p, u_hi, -hi) exact), whole
// turns are dropped (x - rint(x) is exact in fp32 by Sterbenz's lemma), and only
// the fractional turn, at most half a turn, is scaled by 2 pi for sincosf.  The
// position is split into a multiple of 4096 and a remainder so that both parts
// convert to fp32 exactly for any int32 position.  Angle error ~1e-6 rad.
__device__ __forceinline__ float rope_turn_part(float p, float u_hi, float u_lo) {
  const float hi = p * u_hi;
  const float err = fmaf(p, u_hi, -hi);
  const float lo = fmaf(p, u_lo, err);
  return (hi - rintf(hi)) + lo;
}

__device__ __forceinline__ void rope_sincos(int pos, float u_hi, float u_lo, float* s, float* c) {
  const float p_hi = static_cast<float>(pos & ~4095), p_lo = static_cast<float>(pos & 4095);
  float f = rope_turn_part(p_hi, u_hi, u_lo) + rope_turn_part(p_lo, u_hi, u_lo);
  f -= rintf(f);
  sincosf(f * 6.2831853071795865f, s, c);
}

inline mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

// Raise a kernel's dynamic shared-memory limit on the current device, once per
// (device, kernel) unless a larger size is asked for later.  A kernel attribute
// belongs to one device's context, so every GPU the process uses gets its own
// call; the table is guarded, so host threads may launch concurrently.  After the
// first launch on a device no runtime configuration work remains, so a step can
// be captured in a CUDA graph once it has run eagerly there.
inline cudaError_t ensure_smem_limit(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  struct Done {
    const void* fn;
    int dev;
    size_t bytes;
  };
  constexpr int kSlots = 256;
  static std::mutex mu;
  static Done done[kSlots];
  static int n_done = 0;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < n_done; ++i) {
    if (done[i].fn == fn && done[i].dev == dev) {
      if (done[i].bytes >= bytes) return cudaSuccess;
      slot = i;
      break;
    }
  }
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (slot < 0 && n_done < kSlots) slot = n_done++;
  if (slot >= 0) done[slot] = Done{fn, dev, bytes};  // a full table only means repeated calls
  return cudaSuccess;
}

// Launch with programmatic stream serialisation (the kernel may start while the
// previous kernel in the stream drains; it synchronises with griddep_wait()).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---- host launchers (one per kernel family), defined in the .cu files -------
// block_table != nullptr: a paged pool viewed as c (c.B sequences of c.N_max = 64 x
// max_blocks rows; c.data the pool of num_pages pages)
mla_status launch_cache_append(const mla_cache& c, const void* c_kv, const void* k_r, const int32_t* seq_idx,
                               const int32_t* pos, int32_t T, float rope_base, cudaStream_t s,
                               const int32_t* block_table = nullptr, int32_t max_blocks = 0,
                               int32_t num_pages = 0);
mla_status launch_absorb_q(const void* q_nope, const void* q_rope, const int32_t* q_pos, const void* w_uk,
                           void* q_cat, int32_t B, int32_t H, int32_t d_k, int32_t d_c, int32_t d_r,
                           int32_t dtype, float rope_base, cudaStream_t s);
mla_status launch_out_up(const void* o_lat, const void* w_uv, void* o, int32_t B, int32_t H, int32_t d_c,
                         int32_t d_v, int32_t dtype, cudaStream_t s);
mla_status launch_gate(const void* h, const void* w_g, void* o, int32_t B, int32_t d_model, int32_t width,
                       int32_t dtype, cudaStream_t s);
bool headgemm_absorb_supported(int32_t d_k, int32_t d_c, int32_t d_r);
bool headgemm_out_up_supported(int32_t d_c, int32_t d_v);
// The new cache rows an absorb launch also writes (mla_absorb_q_append): as
// launch_cache_append's arguments; block_table != nullptr for a paged pool.
struct AppendRows {
  const mla_cache* cache;
  const void* c_kv;
  const void* k_r;
  const int32_t* seq_idx;
  const int32_t* pos;
  int32_t T;
  const int32_t* block_table;
  int32_t max_blocks, num_pages;
};
mla_status launch_absorb_q_tc(const void* q_nope, const void* q_rope, const int32_t* q_pos, const void* w_uk,
                              void* q_cat, int32_t B, int32_t H, int32_t d_k, int32_t d_c, int32_t d_r,
                              float rope_base, cudaStream_t s, const AppendRows* app = nullptr);
bool headgemm_gate_supported(int32_t d_model, int32_t width);
mla_status launch_gate_tc(const void* h, const void* w_g, void* o, int32_t B, int32_t d_model, int32_t width,
                          cudaStream_t s);
mla_status launch_out_up_tc(const void* o_lat, const void* w_uv, void* o, int32_t B, int32_t H, int32_t d_c,
                            int32_t d_v, cudaStream_t s);
mla_status launch_decode_f32(const float* q_cat, const mla_cache& c, const int32_t* seq_lens, int32_t H,
                             float scale, float* o_lat, float* lse, cudaStream_t s);

mla_status launch_prefill_f32(const float* q_cat, const mla_cache& c, const int32_t* q_start, int32_t S,
                              int32_t causal, int32_t H, float scale, float* o_lat, float* lse, cudaStream_t s);

// cache rows from hidden states (projection, RMSNorm, RoPE, append); block_table as
// launch_cache_append
size_t kv_down_workspace_size(int32_t T, int32_t d_model, int32_t d_c, int32_t d_r, int32_t dtype);
mla_status launch_kv_down(const mla_cache& c, const void* h, const void* w, const void* gamma, float eps,
                          const int32_t* seq_idx, const int32_t* pos, int32_t T, int32_t d_model, float rope_base,
                          void* ws, size_t ws_bytes, cudaStream_t s, const int32_t* block_table = nullptr,
                          int32_t max_blocks = 0, int32_t num_pages = 0);

// explicit (non-absorbed) prefill: K / V rebuilt per head, then causal attention
size_t prefill_explicit_workspace_size(int32_t B, int32_t start, int32_t S, int32_t H);
mla_status launch_prefill_explicit(const void* q_nope, const void* q_rope, const mla_cache& c, const void* w_uk,
                                   const void* w_uv, int32_t start, int32_t S, int32_t causal, int32_t H, float scale,
                                   float rope_base, void* ws, size_t ws_bytes, void* o, float* lse, cudaStream_t s);

// tensor-core decode and prefill (bf16): sizes and launch
void set_fault_injection(int32_t kind);
size_t decode_tc_workspace_size(int32_t B);
size_t prefill_tc_workspace_size(int32_t B, int32_t S);
mla_status launch_decode_tc(const void* q_cat, const mla_cache& c, const int32_t* seq_lens, int32_t H,
                            float scale, void* ws, size_t ws_bytes, void* o_lat, float* lse, cudaStream_t s,
                            const int32_t* block_table = nullptr, int32_t max_blocks = 0, int32_t num_pages = 0,
                            const int32_t* row_begin = nullptr);
// log-sum-exp merge of k partials over disjoint row ranges: o_parts [k][rows][d_c],
// lse_parts [k][rows]
mla_status launch_decode_merge(const void* o_parts, const float* lse_parts, int32_t k, long long rows, int32_t d_c,
                               int32_t dtype, void* o, float* lse, cudaStream_t s);
mla_status launch_prefill_tc(const void* q_cat, const mla_cache& c, const int32_t* q_start, int32_t S,
                             int32_t causal, int32_t H, float scale, void* ws, size_t ws_bytes, void* o_lat,
                             float* lse, cudaStream_t s);

}  // namespace mla

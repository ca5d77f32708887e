// extern "C" entry points of libmla: host-side validation and dispatch to the
// kernels.  Nothing here allocates device memory or synchronises the host
// (except mla_get_device_error, which reads the device error word).
#include <cstdlib>

#include <nvtx3/nvToolsExt.h>

#include "mla_internal.cuh"

namespace {

// Optional NVTX ranges around the compute entry points, so that a profiler can
// select one operation's kernels (ncu --nvtx --nvtx-include "mla_decode_attn/").
// On when MLA_NVTX=1 is in the environment at the first call; otherwise each call
// costs one predictable branch.
bool nvtx_on() {
  static const bool on = [] {
    const char* v = std::getenv("MLA_NVTX");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

struct OpRange {
  bool on;
  explicit OpRange(const char* name) : on(nvtx_on()) {
    if (on) nvtxRangePushA(name);
  }
  ~OpRange() {
    if (on) nvtxRangePop();
  }
  OpRange(const OpRange&) = delete;
  OpRange& operator=(const OpRange&) = delete;
};

using mla::aligned16;
using mla::aligned4;

bool valid_dtype(int32_t dt) { return dt == MLA_BF16 || dt == MLA_F32; }

size_t elem_size(int32_t dt) { return dt == MLA_BF16 ? 2 : 4; }

mla_status check_cache(const mla_cache* c) {
  if (c == nullptr || c->data == nullptr) return MLA_ERR_INVALID_ARG;
  if (!valid_dtype(c->dtype)) return MLA_ERR_INVALID_ARG;
  if (c->B <= 0 || c->N_max <= 0 || c->d_c <= 0 || c->d_r < 0 || (c->d_r & 1) != 0) return MLA_ERR_INVALID_ARG;
  if (c->row_stride < static_cast<int64_t>(c->d_c) + c->d_r) return MLA_ERR_INVALID_ARG;
  if ((c->row_stride * static_cast<int64_t>(elem_size(c->dtype))) % 16 != 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c->data)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Checks a paged cache and views it as the contiguous form the launchers take:
// B sequences of N_max = 64 x max_blocks rows over the page pool.
mla_status check_paged(const mla_paged_cache* p, mla_cache* view) {
  if (p == nullptr || p->data == nullptr || p->block_table == nullptr) return MLA_ERR_INVALID_ARG;
  if (!valid_dtype(p->dtype)) return MLA_ERR_INVALID_ARG;
  if (p->num_pages <= 0 || p->B <= 0 || p->max_blocks <= 0 || p->d_c <= 0 || p->d_r < 0 || (p->d_r & 1) != 0)
    return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p->max_blocks) * MLA_PAGE_ROWS > INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (p->row_stride < static_cast<int64_t>(p->d_c) + p->d_r) return MLA_ERR_INVALID_ARG;
  if ((p->row_stride * static_cast<int64_t>(elem_size(p->dtype))) % 16 != 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(p->data) || !aligned4(p->block_table)) return MLA_ERR_INVALID_ARG;
  view->data = p->data;
  view->dtype = p->dtype;
  view->B = p->B;
  view->N_max = p->max_blocks * MLA_PAGE_ROWS;
  view->d_c = p->d_c;
  view->d_r = p->d_r;
  view->_pad = 0;
  view->row_stride = p->row_stride;
  return MLA_OK;
}

// Shared checks and dispatch of the two kv_down entry points (view = the cache as
// the launchers take it; block_table etc. set for a paged pool).
mla_status kv_down(const mla_cache& view, const void* h, const void* w, const void* gamma, float eps,
                   const int32_t* seq_idx, const int32_t* pos, int32_t T, int32_t d_model, float rope_base,
                   void* ws, size_t ws_bytes, void* stream, const int32_t* block_table = nullptr,
                   int32_t max_blocks = 0, int32_t num_pages = 0) {
  if (T < 0 || d_model <= 0) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (h == nullptr || w == nullptr || gamma == nullptr || seq_idx == nullptr || pos == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !(eps < INFINITY)) return MLA_ERR_INVALID_ARG;  // also rejects NaN
  if (!(rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  if (view.d_r > 128 || (view.d_c & 1) != 0 || view.d_c + view.d_r > 1024) return MLA_ERR_UNSUPPORTED;
  return mla::launch_kv_down(view, h, w, gamma, eps, seq_idx, pos, T, d_model, rope_base, ws, ws_bytes,
                             as_stream(stream), block_table, max_blocks, num_pages);
}

}  // namespace

extern "C" {

MLA_API int32_t mla_abi_version(void) { return 1; }

#ifndef MLA_SOURCE_HASH
#define MLA_SOURCE_HASH "unknown"
#endif
// Tagged so that the build can read it from the library file without loading it.
static const char kSourceHashTag[] = "MLA-SOURCE-HASH:" MLA_SOURCE_HASH;
MLA_API const char* mla_build_source_hash(void) { return kSourceHashTag + 16; }

MLA_API const char* mla_status_string(mla_status st) {
  switch (st) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: invalid argument";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: no kernel for this shape/dtype";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: CUDA call failed";
    case MLA_ERR_DEVICE_TIMEOUT: return "MLA_ERR_DEVICE_TIMEOUT: a kernel's bounded wait expired";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MLA_ERR_DEVICE_INDEX: return "MLA_ERR_DEVICE_INDEX: device-side index or length out of range";
  }
  return "MLA_ERR_UNKNOWN";
}

MLA_API mla_status mla_cache_append(const mla_cache* cache, const void* c_kv, const void* k_r,
                                    const int32_t* seq_idx, const int32_t* pos, int32_t T, float rope_base,
                                    void* stream) {
  const OpRange range("mla_cache_append");
  mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  if (T < 0) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (c_kv == nullptr || seq_idx == nullptr || pos == nullptr) return MLA_ERR_INVALID_ARG;
  if (cache->d_r > 0 && k_r == nullptr) return MLA_ERR_INVALID_ARG;
  if (!(rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  if (cache->d_r > 128) return MLA_ERR_UNSUPPORTED;
  return mla::launch_cache_append(*cache, c_kv, k_r, seq_idx, pos, T, rope_base, as_stream(stream));
}

MLA_API mla_status mla_absorb_q(const void* q_nope, const void* q_rope, const int32_t* q_pos, const void* w_uk,
                                void* q_cat, int32_t B, int32_t H, int32_t d_k, int32_t d_c, int32_t d_r,
                                int32_t dtype, float rope_base, void* stream) {
  const OpRange range("mla_absorb_q");
  if (!valid_dtype(dtype)) return MLA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || d_k <= 0 || d_c <= 0 || d_r < 0 || (d_r & 1) != 0) return MLA_ERR_INVALID_ARG;
  if (q_nope == nullptr || w_uk == nullptr || q_cat == nullptr || q_pos == nullptr) return MLA_ERR_INVALID_ARG;
  if (d_r > 0 && q_rope == nullptr) return MLA_ERR_INVALID_ARG;
  if (!(rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  if (d_r > 128) return MLA_ERR_UNSUPPORTED;
  if (dtype == MLA_BF16) {
    // bf16 runs on the tensor cores only: a shape or an alignment outside that
    // kernel is an error, never a silent switch to the CUDA-core kernel
    if (!mla::headgemm_absorb_supported(d_k, d_c, d_r)) return MLA_ERR_UNSUPPORTED;
    if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_cat) || (d_r > 0 && !aligned4(q_rope)))
      return MLA_ERR_INVALID_ARG;
    return mla::launch_absorb_q_tc(q_nope, q_rope, q_pos, w_uk, q_cat, B, H, d_k, d_c, d_r, rope_base,
                                   as_stream(stream));
  }
  if (static_cast<size_t>(32) * d_k * sizeof(float) > 200 * 1024) return MLA_ERR_UNSUPPORTED;
  return mla::launch_absorb_q(q_nope, q_rope, q_pos, w_uk, q_cat, B, H, d_k, d_c, d_r, dtype, rope_base,
                              as_stream(stream));
}

namespace {

// mla_absorb_q_append on a (contiguous or paged) cache view
mla_status absorb_q_append(const mla_cache& c, const void* c_kv, const void* k_r, const int32_t* seq_idx,
                           const int32_t* pos, int32_t T, const void* q_nope, const void* q_rope,
                           const int32_t* q_pos, const void* w_uk, void* q_cat, int32_t B, int32_t H, int32_t d_k,
                           float rope_base, void* stream, const int32_t* block_table, int32_t max_blocks,
                           int32_t num_pages) {
  const int32_t d_c = c.d_c, d_r = c.d_r;
  if (T < 0 || B <= 0 || H <= 0 || d_k <= 0) return MLA_ERR_INVALID_ARG;
  if (q_nope == nullptr || w_uk == nullptr || q_cat == nullptr || q_pos == nullptr) return MLA_ERR_INVALID_ARG;
  if (d_r > 0 && q_rope == nullptr) return MLA_ERR_INVALID_ARG;
  if (T > 0 && (c_kv == nullptr || seq_idx == nullptr || pos == nullptr || (d_r > 0 && k_r == nullptr)))
    return MLA_ERR_INVALID_ARG;
  if (!(rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  if (d_r > 128) return MLA_ERR_UNSUPPORTED;
  const cudaStream_t s = as_stream(stream);
  if (c.dtype == MLA_BF16) {
    // bf16: one tensor-core launch or MLA_ERR_UNSUPPORTED, as mla_absorb_q
    if (!mla::headgemm_absorb_supported(d_k, d_c, d_r)) return MLA_ERR_UNSUPPORTED;
    if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_cat) || (d_r > 0 && !aligned4(q_rope)) ||
        (T > 0 && (!aligned16(c_kv) || (d_r > 0 && !aligned4(k_r)))))
      return MLA_ERR_INVALID_ARG;
    const mla::AppendRows app = {&c, c_kv, k_r, seq_idx, pos, T, block_table, max_blocks, num_pages};
    return mla::launch_absorb_q_tc(q_nope, q_rope, q_pos, w_uk, q_cat, B, H, d_k, d_c, d_r, rope_base, s,
                                   T > 0 ? &app : nullptr);
  }
  // fp32: the CUDA-core append and absorb kernels, one after the other
  if (static_cast<size_t>(32) * d_k * sizeof(float) > 200 * 1024) return MLA_ERR_UNSUPPORTED;
  if (T > 0) {
    const mla_status st =
        mla::launch_cache_append(c, c_kv, k_r, seq_idx, pos, T, rope_base, s, block_table, max_blocks, num_pages);
    if (st != MLA_OK) return st;
  }
  return mla::launch_absorb_q(q_nope, q_rope, q_pos, w_uk, q_cat, B, H, d_k, d_c, d_r, MLA_F32, rope_base, s);
}

}  // namespace

MLA_API mla_status mla_absorb_q_append(const mla_cache* cache, const void* c_kv, const void* k_r,
                                       const int32_t* seq_idx, const int32_t* pos, int32_t T, const void* q_nope,
                                       const void* q_rope, const int32_t* q_pos, const void* w_uk, void* q_cat,
                                       int32_t B, int32_t H, int32_t d_k, float rope_base, void* stream) {
  const OpRange range("mla_absorb_q_append");
  const mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  return absorb_q_append(*cache, c_kv, k_r, seq_idx, pos, T, q_nope, q_rope, q_pos, w_uk, q_cat, B, H, d_k,
                         rope_base, stream, nullptr, 0, 0);
}

MLA_API mla_status mla_absorb_q_append_paged(const mla_paged_cache* cache, const void* c_kv, const void* k_r,
                                             const int32_t* seq_idx, const int32_t* pos, int32_t T,
                                             const void* q_nope, const void* q_rope, const int32_t* q_pos,
                                             const void* w_uk, void* q_cat, int32_t B, int32_t H, int32_t d_k,
                                             float rope_base, void* stream) {
  const OpRange range("mla_absorb_q_append_paged");
  mla_cache view;
  const mla_status st = check_paged(cache, &view);
  if (st != MLA_OK) return st;
  return absorb_q_append(view, c_kv, k_r, seq_idx, pos, T, q_nope, q_rope, q_pos, w_uk, q_cat, B, H, d_k,
                         rope_base, stream, cache->block_table, cache->max_blocks, cache->num_pages);
}

MLA_API size_t mla_decode_workspace_size(int32_t B, int32_t H, int32_t d_c, int32_t dtype) {
  if (B <= 0 || H <= 0 || d_c <= 0) return 0;
  if (dtype == MLA_F32) return 256;  // the fp32 path needs no scratch; a token size keeps the API uniform
  if (dtype == MLA_BF16 && d_c == 512 && H <= 128) return mla::decode_tc_workspace_size(B);
  return 0;
}

MLA_API mla_status mla_decode_attn(const void* q_cat, const mla_cache* cache, const int32_t* seq_lens, int32_t H,
                                   float scale, void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                                   void* stream) {
  const OpRange range("mla_decode_attn");
  mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  if (q_cat == nullptr || seq_lens == nullptr || o_lat == nullptr || H <= 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_cat) || !aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  if (!(scale > 0.f) && !(scale < 0.f) && scale != 0.f) return MLA_ERR_INVALID_ARG;  // NaN
  if (cache->dtype == MLA_F32) {
    if (cache->d_c > 1024 || cache->d_r > 256 || H > 1024) return MLA_ERR_UNSUPPORTED;
    return mla::launch_decode_f32(static_cast<const float*>(q_cat), *cache, seq_lens, H, scale,
                                  static_cast<float*>(o_lat), lse, as_stream(stream));
  }
  if (cache->d_c != 512 || (cache->d_r != 0 && cache->d_r != 64) || H > 128) return MLA_ERR_UNSUPPORTED;
  return mla::launch_decode_tc(q_cat, *cache, seq_lens, H, scale, workspace, workspace_bytes, o_lat, lse,
                               as_stream(stream));
}

MLA_API mla_status mla_decode_attn_partial(const void* q_cat, const mla_cache* cache, const int32_t* row_begin,
                                           const int32_t* row_end, int32_t H, float scale, void* workspace,
                                           size_t workspace_bytes, void* o_part, float* lse_part, void* stream) {
  const OpRange range("mla_decode_attn_partial");
  mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  if (q_cat == nullptr || row_begin == nullptr || row_end == nullptr || o_part == nullptr || lse_part == nullptr ||
      H <= 0)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_cat) || !aligned16(o_part) || !aligned4(row_begin) || !aligned4(row_end) || !aligned4(lse_part))
    return MLA_ERR_INVALID_ARG;
  if (!(scale > 0.f) && !(scale < 0.f) && scale != 0.f) return MLA_ERR_INVALID_ARG;  // NaN
  if (cache->dtype != MLA_BF16 || cache->d_c != 512 || (cache->d_r != 0 && cache->d_r != 64) || H > 128)
    return MLA_ERR_UNSUPPORTED;
  return mla::launch_decode_tc(q_cat, *cache, row_end, H, scale, workspace, workspace_bytes, o_part, lse_part,
                               as_stream(stream), nullptr, 0, 0, row_begin);
}

MLA_API mla_status mla_decode_merge(const void* o_parts, const float* lse_parts, int32_t k, int32_t B, int32_t H,
                                    int32_t d_c, int32_t dtype, void* o_lat, float* lse, void* stream) {
  const OpRange range("mla_decode_merge");
  if (!valid_dtype(dtype)) return MLA_ERR_INVALID_ARG;
  if (o_parts == nullptr || lse_parts == nullptr || o_lat == nullptr) return MLA_ERR_INVALID_ARG;
  if (k <= 0 || B <= 0 || H <= 0 || d_c <= 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o_lat) || !aligned4(lse_parts) || (lse != nullptr && !aligned4(lse)))
    return MLA_ERR_INVALID_ARG;
  if (d_c % 8 != 0) return MLA_ERR_UNSUPPORTED;
  return mla::launch_decode_merge(o_parts, lse_parts, k, static_cast<long long>(B) * H, d_c, dtype, o_lat, lse,
                                  as_stream(stream));
}

MLA_API size_t mla_prefill_workspace_size(int32_t B, int32_t S, int32_t H, int32_t d_c, int32_t dtype) {
  if (B <= 0 || S <= 0 || H <= 0 || d_c <= 0) return 0;
  if (dtype == MLA_F32) return 256;
  if (dtype == MLA_BF16 && d_c == 512 && H <= 128) return mla::prefill_tc_workspace_size(B, S);
  return 0;
}

MLA_API mla_status mla_prefill_attn(const void* q_cat, const mla_cache* cache, const int32_t* q_start, int32_t S,
                                    int32_t H, float scale, int32_t causal, void* workspace,
                                    size_t workspace_bytes, void* o_lat, float* lse, void* stream) {
  const OpRange range("mla_prefill_attn");
  mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  if (q_cat == nullptr || q_start == nullptr || o_lat == nullptr || H <= 0 || S <= 0) return MLA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_cat) || !aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  if (!(scale > 0.f) && !(scale < 0.f) && scale != 0.f) return MLA_ERR_INVALID_ARG;  // NaN
  if (S > cache->N_max) return MLA_ERR_INVALID_ARG;
  if (static_cast<long long>(cache->B) * S > 0x7fffffffll) return MLA_ERR_UNSUPPORTED;
  if (cache->dtype == MLA_F32) {
    if (cache->d_c > 1024 || cache->d_r > 256 || H > 65535) return MLA_ERR_UNSUPPORTED;
    return mla::launch_prefill_f32(static_cast<const float*>(q_cat), *cache, q_start, S, causal, H, scale,
                                   static_cast<float*>(o_lat), lse, as_stream(stream));
  }
  if (cache->d_c != 512 || (cache->d_r != 0 && cache->d_r != 64) || H > 128) return MLA_ERR_UNSUPPORTED;
  return mla::launch_prefill_tc(q_cat, *cache, q_start, S, causal, H, scale, workspace, workspace_bytes, o_lat,
                                lse, as_stream(stream));
}

MLA_API mla_status mla_out_up(const void* o_lat, const void* w_uv, void* o, int32_t B, int32_t H, int32_t d_c,
                              int32_t d_v, int32_t dtype, void* stream) {
  const OpRange range("mla_out_up");
  if (!valid_dtype(dtype)) return MLA_ERR_INVALID_ARG;
  if (o_lat == nullptr || w_uv == nullptr || o == nullptr) return MLA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || d_c <= 0 || d_v <= 0) return MLA_ERR_INVALID_ARG;
  if (dtype == MLA_BF16) {  // tensor cores only (no silent CUDA-core fallback)
    if (!mla::headgemm_out_up_supported(d_c, d_v)) return MLA_ERR_UNSUPPORTED;
    if (!aligned16(o_lat) || !aligned16(w_uv) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
    return mla::launch_out_up_tc(o_lat, w_uv, o, B, H, d_c, d_v, as_stream(stream));
  }
  if (d_c > 1024) return MLA_ERR_UNSUPPORTED;
  return mla::launch_out_up(o_lat, w_uv, o, B, H, d_c, d_v, dtype, as_stream(stream));
}

MLA_API mla_status mla_gate(const void* h, const void* w_g, void* o, int32_t B, int32_t d_model, int32_t width,
                            int32_t dtype, void* stream) {
  const OpRange range("mla_gate");
  if (!valid_dtype(dtype)) return MLA_ERR_INVALID_ARG;
  if (h == nullptr || w_g == nullptr || o == nullptr) return MLA_ERR_INVALID_ARG;
  if (B <= 0 || d_model <= 0 || width <= 0) return MLA_ERR_INVALID_ARG;
  if (dtype == MLA_BF16) {  // tensor cores only (no silent CUDA-core fallback)
    if (!mla::headgemm_gate_supported(d_model, width)) return MLA_ERR_UNSUPPORTED;
    if (!aligned16(h) || !aligned16(w_g) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
    return mla::launch_gate_tc(h, w_g, o, B, d_model, width, as_stream(stream));
  }
  return mla::launch_gate(h, w_g, o, B, d_model, width, dtype, as_stream(stream));
}

MLA_API mla_status mla_cache_append_paged(const mla_paged_cache* cache, const void* c_kv, const void* k_r,
                                          const int32_t* seq_idx, const int32_t* pos, int32_t T, float rope_base,
                                          void* stream) {
  const OpRange range("mla_cache_append_paged");
  mla_cache view;
  mla_status st = check_paged(cache, &view);
  if (st != MLA_OK) return st;
  if (T < 0) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (c_kv == nullptr || seq_idx == nullptr || pos == nullptr) return MLA_ERR_INVALID_ARG;
  if (view.d_r > 0 && k_r == nullptr) return MLA_ERR_INVALID_ARG;
  if (!(rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  if (view.d_r > 128) return MLA_ERR_UNSUPPORTED;
  return mla::launch_cache_append(view, c_kv, k_r, seq_idx, pos, T, rope_base, as_stream(stream),
                                  cache->block_table, cache->max_blocks, cache->num_pages);
}

MLA_API mla_status mla_decode_attn_paged(const void* q_cat, const mla_paged_cache* cache, const int32_t* seq_lens,
                                         int32_t H, float scale, void* workspace, size_t workspace_bytes,
                                         void* o_lat, float* lse, void* stream) {
  const OpRange range("mla_decode_attn_paged");
  mla_cache view;
  mla_status st = check_paged(cache, &view);
  if (st != MLA_OK) return st;
  if (q_cat == nullptr || seq_lens == nullptr || o_lat == nullptr || H <= 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_cat) || !aligned16(o_lat)) return MLA_ERR_INVALID_ARG;
  if (!(scale > 0.f) && !(scale < 0.f) && scale != 0.f) return MLA_ERR_INVALID_ARG;  // NaN
  if (view.dtype != MLA_BF16 || view.d_c != 512 || (view.d_r != 0 && view.d_r != 64) || H > 128)
    return MLA_ERR_UNSUPPORTED;
  return mla::launch_decode_tc(q_cat, view, seq_lens, H, scale, workspace, workspace_bytes, o_lat, lse,
                               as_stream(stream), cache->block_table, cache->max_blocks, cache->num_pages);
}

MLA_API size_t mla_kv_down_workspace_size(int32_t T, int32_t d_model, int32_t d_c, int32_t d_r, int32_t dtype) {
  if (!valid_dtype(dtype)) return 0;
  return mla::kv_down_workspace_size(T, d_model, d_c, d_r, dtype);
}

MLA_API mla_status mla_kv_down_append(const mla_cache* cache, const void* h, const void* w_dkvr, const void* gamma,
                                      float eps, const int32_t* seq_idx, const int32_t* pos, int32_t T,
                                      int32_t d_model, float rope_base, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  const OpRange range("mla_kv_down_append");
  const mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  return kv_down(*cache, h, w_dkvr, gamma, eps, seq_idx, pos, T, d_model, rope_base, workspace, workspace_bytes,
                 stream);
}

MLA_API mla_status mla_kv_down_append_paged(const mla_paged_cache* cache, const void* h, const void* w_dkvr,
                                            const void* gamma, float eps, const int32_t* seq_idx,
                                            const int32_t* pos, int32_t T, int32_t d_model, float rope_base,
                                            void* workspace, size_t workspace_bytes, void* stream) {
  const OpRange range("mla_kv_down_append_paged");
  mla_cache view;
  const mla_status st = check_paged(cache, &view);
  if (st != MLA_OK) return st;
  return kv_down(view, h, w_dkvr, gamma, eps, seq_idx, pos, T, d_model, rope_base, workspace, workspace_bytes,
                 stream, cache->block_table, cache->max_blocks, cache->num_pages);
}

MLA_API size_t mla_prefill_explicit_workspace_size(int32_t B, int32_t start, int32_t S, int32_t H) {
  return mla::prefill_explicit_workspace_size(B, start, S, H);
}

MLA_API mla_status mla_prefill_explicit(const void* q_nope, const void* q_rope, const mla_cache* cache,
                                        const void* w_uk, const void* w_uv, int32_t start, int32_t S, int32_t causal,
                                        int32_t H, float scale, float rope_base, void* workspace,
                                        size_t workspace_bytes, void* o, float* lse, void* stream) {
  const OpRange range("mla_prefill_explicit");
  const mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  if (q_nope == nullptr || q_rope == nullptr || w_uk == nullptr || w_uv == nullptr || o == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (S <= 0 || start < 0 || H <= 0 || static_cast<int64_t>(start) + S > cache->N_max) return MLA_ERR_INVALID_ARG;
  if (!(scale > 0.f) && !(scale < 0.f) && scale != 0.f) return MLA_ERR_INVALID_ARG;  // NaN
  if (!(rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(o))
    return MLA_ERR_INVALID_ARG;
  if (cache->dtype != MLA_BF16 || cache->d_c != 512 || cache->d_r != 64 || (H & 1) != 0) return MLA_ERR_UNSUPPORTED;
  return mla::launch_prefill_explicit(q_nope, q_rope, *cache, w_uk, w_uv, start, S, causal, H, scale, rope_base,
                                      workspace, workspace_bytes, o, lse, as_stream(stream));
}

MLA_API mla_status mla_debug_inject_fault(int32_t kind) {
  if (kind != 0 && kind != 1) return MLA_ERR_INVALID_ARG;
  mla::set_fault_injection(kind);
  return MLA_OK;
}

MLA_API mla_status mla_get_device_error(uint32_t* detail) {
  if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, mla::g_device_error, sizeof(word)) != cudaSuccess) return MLA_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(mla::g_device_error, &zero, sizeof(zero)) != cudaSuccess) return MLA_ERR_CUDA;
  if (detail != nullptr) *detail = word;
  return static_cast<mla_status>(word & 0xFFu);
}

}  // extern "C"

// Per-head batched GEMMs on the tensor cores (bf16 in, fp32 accumulate):
//
//   absorb_q : q_lat[b][h][c] = sum_d q_nope[b][h][d] W_UK[h][d][c]
//              (0539edu.com sections 3.1 / 5.1: W_UK folded into the query)
//   out_up   : o[b][h][d]     = sum_c o_lat[b][h][c] W_UV[h][d][c]
//              (0539edu.com section 3.1: W_UV applied after attention)
//
// The absorb launch can also append the decode step's new cache rows (the work of
// mla_cache_append, spread over the idle warps of every CTA): the step then has one
// kernel boundary fewer, and the attention that follows waits for both.
//
// Both are computed transposed, D[m][n] = sum_k A_h[m][k] X_h[n][k], with the
// weight dimension as M (128-row tiles) and the batch as N, so that the weights --
// the bytes that dominate -- are streamed once through TMA and every MMA is a full
// M = 128 tcgen05 instruction.  W_UK[h] ([d_k][d_c]) is an MN-major A operand,
// W_UV[h] ([d_v][d_c]) a K-major one; the per-head activations are K-major B
// operands read straight from [B][H][K] through a 3-D tensor map.
#include <atomic>

#include "mla_internal.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace hg {

constexpr int kBM = 128;          // M rows per CTA
constexpr int kBK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int kStagesHG = 8;         // a whole K = 512 in flight
constexpr int kSmemBudgetHG = 200 * 1024;
constexpr int kThreadsHG = 128;

// The new rows cache[seq_idx[i]][pos[i]] = [c_kv[i] || RoPE(k_r[i], pos[i])] written
// by an absorb launch (cache == nullptr: none); the rotation uses the query's table.
struct AppendArgs {
  __nv_bfloat16* cache;
  int32_t B, N_max, d_c, d_r;
  int64_t row_stride;             // elements
  const __nv_bfloat16* c_kv;      // [T][d_c], 16-byte rows
  const __nv_bfloat16* k_r;       // [T][d_r]
  const int32_t* seq_idx;
  const int32_t* pos;
  int32_t T;
  PageMap pages;
};

struct GemmArgs {
  int H, M, K;                    // per-head problem: M x K weights, K-long activations
  int nb;                         // batch rows (N) in total
  int n_tile;                     // N per CTA (multiple of 16, <= 256)
  int stages;                     // ring depth (<= kStagesHG)
  __nv_bfloat16* out;             // out[n * out_n_stride + h * out_h_stride + m]
  long long out_n_stride, out_h_stride;
  // RoPE of the query's position part (absorb only; d_r == 0 otherwise)
  const __nv_bfloat16* q_rope;    // [B][H][d_r]
  const int32_t* q_pos;           // [B]
  int d_r;
  int rope_col;                   // first output column of the rotated part (d_c)
  RopeTable rope;                 // turns per position of each RoPE pair, i < d_r / 2
  int gate;                       // epilogue: out[n][m] *= sigmoid(D[m][n]) instead of storing D
  AppendArgs app;                 // absorb only
};

// The query's position part, q_cat[n][h][d_c + 2j, +1] = RoPE(q_rope[n][h][2j, 2j+1],
// q_pos[n]), for the rows of n-tile n0 of head h, done by the kRopeThreads idle
// threads (warps 2-3) of each of the `parts` m-tile blocks of the head while their
// TMA loads and MMAs are in flight.  When the pair count divides the thread count,
// every thread keeps one pair j (its frequency read once: a kernel parameter read at
// a per-thread index is serialised) and walks rows part * step + t / half,
// + step * parts, ...; the loads of eight rows are issued before any is used.
constexpr int kRopeThreads = 64;
__device__ __forceinline__ void rope_rows(const GemmArgs& g, int h, int n0, int part, int parts, int t) {
  const int half = g.d_r / 2;
  const int n_end = min(n0 + g.n_tile, g.nb);
  constexpr int kU = 8;
  if (kRopeThreads % half == 0) {
    const int j = t % half, step = kRopeThreads / half, stride = step * parts;
    const float u_hi = g.rope.u_hi[j], u_lo = g.rope.u_lo[j];
    for (int nb = n0 + part * step + t / half; nb < n_end; nb += kU * stride) {
      int pos[kU];
      uint32_t x[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int n = nb + u * stride;
        if (n < n_end) {
          pos[u] = g.q_pos[n];
          x[u] = *reinterpret_cast<const uint32_t*>(g.q_rope + (static_cast<long long>(n) * g.H + h) * g.d_r + 2 * j);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int n = nb + u * stride;
        if (n < n_end) {
          float sn, cs;
          rope_sincos(pos[u], u_hi, u_lo, &sn, &cs);
          const float x0 = __uint_as_float(x[u] << 16), x1 = __uint_as_float(x[u] & 0xFFFF0000u);
          *reinterpret_cast<uint32_t*>(g.out + n * g.out_n_stride + h * g.out_h_stride + g.rope_col + 2 * j) =
              pack_bf16x2(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
        }
      }
    }
    return;
  }
  for (int idx = part * kRopeThreads + t; idx < (n_end - n0) * half; idx += parts * kRopeThreads) {
    const int n = n0 + idx / half, j = idx % half;
    float sn, cs;
    rope_sincos(g.q_pos[n], g.rope.u_hi[j], g.rope.u_lo[j], &sn, &cs);
    const uint32_t x = *reinterpret_cast<const uint32_t*>(g.q_rope + (static_cast<long long>(n) * g.H + h) * g.d_r + 2 * j);
    const float x0 = __uint_as_float(x << 16), x1 = __uint_as_float(x & 0xFFFF0000u);
    *reinterpret_cast<uint32_t*>(g.out + n * g.out_n_stride + h * g.out_h_stride + g.rope_col + 2 * j) =
        pack_bf16x2(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
  }
}

// The appended rows, as work items spread over the kRopeThreads idle threads of
// every CTA of the grid: item k is 16-byte chunk u of row i's latent part
// (u < d_c / 8, a copy) or RoPE pair u - d_c / 8 of its key part, with
// (i, u) = (k / U, k % U), U = d_c / 8 + d_r / 2.  A bad sequence, position or page
// skips the item and is recorded, as mla_cache_append does.
__device__ __forceinline__ void append_rows(const GemmArgs& g, int cta, int ctas, int t) {
  const AppendArgs& a = g.app;
  const int chunks = a.d_c / 8, U = chunks + a.d_r / 2;
  const long long items = static_cast<long long>(a.T) * U;
  for (long long k = static_cast<long long>(cta) * kRopeThreads + t; k < items;
       k += static_cast<long long>(ctas) * kRopeThreads) {
    const int i = static_cast<int>(k / U), u = static_cast<int>(k - static_cast<long long>(i) * U);
    // the item's source data does not depend on where the row goes: its load is issued
    // together with the slot's, one round trip for both
    uint4 chunk = make_uint4(0u, 0u, 0u, 0u);
    uint32_t kpair = 0u;
    if (u < chunks)
      chunk = *reinterpret_cast<const uint4*>(a.c_kv + static_cast<int64_t>(i) * a.d_c + 8 * u);
    else
      kpair = *reinterpret_cast<const uint32_t*>(a.k_r + static_cast<int64_t>(i) * a.d_r + 2 * (u - chunks));
    const int32_t b = a.seq_idx[i];
    const int32_t p = a.pos[i];
    if (b < 0 || b >= a.B || p < 0 || p >= a.N_max) {
      record_error(MLA_ERR_DEVICE_INDEX, kSiteAppendIndex);
      continue;
    }
    int64_t row = static_cast<int64_t>(b) * a.N_max + p;
    if (a.pages.table != nullptr) {
      const int32_t pg = a.pages.table[static_cast<int64_t>(b) * a.pages.max_blocks + p / kPageRows];
      if (pg < 0 || pg >= a.pages.num_pages) {
        record_error(MLA_ERR_DEVICE_INDEX, kSitePageIndex);
        continue;
      }
      row = static_cast<int64_t>(pg) * kPageRows + p % kPageRows;
    }
    __nv_bfloat16* dst = a.cache + row * a.row_stride;
    if (u < chunks) {
      *reinterpret_cast<uint4*>(dst + 8 * u) = chunk;
    } else {
      const int j = u - chunks;
      float sn, cs;
      rope_sincos(p, g.rope.u_hi[j], g.rope.u_lo[j], &sn, &cs);
      const float x0 = __uint_as_float(kpair << 16), x1 = __uint_as_float(kpair & 0xFFFF0000u);
      dst[a.d_c + 2 * j] = __float2bfloat16_rn(fmaf(x0, cs, -x1 * sn));
      dst[a.d_c + 2 * j + 1] = __float2bfloat16_rn(fmaf(x0, sn, x1 * cs));
    }
  }
}

template <bool kAMN>
__global__ void __launch_bounds__(kThreadsHG) head_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                                                               const __grid_constant__ CUtensorMap map_b,
                                                               const __grid_constant__ CUtensorMap map_out,
                                                               const __grid_constant__ GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  const int a_bytes = kBM * kBK * 2;               // 16 KB
  const int b_bytes = g.n_tile * kBK * 2;          // n_tile x 128 B
  const int stage_bytes = a_bytes + b_bytes;
  const int nst = g.stages;
  const int tile_bytes = g.n_tile * kBM * 2;       // the transposed output tile reuses the stages
  const uint32_t bars = sbase + (nst * stage_bytes > tile_bytes ? nst * stage_bytes : tile_bytes);
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int* abort = &s_abort;

  const int warp = threadIdx.x >> 5;
  const int mt = blockIdx.x, h = blockIdx.y, nt = blockIdx.z;
  const int m0 = mt * kBM, n0 = nt * g.n_tile;
  const int nk = g.K / kBK;
  const uint32_t tmem_cols = g.n_tile <= 32 ? 32 : (g.n_tile <= 64 ? 64 : (g.n_tile <= 128 ? 128 : 256));

  griddep_launch();
  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(bars + 8 * i, 1);                    // full
      mbar_init(bars + 8 * (kStagesHG + i), 1);      // empty
    }
    mbar_init(bars + 8 * (2 * kStagesHG), 1);        // accumulator done
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), tmem_cols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    const uint32_t leader = elect_one();
    auto load_weights = [&](int k, int st) {
      const uint32_t sa = sbase + st * stage_bytes, full = bars + 8 * st;
      mbar_arrive_expect_tx_if(leader, full, stage_bytes);
      if (kAMN) {
        // W_UK rows h*K + [k*64, k*64+64), latent columns [m0, m0+128) as two 64-wide boxes
        tma_load_2d_if(leader, sa, &map_a, full, m0, h * g.K + k * kBK);
        tma_load_2d_if(leader, sa + a_bytes / 2, &map_a, full, m0 + 64, h * g.K + k * kBK);
      } else {
        // W_UV rows h*M + [m0, m0+128), columns [k*64, k*64+64)
        tma_load_2d_if(leader, sa, &map_a, full, k * kBK, h * g.M + m0);
      }
    };
    auto load_act = [&](int k, int st) {
      const uint32_t sb = sbase + st * stage_bytes + a_bytes;
      tma_load_3d_if(leader, sb, &map_b, bars + 8 * st, k * kBK, h, n0);
    };
    // the weights of the first ring pass are read while the previous kernel drains
    // (no kernel writes them); the activations only after it has completed
    const int first = nk < nst ? nk : nst;
    for (int k = 0; k < first; ++k) load_weights(k, k);
    griddep_wait();
    for (int k = 0; k < first; ++k) load_act(k, k);
    for (int k = first; k < nk; ++k) {
      const int st = k % nst;
      if (!warp_wait(bars + 8 * (kStagesHG + st), ((k / nst) & 1) ^ 1, abort)) break;
      load_weights(k, st);
      load_act(k, st);
    }
  } else if (warp == 1) {
    const uint32_t leader = elect_one();
    const uint32_t idesc = idesc_bf16(kBM, g.n_tile, kAMN, false);
    for (int k = 0; k < nk; ++k) {
      const int st = k % nst;
      if (!warp_wait(bars + 8 * st, (k / nst) & 1, abort)) break;
      tc_fence_after();
      const uint32_t sa = sbase + st * stage_bytes, sb = sa + a_bytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = kAMN ? sdesc_sw128(sa + kk * 16 * 128, a_bytes / 2, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
        mma_ss_if(leader, tmem, ad, sdesc_sw128(sb + kk * 32, 16, 1024), idesc, (k | kk) != 0);
      }
      tc_commit_if(leader, bars + 8 * (kStagesHG + st));
    }
    tc_commit_if(leader, bars + 8 * (2 * kStagesHG));
  } else if (kAMN && (g.d_r > 0 || g.app.cache != nullptr)) {
    griddep_wait();  // q_cat and the cache may still be read by the previous kernel
    if (g.d_r > 0) rope_rows(g, h, n0, mt, gridDim.x, threadIdx.x - 64);
    if (g.app.cache != nullptr)
      append_rows(g, (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x,
                  gridDim.x * gridDim.y * gridDim.z, threadIdx.x - 64);
  }
  __syncwarp();

  // epilogue: warp w holds rows 32w..32w+31 (TMEM lanes), columns = batch rows.  The
  // tile is transposed into the idle stage memory as [n][128 rows] bf16 and leaves
  // in one TMA store (rows n >= nb fall outside the tensor and are clipped).
  const bool ok = warp_wait(bars + 8 * (2 * kStagesHG), 0, abort);
  tc_fence_after();
  griddep_wait();  // the outputs may still be read (or, for the gate, written) by the previous kernel
  if (g.gate) {
    // gate: thread m scales out[n][m] for the tile's batch rows by sigmoid(D[m][n])
    // (a warp reads and writes 64 contiguous bytes per row n)
    if (ok) {
      const int m = m0 + warp * 32 + (threadIdx.x & 31);
      const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
      for (int c0 = 0; c0 < g.n_tile; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int n = n0 + c0 + j;
          if (c0 + j < g.n_tile && n < g.nb) {
            __nv_bfloat16* op = g.out + n * g.out_n_stride + m;
            *op = __float2bfloat16_rn(__bfloat162float(*op) / (1.f + expf(-__uint_as_float(v[j]))));
          }
        }
      }
    }
  } else if (ok) {
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem_raw + (sbase - raw));
    const int ml = warp * 32 + (threadIdx.x & 31);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    for (int c0 = 0; c0 < g.n_tile; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) tile[(c0 + j) * kBM + ml] = __float2bfloat16_rn(__uint_as_float(v[j]));
    }
    fence_proxy_async_cta();
  }
  __syncthreads();
  if (ok && !g.gate && threadIdx.x == 0) {
    tma_store_3d(&map_out, sbase, m0, h, n0);
    bulk_commit();
    bulk_wait_read0();
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) record_error(MLA_ERR_DEVICE_TIMEOUT, kSiteDecodeWait);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> cached{nullptr};  // looked up until it succeeds once
  EncodeTiledFn fn = cached.load(std::memory_order_acquire);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

static bool map_2d(CUtensorMap* m, const void* p, uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B][H][X] output as a 3-D map (X, H, B) with a (128, 1, n_tile) box, no swizzle
// (the staged tile is plain [n][128] bf16).
static bool map_out3d(CUtensorMap* m, void* p, uint64_t X, uint64_t H, uint64_t B, uint32_t n_tile) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {X, H, B};
  const cuuint64_t strides[2] = {X * 2, H * X * 2};
  const cuuint32_t box[3] = {128, 1, n_tile};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// [B][H][K] activations as a 3-D map (K, H, B) with a (64, 1, n_tile) box.
static bool map_act(CUtensorMap* m, const void* p, uint64_t K, uint64_t H, uint64_t B, uint32_t n_tile) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {K, H, B};
  const cuuint64_t strides[2] = {K * 2, H * K * 2};
  const cuuint32_t box[3] = {64, 1, n_tile};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int n_tile_for(int B) {
  int n = B > 256 ? 256 : B;
  return (n + 15) / 16 * 16;
}

// Ring depth: every K step of the tile in flight when shared memory allows.
static int stages_for(int nk, int n_tile) {
  const int per_stage = kBM * kBK * 2 + n_tile * kBK * 2;
  int st = kSmemBudgetHG / per_stage;
  if (st > kStagesHG) st = kStagesHG;
  if (st > nk) st = nk;
  return st < 1 ? 1 : st;
}

template <bool kAMN>
static mla_status launch(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, const GemmArgs& g,
                         int m_tiles, int n_tiles, cudaStream_t s) {
  auto k = head_gemm_kernel<kAMN>;
  const size_t ring = static_cast<size_t>(g.stages) * (kBM * kBK * 2 + g.n_tile * kBK * 2);
  const size_t tile = static_cast<size_t>(g.n_tile) * kBM * 2;
  const size_t smem = (ring > tile ? ring : tile) + 8 * (2 * kStagesHG + 1) + 1024;
  if (ensure_smem_limit(reinterpret_cast<const void*>(k), smem) != cudaSuccess) return MLA_ERR_CUDA;
  return cuda_status(launch_pdl(k, dim3(m_tiles, g.H, n_tiles), dim3(kThreadsHG), smem, s, ma, mb, mo, g));
}

}  // namespace hg

bool headgemm_absorb_supported(int32_t d_k, int32_t d_c, int32_t d_r) {
  return d_k % 64 == 0 && d_c % 128 == 0 && d_r <= 128 && (d_c + d_r) % 8 == 0;  // 16-byte output rows
}

bool headgemm_out_up_supported(int32_t d_c, int32_t d_v) { return d_c % 64 == 0 && d_v % 128 == 0; }

bool headgemm_gate_supported(int32_t d_model, int32_t width) { return d_model % 64 == 0 && width % 128 == 0; }

mla_status launch_absorb_q_tc(const void* q_nope, const void* q_rope, const int32_t* q_pos, const void* w_uk,
                              void* q_cat, int32_t B, int32_t H, int32_t d_k, int32_t d_c, int32_t d_r,
                              float rope_base, cudaStream_t s, const AppendRows* app) {
  using namespace hg;
  GemmArgs g = {};
  if (app != nullptr) {
    const mla_cache& c = *app->cache;
    g.app = {static_cast<__nv_bfloat16*>(c.data), c.B, c.N_max, c.d_c, c.d_r, static_cast<int64_t>(c.row_stride),
             static_cast<const __nv_bfloat16*>(app->c_kv), static_cast<const __nv_bfloat16*>(app->k_r),
             app->seq_idx, app->pos, app->T, {app->block_table, app->max_blocks, app->num_pages}};
  }
  g.H = H;
  g.M = d_c;
  g.K = d_k;
  g.nb = B;
  g.n_tile = n_tile_for(B);
  g.stages = stages_for(d_k / kBK, g.n_tile);
  g.out = static_cast<__nv_bfloat16*>(q_cat);
  g.out_h_stride = d_c + d_r;
  g.out_n_stride = static_cast<long long>(H) * (d_c + d_r);
  g.q_rope = static_cast<const __nv_bfloat16*>(q_rope);
  g.q_pos = q_pos;
  g.d_r = d_r;
  g.rope_col = d_c;
  g.rope = rope_table(d_r, rope_base);
  CUtensorMap ma, mb;
  if (!map_2d(&ma, w_uk, d_c, static_cast<uint64_t>(H) * d_k, 64, 64)) return MLA_ERR_CUDA;
  if (!map_act(&mb, q_nope, d_k, H, B, g.n_tile)) return MLA_ERR_CUDA;
  CUtensorMap mo;
  if (!map_out3d(&mo, q_cat, d_c + d_r, H, B, g.n_tile)) return MLA_ERR_CUDA;
  return launch<true>(ma, mb, mo, g, d_c / kBM, (B + g.n_tile - 1) / g.n_tile, s);
}

mla_status launch_out_up_tc(const void* o_lat, const void* w_uv, void* o, int32_t B, int32_t H, int32_t d_c,
                            int32_t d_v, cudaStream_t s) {
  using namespace hg;
  GemmArgs g = {};
  g.H = H;
  g.M = d_v;
  g.K = d_c;
  g.nb = B;
  g.n_tile = n_tile_for(B);
  g.stages = stages_for(d_c / kBK, g.n_tile);
  g.out = static_cast<__nv_bfloat16*>(o);
  g.out_h_stride = d_v;
  g.out_n_stride = static_cast<long long>(H) * d_v;
  CUtensorMap ma, mb;
  if (!map_2d(&ma, w_uv, d_c, static_cast<uint64_t>(H) * d_v, 64, 128)) return MLA_ERR_CUDA;
  if (!map_act(&mb, o_lat, d_c, H, B, g.n_tile)) return MLA_ERR_CUDA;
  CUtensorMap mo;
  if (!map_out3d(&mo, o, d_v, H, B, g.n_tile)) return MLA_ERR_CUDA;
  return launch<false>(ma, mb, mo, g, d_v / kBM, (B + g.n_tile - 1) / g.n_tile, s);
}

// Gate (tahou.com sections 2.6 and 3.2): z[b][j] = sum_i h[b][i] W_g[i][j] computed
// as D[j][b] with W_g^T as the MN-major A operand (one "head", M = width, K = d_model),
// and o[b][j] *= sigmoid(z) in the epilogue.
mla_status launch_gate_tc(const void* h, const void* w_g, void* o, int32_t B, int32_t d_model, int32_t width,
                          cudaStream_t s) {
  using namespace hg;
  GemmArgs g = {};
  g.H = 1;
  g.M = width;
  g.K = d_model;
  g.nb = B;
  g.n_tile = n_tile_for(B);
  g.stages = stages_for(d_model / kBK, g.n_tile);
  g.out = static_cast<__nv_bfloat16*>(o);
  g.out_h_stride = 0;
  g.out_n_stride = width;
  g.gate = 1;
  CUtensorMap ma, mb, mo;
  if (!map_2d(&ma, w_g, width, d_model, 64, 64)) return MLA_ERR_CUDA;
  if (!map_act(&mb, h, d_model, 1, B, g.n_tile)) return MLA_ERR_CUDA;
  if (!map_out3d(&mo, o, width, 1, B, g.n_tile)) return MLA_ERR_CUDA;  // unused by the gate epilogue
  return launch<true>(ma, mb, mo, g, width / kBM, (B + g.n_tile - 1) / g.n_tile, s);
}

}  // namespace mla

// New tokens' cache rows straight from their hidden states:
//
//   x      = h W_DKV                      (0539edu.com section 2.2: compression)
//   c_KV   = x / sqrt(mean(x^2) + eps) * gamma
//                                         (the same page, section 6.3: RMSNorm after
//                                          the compression projection)
//   k_R    = RoPE(h W_KR, pos)            (hotelren.com section 6.2: one key
//                                          projection shared by all heads; icman.com.cn
//                                          section 2: the key is cached rotated)
//   cache[seq][pos] = [c_KV || k_R]
//
// with W_DKV and W_KR side by side as one [d_model][d_c + d_r] matrix W.
//
// Two launches.  (1) The projection D = h W on the tensor cores, computed
// transposed, D^T[m][n] = sum_k W[k][m] h[n][k]: the R = d_c + d_r output columns are
// M (128-row tiles, W the MN-major A operand streamed once through TMA), the tokens
// are N, and K = d_model is cut into `splits` ranges so that a decode batch of a few
// dozen tokens still spreads the weight stream over every SM.  Each CTA writes its
// fp32 partial tile to the workspace.  (2) One block per token sums the partials in
// a fixed order (deterministic), normalises the latent part, rotates the key part
// and stores the row in the cache dtype.  The projection lets the finishing kernel
// launch (programmatic dependent launch) only once its own wait on the previous
// kernel has returned, so the finishing kernel may read the token's slot, gains and
// rotation before it waits for the partials: of the chain of dependent loads, only
// the partials remain after the projection.  Shapes the tensor-core kernel does not
// take (fp32, odd widths) use a CUDA-core kernel for (1) with a single range.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace kvd {

constexpr int kBM = 128;      // output columns (M) per CTA
constexpr int kBK = 64;       // K per stage: one 128-byte swizzle row of bf16
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kThreads = 128;
constexpr int kMaxR = 1024;   // row width the finishing kernel holds in registers
constexpr int kPairsPerThread = kMaxR / 2 / kThreads;

struct GemmArgs {
  int T;        // tokens (N)
  int R;        // output columns d_c + d_r (M)
  int nk;       // K steps in all (d_model / 64)
  int splits;   // K ranges (grid z)
  int n_tile;   // tokens per CTA (multiple of 16, <= 256)
  int stages;   // ring depth
  float* ws;    // partials [splits][T][R]
};

struct Plan {
  int m_tiles, n_tile, n_tiles, splits, stages;
  bool tc;
};

inline bool tc_shape_ok(int32_t d_model, int32_t R, int32_t dtype) {
  return dtype == MLA_BF16 && d_model % kBK == 0 && R % 8 == 0;  // 16-byte rows for the TMA maps
}

inline Plan plan(int32_t T, int32_t d_model, int32_t R, int32_t dtype) {
  Plan p = {};
  p.tc = tc_shape_ok(d_model, R, dtype);
  if (!p.tc) {
    p.splits = 1;
    return p;
  }
  p.m_tiles = (R + kBM - 1) / kBM;
  const int nt = T > 256 ? 256 : T;
  p.n_tile = (nt + 15) / 16 * 16;
  p.n_tiles = (T + p.n_tile - 1) / p.n_tile;
  const int nk = d_model / kBK;
  const int tiles = p.m_tiles * p.n_tiles;
  int s = (148 + tiles - 1) / tiles;  // about one CTA per SM in all
  if (s > nk) s = nk;
  p.splits = s < 1 ? 1 : s;
  const int per_stage = kBM * kBK * 2 + p.n_tile * kBK * 2;
  int st = kSmemBudget / per_stage;
  const int k_per = (nk + p.splits - 1) / p.splits;
  if (st > kMaxStages) st = kMaxStages;
  if (st > k_per) st = k_per;
  p.stages = st < 1 ? 1 : st;
  return p;
}

inline size_t workspace_bytes(int32_t T, int32_t d_model, int32_t R, int32_t dtype) {
  const Plan p = plan(T, d_model, R, dtype);
  return static_cast<size_t>(p.splits) * static_cast<size_t>(T) * static_cast<size_t>(R) * sizeof(float);
}

// ---------------------------------------------------------------------------
// (1a) tensor-core projection, one (128 columns, n_tile tokens, K range) tile per CTA
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) kvd_gemm_kernel(const __grid_constant__ CUtensorMap map_w,
                                                            const __grid_constant__ CUtensorMap map_h,
                                                            const __grid_constant__ GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int a_bytes = kBM * kBK * 2;       // 16 KB: 64 K rows x 128 columns, as two 64-column boxes
  const int b_bytes = g.n_tile * kBK * 2;  // n_tile tokens x 128 bytes
  const int stage_bytes = a_bytes + b_bytes;
  const int nst = g.stages;
  const uint32_t bars = sbase + nst * stage_bytes;  // full[kMaxStages], empty[kMaxStages], done
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int* abort = &s_abort;

  const int warp = threadIdx.x >> 5;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * g.n_tile, sp = blockIdx.z;
  const int k_lo = sp * g.nk / g.splits, k_hi = (sp + 1) * g.nk / g.splits;
  const int nk = k_hi - k_lo;  // >= 1: splits <= nk
  const uint32_t tmem_cols = g.n_tile <= 32 ? 32 : (g.n_tile <= 64 ? 64 : (g.n_tile <= 128 ? 128 : 256));

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (kMaxStages + i), 1);
    }
    mbar_init(bars + 8 * (2 * kMaxStages), 1);
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
    // ------------------------------------------------------------ TMA producer
    const uint32_t leader = elect_one();
    // W rows [k*64, k*64+64), columns [m0, m0+128) as two 64-wide boxes.  Columns
    // past R read as zeros; a second box wholly past R (R = 576: the last tile) is
    // not loaded at all -- its shared memory then feeds only output rows m >= R,
    // which the epilogue never stores.
    const bool hi_box = m0 + 64 < g.R;
    const uint32_t tx = stage_bytes - (hi_box ? 0 : a_bytes / 2);
    auto load_w = [&](int k, int st) {
      const uint32_t sa = sbase + st * stage_bytes, full = bars + 8 * st;
      mbar_arrive_expect_tx_if(leader, full, tx);
      tma_load_2d_if(leader, sa, &map_w, full, m0, (k_lo + k) * kBK);
      if (hi_box) tma_load_2d_if(leader, sa + a_bytes / 2, &map_w, full, m0 + 64, (k_lo + k) * kBK);
    };
    auto load_h = [&](int k, int st) {
      tma_load_2d_if(leader, sbase + st * stage_bytes + a_bytes, &map_h, bars + 8 * st, (k_lo + k) * kBK, n0);
    };
    // no kernel of this library writes the weights, so the first ring pass of them
    // overlaps the previous kernel's tail; h only after it has completed
    const int first = nk < nst ? nk : nst;
    for (int k = 0; k < first; ++k) load_w(k, k);
    griddep_wait();
    griddep_launch();
    for (int k = 0; k < first; ++k) load_h(k, k);
    for (int k = first; k < nk; ++k) {
      const int st = k % nst;
      if (!warp_wait(bars + 8 * (kMaxStages + st), ((k / nst) & 1) ^ 1, abort)) break;
      load_w(k, st);
      load_h(k, st);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    griddep_wait();
    griddep_launch();
    const uint32_t leader = elect_one();
    const uint32_t idesc = idesc_bf16(kBM, g.n_tile, true, false);
    for (int k = 0; k < nk; ++k) {
      const int st = k % nst;
      if (!warp_wait(bars + 8 * st, (k / nst) & 1, abort)) break;
      tc_fence_after();
      const uint32_t sa = sbase + st * stage_bytes, sb = sa + a_bytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // A: 16 K rows (2 KB) per step, the two 64-column halves a_bytes / 2 apart
        const uint64_t ad = sdesc_sw128(sa + kk * 16 * 128, a_bytes / 2, 1024);
        mma_ss_if(leader, tmem, ad, sdesc_sw128(sb + kk * 32, 16, 1024), idesc, (k | kk) != 0);
      }
      tc_commit_if(leader, bars + 8 * (kMaxStages + st));
    }
    tc_commit_if(leader, bars + 8 * (2 * kMaxStages));
  } else {
    griddep_wait();
    griddep_launch();
  }
  __syncwarp();

  // epilogue: warp w holds output columns m0 + 32w + lane (TMEM lanes), one TMEM
  // column per token; each token's 32 columns leave as one 128-byte store per warp
  const bool ok = warp_wait(bars + 8 * (2 * kMaxStages), 0, abort);
  tc_fence_after();
  griddep_wait();  // the workspace may still be read by the previous kernel
  if (ok) {
    const int m = m0 + warp * 32 + (threadIdx.x & 31);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float* out = g.ws + static_cast<size_t>(sp) * g.T * g.R + m;
    for (int c0 = 0; c0 < g.n_tile; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int n = n0 + c0 + j;
        if (c0 + j < g.n_tile && n < g.T && m < g.R) out[static_cast<size_t>(n) * g.R] = __uint_as_float(v[j]);
      }
    }
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

// ---------------------------------------------------------------------------
// (1b) CUDA-core projection for the shapes (1a) does not take: one thread per
// output column, eight tokens per block, a single K range
// ---------------------------------------------------------------------------
constexpr int kSimtTokens = 8;

template <typename T>
__global__ void __launch_bounds__(kThreads) kvd_simt_kernel(const T* __restrict__ h, const T* __restrict__ w,
                                                            int32_t n_tok, int32_t d_model, int32_t R,
                                                            float* __restrict__ ws) {
  griddep_wait();  // h may come from the previous kernel, which may still read ws
  griddep_launch();  // after the wait: the finishing kernel reads its row slots early
  const int m = blockIdx.x * kThreads + threadIdx.x;
  const int n0 = blockIdx.y * kSimtTokens;
  float acc[kSimtTokens];
#pragma unroll
  for (int u = 0; u < kSimtTokens; ++u) acc[u] = 0.f;
  if (m < R) {
    for (int i = 0; i < d_model; ++i) {
      const float wv = ld_elem(w + static_cast<size_t>(i) * R + m);
#pragma unroll
      for (int u = 0; u < kSimtTokens; ++u)
        if (n0 + u < n_tok) acc[u] = fmaf(ld_elem(h + static_cast<size_t>(n0 + u) * d_model + i), wv, acc[u]);
    }
#pragma unroll
    for (int u = 0; u < kSimtTokens; ++u)
      if (n0 + u < n_tok) ws[static_cast<size_t>(n0 + u) * R + m] = acc[u];
  }
}

// ---------------------------------------------------------------------------
// (2) one block per token: partial sums -> RMSNorm on the latent, RoPE on the key,
// the row into the (contiguous or paged) cache.  Column pairs (2q, 2q+1) are held
// by thread t = q % 128 of each of four groups; group g sums the K ranges g, g + 4,
// g + 8, ... in that order, eight independent loads at a time (the partials sit in
// L2, so a chain of dependent loads would cost an L2 round trip per range), and
// group 0 adds the four group sums in group order.  The summation order is fixed,
// so the result is deterministic.  The latent pairs feed the mean square; the key
// pairs are exactly RoPE's rotation pairs.  The block's first token's slot, gains
// and rotation are read before the wait for the partials (the projection kernels
// trigger this launch only after their own wait has returned).
// ---------------------------------------------------------------------------
constexpr int kFinishGroups = 4;
constexpr int kFinishThreads = kThreads * kFinishGroups;
constexpr int kSplitBatch = 8;

template <typename T>
__global__ void __launch_bounds__(kFinishThreads) kvd_finish_kernel(const float* __restrict__ ws, int32_t splits,
                                                                    int32_t n_tok, int32_t d_c, int32_t d_r,
                                                                    const T* __restrict__ gamma, float eps,
                                                                    T* __restrict__ cache, int32_t B, int32_t N_max,
                                                                    int64_t row_stride,
                                                                    const int32_t* __restrict__ seq_idx,
                                                                    const int32_t* __restrict__ pos,
                                                                    const __grid_constant__ RopeTable rope,
                                                                    PageMap pages) {
  __shared__ float s_hi[64], s_lo[64];
  __shared__ float2 s_part[kFinishGroups - 1][kMaxR / 2];
  __shared__ float s_red[kThreads / 32];
  griddep_launch();
  rope_table_to_smem(rope, d_r / 2, s_hi, s_lo);
  const int R = d_c + d_r;
  const int pairs = R / 2;
  const int g = threadIdx.x / kThreads, t = threadIdx.x % kThreads;
  const int lane = t & 31, warp = t >> 5;
  const size_t split_stride = static_cast<size_t>(n_tok) * R;
  // A token's cache slot, gains and rotation do not depend on the partials, so the
  // block's first token has them read before the wait: the projection signals its
  // dependents only after its own wait, so whatever wrote seq_idx, pos or the page
  // table has completed.  Slot -1: a bad sequence or position, -2: a bad page.
  auto slot = [&](int i, int32_t* p_out) -> int64_t {
    const int32_t b = __ldcg(seq_idx + i);
    const int32_t p = __ldcg(pos + i);
    *p_out = p;
    if (b < 0 || b >= B || p < 0 || p >= N_max) return -1;
    int64_t row = static_cast<int64_t>(b) * N_max + p;
    if (pages.table != nullptr) {
      const int32_t pg = __ldcg(pages.table + static_cast<int64_t>(b) * pages.max_blocks + p / kPageRows);
      if (pg < 0 || pg >= pages.num_pages) return -2;
      row = static_cast<int64_t>(pg) * kPageRows + p % kPageRows;
    }
    return row;
  };
  // per column pair of a group-0 thread: (gamma, gamma) of a latent pair, (cos, sin)
  // of a key pair
  float2 coef[kPairsPerThread];
  auto coefs = [&](int32_t p) {
#pragma unroll
    for (int u = 0; u < kPairsPerThread; ++u) {
      const int q = t + u * kThreads;
      if (q >= pairs) continue;
      if (2 * q < d_c) {
        coef[u] = make_float2(ld_elem(gamma + 2 * q), ld_elem(gamma + 2 * q + 1));
      } else {
        const int j = q - d_c / 2;
        float sn, cs;
        rope_sincos(p, s_hi[j], s_lo[j], &sn, &cs);
        coef[u] = make_float2(cs, sn);
      }
    }
  };
  int i = blockIdx.x;
  int32_t p = 0;
  int64_t row = -1;
  if (i < n_tok) {
    row = slot(i, &p);
    if (g == 0 && row >= 0) coefs(p);
  }
  griddep_wait();  // the partials come from the previous kernel
  for (; i < n_tok; i += gridDim.x) {
    if (i != static_cast<int>(blockIdx.x)) {
      row = slot(i, &p);
      if (g == 0 && row >= 0) coefs(p);
    }
    if (row < 0) {  // block-uniform
      if (threadIdx.x == 0) record_error(MLA_ERR_DEVICE_INDEX, row == -1 ? kSiteAppendIndex : kSitePageIndex);
      continue;
    }
    const float* src = ws + static_cast<size_t>(i) * R;
    float2 v[kPairsPerThread];
#pragma unroll
    for (int u = 0; u < kPairsPerThread; ++u) v[u] = make_float2(0.f, 0.f);
    for (int s0 = g; s0 < splits; s0 += kFinishGroups * kSplitBatch) {
      float2 x[kPairsPerThread][kSplitBatch];
#pragma unroll
      for (int u = 0; u < kPairsPerThread; ++u) {
        const int q = t + u * kThreads;
#pragma unroll
        for (int k = 0; k < kSplitBatch; ++k) {
          const int sp = s0 + k * kFinishGroups;
          x[u][k] = (q < pairs && sp < splits)
                        ? *reinterpret_cast<const float2*>(src + sp * split_stride + 2 * q)
                        : make_float2(0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kPairsPerThread; ++u) {
#pragma unroll
        for (int k = 0; k < kSplitBatch; ++k) {
          if (s0 + k * kFinishGroups < splits) {
            v[u].x += x[u][k].x;
            v[u].y += x[u][k].y;
          }
        }
      }
    }
    if (g > 0) {
#pragma unroll
      for (int u = 0; u < kPairsPerThread; ++u) {
        const int q = t + u * kThreads;
        if (q < pairs) s_part[g - 1][q] = v[u];
      }
    }
    __syncthreads();
    if (g == 0) {
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < kPairsPerThread; ++u) {
        const int q = t + u * kThreads;
        if (q >= pairs) continue;
#pragma unroll
        for (int gg = 0; gg < kFinishGroups - 1; ++gg) {
          v[u].x += s_part[gg][q].x;
          v[u].y += s_part[gg][q].y;
        }
        if (2 * q < d_c) ss = fmaf(v[u].x, v[u].x, fmaf(v[u].y, v[u].y, ss));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_red[warp] = ss;
    }
    __syncthreads();
    if (g == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) tot += s_red[w];
      const float r = rsqrtf(tot / static_cast<float>(d_c) + eps);
      T* dst = cache + row * row_stride;
#pragma unroll
      for (int u = 0; u < kPairsPerThread; ++u) {
        const int q = t + u * kThreads;
        if (q >= pairs) continue;
        if (2 * q < d_c) {
          st_elem(dst + 2 * q, v[u].x * r * coef[u].x);
          st_elem(dst + 2 * q + 1, v[u].y * r * coef[u].y);
        } else {
          const float cs = coef[u].x, sn = coef[u].y;
          st_elem(dst + 2 * q, fmaf(v[u].x, cs, -v[u].y * sn));
          st_elem(dst + 2 * q + 1, fmaf(v[u].x, sn, v[u].y * cs));
        }
      }
    }
    __syncthreads();  // s_part and s_red are rewritten for the next token
  }
}

// (2') the same for projections cut into fewer than kFinishGroups K ranges (prompt-
// sized batches run as one range): one warp per token, four tokens per block, so
// thousands of tokens are in flight; the ranges are added in order (deterministic),
// the mean square is a warp reduction.
constexpr int kWarpPairs = kMaxR / 2 / 32;  // column pairs per lane

template <typename T>
__global__ void __launch_bounds__(kThreads) kvd_finish_warp_kernel(const float* __restrict__ ws, int32_t splits,
                                                                   int32_t n_tok, int32_t d_c, int32_t d_r,
                                                                   const T* __restrict__ gamma, float eps,
                                                                   T* __restrict__ cache, int32_t B, int32_t N_max,
                                                                   int64_t row_stride,
                                                                   const int32_t* __restrict__ seq_idx,
                                                                   const int32_t* __restrict__ pos,
                                                                   const __grid_constant__ RopeTable rope,
                                                                   PageMap pages) {
  __shared__ float s_hi[64], s_lo[64];
  griddep_launch();
  rope_table_to_smem(rope, d_r / 2, s_hi, s_lo);
  griddep_wait();  // the partials come from the previous kernel
  const int lane = threadIdx.x & 31, warps = kThreads / 32;
  const int R = d_c + d_r, pairs = R / 2;
  const size_t split_stride = static_cast<size_t>(n_tok) * R;
  for (int i = blockIdx.x * warps + (threadIdx.x >> 5); i < n_tok; i += gridDim.x * warps) {
    const int32_t b = seq_idx[i];
    const int32_t p = pos[i];
    if (b < 0 || b >= B || p < 0 || p >= N_max) {  // warp-uniform
      if (lane == 0) record_error(MLA_ERR_DEVICE_INDEX, kSiteAppendIndex);
      continue;
    }
    int64_t row = static_cast<int64_t>(b) * N_max + p;
    if (pages.table != nullptr) {
      const int32_t pg = pages.table[static_cast<int64_t>(b) * pages.max_blocks + p / kPageRows];
      if (pg < 0 || pg >= pages.num_pages) {
        if (lane == 0) record_error(MLA_ERR_DEVICE_INDEX, kSitePageIndex);
        continue;
      }
      row = static_cast<int64_t>(pg) * kPageRows + p % kPageRows;
    }
    const float* src = ws + static_cast<size_t>(i) * R;
    float2 v[kWarpPairs];
#pragma unroll
    for (int u = 0; u < kWarpPairs; ++u) v[u] = make_float2(0.f, 0.f);
    for (int sp = 0; sp < splits; ++sp) {
#pragma unroll
      for (int u = 0; u < kWarpPairs; ++u) {
        const int q = lane + 32 * u;
        if (q < pairs) {
          const float2 x = *reinterpret_cast<const float2*>(src + sp * split_stride + 2 * q);
          v[u].x += x.x;
          v[u].y += x.y;
        }
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < kWarpPairs; ++u) {
      const int q = lane + 32 * u;
      if (q < pairs && 2 * q < d_c) ss = fmaf(v[u].x, v[u].x, fmaf(v[u].y, v[u].y, ss));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / static_cast<float>(d_c) + eps);
    T* dst = cache + row * row_stride;
#pragma unroll
    for (int u = 0; u < kWarpPairs; ++u) {
      const int q = lane + 32 * u;
      if (q >= pairs) continue;
      if (2 * q < d_c) {
        st_elem(dst + 2 * q, v[u].x * r * ld_elem(gamma + 2 * q));
        st_elem(dst + 2 * q + 1, v[u].y * r * ld_elem(gamma + 2 * q + 1));
      } else {
        const int j = q - d_c / 2;
        float sn, cs;
        rope_sincos(p, s_hi[j], s_lo[j], &sn, &cs);
        st_elem(dst + 2 * q, fmaf(v[u].x, cs, -v[u].y * sn));
        st_elem(dst + 2 * q + 1, fmaf(v[u].x, sn, v[u].y * cs));
      }
    }
  }
}

}  // namespace kvd

size_t kv_down_workspace_size(int32_t T, int32_t d_model, int32_t d_c, int32_t d_r, int32_t dtype) {
  if (T <= 0 || d_model <= 0 || d_c <= 0 || d_r < 0) return 0;
  return kvd::workspace_bytes(T, d_model, d_c + d_r, dtype);
}

mla_status launch_kv_down(const mla_cache& c, const void* h, const void* w, const void* gamma, float eps,
                          const int32_t* seq_idx, const int32_t* pos, int32_t T, int32_t d_model, float rope_base,
                          void* ws, size_t ws_bytes, cudaStream_t s, const int32_t* block_table, int32_t max_blocks,
                          int32_t num_pages) {
  using namespace kvd;
  const int R = c.d_c + c.d_r;
  if (R > kMaxR || (c.d_c & 1) != 0) return MLA_ERR_UNSUPPORTED;
  Plan p = plan(T, d_model, R, c.dtype);
  // bf16 projects on the tensor cores only: a shape or an alignment outside that
  // kernel is an error, never a silent switch to the CUDA-core projection
  if (c.dtype == MLA_BF16 && !p.tc) return MLA_ERR_UNSUPPORTED;
  if (p.tc && !(aligned16(h) && aligned16(w))) return MLA_ERR_INVALID_ARG;  // the TMA maps need 16-byte bases
  const size_t need = static_cast<size_t>(p.splits) * T * R * sizeof(float);
  if (ws == nullptr || ws_bytes < need || !aligned16(ws)) return MLA_ERR_WORKSPACE;
  float* wsf = static_cast<float*>(ws);
  if (p.tc) {
    GemmArgs g = {};
    g.T = T;
    g.R = R;
    g.nk = d_model / kBK;
    g.splits = p.splits;
    g.n_tile = p.n_tile;
    g.stages = p.stages;
    g.ws = wsf;
    CUtensorMap mw, mh;
    if (!hg::map_2d(&mw, w, R, d_model, 64, 64)) return MLA_ERR_CUDA;
    if (!hg::map_2d(&mh, h, d_model, T, 64, p.n_tile)) return MLA_ERR_CUDA;
    const size_t smem = static_cast<size_t>(p.stages) * (kBM * kBK * 2 + p.n_tile * kBK * 2) +
                        8 * (2 * kMaxStages + 1) + 1024;
    if (ensure_smem_limit(reinterpret_cast<const void*>(kvd_gemm_kernel), smem) != cudaSuccess) return MLA_ERR_CUDA;
    if (launch_pdl(kvd_gemm_kernel, dim3(p.m_tiles, p.n_tiles, p.splits), dim3(kThreads), smem, s, mw, mh, g) !=
        cudaSuccess)
      return MLA_ERR_CUDA;
  } else {
    const dim3 grid((R + kThreads - 1) / kThreads, (T + kSimtTokens - 1) / kSimtTokens);
    const cudaError_t e = launch_pdl(kvd_simt_kernel<float>, grid, dim3(kThreads), 0, s, static_cast<const float*>(h),
                                     static_cast<const float*>(w), T, d_model, R, wsf);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
  }
  const PageMap pages = {block_table, max_blocks, num_pages};
  cudaError_t e;
  const auto* gm = static_cast<const __nv_bfloat16*>(gamma);
  auto* cb = static_cast<__nv_bfloat16*>(c.data);
  const int64_t rs = static_cast<int64_t>(c.row_stride);
  const RopeTable rt = rope_table(c.d_r, rope_base);
  if (p.splits >= kFinishGroups) {  // a K split: four groups share each token's ranges
    const int grid = T < 148 * 16 ? T : 148 * 16;
    if (c.dtype == MLA_BF16)
      e = launch_pdl(kvd_finish_kernel<__nv_bfloat16>, dim3(grid), dim3(kFinishThreads), 0, s, wsf, p.splits, T,
                     c.d_c, c.d_r, gm, eps, cb, c.B, c.N_max, rs, seq_idx, pos, rt, pages);
    else
      e = launch_pdl(kvd_finish_kernel<float>, dim3(grid), dim3(kFinishThreads), 0, s, wsf, p.splits, T, c.d_c,
                     c.d_r, static_cast<const float*>(gamma), eps, static_cast<float*>(c.data), c.B, c.N_max, rs,
                     seq_idx, pos, rt, pages);
  } else {  // few ranges: one warp per token, thousands of tokens in flight
    const int warps = kThreads / 32;
    const int need = (T + warps - 1) / warps;
    const int grid = need < 148 * 32 ? need : 148 * 32;
    if (c.dtype == MLA_BF16)
      e = launch_pdl(kvd_finish_warp_kernel<__nv_bfloat16>, dim3(grid), dim3(kThreads), 0, s, wsf, p.splits, T,
                     c.d_c, c.d_r, gm, eps, cb, c.B, c.N_max, rs, seq_idx, pos, rt, pages);
    else
      e = launch_pdl(kvd_finish_warp_kernel<float>, dim3(grid), dim3(kThreads), 0, s, wsf, p.splits, T, c.d_c,
                     c.d_r, static_cast<const float*>(gamma), eps, static_cast<float*>(c.data), c.B, c.N_max, rs,
                     seq_idx, pos, rt, pages);
  }
  return cuda_status(e);
}

}  // namespace mla

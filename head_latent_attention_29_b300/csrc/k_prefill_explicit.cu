// Prefill without absorption: every head's keys and values are rebuilt from the
// cached latent rows, and the prompt runs standard causal attention per head.
//
//   K_nope[b][t][h][d] = sum_c c_KV[b][t][c] W_UK[h][d][c]     (0539edu.com section 2.2:
//   V     [b][t][h][d] = sum_c c_KV[b][t][c] W_UV[h][d][c]      k = c_KV W_UK, v = c_KV W_UV)
//   k_h,t = [K_nope[b][t][h] || k_R,t]   (the rotated key as cached; hotelren.com
//                                         section 6.2: one key shared by all heads)
//   q_h,i = [q_nope[b][i][h] || RoPE(q_R[b][i][h], start + i)]
//   o[b][i][h] = softmax_t(scale q_h,i . k_h,t, t <= start + i) V,  lse alongside
//
// The same page notes that in prefill the absorbed form costs more compute (every
// score runs over the 576-wide latent row) and that the explicit form is its
// precision fallback: per (query, key) pair and head the explicit form needs
// 2 (d_k + d_r) + 2 d_v = 640 FLOPs against 2 (d_c + d_r) + 2 d_c = 2176.
//
// Two kernels.  (1) kvup_kernel: the K_nope / V rebuild as one tcgen05 GEMM per
// (256 output features, 128 tokens, sequence) tile, A = the cached latent rows
// (K-major, straight from the cache through TMA), B = W_UK or W_UV rows (K-major),
// K = d_c = 512, written as bf16 [B][P][H][128] (P = start + S rows per sequence).
// (2) attn_kernel: one CTA per (sequence, head, 128-query tile); the tiles of one head
//     are consecutive (heaviest first), so resident CTAs share its K / V in L2.
// The query (192 wide, its RoPE part rotated on the way) sits in tensor memory as
// the A operand of S = Q K^T (M = 128 queries, N = 128 keys); S is double-buffered
// in tensor memory so that the softmax of one key tile overlaps the S product of
// the next; P goes to shared memory (bf16) and O += P V accumulates in tensor
// memory (M = 128 queries, N = 128 = d_v, V the MN-major B operand).  The running
// maximum is raised lazily (only when a tile's maximum exceeds it by more than
// 2^8), and O is rescaled in place only then.
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace px {

constexpr int kDK = 128;   // d_k = d_v: per-head key (no-position part) and value width
constexpr int kDR = 64;    // decoupled RoPE width
constexpr int kDC = 512;   // latent width
constexpr int kChunkBytes = 128 * 128;  // one 64-element-wide (128-byte) column block of 128 rows

// ---------------------------------------------------------------------------
// (1) K_nope / V rebuild
// ---------------------------------------------------------------------------
constexpr int kUpM = 128;          // tokens per CTA (M)
constexpr int kUpN = 256;          // output features per CTA (N)
constexpr int kUpStages = 4;
constexpr int kUpNk = kDC / 64;    // 8 K steps of 64
constexpr int kUpStageBytes = kUpM * 128 + kUpN * 128;  // 16 KB of latent rows + 32 KB of weight rows
constexpr int kUpThreads = 128;

struct UpArgs {
  int H;            // heads (even)
  int P;            // rows per sequence rebuilt (start + S)
  __nv_bfloat16* k_nope;  // [B][P][H][128]
  __nv_bfloat16* v;       // [B][P][H][128]
};

__global__ void __launch_bounds__(kUpThreads) kvup_kernel(const __grid_constant__ CUtensorMap map_c,
                                                          const __grid_constant__ CUtensorMap map_wuk,
                                                          const __grid_constant__ CUtensorMap map_wuv,
                                                          const __grid_constant__ UpArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bars = sbase + kUpStages * kUpStageBytes;  // full[4], empty[4], done
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int* abort = &s_abort;
  const int warp = threadIdx.x >> 5;
  const int half_tiles = g.H / 2;  // feature tiles per matrix (H * 128 / 256)
  const int ft = blockIdx.x, t0 = blockIdx.y * kUpM, b = blockIdx.z;
  const bool is_v = ft >= half_tiles;
  const int f0 = (is_v ? ft - half_tiles : ft) * kUpN;  // first output feature (h * 128 + d)

  griddep_launch();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kUpStages; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (kUpStages + i), 1);
    }
    mbar_init(bars + 8 * (2 * kUpStages), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), kUpN);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    const uint32_t leader = elect_one();
    const CUtensorMap* mw = is_v ? &map_wuv : &map_wuk;
    griddep_wait();  // the latent rows may still be written by the previous kernel
    for (int k = 0; k < kUpNk; ++k) {
      const int st = k % kUpStages;
      if (!warp_wait(bars + 8 * (kUpStages + st), ((k / kUpStages) & 1) ^ 1, abort)) break;
      const uint32_t sa = sbase + st * kUpStageBytes, full = bars + 8 * st;
      mbar_arrive_expect_tx_if(leader, full, kUpStageBytes);
      tma_load_3d_if(leader, sa, &map_c, full, k * 64, t0, b);                // 128 rows x 64 latent columns
      tma_load_2d_if(leader, sa + kUpM * 128, mw, full, k * 64, f0);          // 256 weight rows x 64 columns
    }
  } else if (warp == 1) {
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc = idesc_bf16(kUpM, kUpN, false, false);
    for (int k = 0; k < kUpNk; ++k) {
      const int st = k % kUpStages;
      if (!warp_wait(bars + 8 * st, (k / kUpStages) & 1, abort)) break;
      tc_fence_after();
      const uint32_t sa = sbase + st * kUpStageBytes, sb = sa + kUpM * 128;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss_if(leader, tmem, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024), idesc,
                  (k | kk) != 0);
      tc_commit_if(leader, bars + 8 * (kUpStages + st));
    }
    tc_commit_if(leader, bars + 8 * (2 * kUpStages));
  }
  __syncwarp();

  // epilogue: thread r holds token t0 + r (TMEM lane r), 256 consecutive features
  const bool ok = warp_wait(bars + 8 * (2 * kUpStages), 0, abort);
  tc_fence_after();
  griddep_wait();  // the output buffers may still be read by the previous kernel
  const int r = threadIdx.x, t = t0 + r;
  if (ok) {
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    __nv_bfloat16* out = (is_v ? g.v : g.k_nope) + (static_cast<size_t>(b) * g.P + t) * g.H * kDK + f0;
    for (int c0 = 0; c0 < kUpN; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + c0, v);
      tmem_wait_ld();
      if (t < g.P) {
        uint4* dst = reinterpret_cast<uint4*>(out + c0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                              pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                              pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                              pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) record_error(MLA_ERR_DEVICE_TIMEOUT, kSiteDecodeWait);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kUpN);
  }
}

// ---------------------------------------------------------------------------
// (2) causal attention per (sequence, head, 128-query tile)
// ---------------------------------------------------------------------------
constexpr int kQ = 128;            // queries per CTA (M, one per tensor-memory lane)
constexpr int kKT = 128;           // keys per tile (N of S, K of PV)
constexpr int kKStages = 2;        // key tiles in flight; ring load 0 carries the query
constexpr int kVStages = 2;
constexpr int kKBytes = 3 * kChunkBytes;   // K_nope 0-63, 64-127, rotated k_R: 48 KB
constexpr int kVBytes = 2 * kChunkBytes;   // V 0-63, 64-127: 32 KB
constexpr int kPBytes = 2 * kChunkBytes;   // P keys 0-63, 64-127: 32 KB
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKStages * kKBytes;
constexpr int kOffP = kOffV + kVStages * kVBytes;
constexpr int kOffX = kOffP + kPBytes;         // row maxima / sums exchanged by the two halves: [2][2][128] fp32
constexpr int kOffBar = kOffX + 2 * 2 * 128 * 4;
// barriers (8 bytes each)
// The softmax side arrives once per warp (after __syncwarp) on S-free, the maxima
// exchange, P-full and query-ready: 8 arrivals per phase instead of 256.
constexpr int kBarKFull = 0, kBarKEmpty = 2, kBarVFull = 4, kBarVEmpty = 6, kBarSFull = 8, kBarSFree = 10,
              kBarPFull = 12, kBarPvDone = 13, kBarQReady = 14, kBarDrain = 15, kBarX = 16, kNumBars = 18;
constexpr int kAttnSmem = kOffBar + 8 * kNumBars + 1024;  // + alignment slack
// warp 0: Q and K loads, 1: MMA, 2: V loads, 3: idle, 4-11: softmax.  Warps 4-7 take
// score columns 0-63 of their rows (and O columns 0-63), warps 8-11 columns 64-127
// of the same rows (TMEM lanes 32 (w % 4) ...).
constexpr int kAttnThreads = 384;
constexpr int kSoftmaxThreads = 256;
// tensor memory columns
constexpr uint32_t kColS = 0;      // two 128-column S buffers
constexpr uint32_t kColO = 256;    // O, 128 columns
constexpr uint32_t kColQ = 384;    // the query as bf16 pairs: 96 columns
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct AttnArgs {
  int B, S, H, start, P;   // P = start + S rows per sequence
  int causal;
  int q_tiles;             // ceil(S / 128)
  float scale_log2;        // scale * log2(e)
  __nv_bfloat16* o;        // [B][S][H][128]
  float* lse;              // [B][S][H] or nullptr
  RopeTable rope;
};

__device__ __forceinline__ uint32_t bar_at(uint32_t sbase, int i) { return sbase + kOffBar + 8 * i; }

__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ CUtensorMap map_qn,
                                                               const __grid_constant__ CUtensorMap map_qr,
                                                               const __grid_constant__ CUtensorMap map_k,
                                                               const __grid_constant__ CUtensorMap map_v,
                                                               const __grid_constant__ CUtensorMap map_c,
                                                               const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_hi[kDR / 2], s_lo[kDR / 2];
  volatile int* abort = &s_abort;
  const int warp = threadIdx.x >> 5;

  // work item: the query tiles of one (sequence, head) are consecutive, the heaviest
  // (latest) first, so the CTAs resident at any time cover a few heads and share
  // their keys and values in L2 instead of each streaming its own head from HBM
  const int qt = a.q_tiles - 1 - static_cast<int>(blockIdx.x) % a.q_tiles;
  const int rem = static_cast<int>(blockIdx.x) / a.q_tiles;
  const int b = rem / a.H, h = rem % a.H;
  const int q0 = qt * kQ;
  // keys this tile reads: 0 .. last (causal: the last query's position)
  const int q_last = a.start + min(q0 + kQ, a.S) - 1;
  const int n_keys = a.causal ? q_last + 1 : a.P;
  const int nkt = (n_keys + kKT - 1) / kKT;

  griddep_launch();
  for (int i = threadIdx.x; i < kDR / 2; i += blockDim.x) {
    s_hi[i] = a.rope.u_hi[i];
    s_lo[i] = a.rope.u_lo[i];
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_at(sbase, kBarKFull + i), 1);
      mbar_init(bar_at(sbase, kBarKEmpty + i), 1);
      mbar_init(bar_at(sbase, kBarVFull + i), 1);
      mbar_init(bar_at(sbase, kBarVEmpty + i), 1);
      mbar_init(bar_at(sbase, kBarSFull + i), 1);
      mbar_init(bar_at(sbase, kBarSFree + i), kSoftmaxThreads / 32);
      mbar_init(bar_at(sbase, kBarX + i), kSoftmaxThreads / 32);
    }
    mbar_init(bar_at(sbase, kBarPFull), kSoftmaxThreads / 32);
    mbar_init(bar_at(sbase, kBarPvDone), 1);
    mbar_init(bar_at(sbase, kBarQReady), kSoftmaxThreads / 32);
    mbar_init(bar_at(sbase, kBarDrain), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  griddep_wait();  // queries, rebuilt K / V and the cache come from earlier kernels

  if (warp == 0) {
    // ------------------------------------------------------------ query and keys
    const uint32_t leader = elect_one();
    const int qrow = b * a.S + q0;  // first query row of the tile in [B * S]
    // ring load 0: the query's three 64-wide blocks into K stage 0
    {
      const uint32_t full = bar_at(sbase, kBarKFull + 0), dst = sbase + kOffK;
      mbar_arrive_expect_tx_if(leader, full, kKBytes);
      tma_load_3d_if(leader, dst, &map_qn, full, 0, h, qrow);
      tma_load_3d_if(leader, dst + kChunkBytes, &map_qn, full, 64, h, qrow);
      tma_load_3d_if(leader, dst + 2 * kChunkBytes, &map_qr, full, 0, h, qrow);
    }
    for (int j = 0; j < nkt; ++j) {
      const int li = j + 1, st = li % kKStages;
      if (!warp_wait(bar_at(sbase, kBarKEmpty + st), ((li / kKStages) & 1) ^ 1, abort)) break;
      const uint32_t full = bar_at(sbase, kBarKFull + st), dst = sbase + kOffK + st * kKBytes;
      const int krow = b * a.P + j * kKT;
      mbar_arrive_expect_tx_if(leader, full, kKBytes);
      tma_load_3d_if(leader, dst, &map_k, full, 0, h, krow);
      tma_load_3d_if(leader, dst + kChunkBytes, &map_k, full, 64, h, krow);
      tma_load_3d_if(leader, dst + 2 * kChunkBytes, &map_c, full, kDC, j * kKT, b);  // the rotated key
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ values
    const uint32_t leader = elect_one();
    for (int j = 0; j < nkt; ++j) {
      const int st = j % kVStages;
      if (!warp_wait(bar_at(sbase, kBarVEmpty + st), ((j / kVStages) & 1) ^ 1, abort)) break;
      const uint32_t full = bar_at(sbase, kBarVFull + st), dst = sbase + kOffV + st * kVBytes;
      const int krow = b * a.P + j * kKT;
      mbar_arrive_expect_tx_if(leader, full, kVBytes);
      tma_load_3d_if(leader, dst, &map_v, full, 0, h, krow);
      tma_load_3d_if(leader, dst + kChunkBytes, &map_v, full, 64, h, krow);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one();
    constexpr uint32_t idesc_s = idesc_bf16(kQ, kKT, false, false);  // Q (tensor memory) x K^T
    constexpr uint32_t idesc_o = idesc_bf16(kQ, kDK, false, true);   // P x V, V MN-major
    auto issue_pv = [&](int jj) -> bool {
      if (!warp_wait(bar_at(sbase, kBarPFull), jj & 1, abort)) return false;
      const int st = jj % kVStages;
      if (!warp_wait(bar_at(sbase, kBarVFull + st), (jj / kVStages) & 1, abort)) return false;
      tc_fence_after();
      const uint32_t pa = sbase + kOffP, vb = sbase + kOffV + st * kVBytes;
#pragma unroll
      for (int kk = 0; kk < kKT / 16; ++kk)
        mma_ss_if(leader, tmem + kColO, sdesc_sw128(pa + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024),
                  sdesc_sw128(vb + kk * 16 * 128, kChunkBytes, 1024), idesc_o, (jj | kk) != 0);
      tc_commit_if(leader, bar_at(sbase, kBarVEmpty + st));
      tc_commit_if(leader, bar_at(sbase, kBarPvDone));
      return true;
    };
    bool go = warp_wait(bar_at(sbase, kBarQReady), 0, abort);
    if (go && leader) mbar_arrive(bar_at(sbase, kBarKEmpty + 0));  // the query's slot is free again
    for (int j = 0; go && j < nkt; ++j) {
      const int li = j + 1, st = li % kKStages, sb = j & 1;
      if (!warp_wait(bar_at(sbase, kBarKFull + st), (li / kKStages) & 1, abort)) break;
      if (j >= 2 && !warp_wait(bar_at(sbase, kBarSFree + sb), ((j - 2) >> 1) & 1, abort)) break;
      tc_fence_after();
      const uint32_t kb = sbase + kOffK + st * kKBytes, d = tmem + kColS + sb * kKT;
#pragma unroll
      for (int ch = 0; ch < 3; ++ch)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_if(leader, d, tmem + kColQ + ch * 32 + kk * 8, sdesc_sw128(kb + ch * kChunkBytes + kk * 32, 16, 1024),
                    idesc_s, (ch | kk) != 0);
      tc_commit_if(leader, bar_at(sbase, kBarKEmpty + st));
      tc_commit_if(leader, bar_at(sbase, kBarSFull + sb));
      if (j >= 1 && !issue_pv(j - 1)) go = false;
    }
    if (go && nkt > 0) issue_pv(nkt - 1);
    // every MMA this warp issued has completed before teardown
    tc_commit_if(leader, bar_at(sbase, kBarDrain));
    warp_wait(bar_at(sbase, kBarDrain), 0, abort);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax: two threads per query row
    // Thread (half hf, row r) owns score columns [64 hf, 64 hf + 64) of every key tile
    // and O columns [64 hf, 64 hf + 64).  Per tile the two halves exchange their row
    // maxima through shared memory (a barrier of all softmax threads, bounded like
    // every wait), so that both take the same reference; each keeps the sum of its own
    // half, and the halves' sums are added once at the end.
    const int hf = (warp - 4) >> 2;
    const int r = (threadIdx.x - 128) & 127;
    const uint32_t lane_off = static_cast<uint32_t>(r & ~31) << 16;
    const int qi = q0 + r;                               // prompt index of this row
    const int qpos = a.start + min(qi, a.S - 1);         // rows past the prompt mirror its last query
    const int limit = a.causal ? qpos : a.P - 1;         // last key this row reads
    float* xch = reinterpret_cast<float*>(gbase + kOffX);  // [slot][half][row]
    bool ok = true;
    // the query row into tensor memory (half 0: the two no-position blocks; half 1: the
    // RoPE block, rotated at the row's position)
    if (warp_wait(bar_at(sbase, kBarKFull + 0), 0, abort)) {
      for (int ch = hf == 0 ? 0 : 2; ch < (hf == 0 ? 2 : 3); ++ch) {
        const uint8_t* row = gbase + kOffK + ch * kChunkBytes + r * 128;
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 x = *reinterpret_cast<const uint4*>(row + ((u ^ (r & 7)) << 4));
          v[4 * u] = x.x;
          v[4 * u + 1] = x.y;
          v[4 * u + 2] = x.z;
          v[4 * u + 3] = x.w;
        }
        if (ch == 2) {
#pragma unroll
          for (int w = 0; w < 32; ++w) {  // word w holds RoPE pair w
            float sn, cs;
            rope_sincos(a.start + qi, s_hi[w], s_lo[w], &sn, &cs);
            const float x0 = __uint_as_float(v[w] << 16), x1 = __uint_as_float(v[w] & 0xFFFF0000u);
            v[w] = pack_bf16x2(fmaf(x0, cs, -x1 * sn), fmaf(x0, sn, x1 * cs));
          }
        }
        tmem_st32(tmem + lane_off + kColQ + ch * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
    } else {
      ok = false;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar_at(sbase, kBarQReady));

    float m_ref = 0.f, l = 0.f;
    for (int j = 0; ok && j < nkt; ++j) {
      const int sb = j & 1, kbase = j * kKT + hf * 64;
      if (!warp_wait(bar_at(sbase, kBarSFull + sb), (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld64(tmem + lane_off + kColS + sb * kKT + hf * 64, sr);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(bar_at(sbase, kBarSFree + sb));  // this half of S is in registers
      // keys past the row's limit only on the diagonal (causal) or last (non-causal) tile
      if (__any_sync(0xffffffffu, kbase + 63 > limit)) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (kbase + c > limit) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) mx[c] = __uint_as_float(sr[c]);
#pragma unroll
      for (int c = 4; c < 64; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(sr[c]));
      const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
      // both halves' maxima: the same reference on both sides of the row
      xch[(sb * 2 + hf) * kQ + r] = mloc;
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(bar_at(sbase, kBarX + sb));
      if (!warp_wait(bar_at(sbase, kBarX + sb), (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      const float mt = fmaxf(mloc, xch[(sb * 2 + (hf ^ 1)) * kQ + r]);
      float alpha = 1.f;
      if (j == 0) {
        m_ref = mt;  // key 0 is always read: finite
      } else if (mt > m_ref + kRescaleThreshold) {
        alpha = fast_exp2(m_ref - mt);
        m_ref = mt;
      }
      // probabilities as bf16 pairs, and this half's row sum as rounded
      uint32_t pk[32];
      float psum[4] = {0.f, 0.f, 0.f, 0.f};
      const float neg = -m_ref;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const uint32_t w = pack_bf16x2(fast_exp2(fmaf(__uint_as_float(sr[c]), a.scale_log2, neg)),
                                       fast_exp2(fmaf(__uint_as_float(sr[c + 1]), a.scale_log2, neg)));
        pk[c / 2] = w;
        psum[(c / 2) & 3] += __uint_as_float(w << 16) + __uint_as_float(w & 0xFFFF0000u);
      }
      // the previous tile's PV product has finished with P and O
      if (j >= 1 && !warp_wait(bar_at(sbase, kBarPvDone), (j - 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + kColO + hf * 64 + cc * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(tmem + lane_off + kColO + hf * 64 + cc * 32, v);
        }
        tmem_wait_st();
      }
      l = l * alpha + ((psum[0] + psum[1]) + (psum[2] + psum[3]));
      // this half of row r of P (K-major, 128-byte swizzle: keys 64 hf .. 64 hf + 63)
      uint8_t* prow = gbase + kOffP + hf * kChunkBytes + r * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      fence_proxy_async_cta();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(bar_at(sbase, kBarPFull));
    }
    // epilogue: the halves' sums added, O / l and the log-sum-exp, rows inside the prompt
    if (ok && nkt > 0 && warp_wait(bar_at(sbase, kBarPvDone), (nkt - 1) & 1, abort)) {
      const int sx = nkt & 1;  // the exchange slot the last tile did not use
      xch[(sx * 2 + hf) * kQ + r] = l;
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(bar_at(sbase, kBarX + sx));
      if (warp_wait(bar_at(sbase, kBarX + sx), (nkt >> 1) & 1, abort)) {
        const float ltot = l + xch[(sx * 2 + (hf ^ 1)) * kQ + r];
        tc_fence_after();
        const float inv = 1.f / ltot;
        __nv_bfloat16* orow = a.o + ((static_cast<size_t>(b) * a.S + qi) * a.H + h) * kDK + hf * 64;
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + kColO + hf * 64 + cc * 32, v);
          tmem_wait_ld();
          if (qi < a.S) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv),
                                  pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv),
                                  pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv),
                                  pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv));
          }
        }
        if (hf == 0 && qi < a.S && a.lse != nullptr)
          a.lse[(static_cast<size_t>(b) * a.S + qi) * a.H + h] = (m_ref + __log2f(ltot)) * 0.69314718055994531f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && s_abort) record_error(MLA_ERR_DEVICE_TIMEOUT, kSiteDecodeWait);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace px

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static bool tmap(CUtensorMap* m, const void* p, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                 const uint32_t* box) {
  hg::EncodeTiledFn enc = hg::encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t bx[3], es[3];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(p), d, st, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t prefill_explicit_workspace_size(int32_t B, int32_t start, int32_t S, int32_t H) {
  if (B <= 0 || start < 0 || S <= 0 || H <= 0) return 0;
  return 2 * static_cast<size_t>(B) * static_cast<size_t>(start + S) * static_cast<size_t>(H) * px::kDK * 2;
}

mla_status launch_prefill_explicit(const void* q_nope, const void* q_rope, const mla_cache& c, const void* w_uk,
                                   const void* w_uv, int32_t start, int32_t S, int32_t causal, int32_t H, float scale,
                                   float rope_base, void* ws, size_t ws_bytes, void* o, float* lse, cudaStream_t s) {
  using namespace px;
  const int B = c.B, P = start + S;
  if (ws == nullptr || ws_bytes < prefill_explicit_workspace_size(B, start, S, H) || !aligned16(ws))
    return MLA_ERR_WORKSPACE;
  __nv_bfloat16* k_nope = static_cast<__nv_bfloat16*>(ws);
  __nv_bfloat16* v = k_nope + static_cast<size_t>(B) * P * H * kDK;
  const uint64_t R = static_cast<uint64_t>(c.d_c + c.d_r);
  const uint64_t rs = static_cast<uint64_t>(c.row_stride) * 2;
  CUtensorMap map_c_up, map_c_kr, map_wuk, map_wuv, map_qn, map_qr, map_k, map_v;
  {
    const uint64_t dims[3] = {R, static_cast<uint64_t>(c.N_max), static_cast<uint64_t>(B)};
    const uint64_t str[2] = {rs, rs * c.N_max};
    const uint32_t box[3] = {64, 128, 1};
    if (!tmap(&map_c_up, c.data, 3, dims, str, box) || !tmap(&map_c_kr, c.data, 3, dims, str, box))
      return MLA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(kDC), static_cast<uint64_t>(H) * kDK};
    const uint64_t str[1] = {kDC * 2};
    const uint32_t box[2] = {64, 256};
    if (!tmap(&map_wuk, w_uk, 2, dims, str, box) || !tmap(&map_wuv, w_uv, 2, dims, str, box)) return MLA_ERR_CUDA;
  }
  {
    const uint64_t rows = static_cast<uint64_t>(B) * S;
    const uint64_t dn[3] = {kDK, static_cast<uint64_t>(H), rows}, sn[2] = {kDK * 2, static_cast<uint64_t>(H) * kDK * 2};
    const uint64_t dr[3] = {kDR, static_cast<uint64_t>(H), rows}, sr[2] = {kDR * 2, static_cast<uint64_t>(H) * kDR * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!tmap(&map_qn, q_nope, 3, dn, sn, box) || !tmap(&map_qr, q_rope, 3, dr, sr, box)) return MLA_ERR_CUDA;
    const uint64_t dk[3] = {kDK, static_cast<uint64_t>(H), static_cast<uint64_t>(B) * P};
    if (!tmap(&map_k, k_nope, 3, dk, sn, box) || !tmap(&map_v, v, 3, dk, sn, box)) return MLA_ERR_CUDA;
  }
  // (1) K_nope / V for rows 0 .. P-1 of every sequence
  UpArgs u = {H, P, k_nope, v};
  const size_t up_smem = static_cast<size_t>(kUpStages) * kUpStageBytes + 8 * (2 * kUpStages + 1) + 1024;
  if (ensure_smem_limit(reinterpret_cast<const void*>(kvup_kernel), up_smem) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_pdl(kvup_kernel, dim3(H, (P + kUpM - 1) / kUpM, B), dim3(kUpThreads), up_smem, s, map_c_up, map_wuk,
                 map_wuv, u) != cudaSuccess)
    return MLA_ERR_CUDA;
  // (2) attention
  AttnArgs a = {};
  a.B = B;
  a.S = S;
  a.H = H;
  a.start = start;
  a.P = P;
  a.causal = causal ? 1 : 0;
  a.q_tiles = (S + kQ - 1) / kQ;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.rope = rope_table(kDR, rope_base);
  if (ensure_smem_limit(reinterpret_cast<const void*>(attn_kernel), kAttnSmem) != cudaSuccess) return MLA_ERR_CUDA;
  const long long grid = static_cast<long long>(B) * H * a.q_tiles;
  if (grid > 0x7FFFFFFFLL) return MLA_ERR_UNSUPPORTED;
  return cuda_status(launch_pdl(attn_kernel, dim3(static_cast<unsigned>(grid)), dim3(kAttnThreads), kAttnSmem, s,
                                map_qn, map_qr, map_k, map_v, map_c_kr, a));
}

}  // namespace mla

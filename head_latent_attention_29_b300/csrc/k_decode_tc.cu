// Tensor-core MLA decode attention for sm_103a (bf16 operands, fp32 accumulate).
//
// What is computed (absorbed form, 0539edu.com sections 3.1-3.2; decoupled RoPE
// row of the icman.com.cn article, section 2; max-subtracted softmax of the
// hotelren.com guide, section 7.3): for every sequence b and head h,
//   s_t = scale * q_cat[b][h] . cache[b][t]        (d_c + d_r wide)
//   o_lat[b][h] = sum_t softmax(s)_t * cache[b][t][0:d_c],  lse = ln sum exp(s).
//
// How it maps onto B300:
//  * All heads of a sequence share every cache row, so both products are dense
//    contractions with the heads as the M = 128 dimension.
//  * The fp32 output accumulator for 128 heads x 512 latent columns is 256 KB,
//    the whole tensor memory of one SM.  Each unit of work therefore runs on a
//    2-CTA cluster:
//      - CTA 0 (score CTA) holds the absorbed query in tensor memory (A operand
//        of S = Q C^T, 288 columns), computes S for 64-token blocks into a
//        double-buffered 64-column accumulator, runs the online softmax (one
//        thread per head row, no cross-thread reduction), and writes the bf16
//        probabilities P straight into CTA 1's shared memory.
//      - CTA 1 (output CTA) accumulates O += P C[:, 0:512] with two N = 256
//        MMAs per 16-token step into its full 512-column tensor memory, and
//        rescales O in place on the rare blocks where the running maximum of a
//        row grew by more than 2^8.
//    The two contractions (576 and 512 wide) are split across the two SMs with
//    no redundant work.
//  * Cache rows stream in through TMA (128-byte swizzled 64x64 chunks, 3-stage
//    ring per CTA).  The same swizzled chunk is the K-major B operand of
//    S = Q C^T and the MN-major B operand of O = P C.
//  * The token stream of all sequences is cut into equal runs of 64-token blocks,
//    one run per cluster, so every SM pair gets the same work whatever the mix
//    of lengths; each (run, sequence) overlap leaves an unnormalised partial
//    (m, l, O) and a combine kernel merges the partials of each sequence.
#include <cmath>

#include "mla_internal.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace dtc {

constexpr int kBN = 64;                     // tokens per block
constexpr int kDC = 512;                    // latent width
constexpr int kChDC = kDC / 64;             // 8 chunks of 64 columns cover the latent
constexpr int kChunk = kBN * 128;           // bytes of one [64 tok x 64 col] bf16 chunk
constexpr int kStages = 3;
constexpr int kStageDC = kChDC * kChunk;    // 64 KB of latent chunks per stage
constexpr int kM = 128;                     // head rows per MMA
constexpr int kMaxPairs = 160;              // upper bound on clusters per launch
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P stays <= 256

// Shared-memory map (offsets from a 1024-aligned base; identical in both CTAs so
// that remote addresses map one to one).
constexpr int kOffStage = 0;                           // kStages x 64 KB latent chunks
constexpr int kOffRope = kStages * kStageDC;           // score CTA: kStages x 8 KB RoPE chunks
constexpr int kOffP = kStages * kStageDC;              // output CTA: 2 x 16 KB P tiles
constexpr int kPBytes = kM * 128;
constexpr int kOffAlpha = kOffP + 2 * kPBytes;         // output CTA: 2 x 128 fp32 row factors
constexpr int kOffBar = kOffAlpha + 2 * kM * 4;
enum : int {
  kBarFull = 0,                     // [kStages] TMA landed
  kBarEmpty = kBarFull + kStages,   // [kStages] stage consumed by this CTA's MMAs
  kBarSFull = kBarEmpty + kStages,  // [2] score CTA: S buffer written
  kBarSEmpty = kBarSFull + 2,       // [2] score CTA: S buffer read
  kBarQReady = kBarSEmpty + 2,      // score CTA: query loaded into tensor memory
  kBarPFree = kBarQReady + 1,       // [2] score CTA: output CTA released P tile
  kBarPFull = kBarPFree + 2,        // [2] output CTA: P tile and factors written
  kBarPvGo = kBarPFull + 2,         // output CTA: block may be multiplied
  kBarODone = kBarPvGo + 1,         // [2] output CTA: PV of a block completed
  kBarDrain = kBarODone + 2,        // MMA drain at teardown
  kNumBars = kBarDrain + 1,
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 128;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kOffRope + kStages * kChunk <= kOffP + 2 * kPBytes, "score CTA map");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// tensor-memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0;     // score CTA: query, R/2 columns (bf16 pairs)
constexpr uint32_t kColS = 320;   // score CTA: two 64-column S buffers
// output CTA: O occupies columns [0, 512)

struct Misc {                     // at kOffMisc
  uint32_t tmem;
  int abort;
  int flag[2];                    // output CTA: block id + 1 of a block that rescaled
  long long lo, hi, cum0;
  int b0, len0;
};
static_assert(sizeof(Misc) <= 128, "misc");

struct Args {
  const __nv_bfloat16* q_cat;  // [B][H][R]
  const int32_t* seq_lens;     // [B]
  int B, H, N_max, R, nch;     // nch: 64-column chunks per row (R / 64)
  float scale_log2;            // scale * log2(e)
  int32_t* hdr;                // workspace: [0] = total blocks, [1] = runs used
  int32_t* cum;                // workspace: [B + 1] first block of each sequence
  float* part_m;               // [slots][128] running max (log2 units)
  float* part_l;               // [slots][128] running sum
  float* part_o;               // [slots][128][512] unnormalised output
};

__device__ __forceinline__ int clamp_len(int n, int n_max) { return n < 0 ? 0 : (n > n_max ? n_max : n); }

// Walks the 64-token blocks [lo, hi) of the flattened token stream.
struct Cursor {
  const int32_t* seq_lens;
  int n_max;
  long long g, lo, hi, cum;
  int b, len, nblk;
  __device__ void start(const Misc& m, const int32_t* sl, int nm) {
    seq_lens = sl;
    n_max = nm;
    g = lo = m.lo;
    hi = m.hi;
    cum = m.cum0;
    b = m.b0;
    len = m.len0;
    nblk = (len + kBN - 1) / kBN;
  }
  __device__ bool ok() const { return g < hi; }
  __device__ void next() {
    ++g;
    while (g < hi && g >= cum + nblk) {
      cum += nblk;
      ++b;
      len = clamp_len(seq_lens[b], n_max);
      nblk = (len + kBN - 1) / kBN;
    }
  }
  __device__ int t0() const { return static_cast<int>(g - cum) * kBN; }
  __device__ int rows() const { return min(kBN, len - t0()); }
  __device__ bool first() const { return g == lo || g == cum; }
  __device__ bool last() const { return g == hi - 1 || g == cum + nblk - 1; }
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + kOffBar + 8 * i; }

template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait<kCluster>(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Plan the run of this cluster: total blocks T, runs P = min(clusters, T), this
// run's [lo, hi), and the sequence that holds block lo.  One warp.
__device__ void plan_run(const Args& a, Misc* misc, bool write_table) {
  const int lane = threadIdx.x & 31;
  long long T = 0;
  for (int base = 0; base < a.B; base += 32) {
    const int b = base + lane;
    int nb = 0;
    if (b < a.B) {
      const int n = a.seq_lens[b];
      if (write_table && (n < 0 || n > a.N_max)) record_error(MLA_ERR_DEVICE_INDEX, kSiteDecodeLength);
      nb = (clamp_len(n, a.N_max) + kBN - 1) / kBN;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, off);
    T += nb;
  }
  const long long nclus = nclusters_x();
  const long long P = T < nclus ? T : nclus;
  const long long cid = cluster_id_x();
  long long lo = 0, hi = 0;
  if (cid < P) {
    lo = cid * T / P;
    hi = (cid + 1) * T / P;
  }
  int b0 = 0, len0 = 0;
  long long cum0 = 0;
  if (lo < hi || write_table) {
    long long run = 0;
    bool found = false;
    for (int base = 0; base < a.B; base += 32) {
      const int b = base + lane;
      const int n = b < a.B ? clamp_len(a.seq_lens[b], a.N_max) : 0;
      const int nb = (n + kBN - 1) / kBN;
      int incl = nb;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const long long excl = run + incl - nb;
      if (write_table && b < a.B) a.cum[b] = static_cast<int32_t>(excl);
      const bool hit = !found && b < a.B && nb > 0 && excl <= lo && lo < excl + nb;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m != 0u) {
        const int src = __ffs(m) - 1;
        b0 = base + src;
        cum0 = __shfl_sync(0xffffffffu, excl, src);
        len0 = __shfl_sync(0xffffffffu, n, src);
        found = true;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      if (found && !write_table) break;
    }
  }
  if (lane == 0) {
    misc->lo = lo;
    misc->hi = hi;
    misc->b0 = b0;
    misc->cum0 = cum0;
    misc->len0 = len0;
    if (write_table) {
      a.cum[a.B] = static_cast<int32_t>(T);
      a.hdr[0] = static_cast<int32_t>(T);
      a.hdr[1] = static_cast<int32_t>(P);
    }
  }
}

__global__ void __launch_bounds__(256, 1) decode_split_kernel(const __grid_constant__ CUtensorMap map,
                                                              const Args a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  Misc* misc = reinterpret_cast<Misc*>(gbase + kOffMisc);
  volatile int* abort = &misc->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = score CTA, 1 = output CTA
  const bool score_cta = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_addr(sbase, kBarFull + i), 1);
      mbar_init(bar_addr(sbase, kBarEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_addr(sbase, kBarSFull + i), 1);
      mbar_init(bar_addr(sbase, kBarSEmpty + i), 128);
      mbar_init(bar_addr(sbase, kBarPFree + i), 1);
      mbar_init(bar_addr(sbase, kBarPFull + i), 128);
      mbar_init(bar_addr(sbase, kBarODone + i), 1);
    }
    mbar_init(bar_addr(sbase, kBarQReady), 128);
    mbar_init(bar_addr(sbase, kBarPvGo), 128);
    mbar_init(bar_addr(sbase, kBarDrain), 1);
    misc->abort = 0;
    misc->flag[0] = misc->flag[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&map);
  if (warp == 1) {
    tmem_alloc(sbase + kOffMisc + offsetof(Misc, tmem), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2) plan_run(a, misc, cluster_id_x() == 0 && score_cta);
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // peer barriers initialised before any remote arrive

  const uint32_t tmem = misc->tmem;
  const int nch = a.nch;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int nload = score_cta ? nch : kChDC;
      Cursor c;
      c.start(*misc, a.seq_lens, a.N_max);
      for (int k = 0; c.ok(); c.next(), ++k) {
        const int st = k % kStages;
        if (!mbar_wait(bar_addr(sbase, kBarEmpty + st), ((k / kStages) & 1) ^ 1, abort)) break;
        mbar_arrive_expect_tx(bar_addr(sbase, kBarFull + st), nload * kChunk);
        for (int ch = 0; ch < nload; ++ch) {
          const uint32_t dst = ch < kChDC ? sbase + kOffStage + st * kStageDC + ch * kChunk
                                          : sbase + kOffRope + st * kChunk;
          tma_load_3d(dst, &map, bar_addr(sbase, kBarFull + st), ch * 64, c.t0(), c.b);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Cursor c;
      c.start(*misc, a.seq_lens, a.N_max);
      if (score_cta) {
        constexpr uint32_t idesc = idesc_bf16(kM, kBN, false, false);
        int seg = 0;
        for (int k = 0; c.ok(); c.next(), ++k) {
          if (c.first()) {
            if (!mbar_wait(bar_addr(sbase, kBarQReady), seg & 1, abort)) break;
            ++seg;
          }
          const int st = k % kStages, sb = k & 1;
          if (!mbar_wait(bar_addr(sbase, kBarFull + st), (k / kStages) & 1, abort)) break;
          if (!mbar_wait(bar_addr(sbase, kBarSEmpty + sb), ((k >> 1) & 1) ^ 1, abort)) break;
          tc_fence_after();
          const uint32_t d = tmem + kColS + sb * kBN;
          for (int ch = 0; ch < nch; ++ch) {
            const uint32_t chunk = ch < kChDC ? sbase + kOffStage + st * kStageDC + ch * kChunk
                                              : sbase + kOffRope + st * kChunk;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc = sdesc_sw128(chunk + kk * 32, 16, 1024);
              mma_ts(d, tmem + kColQ + ch * 32 + kk * 8, bdesc, idesc, (ch | kk) != 0);
            }
          }
          tc_commit(bar_addr(sbase, kBarEmpty + st));
          tc_commit(bar_addr(sbase, kBarSFull + sb));
        }
      } else {
        constexpr uint32_t idesc = idesc_bf16(kM, 256, false, true);
        for (int k = 0; c.ok(); c.next(), ++k) {
          const int st = k % kStages, sb = k & 1;
          if (!mbar_wait(bar_addr(sbase, kBarPvGo), k & 1, abort)) break;
          if (!mbar_wait(bar_addr(sbase, kBarFull + st), (k / kStages) & 1, abort)) break;
          tc_fence_after();
          const uint32_t pa = sbase + kOffP + sb * kPBytes;
          const uint32_t stage = sbase + kOffStage + st * kStageDC;
          const bool acc0 = !c.first();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = sdesc_sw128(pa + kk * 32, 16, 1024);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint64_t bdesc = sdesc_sw128(stage + half * 4 * kChunk + kk * 16 * 128, kChunk, 1024);
              mma_ss(tmem + half * 256, adesc, bdesc, idesc, (acc0 || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit(bar_addr(sbase, kBarEmpty + st));
          tc_commit(bar_addr(sbase, kBarODone + sb));
          tc_commit_mc(bar_addr(sbase, kBarPFree + sb), static_cast<uint16_t>(1u));  // to the score CTA
        }
      }
      // drain: every MMA this thread issued has completed before teardown
      tc_commit(bar_addr(sbase, kBarDrain));
      mbar_wait(bar_addr(sbase, kBarDrain), 0, abort);
    }
  } else if (warp >= 4) {
    const int r = threadIdx.x - 128;                       // head row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(r & ~31) << 16;
    Cursor c;
    c.start(*misc, a.seq_lens, a.N_max);
    if (score_cta) {
      // ---------------------------------------------------------- softmax
      float m_ref = 0.f, l = 0.f;
      int k = 0;
      for (; c.ok(); c.next(), ++k) {
        if (c.first()) {
          // query of this sequence into tensor memory (rows >= H are zero)
          const uint4* src = reinterpret_cast<const uint4*>(a.q_cat + (static_cast<long long>(c.b) * a.H + r) * a.R);
          for (int j = 0; j < nch; ++j) {
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              uint4 x = make_uint4(0u, 0u, 0u, 0u);
              if (r < a.H) x = __ldg(src + j * 8 + u);
              v[4 * u] = x.x;
              v[4 * u + 1] = x.y;
              v[4 * u + 2] = x.z;
              v[4 * u + 3] = x.w;
            }
            tmem_st32(tmem + lane_off + kColQ + j * 32, v);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar_addr(sbase, kBarQReady));
        }
        const int sb = k & 1;
        if (!warp_wait(bar_addr(sbase, kBarSFull + sb), (k >> 1) & 1, abort)) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld64(tmem + lane_off + kColS + sb * kBN, sr);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar_addr(sbase, kBarSEmpty + sb));

        const int nv = c.rows();
        float mloc = -INFINITY;
#pragma unroll
        for (int j = 0; j < kBN; ++j) {
          const float x = j < nv ? __uint_as_float(sr[j]) * a.scale_log2 : -INFINITY;
          sr[j] = __float_as_uint(x);
          mloc = fmaxf(mloc, x);
        }
        float alpha = 1.f;
        bool rescaled = false;
        if (c.first()) {
          m_ref = mloc;
          l = 0.f;
        } else if (mloc > m_ref + kRescaleThreshold) {
          alpha = fast_exp2(m_ref - mloc);
          m_ref = mloc;
          l *= alpha;
          rescaled = true;
        }
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int j = 0; j < kBN; j += 2) {
          const float p0 = fast_exp2(__uint_as_float(sr[j]) - m_ref);
          const float p1 = fast_exp2(__uint_as_float(sr[j + 1]) - m_ref);
          lsum += p0 + p1;
          pk[j >> 1] = pack_bf16x2(p0, p1);
        }
        l += lsum;
        if (!warp_wait(bar_addr(sbase, kBarPFree + sb), ((k >> 1) & 1) ^ 1, abort)) break;
        // P row r into the output CTA's P tile (K-major, 128-byte swizzle)
        const uint32_t prow = sbase + kOffP + sb * kPBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          st_cluster_v4(prow + ((cc ^ (r & 7)) << 4), 1u, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2],
                        pk[4 * cc + 3]);
        st_cluster_f32(sbase + kOffAlpha + sb * kM * 4 + r * 4, 1u, alpha);
        if (__any_sync(0xffffffffu, rescaled) && lane == 0)
          st_cluster_f32(sbase + kOffMisc + offsetof(Misc, flag) + sb * 4, 1u, __int_as_float(k + 1));
        fence_proxy_async_cluster();
        mbar_arrive_cluster(bar_addr(sbase, kBarPFull + sb), 1u);
        if (c.last() && r < a.H) {
          const long long slot = cluster_id_x() + c.b;
          a.part_m[slot * kM + r] = m_ref;
          a.part_l[slot * kM + r] = l;
        }
      }
      // the output CTA's releases of the last two P tiles have landed before exit
      for (int i = k - 2; i < k; ++i)
        if (i >= 0) warp_wait(bar_addr(sbase, kBarPFree + (i & 1)), (i >> 1) & 1, abort);
    } else {
      // ---------------------------------------------------------- correction + epilogue
      int k = 0;
      for (; c.ok(); c.next(), ++k) {
        const int sb = k & 1, st = k % kStages;
        if (!warp_wait<true>(bar_addr(sbase, kBarPFull + sb), (k >> 1) & 1, abort)) break;
        const bool need = !c.first() && misc->flag[sb] == k + 1;
        if (need) {
          const float alpha = reinterpret_cast<const float*>(gbase + kOffAlpha)[sb * kM + r];
          const int kp = k - 1;  // PV of the previous block has to be complete
          if (!warp_wait(bar_addr(sbase, kBarODone + (kp & 1)), (kp >> 1) & 1, abort)) break;
          tc_fence_after();
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t v[64];
            tmem_ld64(tmem + lane_off + cc * 64, v);
            tmem_wait_ld();
            uint32_t lo32[32], hi32[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              lo32[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
              hi32[j] = __float_as_uint(__uint_as_float(v[32 + j]) * alpha);
            }
            tmem_st32(tmem + lane_off + cc * 64, lo32);
            tmem_st32(tmem + lane_off + cc * 64 + 32, hi32);
          }
          tmem_wait_st();
        }
        const int nv = c.rows();
        if (nv < kBN) {
          // rows past the end of the sequence must not carry NaN/Inf into P C
          if (!warp_wait(bar_addr(sbase, kBarFull + st), (k / kStages) & 1, abort)) break;
          uint8_t* stage = gbase + kOffStage + st * kStageDC;
          const int npieces = (kBN - nv) * kChDC * 8;  // 16-byte pieces
          for (int q = r; q < npieces; q += 128) {
            const int row = nv + q / (kChDC * 8);
            const int rem = q % (kChDC * 8);
            const int ch = rem >> 3, piece = rem & 7;
            *reinterpret_cast<uint4*>(stage + ch * kChunk + row * 128 + piece * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_cta();
        }
        tc_fence_before();
        mbar_arrive(bar_addr(sbase, kBarPvGo));
        if (c.last()) {
          if (!warp_wait(bar_addr(sbase, kBarODone + sb), (k >> 1) & 1, abort)) break;
          tc_fence_after();
          const long long slot = cluster_id_x() + c.b;
          float4* dst = reinterpret_cast<float4*>(a.part_o + (slot * kM + r) * kDC);
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t v[64];
            tmem_ld64(tmem + lane_off + cc * 64, v);
            tmem_wait_ld();
            if (r < a.H) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                dst[cc * 16 + j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                               __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            }
          }
          tc_fence_before();
        }
      }
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && *abort) record_error(MLA_ERR_DEVICE_TIMEOUT, kSiteDecodeWait);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // no remote access into a CTA that has exited
}

// Merge the partials of each sequence: M = max m_s, L = sum l_s 2^(m_s - M),
// o = sum 2^(m_s - M) O_s / L, lse = (M + log2 L) ln 2.  One block per (head, b).
template <typename TOut>
__global__ void __launch_bounds__(128) combine_kernel(const Args a, TOut* __restrict__ o_lat,
                                                      float* __restrict__ lse) {
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const long long T = a.hdr[0], P = a.hdr[1];
  const long long cb = a.cum[b], ce = a.cum[b + 1];
  const int c0 = tid * 4;
  TOut* out = o_lat + (static_cast<long long>(b) * a.H + h) * kDC + c0;
  if (ce <= cb || P <= 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) st_elem(out + i, 0.f);
    if (lse != nullptr && tid == 0) lse[static_cast<long long>(b) * a.H + h] = -INFINITY;
    return;
  }
  // run p covers blocks [p T / P, (p + 1) T / P); run of block g = ceil((g + 1) P / T) - 1
  const long long p_first = ((cb + 1) * P + T - 1) / T - 1;
  const long long p_last = (ce * P + T - 1) / T - 1;
  float M = -INFINITY;
  for (long long p = p_first; p <= p_last; ++p) M = fmaxf(M, a.part_m[(p + b) * kM + h]);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long p = p_first; p <= p_last; ++p) {
    const long long slot = p + b;
    const float w = exp2f(a.part_m[slot * kM + h] - M);
    L += w * a.part_l[slot * kM + h];
    const float4 v = *reinterpret_cast<const float4*>(a.part_o + (slot * kM + h) * kDC + c0);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float inv = 1.f / L;
  st_elem(out + 0, acc.x * inv);
  st_elem(out + 1, acc.y * inv);
  st_elem(out + 2, acc.z * inv);
  st_elem(out + 3, acc.w * inv);
  if (lse != nullptr && tid == 0) lse[static_cast<long long>(b) * a.H + h] = (M + log2f(L)) * 0.69314718055994531f;
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

struct WsLayout {
  size_t hdr, cum, m, l, o, total;
};

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static WsLayout ws_layout(int B) {
  WsLayout w;
  const size_t slots = static_cast<size_t>(kMaxPairs) + static_cast<size_t>(B);
  w.hdr = 0;
  w.cum = 256;
  w.m = w.cum + align256(sizeof(int32_t) * (B + 1));
  w.l = w.m + align256(sizeof(float) * slots * kM);
  w.o = w.l + align256(sizeof(float) * slots * kM);
  w.total = w.o + sizeof(float) * slots * kM * kDC;
  return w;
}

static int pairs_for_device() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
      cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kMaxPairs, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_split_kernel, &cfg) != cudaSuccess || n <= 0) return -1;
  cached[dev] = n < kMaxPairs ? n : kMaxPairs;
  return cached[dev];
}

}  // namespace dtc

size_t decode_tc_workspace_size(int32_t B) { return dtc::ws_layout(B).total; }

mla_status launch_decode_tc(const void* q_cat, const mla_cache& c, const int32_t* seq_lens, int32_t H,
                            float scale, void* ws, size_t ws_bytes, void* o_lat, float* lse, cudaStream_t s) {
  using namespace dtc;
  const WsLayout w = ws_layout(c.B);
  if (ws == nullptr || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MLA_ERR_WORKSPACE;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return MLA_ERR_CUDA;
  const int npairs = pairs_for_device();
  if (npairs <= 0) return MLA_ERR_CUDA;

  const int R = c.d_c + c.d_r;
  CUtensorMap map;
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(c.N_max),
                              static_cast<cuuint64_t>(c.B)};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(c.row_stride) * 2,
                                 static_cast<cuuint64_t>(c.row_stride) * 2 * static_cast<cuuint64_t>(c.N_max)};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBN), 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c.data, gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLA_ERR_INVALID_ARG;

  uint8_t* wsb = static_cast<uint8_t*>(ws);
  Args a;
  a.q_cat = static_cast<const __nv_bfloat16*>(q_cat);
  a.seq_lens = seq_lens;
  a.B = c.B;
  a.H = H;
  a.N_max = c.N_max;
  a.R = R;
  a.nch = R / 64;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.hdr = reinterpret_cast<int32_t*>(wsb + w.hdr);
  a.cum = reinterpret_cast<int32_t*>(wsb + w.cum);
  a.part_m = reinterpret_cast<float*>(wsb + w.m);
  a.part_l = reinterpret_cast<float*>(wsb + w.l);
  a.part_o = reinterpret_cast<float*>(wsb + w.o);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * npairs, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_split_kernel, map, a);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  dim3 grid(H, c.B);
  combine_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a, static_cast<__nv_bfloat16*>(o_lat), lse);
  return cuda_status(cudaGetLastError());
}

}  // namespace mla

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
//        of S = Q C^T, 288 columns), computes S for 64-token blocks into three
//        64-column accumulators, runs the online softmax (one thread per head
//        row, no cross-thread reduction; two warpgroups on alternate blocks), and
//        writes the bf16 probabilities P, with each row's reference maximum and
//        the row sum of the rounded tile, straight into CTA 1's shared memory
//        with st.async, which completes bytes on CTA 1's barrier (no
//        cluster-scope fences on the producer side).
//      - CTA 1 (output CTA) accumulates O += P C[:, 0:512] with two N = 256
//        MMAs per 16-token step into its full 512-column tensor memory, and
//        rescales O in place on the rare blocks where the running maximum of a
//        row grew by more than 2^8.
//    The two contractions (576 and 512 wide) are split across the two SMs with
//    no redundant work.
//  * Cache rows stream in through TMA (128-byte swizzled 64x64 chunks; a 3-slot
//    ring in the score CTA, whose loads go to HBM, and a 2-slot ring in the output
//    CTA, whose loads of the same rows hit L2).  The same swizzled chunk is the
//    K-major B operand of S = Q C^T and the MN-major B operand of O = P C.  The
//    score CTA's ring also
//    carries each problem's query (two slots of 64 rows) on its way to tensor
//    memory, so a new problem costs two ring loads instead of per-thread reads.
//  * A "problem" is one query row group (all heads of one query) against a prefix
//    of one cached sequence: in decode, sequence b's query against its N_b rows; in
//    causal prefill, query i of sequence b against rows [0, start_b + i] (the rows
//    of the prompt itself, already appended).  The blocks of all problems form one
//    token stream that is cut into runs of equal cost (blocks plus a fixed cost per
//    problem), one run per cluster, so every SM pair gets the same work whatever
//    the mix of lengths.  A problem that lies inside one run is normalised and
//    written out directly; one cut by run boundaries leaves an unnormalised
//    partial (m, l, O) per piece, and a combine kernel merges the pieces.
#include <atomic>
#include <cmath>

#include "mla_internal.cuh"
#include "mla_ptx.cuh"

// Timing hooks: empty in the library; an instrumented build may define them to
// record (block, event) timestamps.
#ifndef MLA_TRACE_POINT
#define MLA_TRACE_POINT(block, event) \
  do {                                 \
  } while (0)
#endif

namespace mla {
namespace dtc {

constexpr int kBN = 64;                     // tokens per block
constexpr int kDC = 512;                    // latent width
constexpr int kChDC = kDC / 64;             // 8 chunks of 64 columns cover the latent
constexpr int kChunksPerRow = kDC / 32;     // 32-column groups of a piece row, each with its own fp16 scale
constexpr int kChunk = kBN * 128;           // bytes of one [64 tok x 64 col] bf16 chunk
constexpr int kM = 128;                     // head rows per MMA
constexpr int kMaxPairs = 80;               // upper bound on clusters per launch (148 SMs -> 74)
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P stays <= 256
// Fixed cost of a problem (query in, output out) in 64-row blocks, for the run
// planner.  With more problems than runs they follow each other closely and each
// one's output write stalls the pipeline; with fewer, a run holds at most a couple
// of problems and hides part of it behind the blocks already in flight.
constexpr int kSwitchCostMany = 4;
constexpr int kSwitchCostFew = 3;
constexpr int kThreads = 384;               // 12 warps: see the role map in the kernel

constexpr int kStages = 3;                  // score CTA TMA ring depth (HBM stream)
constexpr int kStagesO = 2;                 // output CTA ring depth (its loads hit L2)
constexpr int kPBufs = 4;                   // P tiles in flight between the CTAs
constexpr int kStageDC = kChDC * kChunk;    // 64 KB of latent chunks per stage
constexpr int kSBufs = 3;                   // score accumulators in tensor memory
constexpr int kPBytes = kM * 128;           // one bf16 P tile (128 heads x 64 tokens)
constexpr int kRefBytes = kM * 4;           // one fp32 value per head row
constexpr int kMsgBytes = kM * 8;           // per-row (reference, row sum of the bf16 tile) sent with a tile
constexpr uint32_t kPTxBytes = kPBytes + kMsgBytes;

// Shared-memory map (offsets from a 1024-aligned base).  Identical in both CTAs so
// that a local offset names the same object in the peer.
constexpr int kOffStage = 0;                           // kStages (score) / kStagesO (output) x 64 KB
constexpr int kOffRope = kStages * kStageDC;           // score CTA: kStages x 8 KB RoPE chunks
constexpr int kOffX = kOffRope + kStages * kChunk;     // score CTA: reference exchange between groups
constexpr int kOffP = kStagesO * kStageDC;             // output CTA: kPBufs P tiles
constexpr int kOffRef = kOffP + kPBufs * kPBytes;      // output CTA: kPBufs x 128 (reference, row sum) pairs
constexpr int kOffEpi = kOffRef + kPBufs * kMsgBytes;  // output CTA: per-row (m, l) for the epilogue helpers
constexpr int kStgBytes = kM * 64;                     // output CTA: one [128 rows][32 columns] bf16 output tile
constexpr int kOffStg = kOffEpi + 2 * kRefBytes;       // output CTA: two staging tiles (one per epilogue group)
constexpr int kOffBar = (kOffX + kRefBytes > kOffEpi + 2 * kRefBytes) ? kOffX + kRefBytes : kOffEpi + 2 * kRefBytes;
static_assert(kOffStg + 2 * kStgBytes <= kOffBar && kOffStg % 16 == 0, "output staging tiles");
static_assert(kOffP % 1024 == 0, "P tiles must sit on 1024-byte boundaries");
enum : int {
  kBarFull = 0,                       // [kStages] stage landed
  kBarEmpty = kBarFull + kStages,     // [kStages] stage consumed by this CTA's MMAs
  kBarSFull = kBarEmpty + kStages,    // [kSBufs] score: S buffer written
  kBarSEmpty = kBarSFull + kSBufs,    // [kSBufs] score: S buffer read
  kBarQReady = kBarSEmpty + kSBufs,   // score: query in tensor memory
  kBarRefReady = kBarQReady + 1,      // [2] score: reference of a block published (per softmax group)
  kBarPFree = kBarRefReady + 2,       // [kPBufs] score: output CTA released a P tile
  kBarPFull = kBarPFree + kPBufs,     // [kPBufs] output: P tile + references landed (tx bytes)
  kBarPvGo = kBarPFull + kPBufs,      // [kPBufs] output: block may be multiplied
  kBarODone = kBarPvGo + kPBufs,      // [kPBufs] output: PV of a block completed
  kBarDrain = kBarODone + kPBufs,     // MMA drain at teardown
  kBarEpiGo = kBarDrain + 1,          // output: (m, l) of a finished problem published to the helper warps
  kBarEpiDone = kBarEpiGo + 1,        // output: the helpers' half of the output is out of tensor memory
  kNumBars = kBarEpiDone + 1,
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 128;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// tensor-memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0;     // score CTA: query, R/2 columns (bf16 pairs)
constexpr uint32_t kColS = 320;   // score CTA: kSBufs 64-column S buffers (columns 320..511)
// output CTA: O occupies columns [0, 512)

struct Misc {                     // at kOffMisc
  uint32_t tmem;
  int abort;
  long long lo, hi, cum0;
  int b0, len0;
  int active;  // this cluster has a run
};
static_assert(sizeof(Misc) <= 128, "misc");

__device__ __forceinline__ int clamp_len(int n, int n_max) { return n < 0 ? 0 : (n > n_max ? n_max : n); }

// The problems of a launch and the rows each one reads.
struct Problems {
  const int32_t* seq_lens;  // decode: [B] rows of sequence b (one problem per sequence)
  const int32_t* q_start;   // prefill: [B] position of sequence b's first query; nullptr in decode
  int S;                    // queries per sequence (1 in decode)
  int causal;               // prefill: query i reads start + i + 1 rows (else start + S)
  int n_max;
  __device__ int raw_len(int pr) const {
    if (q_start == nullptr) return seq_lens[pr];
    const int b = pr / S, i = pr - b * S;
    return q_start[b] + (causal ? i + 1 : S);
  }
  __device__ int len(int pr) const { return clamp_len(raw_len(pr), n_max); }
  __device__ int seq(int pr) const { return q_start == nullptr ? pr : pr / S; }
};

struct Args {
  const __nv_bfloat16* q_cat;  // [NP][H][R]
  Problems pb;
  int NP, H, N_max, R, nch;    // NP problems; nch: 64-column chunks per row (R / 64)
  float scale_log2;            // scale * log2(e)
  int switch_cost;             // fixed cost of a problem for the run planner, in blocks
  int32_t* hdr;                // workspace: [0] total blocks, [1] runs used, [2] problems with no rows
  int32_t* cum;                // workspace: [NP + 1] first block of each problem
  int32_t* bnd;                // workspace: [kMaxPairs][4] per run: problem holding its first block, that
                               //   problem's first block and end, the run's first block
  float* part_m;               // [2 kMaxPairs][128] running max (log2 units)
  float* part_l;               // [2 kMaxPairs][128] running sum
  float* part_s;               // [2 kMaxPairs][16][128] max |O| over each 32 latent columns of a row
  __half* part_o;              // [2 kMaxPairs][256][128][2] O / part_s in fp16: column pairs, head, pair
  __nv_bfloat16* o_lat;        // [NP][H][512]
  float* lse;                  // [NP][H] natural-log LSE, or nullptr
  int fault;                   // injected fault for tests of the failure detection: 1 = the score CTA
                               //   issues no loads, so the waits on them run out (0 in normal use)
  const int32_t* block_table;  // paged cache: [seqs][max_blocks] page of each 64-row block; nullptr when
                               //   the cache is contiguous
  int max_blocks, num_pages;
  const int32_t* row_begin;    // decode over row ranges (the kRanged kernel): [B] first row of sequence b;
                               //   pb.seq_lens then holds the end (exclusive) of its rows
};

// Rows of problem pr in a decode over row ranges: [row0, row0 + len) with
// 0 <= row0 <= row0 + len <= N_max (clamped; out-of-range ranges are recorded by the
// planner).  Without ranges (kRanged = false) the problem's own length from row 0.
template <bool kRanged>
__device__ __forceinline__ int span_row0(const Args& a, int pr) {
  if constexpr (kRanged) return clamp_len(a.row_begin[pr], a.N_max);
  else return 0;
}
template <bool kRanged>
__device__ __forceinline__ int span_len(const Args& a, int pr) {
  if constexpr (kRanged) {
    const int r0 = clamp_len(a.row_begin[pr], a.N_max), e = clamp_len(a.pb.seq_lens[pr], a.N_max);
    return e > r0 ? e - r0 : 0;
  } else {
    return a.pb.len(pr);
  }
}
template <bool kRanged>
__device__ __forceinline__ bool span_bad(const Args& a, int pr) {
  if constexpr (kRanged) {
    const int r0 = a.row_begin[pr], e = a.pb.seq_lens[pr];
    return r0 < 0 || e < r0 || e > a.N_max;
  } else {
    const int n = a.pb.raw_len(pr);
    return n < 0 || n > a.N_max;
  }
}

// Walks the 64-token blocks [lo, hi) of the flattened token stream.
template <bool kRanged>
struct Cursor {
  Problems pbs;
  const int32_t* rbeg;  // kRanged: the first row of each problem
  long long g, lo, hi, cum;
  int b, len, nblk, cs, r0;  // b: problem, cs: its cache sequence, r0: its first row (kRanged)
  __device__ void start(const Misc& m, const Args& a) {
    pbs = a.pb;
    rbeg = a.row_begin;
    g = lo = m.lo;
    hi = m.hi;
    cum = m.cum0;
    b = m.b0;
    len = m.len0;
    nblk = (len + kBN - 1) / kBN;
    cs = pbs.seq(b);
    if constexpr (kRanged) r0 = clamp_len(rbeg[b], pbs.n_max);
  }
  __device__ bool ok() const { return g < hi; }
  __device__ void next() {
    ++g;
    while (g < hi && g >= cum + nblk) {
      cum += nblk;
      ++b;
      if constexpr (kRanged) {
        r0 = clamp_len(rbeg[b], pbs.n_max);
        const int e = clamp_len(pbs.seq_lens[b], pbs.n_max);
        len = e > r0 ? e - r0 : 0;
      } else {
        len = pbs.len(b);
      }
      nblk = (len + kBN - 1) / kBN;
      cs = pbs.seq(b);
    }
  }
  __device__ int t0() const { return static_cast<int>(g - cum) * kBN; }
  __device__ int rows() const { return min(kBN, len - t0()); }
  __device__ bool first() const { return g == lo || g == cum; }
  __device__ bool last() const { return g == hi - 1 || g == cum + nblk - 1; }
  __device__ bool whole() const { return cum >= lo && cum + nblk <= hi; }  // problem inside this run
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) { return base + kOffBar + 8 * i; }

// TMA coordinates (row, plane) of the 64-row block of c: row t0 of sequence plane cs
// in a contiguous cache; row 0 of the block's page in a paged pool (an index
// outside the pool is recorded and page 0 read instead, so the load stays in
// bounds and its barrier completes).
template <bool kRanged>
__device__ __forceinline__ void block_coords(const Args& a, const Cursor<kRanged>& c, int* row, int* plane) {
  if (a.block_table == nullptr) {
    if constexpr (kRanged) *row = c.r0 + c.t0();
    else *row = c.t0();
    *plane = c.cs;
    return;
  }
  int pg = a.block_table[static_cast<long long>(c.cs) * a.max_blocks + c.t0() / kBN];
  if (pg < 0 || pg >= a.num_pages) {
    record_error(MLA_ERR_DEVICE_INDEX, kSitePageIndex);
    pg = 0;
  }
  *row = 0;
  *plane = pg;
}

// Shared address of 64-column chunk ch (8 KB: 64 rows x 128 bytes, 128-byte swizzle)
// of ring slot st: chunks 0-7 in the slot's latent area, chunk 8 in its RoPE area.
__device__ __forceinline__ uint32_t ring_chunk(uint32_t base, int st, int ch) {
  return ch < kChDC ? base + kOffStage + st * kStageDC + ch * kChunk : base + kOffRope + st * kChunk;
}

// Plan the run of this cluster.  Every problem costs its blocks plus a fixed
// sw = a.switch_cost (its query staging and output write, in block units); the total
// cost C is cut into P equal runs, P = min(clusters, T, C / (sw + 1)) so that every
// run holds at least one block.  A run starts at the first block whose cost position
// (problem start + sw + block offset) reaches p C / P.  One warp.
// The writer of the table (one warp per launch) also checks every length, fills the
// block prefix table and counts the problems with no rows.  Reads only the problem
// lengths; writes the workspace only with write_table.
template <bool kRanged>
__device__ void plan_run(const Args& a, Misc* misc, bool write_table) {
  const int lane = threadIdx.x & 31;
  const int sw = a.switch_cost;
  long long T = 0;
  int empties = 0;
  for (int base = 0; base < a.NP; base += 32) {
    const int b = base + lane;
    int nb = 0;
    if (b < a.NP) {
      if (write_table && span_bad<kRanged>(a, b)) record_error(MLA_ERR_DEVICE_INDEX, kSiteDecodeLength);
      nb = (span_len<kRanged>(a, b) + kBN - 1) / kBN;
      empties += nb == 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, off);
    T += nb;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) empties += __shfl_xor_sync(0xffffffffu, empties, off);
  const long long C = T + static_cast<long long>(sw) * (a.NP - empties);
  const long long nclus = nclusters_x();
  long long P = T < nclus ? T : nclus;
  if (P > C / (sw + 1)) P = C / (sw + 1);
  if (T > 0 && P < 1) P = 1;
  const long long cid = cluster_id_x();
  const bool active = cid < P;
  const long long x_lo = active ? cid * C / P : 0, x_hi = active ? (cid + 1) * C / P : 0;
  long long lo = 0, hi = active ? T : 0, cum0 = 0;
  int b0 = 0, len0 = 0;
  if (active || write_table) {
    long long run = 0, crun = 0;  // blocks and cost of the problems before this group of 32
    bool found_lo = !active, found_hi = !active || x_hi >= C;
    for (int base = 0; base < a.NP; base += 32) {
      const int b = base + lane;
      const int n = b < a.NP ? span_len<kRanged>(a, b) : 0;
      const int nb = (n + kBN - 1) / kBN;
      const int cost = nb > 0 ? nb + sw : 0;
      int incl = nb, cincl = cost;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        const int cv = __shfl_up_sync(0xffffffffu, cincl, off);
        if (lane >= off) {
          incl += v;
          cincl += cv;
        }
      }
      const long long excl = run + incl - nb, cexcl = crun + cincl - cost;
      if (write_table && b < a.NP) a.cum[b] = static_cast<int32_t>(excl);
      const unsigned mlo = __ballot_sync(0xffffffffu, !found_lo && cost > 0 && cexcl <= x_lo && x_lo < cexcl + cost);
      if (mlo != 0u) {
        const int src = __ffs(mlo) - 1;
        b0 = base + src;
        cum0 = __shfl_sync(0xffffffffu, excl, src);
        len0 = __shfl_sync(0xffffffffu, n, src);
        const long long into = x_lo - __shfl_sync(0xffffffffu, cexcl, src) - sw;
        lo = cum0 + (into > 0 ? into : 0);
        found_lo = true;
      }
      const unsigned mhi = __ballot_sync(0xffffffffu, !found_hi && cost > 0 && cexcl <= x_hi && x_hi < cexcl + cost);
      if (mhi != 0u) {
        const int src = __ffs(mhi) - 1;
        const long long into = x_hi - __shfl_sync(0xffffffffu, cexcl, src) - sw;
        hi = __shfl_sync(0xffffffffu, excl, src) + (into > 0 ? into : 0);
        found_hi = true;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      crun += __shfl_sync(0xffffffffu, cincl, 31);
      if (found_lo && found_hi && !write_table) break;
    }
  }
  if (lane == 0) {
    misc->lo = lo;
    misc->hi = hi;
    misc->b0 = b0;
    misc->cum0 = cum0;
    misc->len0 = len0;
    misc->active = active ? 1 : 0;
    if (write_table) {
      a.cum[a.NP] = static_cast<int32_t>(T);
      a.hdr[0] = static_cast<int32_t>(T);
      a.hdr[1] = static_cast<int32_t>(P);
      a.hdr[2] = empties;
    }
  }
}

// Slot of the piece of problem c.b that ends this run: 2 p for the problem that holds
// the run's first block (b0), 2 p + 1 for the one cut at the run's end.
template <class C>
__device__ __forceinline__ long long piece_slot(const C& c, int b0) {
  return 2 * static_cast<long long>(cluster_id_x()) + (c.b == b0 ? 0 : 1);
}

// Write latent columns [col0, col0 + 256) of row r of the finished problem c.b from
// tensor memory: o = O / l in bf16 if the whole problem ran here, else the
// unnormalised fp32 piece ([column][head] in its slot, a warp storing 128
// contiguous bytes per column).
template <class C>
__device__ __forceinline__ void store_output(const Args& a, const CUtensorMap* omap, const C& c, int b0,
                                             uint32_t trow, int r, float l, int col0, uint8_t* smem_gen,
                                             uint32_t sbase) {
  if (c.whole()) {
    // o = O / l in bf16, 32 columns at a time: each thread packs its row into a
    // [H rows][32 columns] tile in shared memory (64-byte rows) and one thread writes
    // the tile out with a TMA store (rows past H are outside the box).  The next
    // chunk's tensor-memory load is in flight while a chunk is handed over.
    const float inv = 1.f / l;
    const int grp = col0 != 0 ? 1 : 0;
    uint8_t* stg = smem_gen + kOffStg + grp * kStgBytes;
    const uint32_t stg_s = sbase + kOffStg + grp * kStgBytes;
    const uint32_t bar_id = 1u + grp;
    uint32_t v[32];
    tmem_ld32(trow + col0, v);
    for (int cc = 0; cc < 8; ++cc) {
      tmem_wait_ld();
      uint4 w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w[q].x = pack_bf16x2(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv);
        w[q].y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv);
        w[q].z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv);
        w[q].w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv);
      }
      if (cc + 1 < 8) tmem_ld32(trow + col0 + (cc + 1) * 32, v);
      if (r == 0) bulk_wait_read0();  // the previous store has read the tile
      named_sync(bar_id, 128);
      if (r < a.H) {
        uint4* srow = reinterpret_cast<uint4*>(stg + r * 64);
#pragma unroll
        for (int q = 0; q < 4; ++q) srow[q] = w[q];
      }
      fence_proxy_async_cta();
      named_sync(bar_id, 128);
      if (r == 0) {
        tma_store_2d(omap, stg_s, col0 + cc * 32, c.b * a.H);
        bulk_commit();
      }
    }
  } else {
    // a piece: every 32 columns of the row scaled by their largest magnitude and stored
    // in fp16 (the pieces are merged into bf16 outputs; |O / max| <= 1 keeps fp16 in
    // range and its 11-bit significand well below the output's rounding).  One pass
    // over tensor memory, the next chunk's load in flight while a chunk is stored.
    // Stores go by column pairs, [pair][head][2], so a warp writes 128 contiguous
    // bytes per pair.
    const long long slot = piece_slot(c, b0);
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.part_o) + slot * (kDC / 2 * kM) + (col0 / 2) * kM + r;
    float* sdst = a.part_s + (slot * kChunksPerRow + col0 / 32) * kM + r;
    uint32_t v[32];
    tmem_ld32(trow + col0, v);
    for (int cc = 0; cc < 8; ++cc) {
      tmem_wait_ld();
      float mx = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fabsf(__uint_as_float(v[j])));
      const float inv = mx > 0.f ? 1.f / mx : 0.f;
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const __half2 hv = __floats2half2_rn(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
        w[j / 2] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      if (cc + 1 < 8) tmem_ld32(trow + col0 + (cc + 1) * 32, v);
      if (r < a.H) {
#pragma unroll
        for (int j = 0; j < 16; ++j) dst[(cc * 16 + j) * kM] = w[j];
        sdst[cc * kM] = mx;
      }
    }
  }
}

// Role map (12 warps).  Score CTA: warp 0 TMA, warp 1 S MMA, warp 2 run planning,
// warps 4-7 softmax group A (even blocks), warps 8-11 softmax group B (odd blocks).
// Output CTA: warp 0 TMA, warp 1 PV MMA, warps 4-7 correction + epilogue (latent
// columns 0..255), warps 8-11 epilogue (columns 256..511).
template <bool kRanged>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const __grid_constant__ CUtensorMap map,
                                                                   const __grid_constant__ CUtensorMap qmap,
                                                                   const __grid_constant__ CUtensorMap omap,
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
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(bar_addr(sbase, kBarSFull + i), 1);
      mbar_init(bar_addr(sbase, kBarSEmpty + i), 128);
    }
    for (int i = 0; i < 2; ++i) mbar_init(bar_addr(sbase, kBarRefReady + i), 128);
    // Per-P-tile barriers: the output CTA's correction warps can run up to kPBufs-1
    // blocks ahead of its MMA warp, so every per-block handshake there has one
    // barrier per tile and never more than one phase outstanding.
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(bar_addr(sbase, kBarPFree + i), 1);
      mbar_init(bar_addr(sbase, kBarPFull + i), 1);
      mbar_init(bar_addr(sbase, kBarPvGo + i), 128);
      mbar_init(bar_addr(sbase, kBarODone + i), 1);
    }
    mbar_init(bar_addr(sbase, kBarQReady), 128);
    mbar_init(bar_addr(sbase, kBarDrain), 1);
    mbar_init(bar_addr(sbase, kBarEpiGo), 128);
    mbar_init(bar_addr(sbase, kBarEpiDone), 128);
    misc->abort = 0;
    if (!score_cta) {  // the first kPBufs P tiles are expected before any is sent
      for (int i = 0; i < kPBufs; ++i) mbar_arrive_expect_tx(bar_addr(sbase, kBarPFull + i), kPTxBytes);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map);
    tma_prefetch_desc(&qmap);
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffMisc + offsetof(Misc, tmem), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) MLA_TRACE_POINT(63, score_cta ? 0 : 2);
  // the run plan reads only the problem lengths (seq_lens / q_start, which no kernel
  // of this library writes), so it overlaps the previous kernel's tail
  if (warp == 2) plan_run<kRanged>(a, misc, false);
  griddep_launch();
  // the workspace, o_lat and q_cat may still be in use by the previous kernels
  griddep_wait();
  if (score_cta && warp == 3 && cluster_id_x() == 0) {
    Misc tmp;
    plan_run<kRanged>(a, &tmp, true);  // the block table and run count for the combine
  }
  if (score_cta && threadIdx.x == 64 && misc->active) {  // this run's record for the combine
    int32_t* e = a.bnd + 4 * cluster_id_x();
    e[0] = misc->b0;
    e[1] = static_cast<int32_t>(misc->cum0);
    e[2] = static_cast<int32_t>(misc->cum0 + (misc->len0 + kBN - 1) / kBN);
    e[3] = static_cast<int32_t>(misc->lo);
  }
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // peer barriers initialised before any remote arrive
  if (threadIdx.x == 0) MLA_TRACE_POINT(63, score_cta ? 1 : 3);

  const uint32_t tmem = misc->tmem;
  const int nch = a.nch;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint32_t leader = elect_one();
    const int nload = score_cta ? nch : kChDC;
    const int nst = score_cta ? kStages : kStagesO;
    Cursor<kRanged> c;
    c.start(*misc, a);
    int li = 0;  // ring load index: the score CTA's ring also carries each problem's query
    // 64 cache rows of block c into ring slot st
    auto load_block = [&](const Cursor<kRanged>& cb, int st) {
      int row, plane;
      block_coords(a, cb, &row, &plane);
      mbar_arrive_expect_tx_if(leader, bar_addr(sbase, kBarFull + st), nload * kChunk);
      for (int ch = 0; ch < nload; ++ch)
        tma_load_3d_if(leader, ring_chunk(sbase, st, ch), &map, bar_addr(sbase, kBarFull + st), ch * 64, row, plane);
    };
    bool head_loaded = false;  // the run's first block went out ahead of its query
    const bool skip_loads = score_cta && a.fault == 1;
    for (int k = 0; c.ok() && !skip_loads; c.next(), ++k) {
      if (score_cta && c.first()) {
        if (k == 0) {
          // run start: every slot is free, so the first block (HBM latency) is issued
          // before the query (likely in L2) that precedes it in ring order
          load_block(c, 2 % kStages);
          head_loaded = true;
        }
        // the problem's query, rows 0..63 and 64..127, as 64 x 64 boxes into two ring
        // slots (latent area: 8 boxes, RoPE area: the ninth); the softmax threads move
        // it into tensor memory and the MMA warp releases the slots
        for (int part = 0; part < 2; ++part, ++li) {
          const int st = li % kStages;
          if (!warp_wait(bar_addr(sbase, kBarEmpty + st), ((li / kStages) & 1) ^ 1, abort)) break;
          mbar_arrive_expect_tx_if(leader, bar_addr(sbase, kBarFull + st), nch * kChunk);
          for (int ch = 0; ch < nch; ++ch)
            tma_load_2d_if(leader, ring_chunk(sbase, st, ch), &qmap, bar_addr(sbase, kBarFull + st), ch * 64,
                           c.b * a.H + part * kBN);
        }
      } else if (score_cta && c.g == c.cum + 1 && c.b + 1 < a.NP) {
        // the problem's second block: the next problem's query moves into L2 meanwhile
        prefetch_l2_bulk_if(leader, a.q_cat + static_cast<long long>(c.b + 1) * a.H * a.R,
                            static_cast<uint32_t>(a.H * a.R * 2));
      }
      const int st = (score_cta ? li : k) % nst;
      const int ph = (score_cta ? li : k) / nst;
      ++li;
      if (head_loaded) {
        head_loaded = false;
        continue;
      }
      if (!warp_wait(bar_addr(sbase, kBarEmpty + st), (ph & 1) ^ 1, abort)) break;
      MLA_TRACE_POINT(k, score_cta ? 8 : 7);
      load_block(c, st);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = elect_one();
    Cursor<kRanged> c;
    c.start(*misc, a);
    if (score_cta) {
      // S = Q C^T: M = 128 heads, N = 64 tokens, A (the query) from tensor memory
      constexpr uint32_t idesc = idesc_bf16(kM, kBN, false, false);
      int seg = 0, li = 0;
      for (int k = 0; c.ok(); c.next(), ++k) {
        if (c.first()) {
          // the query left its two ring slots for tensor memory: release them
          if (!warp_wait(bar_addr(sbase, kBarQReady), seg & 1, abort)) break;
          ++seg;
          if (leader) {
            mbar_arrive(bar_addr(sbase, kBarEmpty + li % kStages));
            mbar_arrive(bar_addr(sbase, kBarEmpty + (li + 1) % kStages));
          }
          li += 2;
        }
        const int st = li % kStages, sb = k % kSBufs;
        if (!warp_wait(bar_addr(sbase, kBarFull + st), (li / kStages) & 1, abort)) break;
        MLA_TRACE_POINT(k, 13);
        ++li;
        if (!warp_wait(bar_addr(sbase, kBarSEmpty + sb), ((k / kSBufs) & 1) ^ 1, abort)) break;
        MLA_TRACE_POINT(k, 0);
        tc_fence_after();
        const uint32_t d = tmem + kColS + sb * kBN;
#pragma unroll
        for (int ch = 0; ch < kChDC; ++ch) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_if(leader, d, tmem + kColQ + ch * 32 + kk * 8, sdesc_sw128(ring_chunk(sbase, st, ch) + kk * 32, 16, 1024),
                      idesc, (ch | kk) != 0);
        }
        if (nch > kChDC) {  // the RoPE chunk
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_if(leader, d, tmem + kColQ + kChDC * 32 + kk * 8,
                      sdesc_sw128(ring_chunk(sbase, st, kChDC) + kk * 32, 16, 1024), idesc, 1u);
        }
        tc_commit_if(leader, bar_addr(sbase, kBarEmpty + st));
        tc_commit_if(leader, bar_addr(sbase, kBarSFull + sb));
        MLA_TRACE_POINT(k, 15);
      }
    } else {
      // O += P C: M = 128 heads, N = 256 latent columns per MMA, both operands in smem
      constexpr uint32_t idesc = idesc_bf16(kM, 256, false, true);
      for (int k = 0; c.ok(); c.next(), ++k) {
        const int st = k % kStagesO, pb = k % kPBufs;
        if (!warp_wait(bar_addr(sbase, kBarPvGo + pb), (k / kPBufs) & 1, abort)) break;
        MLA_TRACE_POINT(k, 5);
        if (!warp_wait(bar_addr(sbase, kBarFull + st), (k / kStagesO) & 1, abort)) break;
        MLA_TRACE_POINT(k, 6);
        tc_fence_after();
        const uint32_t pa = sbase + kOffP + pb * kPBytes;
        const uint32_t stage = sbase + kOffStage + st * kStageDC;
        const uint32_t acc0 = c.first() ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t adesc = sdesc_sw128(pa + kk * 32, 16, 1024);
#pragma unroll
          for (int half = 0; half < 2; ++half)
            mma_ss_if(leader, tmem + half * 256, adesc, sdesc_sw128(stage + half * 4 * kChunk + kk * 16 * 128, kChunk, 1024),
                      idesc, acc0 | (kk > 0 ? 1u : 0u));
        }
        MLA_TRACE_POINT(k, 13);
        tc_commit_if(leader, bar_addr(sbase, kBarEmpty + st));
        tc_commit_if(leader, bar_addr(sbase, kBarODone + pb));
        tc_commit_mc_if(leader, bar_addr(sbase, kBarPFree + pb), static_cast<uint16_t>(1u));  // to the score CTA
      }
    }
    // drain: every MMA this warp issued has completed before teardown
    tc_commit_if(leader, bar_addr(sbase, kBarDrain));
    warp_wait(bar_addr(sbase, kBarDrain), 0, abort);
  } else if (warp >= 4 && score_cta) {
    // ------------------------------------------------------------ softmax (two groups)
    // Group g handles blocks k with k % 2 == g.  Consecutive blocks only share the
    // per-row reference m: the group of block k reads block k-1's reference from
    // shared memory, raises it when the block's maximum exceeds it by more than
    // 2^8, publishes it for block k+1, then exponentiates and ships P while the
    // other group works on the next block.
    const int grp = (warp - 4) >> 2;
    const int r = (threadIdx.x - 128) & 127;                    // head row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(r & ~31) << 16;
    float* ref_x = reinterpret_cast<float*>(gbase + kOffX);    // reference exchange between the groups
    Cursor<kRanged> c;
    c.start(*misc, a);
    int k = 0, last_mine = -1, li = 0;  // li: the score ring's load index, as the producer counts it
    for (; c.ok(); c.next(), ++k) {
      const bool first = c.first();
      const int qli = li;  // a problem's query occupies ring loads qli, qli + 1
      li += first ? 3 : 1;
      if ((k & 1) != grp) continue;
      last_mine = k;
      if (first) {
        // the previous block's S product (other group, older query) must be finished
        if (k > 0 && !warp_wait(bar_addr(sbase, kBarSFull + (k - 1) % kSBufs), ((k - 1) / kSBufs) & 1, abort)) break;
        if (r == 0) MLA_TRACE_POINT(k, 9);
        if (!warp_wait(bar_addr(sbase, kBarFull + qli % kStages), (qli / kStages) & 1, abort)) break;
        if (!warp_wait(bar_addr(sbase, kBarFull + (qli + 1) % kStages), ((qli + 1) / kStages) & 1, abort)) break;
        // row r of the query from its slot (rows 0-63, then 64-127); 128-byte swizzle:
        // piece j of a row at row * 128 + ((j ^ row % 8) * 16), so a warp's reads hit
        // distinct banks
        const int qst = (qli + (r >> 6)) % kStages;
        for (int ch = 0; ch < nch; ++ch) {
          const uint8_t* qrow = gbase + (ring_chunk(sbase, qst, ch) - sbase) + (r & 63) * 128;
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(qrow + ((u ^ (r & 7)) << 4));
            v[4 * u] = x.x;
            v[4 * u + 1] = x.y;
            v[4 * u + 2] = x.z;
            v[4 * u + 3] = x.w;
          }
          tmem_st32(tmem + lane_off + kColQ + ch * 32, v);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_addr(sbase, kBarQReady));
        if (r == 0) MLA_TRACE_POINT(k, 10);
      }
      const int sbuf = k % kSBufs, pb = k % kPBufs;
      if (!warp_wait(bar_addr(sbase, kBarSFull + sbuf), (k / kSBufs) & 1, abort)) break;
      if (r == 0) MLA_TRACE_POINT(k, 1);
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld64(tmem + lane_off + kColS + sbuf * kBN, sr);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, kBarSEmpty + sbuf));

      const int nv = c.rows();
      if (nv < kBN) {
#pragma unroll
        for (int j = 0; j < kBN; ++j)
          if (j >= nv) sr[j] = __float_as_uint(-INFINITY);
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(sr[i]);
#pragma unroll
      for (int j = 8; j < kBN; ++j) mx[j & 7] = fmaxf(mx[j & 7], __uint_as_float(sr[j]));
      const float mloc = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * a.scale_log2;
      // reference of block k-1 (published by the other group)
      float m_ref;
      if (k > 0 && !warp_wait(bar_addr(sbase, kBarRefReady + (grp ^ 1)), ((k - 1) >> 1) & 1, abort)) break;
      if (c.first()) {
        m_ref = mloc;
      } else {
        m_ref = ref_x[r];
        if (mloc > m_ref + kRescaleThreshold) m_ref = mloc;
      }
      ref_x[r] = m_ref;  // for block k+1 (ordered by the arrive below)
      mbar_arrive(bar_addr(sbase, kBarRefReady + grp));

      uint32_t pk[32];
      const float neg = -m_ref;
#pragma unroll
      for (int j = 0; j < kBN; j += 2) {
        const float p0 = fast_exp2(fmaf(__uint_as_float(sr[j]), a.scale_log2, neg));
        const float p1 = fast_exp2(fmaf(__uint_as_float(sr[j + 1]), a.scale_log2, neg));
        pk[j >> 1] = pack_bf16x2(p0, p1);
      }
      // the row sum of the probabilities as rounded to bf16, i.e. of the values the
      // PV product multiplies (the output CTA normalises by exactly what it summed)
      float psum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 32; ++j)
        psum[j & 3] += __uint_as_float(pk[j] << 16) + __uint_as_float(pk[j] & 0xFFFF0000u);
      const float ps = (psum[0] + psum[1]) + (psum[2] + psum[3]);
      if (r == 0) MLA_TRACE_POINT(k, 14);
      if (!warp_wait(bar_addr(sbase, kBarPFree + pb), ((k / kPBufs) & 1) ^ 1, abort)) break;
      if (r == 0) MLA_TRACE_POINT(k, 2);
      // P row r into the output CTA's P tile (K-major, 128-byte swizzle) and the row's
      // reference; every store completes its bytes on the output CTA's P barrier
      const uint32_t pbar = bar_addr(sbase, kBarPFull + pb);
      const uint32_t prow = sbase + kOffP + pb * kPBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        st_async_v4(prow + ((cc ^ (r & 7)) << 4), pbar, 1u, pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      st_async_v2(sbase + kOffRef + pb * kMsgBytes + r * 8, pbar, 1u, __float_as_uint(m_ref), __float_as_uint(ps));
      if (r == 0) MLA_TRACE_POINT(k, 3);
    }
    // the output CTA has consumed this group's last tile (its release, an arrival
    // into this CTA, has landed) before this CTA exits
    if (last_mine >= 0)
      warp_wait(bar_addr(sbase, kBarPFree + last_mine % kPBufs), (last_mine / kPBufs) & 1, abort);
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ output CTA: correction + epilogue
    // Tracks the row maximum m (the references it receives) and the row sum l of the
    // bf16 P tiles it multiplies, rescales O in place when a row's reference rose,
    // and writes the unnormalised partial (m, l, O) at the end of each sequence run.
    const int r = threadIdx.x - 128;
    const uint32_t lane_off = static_cast<uint32_t>(r & ~31) << 16;
    Cursor<kRanged> c;
    c.start(*misc, a);
    float m = 0.f, l = 0.f;
    int k = 0, n_epi = 0;
    for (; c.ok(); c.next(), ++k) {
      const int pb = k % kPBufs, st = k % kStagesO;
      if (!warp_wait<true>(bar_addr(sbase, kBarPFull + pb), (k / kPBufs) & 1, abort)) break;
      if (r == 0) MLA_TRACE_POINT(k, 4);
      const float2 msg = reinterpret_cast<const float2*>(gbase + kOffRef + pb * kMsgBytes)[r];
      const float ref = msg.x, ps = msg.y;
      float alpha = 1.f;
      if (!c.first()) alpha = fast_exp2(m - ref);
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        const int kp = k - 1;  // PV of the previous block has to be complete
        if (!warp_wait(bar_addr(sbase, kBarODone + kp % kPBufs), (kp / kPBufs) & 1, abort)) break;
        tc_fence_after();
        for (int cc = 0; cc < 16; ++cc) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + cc * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(tmem + lane_off + cc * 32, v);
        }
        tmem_wait_st();
      }
      const int nv = c.rows();
      if (nv < kBN) {
        // rows past the end of the sequence must not carry NaN/Inf into P C.  Once PV
        // of block k-2 is done the stage can only hold block k (or be loading it).
        if (k >= 2 && !warp_wait(bar_addr(sbase, kBarODone + (k - 2) % kPBufs), ((k - 2) / kPBufs) & 1, abort)) break;
        if (!warp_wait(bar_addr(sbase, kBarFull + st), (k / kStagesO) & 1, abort)) break;
        uint8_t* stage = gbase + kOffStage + st * kStageDC;
        const int npieces = (kBN - nv) * kChDC * 8;  // 16-byte pieces
        for (int q = r; q < npieces; q += 128) {
          const int row = nv + q / (kChDC * 8);
          const int rem = q % (kChDC * 8);
          const int ch = rem >> 3, piece = rem & 7;
          *reinterpret_cast<uint4*>(stage + ch * kChunk + row * 128 + piece * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_cta();  // P arrived through st.async; zeroed rows through generic stores
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, kBarPvGo + pb));
      l = c.first() ? ps : l * alpha + ps;
      m = ref;
      // this buffer's next tile (block k + kPBufs) is sent only after PV of block k
      if (r == 0) mbar_arrive_expect_tx(bar_addr(sbase, kBarPFull + pb), kPTxBytes);
      if (c.last()) {
        if (!warp_wait(bar_addr(sbase, kBarODone + pb), (k / kPBufs) & 1, abort)) break;
        if (r == 0) MLA_TRACE_POINT(k, 11);
        // the row's (m, l) to the helper warps, which write latent columns 256..511
        float* epi = reinterpret_cast<float*>(gbase + kOffEpi);
        epi[r] = m;
        epi[kM + r] = l;
        mbar_arrive(bar_addr(sbase, kBarEpiGo));
        tc_fence_after();
        store_output(a, &omap, c, misc->b0, tmem + lane_off, r, l, 0, gbase, sbase);
        if (r < a.H) {
          if (c.whole()) {
            if (a.lse != nullptr) a.lse[static_cast<long long>(c.b) * a.H + r] = (m + log2f(l)) * 0.69314718055994531f;
          } else {
            const long long slot = piece_slot(c, misc->b0);
            a.part_m[slot * kM + r] = m;
            a.part_l[slot * kM + r] = l;
          }
        }
        tc_fence_before();
        // O is overwritten by the next problem's first PV only after both halves are out
        if (!warp_wait(bar_addr(sbase, kBarEpiDone), n_epi & 1, abort)) break;
        ++n_epi;
        if (r == 0) MLA_TRACE_POINT(k, 12);
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ output CTA: epilogue helpers
    // Warps 8-11 see the same TMEM lanes as warps 4-7 and write the upper half of the
    // latent columns of every finished problem.
    const int r = threadIdx.x - 256;
    const uint32_t lane_off = static_cast<uint32_t>(r & ~31) << 16;
    const float* epi = reinterpret_cast<const float*>(gbase + kOffEpi);
    Cursor<kRanged> c;
    c.start(*misc, a);
    int n_epi = 0;
    for (; c.ok(); c.next()) {
      if (!c.last()) continue;
      if (!warp_wait(bar_addr(sbase, kBarEpiGo), n_epi & 1, abort)) break;
      const float l = epi[kM + r];
      tc_fence_after();
      store_output(a, &omap, c, misc->b0, tmem + lane_off, r, l, kDC / 2, gbase, sbase);
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, kBarEpiDone));
      ++n_epi;
    }
  }

  if (!score_cta && (threadIdx.x == 128 || threadIdx.x == 256)) bulk_wait0();  // output tile stores complete
  __syncthreads();
  if (threadIdx.x == 0) MLA_TRACE_POINT(62, score_cta ? 4 : 5);
  if (threadIdx.x == 0 && *abort) record_error(MLA_ERR_DEVICE_TIMEOUT, kSiteDecodeWait);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // no remote access into a CTA that has exited
}

// Merge the pieces of every problem cut by run boundaries: M = max m_s,
// L = sum l_s 2^(m_s - M), o = sum 2^(m_s - M) O_s / L, lse = (M + log2 L) ln 2.
// Work item (x, p) is latent columns [32 x, 32 x + 32) of the problem that run
// boundary p cuts, if p is the first boundary inside it; items (x, 0) write the zero
// output of problems with no rows.  One block per item.  Thread t owns heads
// 2(t % 64), +1 and kCols columns from kCols (t / 64): a warp reads 256 contiguous
// bytes per column of a piece, and up to kPieces pieces are in flight at once (their
// maximum first, then one weighted sum).  The merged tile is staged in shared memory
// ([head][column], padded rows) and written out as 64-byte runs.  Two shapes of
// item, both within 64 registers a thread: the narrow one (256 threads of 8 columns, two
// pieces per round) fits four blocks on an SM, so a B = 32 launch's ~530 items run
// in one wave; the wide one (512 threads of 4 columns, three pieces per round: a
// problem spans two to four runs, so mostly one round) fits two, and is taken when
// the launch's items fit in one wave of it.
template <bool kWide>
struct CombineShape {
  static constexpr int kThreads = kWide ? 512 : 256;
  static constexpr int kPieces = kWide ? 3 : 2;
  static constexpr int kCols = kWide ? 4 : 8;
  static constexpr int kBlocksPerSm = kWide ? 2 : 4;
};
constexpr int kMergeThreads = 256;

// The grouped merge (combine_groups > 1): group g of the combine merges pieces g,
// g + G, ... of each cut problem into an fp32 partial (its running maximum and sum
// per head, its unnormalised sum per head and column); merge_groups_kernel merges
// the G partials.  cutp[y] is the problem the y-th cut is in (-1: none).
struct GroupArgs {
  int G;
  int32_t* cutp;  // [cuts]
  float* gm;      // [G][cuts][128]
  float* gl;      // [G][cuts][128]
  float* ga;      // [G][cuts][128][512]
  int cuts;
};

template <bool kGrouped, bool kWide>
__device__ __forceinline__ void combine_item(const Args& a, int cb32, int p, long long P, __nv_bfloat16* s_o,
                                             const int32_t* bnd, const GroupArgs& gr, int g, int y) {
  constexpr int kPitch = 40;  // staged row: 32 bf16 columns + 16 bytes of padding
  const int t = threadIdx.x;
  if (p == 0) {
    if (a.hdr[2] == 0) return;
    for (int pr = t; pr < a.NP; pr += CombineShape<kWide>::kThreads) {
      if (a.cum[pr] != a.cum[pr + 1]) continue;
      for (int h = 0; h < a.H; ++h) {
        uint4* dst = reinterpret_cast<uint4*>(a.o_lat + (static_cast<long long>(pr) * a.H + h) * kDC + cb32 * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
        if (a.lse != nullptr && cb32 == 0) a.lse[static_cast<long long>(pr) * a.H + h] = -INFINITY;
      }
    }
    return;
  }
  const int32_t* e = bnd + 4 * p;  // the problem holding run p's first block, its first block and end
  const int pr = e[0];
  const long long cb = e[1], ce = e[2], lo_p = e[3];
  if (cb == lo_p) return;                   // the boundary falls between problems
  if (bnd[4 * (p - 1) + 3] > cb) return;    // an earlier boundary cuts this problem and merges it
  const int p_first = p - 1;
  int p_last = p;                           // the run holding the problem's last block
  while (p_last + 1 < P && bnd[4 * (p_last + 1) + 3] < ce) ++p_last;
  const long long slot_first = 2 * p_first + (bnd[4 * p_first + 3] == cb ? 0 : 1);
  if (kGrouped && g == 0 && cb32 == 0 && t == 0) gr.cutp[y] = pr;

  constexpr int kThreads = CombineShape<kWide>::kThreads, kPieces = CombineShape<kWide>::kPieces,
                kCols = CombineShape<kWide>::kCols;
  const int h0 = (t & 63) * 2, c0 = cb32 * 32 + (t >> 6) * kCols;
  float acc[kCols][2];
#pragma unroll
  for (int j = 0; j < kCols; ++j) acc[j][0] = acc[j][1] = 0.f;
  float M[2] = {-INFINITY, -INFINITY}, L[2] = {0.f, 0.f};
  // this group's pieces: p_first + g, p_first + g + G, ... (all of them when G = 1)
  const int G = kGrouped ? gr.G : 1;
  for (int q0 = p_first + (kGrouped ? g : 0); q0 <= p_last; q0 += kPieces * G) {
    float2 m[kPieces], l[kPieces], sc[kPieces];
    uint2 w[kPieces][kCols / 2];  // column pair jp: heads h0, h0 + 1, two fp16 each
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
      const int q = q0 + u * G;
      if (q <= p_last) {
        const long long slot = q == p_first ? slot_first : 2 * static_cast<long long>(q);
        m[u] = *reinterpret_cast<const float2*>(a.part_m + slot * kM + h0);
        l[u] = *reinterpret_cast<const float2*>(a.part_l + slot * kM + h0);
        sc[u] = *reinterpret_cast<const float2*>(a.part_s + (slot * kChunksPerRow + cb32) * kM + h0);
        // [pair][head][2]: heads h0, h0 + 1 of column pair cp are 4 consecutive halves
        const __half* src = a.part_o + (slot * (kDC / 2 * kM) + static_cast<long long>(c0 / 2) * kM + h0) * 2;
#pragma unroll
        for (int jp = 0; jp < kCols / 2; ++jp) w[u][jp] = *reinterpret_cast<const uint2*>(src + jp * kM * 2);
      } else {
        m[u] = make_float2(-INFINITY, -INFINITY);
        l[u] = sc[u] = make_float2(0.f, 0.f);
#pragma unroll
        for (int jp = 0; jp < kCols / 2; ++jp) w[u][jp] = make_uint2(0u, 0u);
      }
    }
    float mn[2] = {M[0], M[1]};
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
      mn[0] = fmaxf(mn[0], m[u].x);
      mn[1] = fmaxf(mn[1], m[u].y);
    }
    const float al0 = exp2f(M[0] - mn[0]), al1 = exp2f(M[1] - mn[1]);  // 0 before the first round
    L[0] *= al0;
    L[1] *= al1;
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      acc[j][0] *= al0;
      acc[j][1] *= al1;
    }
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
      const float w0 = exp2f(m[u].x - mn[0]), w1 = exp2f(m[u].y - mn[1]);  // 0 for absent pieces
      L[0] = fmaf(w0, l[u].x, L[0]);
      L[1] = fmaf(w1, l[u].y, L[1]);
      const float s0 = w0 * sc[u].x, s1 = w1 * sc[u].y;  // the piece's 32-column scale folded in
#pragma unroll
      for (int jp = 0; jp < kCols / 2; ++jp) {
        const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&w[u][jp].x));  // head h0
        const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&w[u][jp].y));  // head h0 + 1
        acc[2 * jp][0] = fmaf(s0, a0.x, acc[2 * jp][0]);
        acc[2 * jp + 1][0] = fmaf(s0, a0.y, acc[2 * jp + 1][0]);
        acc[2 * jp][1] = fmaf(s1, a1.x, acc[2 * jp][1]);
        acc[2 * jp + 1][1] = fmaf(s1, a1.y, acc[2 * jp + 1][1]);
      }
    }
    M[0] = mn[0];
    M[1] = mn[1];
  }
  if (kGrouped) {
    // this group's partial, in the log2 units of the pieces (a group with no piece
    // leaves M = -inf, L = 0, acc = 0)
    const long long gi = static_cast<long long>(g) * gr.cuts + y;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float* dst = gr.ga + (gi * kM + h0 + i) * kDC + c0;
#pragma unroll
      for (int j = 0; j < kCols; j += 4)
        *reinterpret_cast<float4*>(dst + j) = make_float4(acc[j][i], acc[j + 1][i], acc[j + 2][i], acc[j + 3][i]);
    }
    if (cb32 == 0 && t < 64) {
      *reinterpret_cast<float2*>(gr.gm + gi * kM + h0) = make_float2(M[0], M[1]);
      *reinterpret_cast<float2*>(gr.gl + gi * kM + h0) = make_float2(L[0], L[1]);
    }
    return;
  }
  __syncthreads();  // the previous item's tile has been written out
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float inv = 1.f / L[i];
    uint32_t pk[kCols / 2];
#pragma unroll
    for (int j = 0; j < kCols / 2; ++j) pk[j] = pack_bf16x2(acc[2 * j][i] * inv, acc[2 * j + 1][i] * inv);
    __nv_bfloat16* dst = s_o + (h0 + i) * kPitch + (t >> 6) * kCols;
    if constexpr (kCols == 8)
      *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    else
      *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  }
  if (a.lse != nullptr && cb32 == 0 && t < 64) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (h0 + i < a.H)
        a.lse[static_cast<long long>(pr) * a.H + h0 + i] = (M[i] + log2f(L[i])) * 0.69314718055994531f;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kM * 4 / kThreads; ++k) {
    const int id = k * kThreads + t, row = id >> 2, q = id & 3;
    if (row < a.H)
      *reinterpret_cast<uint4*>(a.o_lat + (static_cast<long long>(pr) * a.H + row) * kDC + cb32 * 32 + q * 8) =
          *reinterpret_cast<const uint4*>(s_o + row * kPitch + q * 8);
  }
}

// Block (x, j) merges columns [32 x, 32 x + 32) of the j-th problem that needs a
// merge (found from the run table: boundary p cuts a problem and is the first
// boundary inside it); the last row of blocks writes the problems with no rows.
template <bool kGrouped, bool kWide>
__global__ void __launch_bounds__(CombineShape<kWide>::kThreads, CombineShape<kWide>::kBlocksPerSm)
    combine_kernel(const Args a, const GroupArgs gr) {
  __shared__ __align__(16) __nv_bfloat16 s_o[kM * 40];
  __shared__ int32_t s_bnd[4 * kMaxPairs];
  __shared__ int s_p;
  griddep_launch();
  griddep_wait();  // the pieces of the split kernel
  // the run table in one round of loads (entries past the run count are not used)
  for (int i = threadIdx.x; i < 4 * kMaxPairs; i += CombineShape<kWide>::kThreads) s_bnd[i] = a.bnd[i];
  if (threadIdx.x == 0) s_p = 0;
  const int P = a.hdr[1];
  __syncthreads();
  if (blockIdx.y == gridDim.y - 1) {
    if (blockIdx.z == 0) combine_item<kGrouped, kWide>(a, blockIdx.x, 0, P, s_o, s_bnd, gr, 0, 0);
    return;
  }
  // boundary p (1 <= p < P) needs a merge if it cuts a problem that starts in run p - 1
  static_assert(kMaxPairs <= 96, "three warps rank the boundaries");
  if (threadIdx.x < 96) {  // whole warps 0..2
    const int p = threadIdx.x;
    const bool need = p >= 1 && p < P && p < kMaxPairs && s_bnd[4 * p + 1] != s_bnd[4 * p + 3] &&
                      s_bnd[4 * (p - 1) + 3] <= s_bnd[4 * p + 1];
    const unsigned m0 = __ballot_sync(0xffffffffu, need);
    const int w = threadIdx.x >> 5;
    __shared__ unsigned s_masks[4];
    if ((threadIdx.x & 31) == 0) s_masks[w] = m0;
    asm volatile("bar.sync 1, 96;" ::: "memory");
    // rank of this boundary among those that need a merge
    int rank = __popc(m0 & ((1u << (threadIdx.x & 31)) - 1u));
    for (int v = 0; v < w; ++v) rank += __popc(s_masks[v]);
    if (need && rank == static_cast<int>(blockIdx.y)) s_p = p;
  }
  __syncthreads();
  // -1 unless this row's item writes its problem (the same thread, later): fewer cuts
  // than rows leave the rest of the rows without one
  if (kGrouped && blockIdx.z == 0 && blockIdx.x == 0 && threadIdx.x == 0) gr.cutp[blockIdx.y] = -1;
  if (s_p > 0) combine_item<kGrouped, kWide>(a, blockIdx.x, s_p, P, s_o, s_bnd, gr, blockIdx.z, blockIdx.y);
}

// The second step of the grouped merge: block (x, y) merges the G partials of
// columns [32 x, 32 x + 32) of the y-th cut problem, thread t heads 2(t % 64), +1
// and columns 8(t / 64)..+7, two partials per round.
__global__ void __launch_bounds__(kMergeThreads) merge_groups_kernel(const Args a, const GroupArgs gr) {
  __shared__ __align__(16) __nv_bfloat16 s_o[kM * 40];
  constexpr int kPitch = 40;
  griddep_launch();
  griddep_wait();  // the group partials
  const int y = blockIdx.y, cb32 = blockIdx.x, t = threadIdx.x;
  const int pr = gr.cutp[y];
  if (pr < 0) return;
  const int h0 = (t & 63) * 2, c0 = cb32 * 32 + (t >> 6) * 8;
  float acc[8][2];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = 0.f;
  float M[2] = {-INFINITY, -INFINITY}, L[2] = {0.f, 0.f};
  for (int g0 = 0; g0 < gr.G; g0 += 2) {
    float2 m[2], l[2];
    float4 v[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long gi = static_cast<long long>(g0 + u) * gr.cuts + y;
      m[u] = *reinterpret_cast<const float2*>(gr.gm + gi * kM + h0);
      l[u] = *reinterpret_cast<const float2*>(gr.gl + gi * kM + h0);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float* src = gr.ga + (gi * kM + h0 + i) * kDC + c0;
        v[u][2 * i] = *reinterpret_cast<const float4*>(src);
        v[u][2 * i + 1] = *reinterpret_cast<const float4*>(src + 4);
      }
    }
    float mn[2] = {M[0], M[1]};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      mn[0] = fmaxf(mn[0], m[u].x);
      mn[1] = fmaxf(mn[1], m[u].y);
    }
    // a partial with no pieces (M = -inf) weighs 0; so does the start (M = -inf)
    const float al0 = M[0] == -INFINITY ? 0.f : exp2f(M[0] - mn[0]);
    const float al1 = M[1] == -INFINITY ? 0.f : exp2f(M[1] - mn[1]);
    L[0] *= al0;
    L[1] *= al1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[j][0] *= al0;
      acc[j][1] *= al1;
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float w0 = m[u].x == -INFINITY ? 0.f : exp2f(m[u].x - mn[0]);
      const float w1 = m[u].y == -INFINITY ? 0.f : exp2f(m[u].y - mn[1]);
      L[0] = fmaf(w0, l[u].x, L[0]);
      L[1] = fmaf(w1, l[u].y, L[1]);
      const float x0[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
      const float x1[8] = {v[u][2].x, v[u][2].y, v[u][2].z, v[u][2].w, v[u][3].x, v[u][3].y, v[u][3].z, v[u][3].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[j][0] = fmaf(w0, x0[j], acc[j][0]);
        acc[j][1] = fmaf(w1, x1[j], acc[j][1]);
      }
    }
    M[0] = mn[0];
    M[1] = mn[1];
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float inv = 1.f / L[i];
    uint4 pk;
    pk.x = pack_bf16x2(acc[0][i] * inv, acc[1][i] * inv);
    pk.y = pack_bf16x2(acc[2][i] * inv, acc[3][i] * inv);
    pk.z = pack_bf16x2(acc[4][i] * inv, acc[5][i] * inv);
    pk.w = pack_bf16x2(acc[6][i] * inv, acc[7][i] * inv);
    *reinterpret_cast<uint4*>(s_o + (h0 + i) * kPitch + (t >> 6) * 8) = pk;
  }
  if (a.lse != nullptr && cb32 == 0 && t < 64) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (h0 + i < a.H)
        a.lse[static_cast<long long>(pr) * a.H + h0 + i] = (M[i] + log2f(L[i])) * 0.69314718055994531f;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int id = k * kMergeThreads + t, row = id >> 2, q = id & 3;
    if (row < a.H)
      *reinterpret_cast<uint4*>(a.o_lat + (static_cast<long long>(pr) * a.H + row) * kDC + cb32 * 32 + q * 8) =
          *reinterpret_cast<const uint4*>(s_o + row * kPitch + q * 8);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> cached{nullptr};  // looked up until it succeeds once
  EncodeTiledFn fn = cached.load(std::memory_order_acquire);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// Pieces of one cut problem are merged by G groups of blocks (every G-th piece each)
// and a second kernel merges the G partials, when few problems share many runs (a
// long single sequence is cut into as many pieces as there are runs, and one block
// per 32 columns would merge them a few at a time, one L2 round trip per round).  G
// from the pieces a problem can expect, e = runs / problems: 1 below 16 pieces
// (the merge then costs less than the second launch), else a power of two near e / 8.
constexpr int kMaxGroups = 16;
__host__ __device__ constexpr int combine_groups(long long np, int npairs) {
  const long long e = np > 0 ? (npairs + np - 1) / np : 1;
  if (e < 16) return 1;
  int g = 1;
  while (2 * g <= e / 8 && 2 * g <= kMaxGroups) g *= 2;
  return g;
}

struct WsLayout {
  size_t hdr, bnd, cum, m, l, s, o;
  size_t cutp, gm, gl, ga;  // grouped merge (combine_groups > 1): cut problems, group partials
  size_t total;
};

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace of a launch over np problems: header, block table, and two partial
// slots per run (the problem holding the run's first block and the one cut at its
// end).
constexpr WsLayout ws_layout(long long np) {
  WsLayout w = {};
  const size_t slots = 2 * static_cast<size_t>(kMaxPairs);
  w.hdr = 0;
  w.bnd = 256;
  w.cum = w.bnd + align256(sizeof(int32_t) * 4 * kMaxPairs);
  w.m = w.cum + align256(sizeof(int32_t) * static_cast<size_t>(np + 1));
  w.l = w.m + align256(sizeof(float) * slots * kM);
  w.s = w.l + align256(sizeof(float) * slots * kM);
  w.o = w.s + align256(sizeof(float) * slots * kChunksPerRow * kM);
  const size_t end = w.o + align256(2 * slots * kM * kDC);  // fp16
  // the grouped merge of problems cut into many pieces (sized for the most runs a
  // launch can have)
  const long long g = combine_groups(np, kMaxPairs);
  const long long ncut = np < kMaxPairs ? np : kMaxPairs;
  const size_t gp = g > 1 ? static_cast<size_t>(g * ncut) : 0;
  w.cutp = end;
  w.gm = w.cutp + (g > 1 ? align256(sizeof(int32_t) * static_cast<size_t>(ncut)) : 0);
  w.gl = w.gm + align256(sizeof(float) * gp * kM);
  w.ga = w.gl + align256(sizeof(float) * gp * kM);
  w.total = w.ga + sizeof(float) * gp * kM * kDC;
  return w;
}

// Fault injection for the tests of the bounded waits (see mla_debug_inject_fault):
// one process-wide switch, read by every later launch on any host thread.
static std::atomic<int> g_inject_fault{0};

static int pairs_for_device() {
  static std::atomic<int> cached[64];  // zero-initialised: not yet computed
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  const int known = cached[dev].load(std::memory_order_acquire);
  if (known > 0) return known;
  // both instantiations have the same resources; the unranged one stands for both
  if (ensure_smem_limit(reinterpret_cast<const void*>(decode_split_kernel<false>), kSmemAlloc) != cudaSuccess ||
      ensure_smem_limit(reinterpret_cast<const void*>(decode_split_kernel<true>), kSmemAlloc) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kMaxPairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_split_kernel<false>, &cfg) != cudaSuccess || n <= 0) return -1;
  const int pairs = n < kMaxPairs ? n : kMaxPairs;
  cached[dev].store(pairs, std::memory_order_release);  // concurrent first calls compute the same value
  return pairs;
}

}  // namespace dtc

size_t decode_tc_workspace_size(int32_t B) { return dtc::ws_layout(B).total; }

void set_fault_injection(int32_t kind) { dtc::g_inject_fault.store(kind == 1 ? 1 : 0, std::memory_order_relaxed); }

size_t prefill_tc_workspace_size(int32_t B, int32_t S) {
  return dtc::ws_layout(static_cast<long long>(B) * S).total;
}

// A paged pool (table != nullptr) is passed as c with c.data the pool, c.B the
// sequences and c.N_max = 64 x max_blocks.
struct PagedView {
  const int32_t* table;
  int32_t max_blocks, num_pages;
};

static mla_status launch_attn_tc(const void* q_cat, const mla_cache& c, const dtc::Problems& pbs, long long np,
                                 int32_t H, float scale, void* ws, size_t ws_bytes, void* o_lat, float* lse,
                                 cudaStream_t s, const PagedView& pv = PagedView{nullptr, 0, 0},
                                 const int32_t* row_begin = nullptr) {
  using namespace dtc;
  const WsLayout w = ws_layout(np);
  if (ws == nullptr || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MLA_ERR_WORKSPACE;
  // block indices are 32-bit on the device
  if (np * ((static_cast<long long>(c.N_max) + kBN - 1) / kBN) >= (1ll << 31)) return MLA_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return MLA_ERR_CUDA;
  const int npairs = pairs_for_device();
  if (npairs <= 0) return MLA_ERR_CUDA;

  const int R = c.d_c + c.d_r;
  CUtensorMap map;
  // contiguous: (R, N_max, B), one plane per sequence; paged: (R, 64, pages), one
  // plane per page, every 64-row block a whole page
  const bool paged = pv.table != nullptr;
  const cuuint64_t plane_rows = paged ? static_cast<cuuint64_t>(kBN) : static_cast<cuuint64_t>(c.N_max);
  const cuuint64_t planes = paged ? static_cast<cuuint64_t>(pv.num_pages) : static_cast<cuuint64_t>(c.B);
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(R), plane_rows, planes};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(c.row_stride) * 2,
                                 static_cast<cuuint64_t>(c.row_stride) * 2 * plane_rows};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBN), 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c.data, gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLA_ERR_INVALID_ARG;

  // the queries as [NP * H rows][R]: each problem's query is staged through the score
  // CTA's ring as 64 x 64 boxes
  CUtensorMap qmap;
  const cuuint64_t qdim[2] = {static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(np) * static_cast<cuuint64_t>(H)};
  const cuuint64_t qstride[1] = {static_cast<cuuint64_t>(R) * 2};
  const cuuint32_t qbox[2] = {64, static_cast<cuuint32_t>(kBN)};
  const cuuint32_t qes[2] = {1, 1};
  if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q_cat), qdim, qstride, qbox, qes,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLA_ERR_INVALID_ARG;

  // o_lat as [NP * H rows][512] for the TMA stores of whole problems: H rows x 32 columns
  CUtensorMap omap;
  const cuuint64_t odim[2] = {static_cast<cuuint64_t>(kDC), static_cast<cuuint64_t>(np) * static_cast<cuuint64_t>(H)};
  const cuuint64_t ostride[1] = {static_cast<cuuint64_t>(kDC) * 2};
  const cuuint32_t obox[2] = {32, static_cast<cuuint32_t>(H)};
  if (enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o_lat, odim, ostride, obox, qes, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return MLA_ERR_INVALID_ARG;

  uint8_t* wsb = static_cast<uint8_t*>(ws);
  Args a;
  a.q_cat = static_cast<const __nv_bfloat16*>(q_cat);
  a.pb = pbs;
  a.NP = static_cast<int>(np);
  a.H = H;
  a.N_max = c.N_max;
  a.R = R;
  a.nch = R / 64;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.switch_cost = np > npairs ? kSwitchCostMany : kSwitchCostFew;
  a.hdr = reinterpret_cast<int32_t*>(wsb + w.hdr);
  a.cum = reinterpret_cast<int32_t*>(wsb + w.cum);
  a.bnd = reinterpret_cast<int32_t*>(wsb + w.bnd);
  a.part_m = reinterpret_cast<float*>(wsb + w.m);
  a.part_l = reinterpret_cast<float*>(wsb + w.l);
  a.part_s = reinterpret_cast<float*>(wsb + w.s);
  a.part_o = reinterpret_cast<__half*>(wsb + w.o);
  a.o_lat = static_cast<__nv_bfloat16*>(o_lat);
  a.lse = lse;
  a.fault = g_inject_fault.load(std::memory_order_relaxed);
  a.block_table = pv.table;
  a.max_blocks = pv.max_blocks;
  a.num_pages = pv.num_pages;
  a.row_begin = row_begin;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * npairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = row_begin != nullptr ? cudaLaunchKernelEx(&cfg, decode_split_kernel<true>, map, qmap, omap, a)
                                       : cudaLaunchKernelEx(&cfg, decode_split_kernel<false>, map, qmap, omap, a);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  // at most min(runs - 1, problems) problems need a merge; one more row for empty problems
  const long long ncut = np < npairs - 1 ? np : npairs - 1;
  const unsigned rows = static_cast<unsigned>(ncut > 0 ? ncut : 0) + 1u;
  GroupArgs gr = {};
  gr.G = combine_groups(np, npairs);
  gr.cuts = static_cast<int>(rows - 1);
  if (gr.G > 1) {
    gr.cutp = reinterpret_cast<int32_t*>(wsb + w.cutp);
    gr.gm = reinterpret_cast<float*>(wsb + w.gm);
    gr.gl = reinterpret_cast<float*>(wsb + w.gl);
    gr.ga = reinterpret_cast<float*>(wsb + w.ga);
  }
  // the wide item shape when the launch's items fit in one wave of it (two blocks an
  // SM, about two SMs a cluster)
  const dim3 grid(kDC / 32, rows, static_cast<unsigned>(gr.G));
  const bool wide = static_cast<long long>(grid.x) * grid.y * grid.z <= 2LL * 2 * npairs;
  cudaError_t err;
  if (gr.G == 1)
    err = wide ? launch_pdl(combine_kernel<false, true>, grid, dim3(CombineShape<true>::kThreads), 0, s, a, gr)
             : launch_pdl(combine_kernel<false, false>, grid, dim3(CombineShape<false>::kThreads), 0, s, a, gr);
  else
    err = wide ? launch_pdl(combine_kernel<true, true>, grid, dim3(CombineShape<true>::kThreads), 0, s, a, gr)
             : launch_pdl(combine_kernel<true, false>, grid, dim3(CombineShape<false>::kThreads), 0, s, a, gr);
  if (err != cudaSuccess || gr.G == 1 || rows == 1) return cuda_status(err);
  return cuda_status(launch_pdl(merge_groups_kernel, dim3(kDC / 32, rows - 1), dim3(kMergeThreads), 0, s, a, gr));
}

mla_status launch_decode_tc(const void* q_cat, const mla_cache& c, const int32_t* seq_lens, int32_t H,
                            float scale, void* ws, size_t ws_bytes, void* o_lat, float* lse, cudaStream_t s,
                            const int32_t* block_table, int32_t max_blocks, int32_t num_pages,
                            const int32_t* row_begin) {
  dtc::Problems p = {};
  p.seq_lens = seq_lens;
  p.q_start = nullptr;
  p.S = 1;
  p.causal = 0;
  p.n_max = c.N_max;
  return launch_attn_tc(q_cat, c, p, c.B, H, scale, ws, ws_bytes, o_lat, lse, s,
                        PagedView{block_table, max_blocks, num_pages}, row_begin);
}

mla_status launch_prefill_tc(const void* q_cat, const mla_cache& c, const int32_t* q_start, int32_t S,
                             int32_t causal, int32_t H, float scale, void* ws, size_t ws_bytes, void* o_lat,
                             float* lse, cudaStream_t s) {
  dtc::Problems p = {};
  p.seq_lens = nullptr;
  p.q_start = q_start;
  p.S = S;
  p.causal = causal != 0;
  p.n_max = c.N_max;
  return launch_attn_tc(q_cat, c, p, static_cast<long long>(c.B) * S, H, scale, ws, ws_bytes, o_lat, lse, s);
}

}  // namespace mla

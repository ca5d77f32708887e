// CUDA-core kernels of libmla: cache append with RoPE, query absorption,
// W_UV up-projection, the sigmoid output gate, and the fp32 decode attention.
//
// These steps are memory-bound at the decode shapes (they stream W_UK, W_UV or
// W_g once) or tiny (the fp32 path), so they run on the CUDA cores with
// coalesced loads and fp32 arithmetic.
#include <cmath>

#include "mla_internal.cuh"
#include "mla_ptx.cuh"

namespace mla {

// ============================================================================
// Cache append: cache[seq][pos] = [c_kv || RoPE(k_r, pos)]
// (icman.com.cn MLA article, section 2: the 64-wide key is cached with RoPE
// applied; 0539edu.com section 5.2: the cache is written by position.)  With a
// block table the cache is paged: row pos of sequence seq is row pos % 64 of page
// table[seq][pos / 64] of the pool.
// ============================================================================
struct PageMap {
  const int32_t* table;  // [B][max_blocks] page of each 64-row block, or nullptr (contiguous cache)
  int32_t max_blocks;
  int32_t num_pages;
};

template <typename T>
__global__ void __launch_bounds__(128) cache_append_kernel(T* __restrict__ cache, int32_t B, int32_t N_max,
                                                           int32_t d_c, int32_t d_r, int64_t row_stride,
                                                           const T* __restrict__ c_kv, const T* __restrict__ k_r,
                                                           const int32_t* __restrict__ seq_idx,
                                                           const int32_t* __restrict__ pos, int32_t n_rows,
                                                           const __grid_constant__ RopeTable rope, int vec_ok,
                                                           PageMap pages) {
  __shared__ float s_hi[64], s_lo[64];
  griddep_launch();
  rope_table_to_smem(rope, d_r / 2, s_hi, s_lo);
  griddep_wait();  // the rows written here may still be read by the previous kernel
  for (int64_t i = blockIdx.x; i < n_rows; i += gridDim.x) {
    const int32_t b = seq_idx[i];
    const int32_t p = pos[i];
    if (b < 0 || b >= B || p < 0 || p >= N_max) {
      if (threadIdx.x == 0) record_error(MLA_ERR_DEVICE_INDEX, kSiteAppendIndex);
      continue;
    }
    int64_t row = static_cast<int64_t>(b) * N_max + p;
    if (pages.table != nullptr) {
      const int32_t pg = pages.table[static_cast<int64_t>(b) * pages.max_blocks + p / kPageRows];
      if (pg < 0 || pg >= pages.num_pages) {
        if (threadIdx.x == 0) record_error(MLA_ERR_DEVICE_INDEX, kSitePageIndex);
        continue;
      }
      row = static_cast<int64_t>(pg) * kPageRows + p % kPageRows;
    }
    T* dst = cache + row * row_stride;
    const T* src = c_kv + i * d_c;
    if (vec_ok) {
      const int nvec = d_c * static_cast<int>(sizeof(T)) / 16;
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) d4[v] = s4[v];
    } else {
      for (int c = threadIdx.x; c < d_c; c += blockDim.x) dst[c] = src[c];
    }
    // rotate pairs (2j, 2j+1) by pos * theta_j
    const T* kr = k_r + i * d_r;
    for (int j = threadIdx.x; j < d_r / 2; j += blockDim.x) {
      float sn, cs;
      rope_sincos(p, s_hi[j], s_lo[j], &sn, &cs);
      const float x0 = ld_elem(kr + 2 * j), x1 = ld_elem(kr + 2 * j + 1);
      st_elem(dst + d_c + 2 * j, fmaf(x0, cs, -x1 * sn));
      st_elem(dst + d_c + 2 * j + 1, fmaf(x0, sn, x1 * cs));
    }
  }
}

mla_status launch_cache_append(const mla_cache& c, const void* c_kv, const void* k_r, const int32_t* seq_idx,
                               const int32_t* pos, int32_t T, float rope_base, cudaStream_t s,
                               const int32_t* block_table, int32_t max_blocks, int32_t num_pages) {
  const PageMap pages = {block_table, max_blocks, num_pages};
  const int grid = static_cast<int>(T < 148 * 16 ? T : 148 * 16);
  const size_t esz = c.dtype == MLA_BF16 ? 2 : 4;
  const int vec_ok = ((c.d_c * esz) % 16 == 0) && ((c.row_stride * esz) % 16 == 0) && aligned16(c_kv) &&
                     aligned16(c.data);
  if (c.dtype == MLA_BF16) {
    const cudaError_t e = launch_pdl(cache_append_kernel<__nv_bfloat16>, dim3(grid), dim3(128), 0, s,
                                     static_cast<__nv_bfloat16*>(c.data), c.B, c.N_max, c.d_c, c.d_r,
                                     static_cast<int64_t>(c.row_stride), static_cast<const __nv_bfloat16*>(c_kv),
                                     static_cast<const __nv_bfloat16*>(k_r), seq_idx, pos, T,
                                     rope_table(c.d_r, rope_base), vec_ok, pages);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
  } else {
    cache_append_kernel<float><<<grid, 128, 0, s>>>(static_cast<float*>(c.data), c.B, c.N_max, c.d_c, c.d_r,
                                                    c.row_stride, static_cast<const float*>(c_kv),
                                                    static_cast<const float*>(k_r), seq_idx, pos, T,
                                                    rope_table(c.d_r, rope_base), vec_ok, pages);
  }
  return cuda_status(cudaGetLastError());
}

// ============================================================================
// Query absorption: q_cat[b][h] = [q_nope[b][h] . W_UK[h] || RoPE(q_rope[b][h], q_pos[b])]
// (0539edu.com sections 3.1 and 5.1: W_UK folded into the query, weight view
// [h, d_k, d_c].)  One block per (128 latent columns, head); the head's queries
// for 32 sequences at a time sit in shared memory and W_UK is streamed once.
// ============================================================================
constexpr int kAbsorbBatch = 32;

template <typename T>
__global__ void __launch_bounds__(128) absorb_q_kernel(const T* __restrict__ q_nope, const T* __restrict__ q_rope,
                                                       const int32_t* __restrict__ q_pos,
                                                       const T* __restrict__ w_uk, T* __restrict__ q_cat, int B,
                                                       int H, int d_k, int d_c, int d_r,
                                                       const __grid_constant__ RopeTable rope) {
  extern __shared__ float qs[];  // [kAbsorbBatch][d_k]
  __shared__ float s_hi[64], s_lo[64];
  rope_table_to_smem(rope, d_r / 2, s_hi, s_lo);
  const int h = blockIdx.y;
  const int c = blockIdx.x * 128 + threadIdx.x;
  const int R = d_c + d_r;
  for (int b0 = 0; b0 < B; b0 += kAbsorbBatch) {
    const int nb = min(kAbsorbBatch, B - b0);
    __syncthreads();
    for (int idx = threadIdx.x; idx < kAbsorbBatch * d_k; idx += blockDim.x) {
      const int bb = idx / d_k, d = idx - bb * d_k;
      qs[idx] = bb < nb ? ld_elem(q_nope + (static_cast<int64_t>(b0 + bb) * H + h) * d_k + d) : 0.f;
    }
    __syncthreads();
    if (c < d_c) {
      float acc[kAbsorbBatch];
#pragma unroll
      for (int bb = 0; bb < kAbsorbBatch; ++bb) acc[bb] = 0.f;
      const T* w = w_uk + static_cast<int64_t>(h) * d_k * d_c + c;
      for (int d = 0; d < d_k; ++d) {
        const float wv = ld_elem(w + static_cast<int64_t>(d) * d_c);
#pragma unroll
        for (int bb = 0; bb < kAbsorbBatch; ++bb) acc[bb] = fmaf(qs[bb * d_k + d], wv, acc[bb]);
      }
#pragma unroll
      for (int bb = 0; bb < kAbsorbBatch; ++bb)
        if (bb < nb) st_elem(q_cat + (static_cast<int64_t>(b0 + bb) * H + h) * R + c, acc[bb]);
    }
  }
  if (blockIdx.x == 0 && d_r > 0) {
    const int half = d_r / 2;
    for (int idx = threadIdx.x; idx < B * half; idx += blockDim.x) {
      const int b = idx / half, j = idx - b * half;
      float sn, cs;
      rope_sincos(q_pos[b], s_hi[j], s_lo[j], &sn, &cs);
      const T* qr = q_rope + (static_cast<int64_t>(b) * H + h) * d_r;
      const float x0 = ld_elem(qr + 2 * j), x1 = ld_elem(qr + 2 * j + 1);
      T* dst = q_cat + (static_cast<int64_t>(b) * H + h) * R + d_c;
      st_elem(dst + 2 * j, fmaf(x0, cs, -x1 * sn));
      st_elem(dst + 2 * j + 1, fmaf(x0, sn, x1 * cs));
    }
  }
}

mla_status launch_absorb_q(const void* q_nope, const void* q_rope, const int32_t* q_pos, const void* w_uk,
                           void* q_cat, int32_t B, int32_t H, int32_t d_k, int32_t d_c, int32_t d_r,
                           int32_t dtype, float rope_base, cudaStream_t s) {
  if (dtype != MLA_F32) return MLA_ERR_UNSUPPORTED;  // bf16 runs on the tensor cores only
  dim3 grid((d_c + 127) / 128, H);
  const size_t smem = sizeof(float) * kAbsorbBatch * d_k;
  auto k = absorb_q_kernel<float>;
  ensure_smem_limit(reinterpret_cast<const void*>(k), smem);
  k<<<grid, 128, smem, s>>>(static_cast<const float*>(q_nope), static_cast<const float*>(q_rope), q_pos,
                            static_cast<const float*>(w_uk), static_cast<float*>(q_cat), B, H, d_k, d_c, d_r,
                            rope_table(d_r, rope_base));
  return cuda_status(cudaGetLastError());
}

// ============================================================================
// W_UV after attention: o[b][h][d] = sum_c o_lat[b][h][c] * W_UV[h][d][c]
// (0539edu.com section 3.1, attn v = (attn c_KV) W_UV.)  One warp per output
// column d holds W_UV[h][d][:] in registers; the head's o_lat rows for 32
// sequences at a time sit in shared memory.
// ============================================================================
constexpr int kOutBatch = 32;

template <typename T>
__global__ void __launch_bounds__(256) out_up_kernel(const T* __restrict__ o_lat, const T* __restrict__ w_uv,
                                                     T* __restrict__ o, int B, int H, int d_c, int d_v) {
  extern __shared__ float os[];  // [kOutBatch][d_c]
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = blockIdx.x * 8 + warp;
  float w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int c = lane + 32 * i;
    w[i] = (d < d_v && c < d_c) ? ld_elem(w_uv + (static_cast<int64_t>(h) * d_v + d) * d_c + c) : 0.f;
  }
  for (int b0 = 0; b0 < B; b0 += kOutBatch) {
    const int nb = min(kOutBatch, B - b0);
    __syncthreads();
    for (int idx = threadIdx.x; idx < nb * d_c; idx += blockDim.x) {
      const int bb = idx / d_c, c = idx - bb * d_c;
      os[idx] = ld_elem(o_lat + (static_cast<int64_t>(b0 + bb) * H + h) * d_c + c);
    }
    __syncthreads();
    for (int bb = 0; bb < nb; ++bb) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = lane + 32 * i;
        if (c < d_c) part = fmaf(os[bb * d_c + c], w[i], part);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == 0 && d < d_v) st_elem(o + (static_cast<int64_t>(b0 + bb) * H + h) * d_v + d, part);
    }
  }
}

mla_status launch_out_up(const void* o_lat, const void* w_uv, void* o, int32_t B, int32_t H, int32_t d_c,
                         int32_t d_v, int32_t dtype, cudaStream_t s) {
  if (dtype != MLA_F32) return MLA_ERR_UNSUPPORTED;  // bf16 runs on the tensor cores only
  dim3 grid((d_v + 7) / 8, H);
  const size_t smem = sizeof(float) * kOutBatch * d_c;
  auto k = out_up_kernel<float>;
  ensure_smem_limit(reinterpret_cast<const void*>(k), smem);
  k<<<grid, 256, smem, s>>>(static_cast<const float*>(o_lat), static_cast<const float*>(w_uv),
                            static_cast<float*>(o), B, H, d_c, d_v);
  return cuda_status(cudaGetLastError());
}

// ============================================================================
// Output gate: o[b][j] *= sigmoid(sum_i h[b][i] W_g[i][j])
// (tahou.com sections 2.6 / 3.2: full-rank, channel-wise, input-dependent.)
// A block owns 32 output channels; its 8 warps split the d_model reduction and
// meet in shared memory; W_g is read once with 32 consecutive channels per warp.
// ============================================================================
constexpr int kGateBatch = 16;
constexpr int kGateTile = 256;

template <typename T>
__global__ void __launch_bounds__(256) gate_kernel(const T* __restrict__ hin, const T* __restrict__ w_g,
                                                   T* __restrict__ o, int B, int d_model, int width) {
  __shared__ float hs[kGateBatch][kGateTile];
  __shared__ float red[8][kGateBatch][32];
  const int jj = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + jj;
  for (int b0 = 0; b0 < B; b0 += kGateBatch) {
    const int nb = min(kGateBatch, B - b0);
    float acc[kGateBatch];
#pragma unroll
    for (int bb = 0; bb < kGateBatch; ++bb) acc[bb] = 0.f;
    for (int i0 = 0; i0 < d_model; i0 += kGateTile) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < kGateBatch * kGateTile; idx += blockDim.x) {
        const int bb = idx / kGateTile, ii = idx - bb * kGateTile;
        hs[bb][ii] = (bb < nb && i0 + ii < d_model)
                         ? ld_elem(hin + static_cast<int64_t>(b0 + bb) * d_model + i0 + ii)
                         : 0.f;
      }
      __syncthreads();
      for (int ii = g * 32; ii < g * 32 + 32; ++ii) {
        const int i = i0 + ii;
        if (i >= d_model) break;
        const float wv = j < width ? ld_elem(w_g + static_cast<int64_t>(i) * width + j) : 0.f;
#pragma unroll
        for (int bb = 0; bb < kGateBatch; ++bb) acc[bb] = fmaf(hs[bb][ii], wv, acc[bb]);
      }
    }
#pragma unroll
    for (int bb = 0; bb < kGateBatch; ++bb) red[g][bb][jj] = acc[bb];
    __syncthreads();
    if (g == 0 && j < width) {
      for (int bb = 0; bb < nb; ++bb) {
        float z = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) z += red[q][bb][jj];
        T* op = o + static_cast<int64_t>(b0 + bb) * width + j;
        st_elem(op, ld_elem(op) * (1.f / (1.f + expf(-z))));
      }
    }
    __syncthreads();
  }
}

mla_status launch_gate(const void* h, const void* w_g, void* o, int32_t B, int32_t d_model, int32_t width,
                       int32_t dtype, cudaStream_t s) {
  if (dtype != MLA_F32) return MLA_ERR_UNSUPPORTED;  // bf16 runs on the tensor cores only
  const int grid = (width + 31) / 32;
  gate_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(h), static_cast<const float*>(w_g),
                                          static_cast<float*>(o), B, d_model, width);
  return cuda_status(cudaGetLastError());
}

// ============================================================================
// fp32 decode attention (CUDA cores).  One block per (head, sequence); 128
// tokens at a time, one token per thread for the score, online softmax with the
// running maximum (hotelren.com section 7.3), then the block accumulates
// o_lat += p_t c_KV,t with each thread owning d_c/128 latent columns.
// ============================================================================
__device__ __forceinline__ float block_reduce_max128(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}

__device__ __forceinline__ float block_reduce_sum128(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  return (red[0] + red[1]) + (red[2] + red[3]);
}

__global__ void __launch_bounds__(128) decode_f32_kernel(const float* __restrict__ q_cat,
                                                         const float* __restrict__ cache, int32_t N_max,
                                                         int32_t d_c, int32_t d_r, int64_t row_stride,
                                                         const int32_t* __restrict__ seq_lens,
                                                         const int32_t* __restrict__ q_start, int32_t S,
                                                         int32_t causal, int32_t H, float scale,
                                                         float* __restrict__ o_lat, float* __restrict__ lse) {
  extern __shared__ float sm[];
  const int R = d_c + d_r;
  float* qs = sm;           // [R]
  float* ps = sm + R;       // [128]
  float* red = ps + 128;    // [4]
  // problem pr: decode sequence pr (q_start == nullptr), or query pr % S of
  // sequence pr / S reading start + pr % S + 1 rows (causal) or start + S rows
  const int pr = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int b = q_start == nullptr ? pr : pr / S;
  int n = q_start == nullptr ? seq_lens[pr] : q_start[b] + (causal ? pr - b * S + 1 : S);
  if (n < 0 || n > N_max) {
    if (tid == 0) record_error(MLA_ERR_DEVICE_INDEX, kSiteDecodeLength);
    n = n < 0 ? 0 : N_max;
  }
  for (int k = tid; k < R; k += 128) qs[k] = q_cat[(static_cast<int64_t>(pr) * H + h) * R + k];
  __syncthreads();
  constexpr int kMaxPer = 8;  // d_c <= 1024
  float acc[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) acc[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  const float* base = cache + static_cast<int64_t>(b) * N_max * row_stride;
  for (int t0 = 0; t0 < n; t0 += 128) {
    const int t = t0 + tid;
    float s = -INFINITY;
    if (t < n) {
      const float* row = base + static_cast<int64_t>(t) * row_stride;
      float dot = 0.f;
      for (int k = 0; k < R; ++k) dot = fmaf(qs[k], row[k], dot);
      s = dot * scale;
    }
    const float mt = block_reduce_max128(s, red);
    const float m_new = fmaxf(m, mt);
    const float alpha = expf(m - m_new);  // 0 on the first tile (m = -inf)
    const float p = t < n ? expf(s - m_new) : 0.f;
    ps[tid] = p;
    const float lt = block_reduce_sum128(p, red);
    l = l * alpha + lt;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) acc[i] *= alpha;
    const int cnt = min(128, n - t0);
    for (int tt = 0; tt < cnt; ++tt) {
      const float pt = ps[tt];
      const float* row = base + static_cast<int64_t>(t0 + tt) * row_stride;
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        const int c = tid + 128 * i;
        if (c < d_c) acc[i] = fmaf(pt, row[c], acc[i]);
      }
    }
    m = m_new;
    __syncthreads();
  }
  const float inv = n > 0 ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int c = tid + 128 * i;
    if (c < d_c) o_lat[(static_cast<int64_t>(pr) * H + h) * d_c + c] = acc[i] * inv;
  }
  if (lse != nullptr && tid == 0) lse[static_cast<int64_t>(pr) * H + h] = n > 0 ? m + logf(l) : -INFINITY;
}

mla_status launch_decode_f32(const float* q_cat, const mla_cache& c, const int32_t* seq_lens, int32_t H,
                             float scale, float* o_lat, float* lse, cudaStream_t s) {
  const int R = c.d_c + c.d_r;
  const size_t smem = sizeof(float) * (R + 128 + 4);
  dim3 grid(c.B, H);
  decode_f32_kernel<<<grid, 128, smem, s>>>(q_cat, static_cast<const float*>(c.data), c.N_max, c.d_c, c.d_r,
                                            c.row_stride, seq_lens, nullptr, 1, 0, H, scale, o_lat, lse);
  return cuda_status(cudaGetLastError());
}

mla_status launch_prefill_f32(const float* q_cat, const mla_cache& c, const int32_t* q_start, int32_t S,
                              int32_t causal, int32_t H, float scale, float* o_lat, float* lse, cudaStream_t s) {
  const int R = c.d_c + c.d_r;
  const size_t smem = sizeof(float) * (R + 128 + 4);
  dim3 grid(static_cast<unsigned>(c.B) * S, H);
  decode_f32_kernel<<<grid, 128, smem, s>>>(q_cat, static_cast<const float*>(c.data), c.N_max, c.d_c, c.d_r,
                                            c.row_stride, nullptr, q_start, S, causal, H, scale, o_lat, lse);
  return cuda_status(cudaGetLastError());
}

}  // namespace mla

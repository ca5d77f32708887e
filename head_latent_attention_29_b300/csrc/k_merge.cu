// Merge of attention partials computed over disjoint row ranges of the same
// sequences (in log-sum-exp form: each partial is its own softmax-normalised
// o_s with lse_s = ln sum exp(s_t) over its rows).  The merged result is the
// attention over the union of the rows:
//   M = max_s lse_s,  w_s = exp(lse_s - M),
//   o = sum_s w_s o_s / sum_s w_s,   lse = M + ln sum_s w_s
// -- the max-subtracted softmax of the hotelren.com guide (section 7.3) applied
// across row subsets.  This is the merge step of decode sharded by sequence
// position: the sequence-parallel remark of the 0539edu.com page (section 8).
#include "mla_internal.cuh"
#include "mla_ptx.cuh"

namespace mla {
namespace mrg {

constexpr int kThreads = 256;
constexpr int kCols = 8;  // columns per thread: one 16-byte load of bf16, two of fp32

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[kCols]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[kCols]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[kCols]) {
  *reinterpret_cast<uint4*>(p) =
      make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ void store8(float* p, const float (&v)[kCols]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// One thread per (row, 8 consecutive columns): a warp covers 256 contiguous
// columns of a row in every partial it reads.
template <typename T>
__global__ void __launch_bounds__(kThreads) merge_kernel(const T* __restrict__ o_parts,
                                                         const float* __restrict__ lse_parts, int k, long long rows,
                                                         int d_c, T* __restrict__ o, float* __restrict__ lse) {
  griddep_launch();
  griddep_wait();  // the partials may come from the kernels just before
  const int groups = d_c / kCols;
  const long long gid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const long long row = gid / groups;
  if (row >= rows) return;
  const int c0 = static_cast<int>(gid - row * groups) * kCols;
  float M = -INFINITY;
  for (int s = 0; s < k; ++s) M = fmaxf(M, lse_parts[s * rows + row]);
  float acc[kCols] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (M == -INFINITY) {  // no rows in any partial: the empty softmax
    store8(o + row * d_c + c0, acc);
    if (lse != nullptr && c0 == 0) lse[row] = -INFINITY;
    return;
  }
  float L = 0.f;
  for (int s = 0; s < k; ++s) {
    const float w = expf(lse_parts[s * rows + row] - M);  // 0 for an empty partial
    if (w == 0.f) continue;
    float v[kCols];
    load8(o_parts + (s * rows + row) * d_c + c0, v);
    L += w;
#pragma unroll
    for (int j = 0; j < kCols; ++j) acc[j] = fmaf(w, v[j], acc[j]);
  }
  const float inv = 1.f / L;
#pragma unroll
  for (int j = 0; j < kCols; ++j) acc[j] *= inv;
  store8(o + row * d_c + c0, acc);
  if (lse != nullptr && c0 == 0) lse[row] = M + logf(L);
}

}  // namespace mrg

mla_status launch_decode_merge(const void* o_parts, const float* lse_parts, int32_t k, long long rows, int32_t d_c,
                               int32_t dtype, void* o, float* lse, cudaStream_t s) {
  const long long threads = rows * (d_c / mrg::kCols);
  const long long blocks = (threads + mrg::kThreads - 1) / mrg::kThreads;
  if (blocks > 0x7FFFFFFFLL) return MLA_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e;
  if (dtype == MLA_BF16)
    e = launch_pdl(mrg::merge_kernel<__nv_bfloat16>, grid, dim3(mrg::kThreads), 0, s,
                   static_cast<const __nv_bfloat16*>(o_parts), lse_parts, k, rows, d_c,
                   static_cast<__nv_bfloat16*>(o), lse);
  else
    e = launch_pdl(mrg::merge_kernel<float>, grid, dim3(mrg::kThreads), 0, s, static_cast<const float*>(o_parts),
                   lse_parts, k, rows, d_c, static_cast<float*>(o), lse);
  return cuda_status(e);
}

}  // namespace mla

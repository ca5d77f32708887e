// Allocation-free decode attention.
//
// Some callers cannot allocate device memory at the moment they need attention:
// code running under a custom allocator that must not be re-entered from there,
// runtimes whose device memory is fixed when they start, or embedders that only
// own the input/output buffers handed to them by a host framework.  For them
// mla_decode_attn_noalloc runs the same tensor-core decode kernels as
// mla_decode_attn, but takes its split-KV scratch from a buffer that is part of
// the library image itself (a file-scope device array), so the call allocates
// nothing.
//
// The buffer holds the workspace of any batch of up to kNoAllocMaxBatch sequences
// (about 25 MB: batches of a few long sequences add the partials of the grouped
// merge).  Every GPU that loads the library keeps it until the process
// exits.  All calls on a device share it, so calls whose kernels could overlap on
// the GPU (different streams without ordering between them) race on it.  The
// kernels overwrite every scratch word they later read (run table, partial
// maxima, sums and outputs), so nothing has to be cleared between calls.
#include <mutex>

#include "mla_internal.cuh"

namespace mla {

constexpr int kNoAllocMaxBatch = 32;
// the largest workspace of any batch up to kNoAllocMaxBatch (small batches add the
// partials of the grouped merge)
constexpr size_t noalloc_scratch_bytes() {
  size_t m = 0;
  for (int b = 1; b <= kNoAllocMaxBatch; ++b) {
    const size_t t = dtc::ws_layout(b).total;
    if (t > m) m = t;
  }
  return m;
}
constexpr size_t kNoAllocScratchBytes = noalloc_scratch_bytes();

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch buffer for the current device, looked up once per
// device (host code may not use the symbol itself as a device pointer).
static mla_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* ptr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    ptr[dev] = p;
  }
  *out = ptr[dev];
  return MLA_OK;
}

}  // namespace mla

extern "C" {

MLA_API mla_status mla_decode_attn_noalloc(const void* q_cat, const mla_cache* cache, const int32_t* seq_lens,
                                           int32_t H, float scale, void* o_lat, float* lse, void* stream) {
  const OpRange range("mla_decode_attn_noalloc");
  if (cache == nullptr || q_cat == nullptr || seq_lens == nullptr || o_lat == nullptr) return MLA_ERR_INVALID_ARG;
  if (cache->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (cache->B > mla::kNoAllocMaxBatch) return MLA_ERR_WORKSPACE;  // beyond the built-in scratch
  void* ws = nullptr;
  const mla_status st = mla::noalloc_scratch(&ws);
  if (st != MLA_OK) return st;
  return mla_decode_attn(q_cat, cache, seq_lens, H, scale, ws, mla::kNoAllocScratchBytes, o_lat, lse, stream);
}

}  // extern "C"

// Single translation unit of libmla: the kernels share one device error word,
// so all sources are compiled together.
#include "k_simt.cu"
#include "k_decode_tc.cu"
#include "k_headgemm.cu"
#include "k_kvdown.cu"
#include "k_prefill_explicit.cu"
#include "k_merge.cu"
#include "mla_api.cu"
#include "mla_noalloc.cu"

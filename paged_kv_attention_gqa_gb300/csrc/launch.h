// Kernel launchers of libpkv (host side), called by the C ABI in pkv_api.cu.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "plan.h"

namespace pkv {

int decode_stages(const Shape &s);
cudaError_t set_smem_limit(const void *fn, size_t smem, cudaStream_t st);
size_t decode_smem_bytes(const Shape &s);
size_t prefill_smem_bytes(const Shape &s);

cudaError_t launch_append(const Shape &s, const Plan &p, void *ws, const void *k, const void *v, void *kv_layer,
                          cudaStream_t st);
// Decode pass (and the split-KV merge) of a DECODE or MIXED plan; `tm` boxes a whole
// page of all kv heads.
cudaError_t launch_decode(const Shape &s, const Plan &p, const CUtensorMap &tm, void *ws, const void *q, void *out,
                          float *lse, cudaStream_t st);
// Prefill pass of a PREFILL, MIXED or DENSE plan; `tm_kv` boxes 16 rows of one kv head of
// the layer slice (paged; V rows follow K rows by page_size) or of contiguous K (dense,
// with `tm_v` over contiguous V); `tm_q` boxes (64 columns, g heads, 128/g tokens) of q
// viewed as [tokens][Hq][D].
cudaError_t launch_prefill(const Shape &s, const Plan &p, const CUtensorMap &tm_kv, const CUtensorMap &tm_v,
                           const CUtensorMap &tm_q, void *ws, void *out, float *lse, cudaStream_t st);
// Copy the first `num_tokens` positions of a page list into contiguous K and V
// ([num_tokens, Hkv, D] each).
cudaError_t launch_gather(const Shape &s, const void *kv_layer, const int32_t *pages, int num_tokens, void *k_out,
                          void *v_out, cudaStream_t st);

// File-scope device scratch used by pkv_run_decode_static (see decode.cu).
size_t static_scratch_bytes();
cudaError_t static_scratch(void **ptr);

}  // namespace pkv

// Kernel launchers of libpkv (host side), called by the C ABI in pkv_api.cu.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "plan.h"

// Every (head_dim, group size) the kernels are compiled for.
#define PKV_FOR_EACH_GROUP(X, DD) X(DD, 1) X(DD, 2) X(DD, 3) X(DD, 4) X(DD, 5) X(DD, 6) X(DD, 7) X(DD, 8) X(DD, 16)
#define PKV_FOR_EACH_HEAD_DIM_AND_GROUP(X) PKV_FOR_EACH_GROUP(X, 64) PKV_FOR_EACH_GROUP(X, 128) PKV_FOR_EACH_GROUP(X, 256)

namespace pkv {

// Launch `kernel` with programmatic stream serialization (see griddep_wait in ptx.cuh):
// every kernel of this library waits for its predecessor on the stream in-kernel, after
// its prologue, so the launch itself may overlap the predecessor's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int decode_stages(const Shape &s);
cudaError_t set_smem_limit(const void *fn, size_t smem, cudaStream_t st);
size_t decode_smem_bytes(const Shape &s);
size_t prefill_smem_bytes(const Shape &s);

cudaError_t launch_append(const Shape &s, const Plan &p, void *ws, const void *k, const void *v, void *kv_layer,
                          cudaStream_t st);
// Append from device index arrays, no plan (pkv_kv_append); see append_indexed_kernel.
cudaError_t launch_append_indexed(const Shape &s, const void *k, const void *v, int num_tokens, void *kv_layer,
                                  const int32_t *qo_indptr, const int32_t *kv_indptr, const int32_t *kv_indices,
                                  const int32_t *last_page_len, int batch, cudaStream_t st);
// Decode pass (and the split-KV merge) of a DECODE or MIXED plan; `tm` boxes
// (64 columns, Shape::dec_box_rows() rows, Shape::dec_heads() heads) of the layer slice.
// `kv_layer` is the slice `tm` maps (read directly for pages below 8 slots).  With k_new /
// v_new given (a DECODE plan), the kernel also appends the plan's new tokens (the pieces
// holding each row's last position store them into kv_layer).
cudaError_t launch_decode(const Shape &s, const Plan &p, const CUtensorMap &tm, void *ws, const void *q,
                          void *kv_layer, void *out, float *lse, cudaStream_t st, const void *k_new = nullptr,
                          const void *v_new = nullptr);
// Prefill pass of a PREFILL, MIXED or DENSE plan; `tm_kv` boxes Shape::pf_box_rows() rows
// of one kv head of the layer slice (paged; V rows follow K rows by page_size) or 16 rows
// of contiguous K (dense, with `tm_v` over contiguous V); `tm_q` boxes (64 columns, g
// heads, 128/g tokens) of q viewed as [tokens][Hq][D].  Paged plans with pages smaller than
// 8 slots read `kv_layer` directly (16-byte copies) instead of `tm_kv`.
cudaError_t launch_prefill(const Shape &s, const Plan &p, const CUtensorMap &tm_kv, const CUtensorMap &tm_v,
                           const CUtensorMap &tm_q, const void *kv_layer, void *ws, void *out, float *lse,
                           cudaStream_t st);
// Copy the first `num_tokens` positions of a page list into contiguous K and V
// ([num_tokens, Hkv, D] each).
cudaError_t launch_gather(const Shape &s, const void *kv_layer, const int32_t *pages, int num_tokens, void *k_out,
                          void *v_out, cudaStream_t st);

// Self-test of the device error path (pkv_selftest_wait_timeout).
cudaError_t launch_selftest_wait(const Plan &p, void *ws, uint32_t polls, cudaStream_t st);

// File-scope device scratch used by pkv_run_decode_static (see decode.cu).
size_t static_scratch_bytes();
cudaError_t static_scratch(void **ptr);

}  // namespace pkv

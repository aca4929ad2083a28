// Prefill kernel instances for paged plans with pages below 8 slots (cp.async gather
// producers); kept apart from the TMA instances so that the two compile in parallel.
#include "prefill_kernel.cuh"

namespace pkv {

cudaError_t launch_prefill_gather(int head_dim, int group, const CUtensorMap &tkv, const CUtensorMap &tv,
                                  const CUtensorMap &tq, const dev::PrefillArgs &a, int grid, size_t smem,
                                  cudaStream_t st) {
    cudaError_t e = cudaErrorInvalidValue;
#define PKV_PF(DD, GG) \
    if (head_dim == DD && group == GG) e = launch_prefill_t<DD, GG, true>(tkv, tv, tq, a, grid, smem, st);
    PKV_FOR_EACH_HEAD_DIM_AND_GROUP(PKV_PF)
#undef PKV_PF
    return e;
}

}  // namespace pkv

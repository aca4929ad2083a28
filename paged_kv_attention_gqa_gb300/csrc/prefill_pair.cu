// Instances of the two-query-tile prefill kernel (prefill_pair.cuh) for head_dim 64 and 128
// and every group size, compiled in their own translation unit.
#include "launch.h"
#include "prefill_pair.cuh"

namespace pkv {

size_t prefill_pair_smem_bytes(int head_dim) {
    return 1024 + (head_dim == 64 ? dev::PpSmem<64>::BYTES : dev::PpSmem<128>::BYTES);
}
static_assert(1024 + dev::PpSmem<128>::BYTES <= 227 * 1024, "the paired prefill fits shared memory");
static_assert(1024 + dev::PpSmem<64>::BYTES > 228 * 1024 / 2, "one paired prefill CTA per SM (512 TMEM columns)");

template <int D, int G>
static cudaError_t launch_pair_t(const CUtensorMap &tkv, const CUtensorMap &tv, const CUtensorMap &tq,
                                 const dev::PrefillArgs &a, int grid, cudaStream_t st) {
    auto fn = dev::prefill_pair_kernel<D, G>;
    const size_t smem = prefill_pair_smem_bytes(D);
    cudaError_t e = set_smem_limit((const void *)fn, smem, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(fn, dim3(grid), dim3(dev::kPpThreads), smem, st, tkv, tv, tq, a);
}

cudaError_t launch_prefill_pair(int head_dim, int group, const CUtensorMap &tkv, const CUtensorMap &tv,
                                const CUtensorMap &tq, const dev::PrefillArgs &a, int grid, cudaStream_t st) {
    cudaError_t e = cudaErrorInvalidValue;
#define PKV_PP(DD, GG) \
    if (head_dim == DD && group == GG) e = launch_pair_t<DD, GG>(tkv, tv, tq, a, grid, st);
    PKV_FOR_EACH_GROUP(PKV_PP, 64)
    PKV_FOR_EACH_GROUP(PKV_PP, 128)
#undef PKV_PP
    return e;
}

}  // namespace pkv

// Instances of the head_dim-256 prefill kernel (prefill_wide.cuh) for every group size,
// compiled in their own translation unit.
#include "launch.h"
#include "prefill_wide.cuh"

namespace pkv {

static constexpr size_t kWideSmem = 1024 + dev::PwSmem::BYTES;
static_assert(kWideSmem <= 227 * 1024, "the head_dim-256 prefill fits shared memory");
static_assert(kWideSmem > 228 * 1024 / 2, "one head_dim-256 prefill CTA per SM (512 TMEM columns)");

template <int G>
static cudaError_t launch_wide_t(const CUtensorMap &tkv, const CUtensorMap &tv, const CUtensorMap &tq,
                                 const dev::PrefillArgs &a, int grid, cudaStream_t st) {
    auto fn = dev::prefill_wide_kernel<G>;
    cudaError_t e = set_smem_limit((const void *)fn, kWideSmem, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(fn, dim3(grid), dim3(dev::kPwThreads), kWideSmem, st, tkv, tv, tq, a);
}

cudaError_t launch_prefill_wide(int group, const CUtensorMap &tkv, const CUtensorMap &tv, const CUtensorMap &tq,
                                const dev::PrefillArgs &a, int grid, cudaStream_t st) {
    cudaError_t e = cudaErrorInvalidValue;
#define PKV_PW(DD, GG) \
    if (group == GG) e = launch_wide_t<GG>(tkv, tv, tq, a, grid, st);
    PKV_FOR_EACH_GROUP(PKV_PW, 256)
#undef PKV_PW
    return e;
}

}  // namespace pkv

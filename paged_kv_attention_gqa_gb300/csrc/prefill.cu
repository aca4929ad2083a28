// Ragged paged prefill launcher (FlashInferPrefillWrapper.run, FlashInferMixedWrapper's
// prefill pass, DenseAttentionManager): head_dim 64 / 128 with K / V by TMA go to the
// two-query-tile kernel (prefill_pair.cuh), head_dim 256 by TMA to prefill_wide.cuh, pages
// below 8 slots to the cp.async-gather instances of prefill_kernel.cuh (prefill_gather.cu).
#include "../../include/pkv.h"
#include "prefill_kernel.cuh"

namespace pkv {
size_t prefill_smem_bytes(const Shape &s) {
    // the cp.async-gather kernel: at least 100 KB, so that no more than two CTAs (2 x 256 TMEM
    // columns) share an SM; head_dim 256 (512 columns) takes more than half an SM's shared memory
    const size_t need = 1024 + (s.head_dim == 64    ? dev::PfSmem<64>::BYTES
                                : s.head_dim == 128 ? dev::PfSmem<128>::BYTES
                                                    : dev::PfSmem<256>::BYTES);
    return need < 100 * 1024 ? 100 * 1024 : need;
}
static_assert(1024 + dev::PfSmem<256>::BYTES > 228 * 1024 / 2, "one head_dim-256 gather-prefill CTA per SM");
static_assert(1024 + dev::PfSmem<256>::BYTES <= 227 * 1024, "the head_dim-256 gather prefill fits shared memory");

cudaError_t launch_prefill(const Shape &s, const Plan &p, const CUtensorMap &tm_kv, const CUtensorMap &tm_v,
                           const CUtensorMap &tm_q, const void *kv_layer, void *ws, void *out, float *lse,
                           cudaStream_t st) {
    const int grid = s.graph_static ? static_counts(s, p.mode).pf_tiles : p.pf_tiles;
    if (grid == 0) return cudaSuccess;
    uint8_t *w = static_cast<uint8_t *>(ws);
    dev::PrefillArgs a;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.tiles = reinterpret_cast<const PrefillTile *>(w + p.lay.pf_tiles);
    a.pages = reinterpret_cast<const int32_t *>(w + p.lay.pf_pages);
    a.hdr = reinterpret_cast<PlanHeader *>(w + p.lay.err);
    a.kv_layer = static_cast<const uint8_t *>(kv_layer);
    a.num_qo_heads = s.num_qo_heads;
    a.num_kv_heads = s.num_kv_heads;
    a.page_size = s.page_size;
    a.page_shift = s.page_shift();
    a.box_rows = s.pf_box_rows();
    a.gather = s.pf_gather() ? 1 : 0;
    if (a.gather && p.mode != PKV_MODE_DENSE && !kv_layer) return cudaErrorInvalidValue;
    // a row coordinate past the tensor (TMA fills zeros); dense plans never use it
    a.oob_row = s.num_cache_pages * 2 * s.page_size;
    const int g = s.group();
    if (s.pf_pair(p.mode == PKV_MODE_DENSE))  // two query tiles per CTA (prefill_pair.cuh)
        return launch_prefill_pair(s.head_dim, g, tm_kv, tm_v, tm_q, a, grid, st);
    if (a.gather && p.mode != PKV_MODE_DENSE)  // dense plans always read K / V by TMA
        return launch_prefill_gather(s.head_dim, g, tm_kv, tm_v, tm_q, a, grid, prefill_smem_bytes(s), st);
    if (s.head_dim == 256)  // 128-key tiles, two S buffers (prefill_wide.cuh)
        return launch_prefill_wide(g, tm_kv, tm_v, tm_q, a, grid, st);
    return cudaErrorInvalidValue;  // every shape pkv_create accepts is taken above
}

}  // namespace pkv

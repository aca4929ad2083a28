// Batched paged decode with split-KV, the split-KV merge, and the last-page append.
//
// Decode (FlashInferDecodeWrapper.run; mstar.engine.resources.attn.wrappers): every row
// has one query token; q head h attends, through kv head h / g, to the row's visible
// positions [lo, L-1] (lo = max(0, L-1-window_left), or 0), o = softmax(sm_scale q K^T) V,
// lse = ln sum exp.
//
// Design for GB300:
//  * A persistent grid of one CTA per SM (x: runs of pages, y: groups of kv heads when a
//    CTA cannot hold all of them).  The planner hands each CTA a contiguous run of the
//    batch's visible pages (balanced to +-1 page); a row cut by a CTA boundary writes an
//    fp32 partial (o normalised, lse) into the workspace, merged afterwards.
//  * The slots of one page are contiguous for ALL kv heads (K: page_size x Hkv x D, then
//    V), so a CTA streams 16-key chunks of its heads: one producer thread issues TMA
//    boxes (64-column halves, 128-byte swizzle) into a ring of stages, completion on an
//    mbarrier; consumers release a stage through a second mbarrier.  A chunk is one box
//    per 64-column half holding its K rows then its V rows (page size 16: a whole page),
//    one box of K and one of V (page size > 16) or two of each (8); pages below 8 slots
//    are copied by the whole producer warp with 16-byte cp.async into the same layout.
//  * One consumer warp per kv head.  The g query heads of the group are the M dimension of
//    a 16x8x16 bf16 tensor-core MMA (padded to 16 rows); keys are N for QK^T and K for PV.
//    Online softmax in the exp2 domain with quad shuffles.
//  * Slots of a chunk past the piece's end are zeroed in shared memory before PV (their
//    scores are masked to -inf; zeroing V keeps 0 * NaN out of the MMA).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"
#include "plan.h"
#include "ptx.cuh"

namespace pkv {
namespace dev {

struct DecodeArgs {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    float *lse;
    const DecodeTile *tiles;
    const int32_t *cta_ptr;
    const int32_t *cta_rows;  // [CTA][kDecodeHeadChunks]: cache rows of its first chunks, -1 past its end
    const int32_t *pages;
    float *part_o;
    float *part_lse;
    PlanHeader *hdr;  // per-plan values (error word, sm_scale) in the workspace
    // fused append (null when the plan's tokens were appended by append_kernel): the new
    // tokens' K / V rows, the layer slice and each token's slot row in it
    const uint4 *k_new;
    const uint4 *v_new;
    uint4 *kv_layer;
    const int32_t *append_rows;
    int num_qo_heads;
    int num_kv_heads;
    int heads;         // kv heads per CTA; blockIdx.y selects the group
    int page_size;
    int page_shift;    // log2 page_size
    int box_rows;      // rows per head of one TMA box
    int kpb_shift;     // log2 of the keys one box holds per head
    int gather;        // 1: pages below 8 slots, copied by the producer warps (cp.async)
    int kv_in_box;     // 1: one box holds a chunk's K rows, then its V rows (page size 16)
    int producers;     // producer warps (warps heads .. heads + producers - 1)
    int box_stride;    // bytes between boxes in a stage
    int stages;
    uint32_t stage_bytes;
};

constexpr float kLn2 = 0.6931471805599453f;
constexpr int kDecodeMaxStages = 16;
static_assert(kDecodeHeadChunks == 4, "a CTA's head rows are read as one int4");

// C consecutive fp32 columns of a partial (C = 2, 4 or 8; 8- or 16-byte aligned), read at L2.
template <int C>
__device__ __forceinline__ void load_cols(float (&x)[C], const float *src) {
    if constexpr (C == 2) {
        const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
        x[0] = t.x;
        x[1] = t.y;
    } else {
#pragma unroll
        for (int i = 0; i < C / 4; ++i) {
            const float4 t = __ldcg(reinterpret_cast<const float4 *>(src) + i);
            x[4 * i] = t.x;
            x[4 * i + 1] = t.y;
            x[4 * i + 2] = t.z;
            x[4 * i + 3] = t.w;
        }
    }
}

// Byte offset, inside one 64-column half of a stage, of key `tok` (0..15) of local head
// `hk`, and its 128-byte swizzle phase (`vrow`: a row offset inside the box, 16 for V rows when a
// box holds a chunk's K and V rows, else 0).
struct RowAddr {
    uint32_t off;
    uint32_t phase;
};
__device__ __forceinline__ RowAddr key_row(const DecodeArgs &a, int hk, int tok, int vrow) {
    const int b = tok >> a.kpb_shift;
    const int row = hk * a.box_rows + vrow + (tok & ((1 << a.kpb_shift) - 1));
    return RowAddr{(uint32_t)(b * a.box_stride + row * 128), (uint32_t)(row & 7)};
}

// SMALL: pages below 16 slots (several TMA boxes per chunk at 8 slots, cp.async producer
// warps below 8); otherwise one box of K and one of V per chunk.
template <int D, int G, bool SMALL>
__global__ void __launch_bounds__((D > 128 ? 4 + (SMALL ? 2 : 1) : 8 + (SMALL ? 4 : 1)) * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
    constexpr int KS = D / 16;  // k-steps of QK^T
    constexpr int NT = D / 8;   // 8-wide output column tiles
    constexpr int HALVES = D / 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.stages * a.stage_bytes);
    uint64_t *empty = full + a.stages;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int Hc = a.heads;
    const int hg = blockIdx.y;
    const int P = a.page_size;
    const int t_begin = a.cta_ptr[blockIdx.x];
    const int t_end = a.cta_ptr[blockIdx.x + 1];
    // The plan's arrays come from the host's copy, never from a kernel, so they are read before
    // waiting for the previous kernel: the TMA producer's first chunks need only their cache
    // rows, which the planner stored beside the CTA's tile range (no dependent tile and
    // page-id loads before the first copies), and its first tile is loaded meanwhile.
    // Inputs and the cache may come from the previous kernel (an append, a merge) and are read
    // only after the wait.
    int4 head_rows = make_int4(-1, -1, -1, -1);
    if (!SMALL && warp == Hc && lane == 0)
        head_rows = reinterpret_cast<const int4 *>(a.cta_rows)[blockIdx.x];
    if (t_begin >= t_end) return;  // an idle CTA of a launch at the handle's maxima
    int *err = &a.hdr->err;
    const float scale_log2 = a.hdr->scale_log2;
    // stage layout: [K or V][64-column half][box]; with K and V in one box: [half][box]
    const int kpb = 1 << a.kpb_shift;
    const int nb = kDecodeKeysPerStage / kpb;
    const uint32_t half_stride = (uint32_t)nb * a.box_stride;
    const uint32_t v_region = a.kv_in_box ? 0u : HALVES * half_stride;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], SMALL && a.gather ? 32 * a.producers : 1);  // gather: one per producer lane
            mbar_init(&empty[s], Hc);
        }
        fence_barrier_init();
        prefetch_tmap(&tmap);
    }
    __syncthreads();
    DecodeTile first_tile{};
    if (!SMALL && warp == Hc && lane == 0) first_tile = a.tiles[t_begin];
    griddep_wait();
    griddep_launch();

    if (SMALL && a.gather && warp >= Hc) {
        // ---------------- producers, pages below 8 slots: cp.async by `producers` warps ---
        // (warp pw copies heads pw, pw + producers, ... of every chunk)
        const int pw = warp - Hc;
        // Lane = (key slot, 16-byte column chunk c), c fastest so that consecutive lanes copy
        // consecutive bytes of one cache row; a warp instruction covers KPI keys.  The slot
        // rows of the lane's keys are looked up once per chunk; keys past the piece's end
        // read nothing and land as zeros.
        constexpr int CH = D / 8;                       // 16-byte chunks per head row
        constexpr int KPI = 32 / CH;                    // keys per warp instruction
        constexpr int NI = kDecodeKeysPerStage / KPI;   // key iterations per chunk
        const int c = lane % CH, kslot = lane / CH;
        const size_t row_bytes = (size_t)a.num_kv_heads * D * 2;  // one slot row, all heads
        const uint8_t *base = reinterpret_cast<const uint8_t *>(a.kv_layer) + (size_t)hg * Hc * D * 2 + c * 16;
        uint32_t it = 0;
        bool ok = true;
        for (int ti = t_begin; ti < t_end && ok; ++ti) {
            const DecodeTile t = a.tiles[ti];
            const ChunkRange cr = chunk_range(t, P);
            for (int k = cr.k0; k < cr.nk; ++k, ++it) {
                const int s = it % a.stages;
                const uint32_t use = it / a.stages;
                const int pos0 = cr.base + k * kDecodeKeysPerStage;
                int row[NI];
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const int pos = pos0 + kslot + KPI * i;
                    row[i] = pos < cr.end ? a.pages[t.kv_base + (pos >> a.page_shift)] * 2 * P + (pos & (P - 1)) : -1;
                }
                // every lane waits on the barrier itself (they wake together); the vote keeps
                // the warp on one path if a wait gives up
                const bool w = use == 0 || mbar_wait(&empty[s], (use - 1) & 1, err, kErrWaitEmpty);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
                const uint32_t st = smem_u32(smem + (size_t)s * a.stage_bytes) + (c >> 3) * half_stride;
                for (int kv = 0; kv < 2; ++kv)
                    for (int hh = pw; hh < Hc; hh += a.producers) {
                        const uint8_t *src_h = base + (size_t)hh * D * 2 + (size_t)kv * P * row_bytes;
                        const uint32_t dst_h = st + kv * HALVES * half_stride + hh * kDecodeKeysPerStage * 128;
#pragma unroll
                        for (int i = 0; i < NI; ++i) {
                            const int key = kslot + KPI * i;
                            const bool valid = row[i] >= 0;
                            cp_async16(dst_h + key * 128 + (((c & 7) ^ (key & 7)) << 4),
                                       valid ? src_h + (size_t)row[i] * row_bytes : base, valid ? 16u : 0u);
                        }
                    }
                cp_async_mbar_arrive(&full[s]);
            }
        }
        cp_async_wait_all();
        // Drain: every stage issued must have been consumed before the CTA exits.
        if (pw == 0 && lane == 0) {
            const uint32_t issued = it;
            for (uint32_t d = issued > (uint32_t)a.stages ? issued - a.stages : 0; d < issued; ++d) {
                const int s = d % a.stages;
                if (!mbar_wait(&empty[s], (d / a.stages) & 1, err, kErrWaitDrain)) break;
            }
        }
        return;
    }
    if (warp >= Hc) {
        if (warp > Hc) return;
        // ---------------- producer ----------------
        if (lane == 0) {
            const int nkv = a.kv_in_box ? 1 : 2;  // boxes per 64-column half
            const uint32_t box_bytes = (uint32_t)a.box_rows * Hc * 128;
            uint32_t it = 0;
            if (!SMALL) {
                // the first chunks into the empty stages, from the planner's rows
                const int hr[kDecodeHeadChunks] = {head_rows.x, head_rows.y, head_rows.z, head_rows.w};
                int nhead = 0;
#pragma unroll
                for (int i = 0; i < kDecodeHeadChunks; ++i)
                    if (nhead == i && i < a.stages && hr[i] >= 0) {
                        uint8_t *st = smem + (size_t)i * a.stage_bytes;
                        mbar_arrive_expect_tx(&full[i], (uint32_t)(nkv * HALVES) * box_bytes);
                        for (int kv = 0; kv < nkv; ++kv)
#pragma unroll
                            for (int h = 0; h < HALVES; ++h)
                                tma_load_3d(st + (kv * HALVES + h) * half_stride, &tmap, &full[i], h * 64,
                                            hr[i] + kv * P, hg * Hc);
                        nhead = i + 1;
                    }
                // then one box (of K and of V) per chunk: its page id is loaded after the slot frees
                for (int ti = t_begin; ti < t_end; ++ti) {
                    const DecodeTile t = ti == t_begin ? first_tile : a.tiles[ti];
                    const ChunkRange cr = chunk_range(t, P);
                    bool ok = true;
                    for (int k = cr.k0; k < cr.nk; ++k, ++it) {
                        if (it < (uint32_t)nhead) continue;  // issued above
                        const int s = it % a.stages;
                        const uint32_t use = it / a.stages;
                        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, err, kErrWaitEmpty)) {
                            ok = false;
                            break;
                        }
                        const int pos0 = cr.base + k * kDecodeKeysPerStage;
                        const int row = a.pages[t.kv_base + (pos0 >> a.page_shift)] * 2 * P + (pos0 & (P - 1));
                        uint8_t *st = smem + (size_t)s * a.stage_bytes;
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(nkv * HALVES) * box_bytes);
                        for (int kv = 0; kv < nkv; ++kv)
#pragma unroll
                            for (int h = 0; h < HALVES; ++h)
                                tma_load_3d(st + (kv * HALVES + h) * half_stride, &tmap, &full[s], h * 64,
                                            row + kv * P, hg * Hc);
                    }
                    if (!ok) break;
                }
            } else {
                // several boxes per chunk (pages below 16 slots): once the slot frees, all the
                // chunk's page ids (up to 16 at page size 1) are loaded together, then its boxes
                // are issued (not one dependent load per box)
                for (int ti = t_begin; ti < t_end; ++ti) {
                    const DecodeTile t = a.tiles[ti];
                    const ChunkRange cr = chunk_range(t, P);
                    bool ok = true;
                    for (int k = cr.k0; k < cr.nk; ++k, ++it) {
                        const int s = it % a.stages;
                        const uint32_t use = it / a.stages;
                        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, err, kErrWaitEmpty)) {
                            ok = false;
                            break;
                        }
                        const int pos0 = cr.base + k * kDecodeKeysPerStage;
                        const int nbox = min(nb, (cr.end - pos0 + kpb - 1) / kpb);
                        int page[kDecodeKeysPerStage];
#pragma unroll
                        for (int b = 0; b < kDecodeKeysPerStage; ++b)
                            if (b < nbox) page[b] = a.pages[t.kv_base + ((pos0 + b * kpb) >> a.page_shift)];
                        uint8_t *st = smem + (size_t)s * a.stage_bytes;
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(nbox * nkv * HALVES) * box_bytes);
#pragma unroll
                        for (int b = 0; b < kDecodeKeysPerStage; ++b)
                            if (b < nbox) {
                                const int row = page[b] * 2 * P + ((pos0 + b * kpb) & (P - 1));
                                for (int kv = 0; kv < nkv; ++kv)
#pragma unroll
                                    for (int h = 0; h < HALVES; ++h)
                                        tma_load_3d(st + (kv * HALVES + h) * half_stride + b * a.box_stride, &tmap,
                                                    &full[s], h * 64, row + kv * P, hg * Hc);
                            }
                    }
                    if (!ok) break;
                }
            }
            // Drain: every stage issued must have been consumed before the CTA exits.
            const uint32_t issued = it;
            for (uint32_t d = issued > (uint32_t)a.stages ? issued - a.stages : 0; d < issued; ++d) {
                const int s = d % a.stages;
                if (!mbar_wait(&empty[s], (d / a.stages) & 1, err, kErrWaitDrain)) break;
            }
        }
        return;
    }
    if (warp >= Hc) return;

// ---------------- consumers: warp = kv head ----------------
    const int hk = warp;               // kv head within the CTA's group (its row in a box)
    const int hkg = hg * Hc + warp;    // kv head
    const int gid = lane >> 2;   // row of the MMA fragment (query head within the group)
    const int tid4 = lane & 3;
    const int Hq = a.num_qo_heads;
    // ldmatrix lane roles: the key row each lane addresses and its 16-byte column chunk
    const int k_tok = (lane & 7) + ((lane >> 4) << 3);
    const int k_chk = (lane >> 3) & 1;
    const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_chk = lane >> 4;
    const int vrow = a.kv_in_box ? kDecodeKeysPerStage : 0;  // V rows after K rows in one box
    const RowAddr ka = key_row(a, hk, k_tok, 0);
    RowAddr va = key_row(a, hk, v_tok, vrow);
    va.off += v_region;

    uint32_t it = 0;
    bool ok = true;
    for (int ti = t_begin; ti < t_end; ++ti) {
        const DecodeTile t = a.tiles[ti];
        const ChunkRange cr = chunk_range(t, P);
        // Query fragments: rows = the g heads of this kv head (rows >= G are zero).
        uint32_t qa[KS][4];
        {
            const __nv_bfloat16 *qrow = a.q + ((size_t)t.q_token * Hq + (size_t)hkg * G) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int c0 = ks * 16 + tid4 * 2;
                qa[ks][0] = gid < G ? *reinterpret_cast<const uint32_t *>(qrow + (size_t)gid * D + c0) : 0u;
                qa[ks][2] = gid < G ? *reinterpret_cast<const uint32_t *>(qrow + (size_t)gid * D + c0 + 8) : 0u;
                qa[ks][1] = gid + 8 < G ? *reinterpret_cast<const uint32_t *>(qrow + (size_t)(gid + 8) * D + c0) : 0u;
                qa[ks][3] =
                    gid + 8 < G ? *reinterpret_cast<const uint32_t *>(qrow + (size_t)(gid + 8) * D + c0 + 8) : 0u;
            }
        }
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        for (int k = cr.k0; k < cr.nk; ++k, ++it) {
            const int s = it % a.stages;
            // a wait that gives up clears ok; the warp still walks its tiles so that the
            // consumer warps keep meeting at their named barriers (no time limit there)
            ok = ok && mbar_wait(&full[s], (it / a.stages) & 1, err, kErrWaitFull);
            uint8_t *st = smem + (size_t)s * a.stage_bytes;
            const uint32_t sbase = smem_u32(st);
            const int pos0 = cr.base + k * kDecodeKeysPerStage;
            const int nvalid = cr.end - pos0;  // keys of this chunk inside the piece
            // fused append: the row's new token (position L-1, in this piece's last chunk)
            // replaces the slot's stale rows in the stage and is stored to the cache; only
            // this CTA reads this head of that page, and its TMA read came first
            const bool patch = a.k_new && t.append_token >= 0 && t.length - 1 - pos0 < kDecodeKeysPerStage;
            if (patch) {
                constexpr int CH = D / 8;  // 16-byte chunks per row
                const int tok = t.length - 1 - pos0;
                const size_t src = ((size_t)t.append_token * a.num_kv_heads + hkg) * CH;
                const size_t row = (size_t)a.append_rows[t.append_token];
                for (int i = lane; i < 2 * CH; i += 32) {
                    const int kv = i / CH, c = i % CH;
                    const uint4 val = (kv ? a.v_new : a.k_new)[src + c];
                    const RowAddr r = key_row(a, hk, tok, kv ? vrow : 0);
                    *reinterpret_cast<uint4 *>(st + (kv ? v_region : 0u) + (c >> 3) * half_stride + r.off +
                                               (((c & 7) ^ r.phase) << 4)) = val;
                    a.kv_layer[((row + (kv ? P : 0)) * a.num_kv_heads + hkg) * CH + c] = val;
                }
                __syncwarp();
            }
            if (nvalid < kDecodeKeysPerStage) {
                // zero this head's V rows past the piece's end (stale, unloaded or poisoned)
                const int nz = (kDecodeKeysPerStage - nvalid) * (D / 8);
                for (int i = lane; i < nz; i += 32) {
                    const RowAddr z = key_row(a, hk, nvalid + i / (D / 8), vrow);
                    const int chunk = i % (D / 8);
                    *reinterpret_cast<uint4 *>(st + v_region + (chunk >> 3) * half_stride + z.off +
                                               (((chunk & 7) ^ z.phase) << 4)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // S = Q K^T over the chunk's 16 keys: two n-tiles of 8 keys.
            float sc[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int chunk = ks * 2 + k_chk;
                const uint32_t addr = sbase + (chunk >> 3) * half_stride + ka.off + (((chunk & 7) ^ ka.phase) << 4);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(addr, b0, b1, b2, b3);
                mma_bf16_16816(sc[0], qa[ks], b0, b1);
                mma_bf16_16816(sc[1], qa[ks], b2, b3);
            }
            // mask + online softmax (exp2 domain)
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int pos = pos0 + n * 8 + tid4 * 2 + e;
                    const bool vis = pos >= t.lo && pos < cr.end;
                    sc[n][e] = vis ? sc[n][e] * scale_log2 : -INFINITY;
                    sc[n][e + 2] = vis ? sc[n][e + 2] * scale_log2 : -INFINITY;
                    mx0 = fmaxf(mx0, sc[n][e]);
                    mx1 = fmaxf(mx1, sc[n][e + 2]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = fast_exp2(m0 - ref0), al1 = fast_exp2(m1 - ref1);
            m0 = mn0;
            m1 = mn1;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    sc[n][e] = fast_exp2(sc[n][e] - ref0);
                    sc[n][e + 2] = fast_exp2(sc[n][e + 2] - ref1);
                    ps0 += sc[n][e];
                    ps1 += sc[n][e + 2];
                }
            l0 = l0 * al0 + ps0;
            l1 = l1 * al1 + ps1;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                acc[n][0] *= al0;
                acc[n][1] *= al0;
                acc[n][2] *= al1;
                acc[n][3] *= al1;
            }
            uint32_t pa[4];
            pa[0] = pack_bf16(sc[0][0], sc[0][1]);
            pa[1] = pack_bf16(sc[0][2], sc[0][3]);
            pa[2] = pack_bf16(sc[1][0], sc[1][1]);
            pa[3] = pack_bf16(sc[1][2], sc[1][3]);
            // O += P V
#pragma unroll
            for (int dj = 0; dj < D / 16; ++dj) {
                const int chunk = dj * 2 + v_chk;
                const uint32_t addr = sbase + (chunk >> 3) * half_stride + va.off + (((chunk & 7) ^ va.phase) << 4);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                mma_bf16_16816(acc[2 * dj], pa, b0, b1);
                mma_bf16_16816(acc[2 * dj + 1], pa, b2, b3);
            }
            if (nvalid < kDecodeKeysPerStage || patch) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // finalise the piece
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        const float inv0 = 1.f / l0, inv1 = 1.f / l1;
        const float lse0 = (m0 + __log2f(l0)) * kLn2;
        const float lse1 = (m1 + __log2f(l1)) * kLn2;
        const int h0 = hkg * G + gid, h1 = hkg * G + gid + 8;
        if (t.partial < 0) {
            if (t.out_token >= 0) {
                __nv_bfloat16 *o = a.out + (size_t)t.out_token * Hq * D;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int c = n * 8 + tid4 * 2;
                    if (gid < G)
                        *reinterpret_cast<uint32_t *>(o + (size_t)h0 * D + c) =
                            pack_bf16(acc[n][0] * inv0, acc[n][1] * inv0);
                    if (gid + 8 < G)
                        *reinterpret_cast<uint32_t *>(o + (size_t)h1 * D + c) =
                            pack_bf16(acc[n][2] * inv1, acc[n][3] * inv1);
                }
                if (a.lse && tid4 == 0) {
                    if (gid < G) a.lse[(size_t)t.out_token * Hq + h0] = lse0;
                    if (gid + 8 < G) a.lse[(size_t)t.out_token * Hq + h1] = lse1;
                }
            }
        } else {
            float *po = a.part_o + (size_t)t.partial * Hq * D;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int c = n * 8 + tid4 * 2;
                if (gid < G)
                    *reinterpret_cast<float2 *>(po + (size_t)h0 * D + c) = make_float2(acc[n][0] * inv0, acc[n][1] * inv0);
                if (gid + 8 < G)
                    *reinterpret_cast<float2 *>(po + (size_t)h1 * D + c) = make_float2(acc[n][2] * inv1, acc[n][3] * inv1);
            }
            if (tid4 == 0) {
                if (gid < G) a.part_lse[(size_t)t.partial * Hq + h0] = lse0;
                if (gid + 8 < G) a.part_lse[(size_t)t.partial * Hq + h1] = lse1;
            }
        }
    }
}

// Merge the split-KV partials of each cut row after the decode kernel: with
// w_j = exp(lse_j - max lse), o = sum_j w_j o_j / sum_j w_j and
// lse = max lse + ln sum_j w_j.  One warp per (cut row, q head), eight to a CTA: lane j
// holds piece j's lse, and every lane requests its D/32 columns of the row's first B pieces
// together with the lse values, before the weights are known, so that a row of up to B pieces
// costs one round trip to L2 after its MergeRow; longer rows take one more per B pieces (each
// batch's loads issued together).  B pieces hold B * D/32 registers: the small instance
// (64) keeps enough warps resident for the many rows of a batch, the large one (128) takes
// the rows of many pieces of long contexts in one batch.
constexpr int kMergeWarps = 8;
constexpr int merge_batch(int D, bool large) {
    return (large ? 128 : 64) / (D / 32) < 32 ? (large ? 128 : 64) / (D / 32) : 32;
}

template <int D, int B>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const PlanHeader *hdr, const MergeRow *rows,
                                                                 const float *part_o, const float *part_lse,
                                                                 __nv_bfloat16 *out, float *lse, int Hq) {
    constexpr int C = D / 32;  // columns per lane: 2, 4 or 8
    static_assert(B >= 1 && B <= 32, "a batch's weights come from one lane each");
    const int lane = threadIdx.x & 31;
    const long long u = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    const int m = (int)(u / Hq), h = (int)(u % Hq);
    // the plan's own values (copied before the decode launch) are read before waiting for the
    // decode kernel; the partials it writes only after
    const bool active = m < hdr->num_merge;
    MergeRow mr{};
    if (active) mr = rows[m];
    griddep_wait();
    griddep_launch();
    if (!active || mr.out_token < 0) return;
    const int count = mr.count;
    const float *lse_of = part_lse + (size_t)mr.first * Hq + h;              // piece j at lse_of[j * Hq]
    const float *o_of = part_o + ((size_t)mr.first * Hq + h) * D + lane * C;  // piece j at o_of[j * Hq * D]
    auto load = [&](float (&dst)[C], int j) { load_cols<C>(dst, o_of + (size_t)j * Hq * D); };
    const float lj = lane < count ? __ldcg(lse_of + (size_t)lane * Hq) : -INFINITY;
    float x[B][C];
#pragma unroll
    for (int j = 0; j < B; ++j)
        if (j < count) load(x[j], j);
    // M = max_j lse_j and sum_j w_j over the warp (pieces past 32: one more lse each per lane)
    float M = lj;
    for (int j = lane + 32; j < count; j += 32) M = fmaxf(M, __ldcg(lse_of + (size_t)j * Hq));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wl = lane < count ? __expf(lj - M) : 0.f;
    float sum = wl;
    for (int j = lane + 32; j < count; j += 32) sum += __expf(__ldcg(lse_of + (size_t)j * Hq) - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    for (int j0 = 0;;) {
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const float w0 = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);
            if (j0 + j < count) {
                const float w = j0 + j < 32 ? w0 : __expf(__ldcg(lse_of + (size_t)(j0 + j) * Hq) - M);
#pragma unroll
                for (int c = 0; c < C; ++c) acc[c] += w * x[j][c];
            }
        }
        j0 += B;
        if (j0 >= count) break;
#pragma unroll
        for (int j = 0; j < B; ++j)  // the next batch (rows of many pieces)
            if (j0 + j < count) load(x[j], j0 + j);
    }
    const float inv = 1.f / sum;
    uint32_t packed[C / 2];
#pragma unroll
    for (int c = 0; c < C; c += 2) packed[c / 2] = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
    __nv_bfloat16 *dst = out + ((size_t)mr.out_token * Hq + h) * D + lane * C;
    if constexpr (C == 2) {
        *reinterpret_cast<uint32_t *>(dst) = packed[0];
    } else if constexpr (C == 4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
    } else {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    if (lse && lane == 0) lse[(size_t)mr.out_token * Hq + h] = M + __logf(sum);
}


// Last-page append: one thread per 16-byte chunk of a new token's K and V rows (num_kv_heads
// x D bf16 each), all chunks in flight at once, written to slot rows[t] of the layer slice
// viewed as [pages * 2 * page_size] rows (V rows page_size further).
__global__ void __launch_bounds__(256) append_kernel(const PlanHeader *hdr, const uint4 *k, const uint4 *v, uint4 *cache,
                                                     const int32_t *rows, int vec_per_token, int page_size) {
    griddep_wait();
    griddep_launch();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int t = (int)(i / vec_per_token), c = (int)(i % vec_per_token);
    if (t >= hdr->num_append) return;
    const size_t row = (size_t)rows[t];
    const uint4 kk = k[(size_t)t * vec_per_token + c];
    const uint4 vv = v[(size_t)t * vec_per_token + c];
    cache[row * vec_per_token + c] = kk;
    cache[(row + page_size) * vec_per_token + c] = vv;
}

// Last-page append straight from the DEVICE index arrays (no plan): one thread per 16-byte
// chunk of a new token's K and V rows.  Token t belongs to the row r with qo_indptr[r] <=
// t < qo_indptr[r+1] (row t when qo_indptr is null: one token per row), sits at position
// p = L_r - n_r + (t - qo_indptr[r]) of that row and lands in page
// kv_indices[kv_indptr[r] + p / page_size] at slot p % page_size.  The arrays were not seen
// by the host, so every index is checked before it is used: a token whose row arrays are
// inconsistent (non-monotone offsets, a fill outside 1..page_size, a position outside the
// row, a page id outside the cache) is not written, and nothing is read or written out of
// bounds.
__global__ void __launch_bounds__(256)
    append_indexed_kernel(const uint4 *k, const uint4 *v, uint4 *cache, const int32_t *qo_indptr,
                          const int32_t *kv_indptr, const int32_t *kv_indices, const int32_t *last_page_len, int batch,
                          int num_tokens, int vec_per_token, int page_size, int page_shift, int num_cache_pages) {
    griddep_wait();
    griddep_launch();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int t = (int)(i / vec_per_token), c = (int)(i % vec_per_token);
    if (t >= num_tokens) return;
    int r, n, first;
    if (qo_indptr) {
        if (t >= __ldg(qo_indptr + batch)) return;
        int lo = 0, hi = batch - 1;  // the last row whose offset is <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(qo_indptr + mid) <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        r = lo;
        first = __ldg(qo_indptr + r);
        n = __ldg(qo_indptr + r + 1) - first;
        if (first > t || t >= first + n) return;
    } else {
        if (t >= batch) return;
        r = t;
        first = t;
        n = 1;
    }
    const int kb = __ldg(kv_indptr + r), ke = __ldg(kv_indptr + r + 1), nnz = __ldg(kv_indptr + batch);
    const int fill = __ldg(last_page_len + r);
    if (kb < 0 || ke <= kb || ke > nnz || fill < 1 || fill > page_size) return;
    const long long L = (long long)(ke - kb - 1) * page_size + fill;
    const long long p = L - n + (t - first);
    if (p < 0 || p >= L) return;
    const int page = __ldg(kv_indices + kb + (int)(p >> page_shift));
    if (page < 0 || page >= num_cache_pages) return;
    const size_t row = (size_t)page * 2 * page_size + (size_t)(p & (page_size - 1));
    const uint4 kk = k[(size_t)t * vec_per_token + c];
    const uint4 vv = v[(size_t)t * vec_per_token + c];
    cache[row * vec_per_token + c] = kk;
    cache[(row + page_size) * vec_per_token + c] = vv;
}

// Gather of a frozen prefix (DenseAttentionManager): one warp per position t copies
// K and V of slot t % page_size of page pages[t / page_size] to row t of k_out / v_out.
__global__ void __launch_bounds__(256) gather_kernel(const uint4 *cache, const int32_t *pages, int num_tokens,
                                                     int vec_per_token, int page_size, uint4 *k_out, uint4 *v_out) {
    griddep_wait();
    griddep_launch();
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= num_tokens) return;
    const size_t row = (size_t)pages[t / page_size] * 2 * page_size + t % page_size;
    const int lane = threadIdx.x & 31;
    const uint4 *ks = cache + row * vec_per_token;
    const uint4 *vs = cache + (row + page_size) * vec_per_token;
    uint4 *kd = k_out + (size_t)t * vec_per_token;
    uint4 *vd = v_out + (size_t)t * vec_per_token;
    for (int i = lane; i < vec_per_token; i += 32) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
}

// Self-test of the device error path: one thread waits, with `polls` polls, on an mbarrier
// nothing ever arrives on; the wait gives up, records kErrWaitSelfTest in the plan's error
// word and the kernel returns (no fault, no hang, the context stays usable).
__global__ void __launch_bounds__(32) selftest_wait_kernel(PlanHeader *hdr, uint32_t polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        mbar_wait(&bar, 0, &hdr->err, kErrWaitSelfTest, polls);
    }
}

}  // namespace dev

cudaError_t launch_selftest_wait(const Plan &p, void *ws, uint32_t polls, cudaStream_t st) {
    dev::selftest_wait_kernel<<<1, 32, 0, st>>>(
        reinterpret_cast<PlanHeader *>(static_cast<uint8_t *>(ws) + p.lay.err), polls);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// launchers

cudaError_t launch_gather(const Shape &s, const void *kv_layer, const int32_t *pages, int num_tokens, void *k_out,
                          void *v_out, cudaStream_t st) {
    if (num_tokens <= 0) return cudaSuccess;
    const int vec = s.num_kv_heads * s.head_dim * 2 / 16;
    const int wpb = 8;
    return launch_pdl(dev::gather_kernel, dim3((num_tokens + wpb - 1) / wpb), dim3(wpb * 32), 0, st,
                      static_cast<const uint4 *>(kv_layer), pages, num_tokens, vec, s.page_size,
                      static_cast<uint4 *>(k_out), static_cast<uint4 *>(v_out));
}

static uint32_t decode_stage_bytes(const Shape &s) { return s.dec_stage_bytes(); }

int decode_stages(const Shape &s) {
    const uint32_t sb = decode_stage_bytes(s);
    int st = (int)(kDecodeRingBytes / (uint32_t)s.dec_ctas_per_sm() / sb);
    return st < 2 ? 0 : (st > dev::kDecodeMaxStages ? dev::kDecodeMaxStages : st);
}

size_t decode_smem_bytes(const Shape &s) {
    return 1024 + (size_t)decode_stages(s) * decode_stage_bytes(s) + 2 * 8 * dev::kDecodeMaxStages + 16;
}

// Raise a kernel's dynamic shared-memory limit; skipped while `st` is being captured
// into a CUDA graph (a launch before the capture has set it already).
cudaError_t set_smem_limit(const void *fn, size_t smem, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int D, int G, bool SMALL>
static cudaError_t launch_decode_t(const CUtensorMap &tm, const dev::DecodeArgs &a, dim3 grid, int warps, size_t smem,
                                   cudaStream_t st) {
    auto fn = dev::decode_kernel<D, G, SMALL>;
    cudaError_t e = set_smem_limit((const void *)fn, smem, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(fn, grid, dim3(warps * 32), smem, st, tm, a);
}

cudaError_t launch_decode(const Shape &s, const Plan &p, const CUtensorMap &tm, void *ws, const void *q,
                          void *kv_layer, void *out, float *lse, cudaStream_t st, const void *k_new,
                          const void *v_new) {
    const StaticCounts sc = static_counts(s, p.mode);
    const int grid = s.graph_static ? sc.dec_ctas : p.dec_ctas;
    if (grid == 0) return cudaSuccess;
    uint8_t *w = static_cast<uint8_t *>(ws);
    dev::DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.tiles = reinterpret_cast<const DecodeTile *>(w + p.lay.dec_tiles);
    a.cta_ptr = reinterpret_cast<const int32_t *>(w + p.lay.dec_cta_ptr);
    a.cta_rows = reinterpret_cast<const int32_t *>(w + p.lay.dec_cta_rows);
    a.pages = reinterpret_cast<const int32_t *>(w + p.lay.dec_pages);
    a.part_o = reinterpret_cast<float *>(w + p.lay.part_o);
    a.part_lse = reinterpret_cast<float *>(w + p.lay.part_lse);
    a.hdr = reinterpret_cast<PlanHeader *>(w + p.lay.err);
    a.k_new = static_cast<const uint4 *>(k_new);
    a.v_new = static_cast<const uint4 *>(v_new);
    a.kv_layer = static_cast<uint4 *>(kv_layer);
    a.append_rows = reinterpret_cast<const int32_t *>(w + p.lay.append_rows);
    a.num_qo_heads = s.num_qo_heads;
    a.num_kv_heads = s.num_kv_heads;
    a.heads = s.dec_heads();
    a.page_size = s.page_size;
    a.page_shift = s.page_shift();
    a.box_rows = s.dec_box_rows();
    a.kpb_shift = __builtin_ctz((unsigned)s.dec_keys_per_box());
    a.gather = s.dec_gather() ? 1 : 0;
    a.kv_in_box = s.dec_kv_in_box() ? 1 : 0;
    a.producers = s.dec_producer_warps();
    a.box_stride = s.dec_box_stride();
    a.stages = decode_stages(s);
    a.stage_bytes = decode_stage_bytes(s);
    if (a.stages == 0) return cudaErrorInvalidValue;
    const int warps = a.heads + a.producers;
    const size_t smem = decode_smem_bytes(s);
    cudaError_t e = cudaErrorInvalidValue;
    const int g = s.group();
#define PKV_DEC(DD, GG)                                                                                  \
    if (s.head_dim == DD && g == GG)                                                                      \
        e = s.page_size < 16                                                                               \
                ? launch_decode_t<DD, GG, true>(tm, a, dim3(grid, s.dec_head_groups()), warps, smem, st)          \
                : launch_decode_t<DD, GG, false>(tm, a, dim3(grid, s.dec_head_groups()), warps, smem, st);
    PKV_FOR_EACH_HEAD_DIM_AND_GROUP(PKV_DEC)
#undef PKV_DEC
    if (e != cudaSuccess) return e;
    // the merge of the rows cut into several pieces (graph mode always launches it at the
    // maxima; its warps past the plan's cut rows return at once)
    const int merges = s.graph_static ? sc.num_merge : p.num_merge;
    if (merges) {
        const long long warps = (long long)merges * s.num_qo_heads;
        const dim3 mgrid((unsigned)((warps + dev::kMergeWarps - 1) / dev::kMergeWarps));
        // the large batch for rows of more pieces than the small one holds (graph mode, whose
        // launch serves every later plan, keeps the small one)
        const bool large = !s.graph_static && p.max_pieces > dev::merge_batch(s.head_dim, false);
        using dev::merge_batch;
        auto mk = s.head_dim == 64    ? dev::merge_kernel<64, merge_batch(64, false)>
                  : s.head_dim == 128 ? (large ? dev::merge_kernel<128, merge_batch(128, true)>
                                               : dev::merge_kernel<128, merge_batch(128, false)>)
                                      : (large ? dev::merge_kernel<256, merge_batch(256, true)>
                                               : dev::merge_kernel<256, merge_batch(256, false)>);
        e = launch_pdl(mk, mgrid, dim3(dev::kMergeWarps * 32), 0, st, static_cast<const PlanHeader *>(a.hdr),
                       reinterpret_cast<const MergeRow *>(w + p.lay.merge_rows), static_cast<const float *>(a.part_o),
                       static_cast<const float *>(a.part_lse), a.out, lse, s.num_qo_heads);
    }
    return e;
}

cudaError_t launch_append(const Shape &s, const Plan &p, void *ws, const void *k, const void *v, void *kv_layer,
                          cudaStream_t st) {
    const int tokens = s.graph_static ? static_counts(s, p.mode).tokens : p.num_append;
    if (tokens == 0) return cudaSuccess;
    uint8_t *w = static_cast<uint8_t *>(ws);
    const int vec = s.num_kv_heads * s.head_dim * 2 / 16;
    const long long chunks = (long long)tokens * vec;
    const int grid = (int)((chunks + 255) / 256);
    return launch_pdl(dev::append_kernel, dim3(grid), dim3(256), 0, st,
                      reinterpret_cast<const PlanHeader *>(w + p.lay.err), static_cast<const uint4 *>(k),
                      static_cast<const uint4 *>(v), static_cast<uint4 *>(kv_layer),
                      reinterpret_cast<const int32_t *>(w + p.lay.append_rows), vec, s.page_size);
}

cudaError_t launch_append_indexed(const Shape &s, const void *k, const void *v, int num_tokens, void *kv_layer,
                                  const int32_t *qo_indptr, const int32_t *kv_indptr, const int32_t *kv_indices,
                                  const int32_t *last_page_len, int batch, cudaStream_t st) {
    if (num_tokens == 0 || batch == 0) return cudaSuccess;
    const int vec = s.num_kv_heads * s.head_dim * 2 / 16;
    const long long chunks = (long long)num_tokens * vec;
    const int grid = (int)((chunks + 255) / 256);
    return launch_pdl(dev::append_indexed_kernel, dim3(grid), dim3(256), 0, st, static_cast<const uint4 *>(k),
                      static_cast<const uint4 *>(v), static_cast<uint4 *>(kv_layer), qo_indptr, kv_indptr, kv_indices,
                      last_page_len, batch, num_tokens, vec, s.page_size, s.page_shift(), s.num_cache_pages);
}

}  // namespace pkv

// ------------------------------------------------------------------------------------
// Scratch for callers that cannot allocate device memory (pkv_run_decode_static).
//
// The plan image and the split-KV partials of such a call live in this file-scope
// array instead of a caller workspace.  Every GPU that loads the library holds it until
// the process exits.  Host code must not use the array's name as an address: its
// device address is fetched once per device with cudaGetSymbolAddress.
namespace pkv {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// Device address of g_decode_scratch in the current device's context.  The first call in
// a context resolves it (with that device current) and caches it under the context's
// unique id; a later call in another context -- another device, or the same device after
// cudaDeviceReset made a new primary context -- resolves it again, so a cached address
// never outlives the context it belongs to.
namespace {
using CtxGetCurrent = CUresult (*)(CUcontext *);
using CtxGetId = CUresult (*)(CUcontext, unsigned long long *);
template <typename F>
cudaError_t driver_fn(const char *name, F *out) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    *out = reinterpret_cast<F>(fn);
    return cudaSuccess;
}
}  // namespace

cudaError_t static_scratch(void **ptr) {
    static CtxGetCurrent ctx_get = nullptr;
    static CtxGetId ctx_id = nullptr;
    static std::mutex mu;
    static struct {
        unsigned long long id;
        void *addr;
    } cached[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!ctx_get && (e = driver_fn("cuCtxGetCurrent", &ctx_get)) != cudaSuccess) return e;
    if (!ctx_id && (e = driver_fn("cuCtxGetId", &ctx_id)) != cudaSuccess) return e;
    auto current_id = [&](unsigned long long *id) {
        CUcontext ctx = nullptr;
        return ctx_get(&ctx) == CUDA_SUCCESS && ctx && ctx_id(ctx, id) == CUDA_SUCCESS;
    };
    unsigned long long id = 0;
    if (current_id(&id) && cached[dev].addr && cached[dev].id == id) {
        *ptr = cached[dev].addr;
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // makes the primary context current if needed
    if (e != cudaSuccess) return e;
    if (!current_id(&id)) return cudaErrorDeviceUninitialized;
    cached[dev].id = id;
    cached[dev].addr = p;
    *ptr = p;
    return cudaSuccess;
}

}  // namespace pkv

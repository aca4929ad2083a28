#pragma once
// Ragged paged prefill over a cached prefix (FlashInferPrefillWrapper.run), also the
// prefill pass of the mixed step (FlashInferMixedWrapper).
//
// New token i of row r sits at position p = L_r - n_r + i and sees keys [lo, p] (causal,
// bottom-right aligned: "the cached prefix plus themselves") or [lo, L_r - 1]
// (non-causal), lo = max(0, p - window_left) or 0.
//
// A CTA computes one tile: up to BQ = 128 / g consecutive new tokens of one row times
// the g query heads of one kv head = 128 query rows (row m = token * g + head), which
// share every K/V tile.  Blackwell design, two CTAs per SM:
//  * warp 4 (one thread) loads Q once and streams 64-key K and V tiles (boxes of 16 or 8
//    slots of the kv head, 64-column halves, 128-byte swizzle) by TMA into a two-stage
//    ring; a page past the row's end is fetched at an out-of-range coordinate, which TMA
//    fills with zeros.  Pages of 1, 2 or 4 slots are gathered instead by the whole warp
//    with 16-byte cp.async copies into the same swizzled layout (keys past the row's end
//    zero-filled);
//  * warp 5 owns 256 tensor-memory columns (512 at head_dim 256): S double-buffered
//    (2 x 64 fp32 columns) and O (D fp32 columns); one thread issues S_j = Q K_j^T
//    (tcgen05.mma, both operands in
//    shared memory, K-major) and then O += P_{j-1} V_{j-1} (P read from tensor memory,
//    V from shared memory MN-major), committing each group to mbarriers;
//  * warps 0-3 (thread = query row = TMEM lane) read S, mask, run the online softmax in
//    the exp2 domain and write P as packed bf16 over the S columns they just read.  The
//    running maximum is only moved (and O rescaled in tensor memory) when it grows by
//    more than 2^8, so most tiles never touch O;
//  * the epilogue reads O, divides by the row sum and stores bf16 rows and the lse.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "plan.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace dev {

struct PrefillArgs {
    __nv_bfloat16 *out;
    float *lse;
    const PrefillTile *tiles;
    const int32_t *pages;
    PlanHeader *hdr;  // per-plan values (tile count, causal, window, sm_scale) in the workspace
    const uint8_t *kv_layer;  // the layer slice, for the cp.async gather of small pages
    int num_qo_heads;
    int num_kv_heads;
    int page_size;
    int page_shift;  // log2 page_size
    int box_rows;  // rows of one paged TMA box (16, or 8 for 8-slot pages)
    int gather;    // pages below 8 slots: cp.async gather instead of TMA
    int oob_row;   // a row coordinate past the cache: TMA fills it with zeros
};

template <int N>
struct IntConst {
    static constexpr int value = N;
};

constexpr int kPfThreads = 192;  // warps 0-3 softmax, 4 producer, 5 MMA
// pages below 8 slots: warps 6-8 join warp 4 as cp.async producers
constexpr int kPfGatherWarps = 4;
constexpr int kPfGatherThreads = kPfThreads + 32 * (kPfGatherWarps - 1);
constexpr int kPfKeys = kPrefillKeysPerStage;  // 64 keys per K/V tile
constexpr int kPfStages = 2;
// tensor-memory columns a CTA allocates: S (2 x 64) + O (D), rounded up to a power of two
template <int D>
struct PfTmem {
    static constexpr uint32_t COLS = D > 128 ? 512u : 256u;
};
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2f = 0.6931471805599453f;

template <int D>
struct PfSmem {
    static constexpr int HALVES = D / 64;
    static constexpr uint32_t Q_BYTES = 128u * D * 2;
    static constexpr uint32_t KV_BYTES = (uint32_t)kPfKeys * D * 2;  // one K or V tile
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t K_OFF = Q_BYTES;
    static constexpr uint32_t V_OFF = K_OFF + kPfStages * KV_BYTES;
    static constexpr uint32_t BAR_OFF = V_OFF + kPfStages * KV_BYTES;
    static constexpr uint32_t BYTES = BAR_OFF + 256;
};

// GATHER: paged plans with pages below 8 slots (cp.async producers instead of TMA).
template <int D, int G, bool GATHER>
__global__ void __launch_bounds__(GATHER ? kPfGatherThreads : kPfThreads, D > 128 ? 1 : 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, const PrefillArgs a) {
    using L = PfSmem<D>;
    constexpr int HALVES = L::HALVES;
    constexpr int BQ = kPrefillRowsPerTile / G;
    constexpr uint32_t Q_TX = (uint32_t)BQ * G * D * 2;  // rows BQ*G..127 stay unused
    constexpr int KSTEPS = D / 16;
    constexpr uint32_t kTmemCols = PfTmem<D>::COLS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    // Each MMA group commits to one barrier that every party waiting on it polls by
    // parity: s_full[s] (S_j done: the softmax may read it, K slot s is free again) and
    // pv_done[s] (PV_j done: V slot s is free, S buffer s may be overwritten, O holds
    // P_0..P_j V).  A waiter is never two phases behind, because the next phase of either
    // barrier needs data that the waiter itself has yet to provide.
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;   // [2]
    uint64_t *v_full = bars + 3;   // [2]
    uint64_t *s_full = bars + 5;   // [2]
    uint64_t *p_full = bars + 7;   // [2]
    uint64_t *pv_done = bars + 9;  // [2]
    // o_final completes once, after the last PV.  The epilogue cannot wait on pv_done by
    // parity: when it gets there, two PVs may still be outstanding, and phase (nt-1)/2 of
    // one buffer's barrier has the same parity as an already completed earlier phase.
    uint64_t *o_final = bars + 11;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 12);

    if ((int)blockIdx.x >= a.hdr->pf_tiles) return;  // an idle CTA of a launch at the maxima
    const PrefillTile t = a.tiles[blockIdx.x];
    int *const err = &a.hdr->err;
    const int causal = a.hdr->causal;
    const int window_left = a.hdr->window_left;
    // dense varlen plans: K and V rows come from two contiguous tensors (tm_kv, tm_v),
    // tile keys at rows kv_base + key; paged plans: both from the layer slice (tm_kv)
    const bool dense = a.hdr->dense != 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int P = a.page_size;
    const int kt0 = t.key_begin / kPfKeys;
    const int nt = (t.key_end + kPfKeys - 1) / kPfKeys - kt0;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&k_full[s], GATHER ? kPfGatherWarps : 1);  // gather: one per producer warp
            mbar_init(&v_full[s], GATHER ? kPfGatherWarps : 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 4);
            mbar_init(&pv_done[s], 1);
        }
        mbar_init(o_final, 1);
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();  // q, the cache (or K / V) may come from the previous kernel
    griddep_launch();
    const uint32_t tmem = *tmem_holder;
    const uint32_t S_col[2] = {tmem, tmem + 64};
    const uint32_t O_col = tmem + 128;

    if (warp == 4 || (GATHER && warp >= 6)) {
        // ------------------------------------------------ producer(s)
        if (warp == 4) {
        if constexpr (BQ * G < kPrefillRowsPerTile) {
            // a group size that does not divide 128 leaves Q rows BQ*G..127 unloaded: zero
            // them (their S rows are never stored, but must not hold Inf or NaN)
            constexpr int ZROWS = kPrefillRowsPerTile - BQ * G;
            for (int i = lane; i < HALVES * ZROWS * 8; i += 32) {
                const int h = i / (ZROWS * 8), r = BQ * G + (i / 8) % ZROWS, c = i % 8;
                *reinterpret_cast<uint4 *>(sm + L::Q_OFF + h * (L::Q_BYTES / HALVES) + r * 128 + c * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        if (lane == 0) {
            prefetch_tmap(&tm_kv);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_q);
            mbar_arrive_expect_tx(q_full, Q_TX);
#pragma unroll
            for (int h = 0; h < HALVES; ++h)
                tma_load_3d(sm + L::Q_OFF + h * (L::Q_BYTES / HALVES), &tm_q, q_full, h * 64, t.kv_head * G,
                            t.q_begin);
        }
        }
        const int npages = (t.length + P - 1) >> a.page_shift;
        if constexpr (!GATHER) {
            // TMA: a 64-key tile is NB boxes of 64 / NB rows (16, or 8 for 8-slot pages)
            auto stream_tiles = [&](auto nb) {
                constexpr int NB = decltype(nb)::value;
                constexpr int R = kPfKeys / NB;
                // cache rows of tile j's boxes (-1: past the row's pages)
                auto tile_rows = [&](int j, int (&rows)[NB]) {
                    const int key0 = (kt0 + j) * kPfKeys;
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const int kb = key0 + b * R;
                        if (dense)
                            rows[b] = t.kv_base + kb;  // past the segment: masked keys, finite V
                        else
                            rows[b] = (kb >> a.page_shift) < npages
                                          ? a.pages[t.kv_base + (kb >> a.page_shift)] * 2 * P + (kb & (P - 1))
                                          : -1;
                    }
                };
                int rows[NB], next[NB];
                tile_rows(0, rows);
                for (int j = 0; j < nt; ++j) {
                    const int s = j & 1;
                    const uint32_t use = j >> 1;
                    if (use > 0 && !mbar_wait(&s_full[s], (use - 1) & 1, err, kErrWaitEmpty)) break;
                    uint8_t *kd = sm + L::K_OFF + s * L::KV_BYTES;
                    mbar_arrive_expect_tx(&k_full[s], L::KV_BYTES);
#pragma unroll
                    for (int b = 0; b < NB; ++b)
#pragma unroll
                        for (int h = 0; h < HALVES; ++h)
                            tma_load_3d(kd + h * (L::KV_BYTES / HALVES) + b * R * 128, &tm_kv, &k_full[s], h * 64,
                                        rows[b] >= 0 ? rows[b] : a.oob_row, t.kv_head);
                    // the next tile's page ids load while this tile's V slot drains: by the
                    // time the next K slot is free (it frees before this V slot) they are here
                    if (j + 1 < nt) tile_rows(j + 1, next);
                    if (use > 0 && !mbar_wait(&pv_done[s], (use - 1) & 1, err, kErrWaitEmpty)) break;
                    uint8_t *vd = sm + L::V_OFF + s * L::KV_BYTES;
                    mbar_arrive_expect_tx(&v_full[s], L::KV_BYTES);
#pragma unroll
                    for (int b = 0; b < NB; ++b)
#pragma unroll
                        for (int h = 0; h < HALVES; ++h)
                            tma_load_3d(vd + h * (L::KV_BYTES / HALVES) + b * R * 128, dense ? &tm_v : &tm_kv,
                                        &v_full[s], h * 64, rows[b] < 0 ? a.oob_row : rows[b] + (dense ? 0 : P),
                                        t.kv_head);
#pragma unroll
                    for (int b = 0; b < NB; ++b) rows[b] = next[b];
                }
            };
            if (lane == 0) {
                if (dense || a.box_rows == 16)
                    stream_tiles(IntConst<4>{});
                else
                    stream_tiles(IntConst<8>{});
            }
        } else {
            // cp.async gather (pages of 1, 2 or 4 slots) by warps 4, 6, 7, 8.  Lane = (key slot,
            // 16-byte column chunk c), a warp instruction covering KPI keys; producer warp pw
            // takes key groups pw, pw + 4, ... of each 64-key tile, looks their slot rows up once
            // and copies K and V rows to their swizzled places (keys at or past the row's end
            // read nothing and land as zeros).  Its copies must have landed, and be made visible
            // to the tensor cores' proxy, before it counts on the tile's full barriers.
            constexpr int CH = D / 8;                     // 16-byte chunks per head row
            constexpr int KPI = 32 / CH;                  // keys per warp instruction
            constexpr int NI = kPfKeys / KPI / kPfGatherWarps;  // key groups per producer warp
            const int pw = warp == 4 ? 0 : warp - 5;
            const int c = lane % CH, kslot = lane / CH;
            const size_t row_bytes = (size_t)a.num_kv_heads * D * 2;  // bytes per cache row
            const size_t v_off = (size_t)P * row_bytes;
            const uint8_t *base = a.kv_layer + (size_t)t.kv_head * D * 2 + c * 16;
            for (int j = 0; j < nt; ++j) {
                const int s = j & 1;
                const uint32_t use = j >> 1;
                const int key0 = (kt0 + j) * kPfKeys;
                int row[NI];
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const int pos = key0 + kslot + KPI * (pw + kPfGatherWarps * i);
                    row[i] = pos < t.length ? a.pages[t.kv_base + (pos >> a.page_shift)] * 2 * P + (pos & (P - 1)) : -1;
                }
                // every lane waits on the barriers itself (they wake together); the vote keeps
                // the warp on one path if a wait gives up
                const bool ok = use == 0 || (mbar_wait(&s_full[s], (use - 1) & 1, err, kErrWaitEmpty) &&
                                             mbar_wait(&pv_done[s], (use - 1) & 1, err, kErrWaitEmpty));
                if (!__all_sync(0xffffffffu, ok)) break;
                const uint32_t kd = smem_u32(sm + L::K_OFF + s * L::KV_BYTES) + (c >> 3) * (L::KV_BYTES / HALVES);
                const uint32_t vd = smem_u32(sm + L::V_OFF + s * L::KV_BYTES) + (c >> 3) * (L::KV_BYTES / HALVES);
#pragma unroll
                for (int i = 0; i < NI; ++i) {
                    const int key = kslot + KPI * (pw + kPfGatherWarps * i);
                    const bool valid = row[i] >= 0;
                    const uint8_t *src = valid ? base + (size_t)row[i] * row_bytes : base;
                    const uint32_t dst = swz128(key, c & 7);
                    cp_async16(kd + dst, src, valid ? 16u : 0u);
                    cp_async16(vd + dst, valid ? src + v_off : base, valid ? 16u : 0u);
                }
                cp_async_wait_all();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&k_full[s]);
                    mbar_arrive(&v_full[s]);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issue (one thread) + V tails
        constexpr uint32_t ID_S = idesc_bf16_f32(128, kPfKeys, 0, 0);
        constexpr uint32_t ID_O = idesc_bf16_f32(128, D, 0, 1);
        const uint32_t sQ = smem_u32(sm + L::Q_OFF);
        const uint32_t tail_begin = t.length;
        const uint32_t tail_end = (uint32_t)((t.length + P - 1) & ~(P - 1));
        bool ok = mbar_wait(q_full, 0, err, kErrWaitFull);
        auto issue_pv = [&](int i) {
            const int s = i & 1;
            ok = ok && mbar_wait(&p_full[s], (i >> 1) & 1, err, kErrWaitFull);
            ok = ok && mbar_wait(&v_full[s], (i >> 1) & 1, err, kErrWaitFull);
            if (!ok) return;
            uint8_t *vs = sm + L::V_OFF + s * L::KV_BYTES;
            // zero V rows of the row's last page past its end (poisoned or stale slots)
            const int key0 = (kt0 + i) * kPfKeys;
            const int zb = max((int)tail_begin, key0), ze = min((int)tail_end, key0 + kPfKeys);
            if (zb < ze) {
                const int nz = (ze - zb) * (D / 8);
                for (int e = lane; e < nz; e += 32) {
                    const int k = zb - key0 + e / (D / 8);
                    const int chunk = e % (D / 8);
                    *reinterpret_cast<uint4 *>(vs + (chunk >> 3) * (L::KV_BYTES / HALVES) + swz128(k, chunk & 7)) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sV = smem_u32(vs);
#pragma unroll
                for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                    const uint64_t bd = smem_desc(sV + kk * 2048, L::KV_BYTES / HALVES, 1024, kSwizzle128B);
                    mma_ts(O_col, S_col[s] + kk * 8, bd, ID_O, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&pv_done[s]);
            }
            __syncwarp();
        };
        for (int j = 0; j < nt && ok; ++j) {
            const int s = j & 1;
            ok = mbar_wait(&k_full[s], (j >> 1) & 1, err, kErrWaitFull);
            // S_j overwrites the columns that PV_{j-2} reads as its A operand (P_{j-2}); MMAs
            // with different accumulators are not ordered for us, so wait for PV_{j-2}
            if (ok && j >= 2) ok = mbar_wait(&pv_done[s], ((j - 2) >> 1) & 1, err, kErrWaitFull);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sK = smem_u32(sm + L::K_OFF + s * L::KV_BYTES);
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const uint32_t off = (kk % 4) * 32;  // 16 columns = 32 bytes along the swizzled row
                    const uint64_t ad = smem_desc(sQ + (kk / 4) * (L::Q_BYTES / HALVES) + off, 16, 1024, kSwizzle128B);
                    const uint64_t bd =
                        smem_desc(sK + (kk / 4) * (L::KV_BYTES / HALVES) + off, 16, 1024, kSwizzle128B);
                    mma_ss(S_col[s], ad, bd, ID_S, kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[s]);
            }
            __syncwarp();
            if (j >= 1) issue_pv(j - 1);
        }
        if (ok && nt >= 1) issue_pv(nt - 1);
        if (ok && lane == 0) mma_commit(o_final);
    } else if (warp < 4) {
        // ------------------------------------------------ softmax + epilogue (warps 0-3)
        const int m = threadIdx.x;  // query row = TMEM lane
        const int tok = m / G;
        const int hd = t.kv_head * G + m % G;
        const bool live = tok < t.n_q;
        const int pos = t.pos0 + tok;
        const int hi = causal == 1 ? pos : t.length - 1;
        const int lo = window_left >= 0 ? max(0, pos - window_left) : 0;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float sl = a.hdr->scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int s = j & 1;
            const int key0 = (kt0 + j) * kPfKeys;
            if (!mbar_wait(&s_full[s], (j >> 1) & 1, err, kErrWaitFull)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(S_col[s] + lane_off, r0);
            tmem_ld32(S_col[s] + lane_off + 32, r1);
            tmem_wait_ld();
            float sv[64];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                sv[c] = __uint_as_float(r0[c]);
                sv[32 + c] = __uint_as_float(r1[c]);
            }
            if (key0 < lo || key0 + kPfKeys - 1 > hi || key0 + kPfKeys > t.length) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const int k = key0 + c;
                    sv[c] = (k >= lo && k <= hi && k < t.length) ? sv[c] : -INFINITY;
                }
            }
            float mx;
            {
                float a0 = sv[0], a1 = sv[1], a2 = sv[2], a3 = sv[3];
#pragma unroll
                for (int c = 4; c < 64; c += 8) {
                    a0 = max3f(a0, sv[c], sv[c + 1]);
                    a1 = max3f(a1, sv[c + 2], sv[c + 3]);
                    a2 = max3f(a2, sv[c + 4], sv[c + 5]);
                    a3 = max3f(a3, sv[c + 6], sv[c + 7]);
                }
                mx = max3f(fmaxf(a0, a1), a2, a3);
            }
            const float m_tile = mx * sl;  // -inf when the whole tile is masked for this row
            // move the running max only when it grows by more than the threshold
            const bool grow = m_tile > m_run + kRescaleThreshold;
            const bool warp_grow = __any_sync(0xffffffffu, grow) && j > 0;
            float alpha = 1.f;
            if (j == 0 || warp_grow) {
                const float m_new = fmaxf(m_run, m_tile);
                if (m_new != -INFINITY) {
                    alpha = ex2_ftz(m_run - m_new);  // 0 when m_run = -inf
                    m_run = m_new;
                }
            }
            const float mref = m_run == -INFINITY ? 0.f : m_run;
            // p = 2^(s * sl - mref), two columns per packed FMA; sums in four packed chains
            const uint64_t sl2 = f2_make(sl, sl), nm2 = f2_make(-mref, -mref);
            uint64_t acc[4] = {0, 0, 0, 0};
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float x0, x1;
                f2_split(ffma2(f2_make(sv[2 * c], sv[2 * c + 1]), sl2, nm2), x0, x1);
                const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
                acc[c & 3] = fadd2(acc[c & 3], f2_make(p0, p1));
                pk[c] = pack_bf16(p0, p1);
            }
            float u0, u1;
            f2_split(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), u0, u1);
            const float psum = u0 + u1;
            l_run = l_run * alpha + psum;
            tmem_st32(S_col[s] + lane_off, pk);
            tmem_wait_st();
            if (warp_grow) {
                // O holds P_0..P_{j-1} V: wait for the last of those MMAs, then scale O rows
                if (!mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err, kErrWaitFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(O_col + lane_off + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tmem_st32(O_col + lane_off + c0, o);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[s]);
        }
        // epilogue
        if (ok && mbar_wait(o_final, 0, err, kErrWaitFull)) {
            tc_fence_after();
            const bool none = l_run == 0.f;  // no visible key (empty context): o = 0, lse = -inf
            const float inv = none ? 0.f : 1.f / l_run;
            __nv_bfloat16 *orow = a.out + ((size_t)(t.q_begin + tok) * a.num_qo_heads + hd) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(O_col + lane_off + c0, o);
                tmem_wait_ld();
                uint32_t pkd[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)  // select, not multiply: unwritten O may hold NaN bits
                    pkd[c] = none ? 0u : pack_bf16(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
                if (live) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        dst[c] = make_uint4(pkd[4 * c], pkd[4 * c + 1], pkd[4 * c + 2], pkd[4 * c + 3]);
                }
            }
            if (live && a.lse)
                a.lse[(size_t)(t.q_begin + tok) * a.num_qo_heads + hd] =
                    none ? -INFINITY : (m_run + __log2f(l_run)) * kLn2f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace dev

// Two query tiles per CTA, head_dim 64 / 128 read by TMA: prefill_pair.cu.
cudaError_t launch_prefill_pair(int head_dim, int group, const CUtensorMap &tkv, const CUtensorMap &tv,
                                const CUtensorMap &tq, const dev::PrefillArgs &a, int grid, cudaStream_t st);
// One query tile per CTA with two S buffers, head_dim 256 read by TMA: prefill_wide.cu.
cudaError_t launch_prefill_wide(int group, const CUtensorMap &tkv, const CUtensorMap &tv, const CUtensorMap &tq,
                                const dev::PrefillArgs &a, int grid, cudaStream_t st);
// Instances with GATHER = true live in prefill_gather.cu (compiled in parallel).
cudaError_t launch_prefill_gather(int head_dim, int group, const CUtensorMap &tkv, const CUtensorMap &tv,
                                  const CUtensorMap &tq, const dev::PrefillArgs &a, int grid, size_t smem,
                                  cudaStream_t st);

template <int D, int G, bool GATHER>
inline cudaError_t launch_prefill_t(const CUtensorMap &tkv, const CUtensorMap &tv, const CUtensorMap &tq,
                                    const dev::PrefillArgs &a, int grid, size_t smem, cudaStream_t st) {
    auto fn = dev::prefill_tc_kernel<D, G, GATHER>;
    cudaError_t e = set_smem_limit((const void *)fn, smem, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(fn, dim3(grid), dim3(GATHER ? dev::kPfGatherThreads : dev::kPfThreads), smem, st, tkv, tv, tq,
                      a);
}

}  // namespace pkv

#pragma once
// Ragged paged prefill over a cached prefix (FlashInferPrefillWrapper.run), the prefill pass of
// the mixed step (FlashInferMixedWrapper) and dense varlen attention (DenseAttentionManager), for
// head_dim 256 with K / V read by TMA.
//
// New token i of row r sits at position p = L_r - n_r + i and sees keys [lo, p] (causal,
// bottom-right aligned: "the cached prefix plus themselves") or [lo, L_r - 1] (non-causal),
// lo = max(0, p - window_left) or 0.
//
// A work tile is up to BQ = 128 / g consecutive new tokens of one row times the g query heads of
// one kv head: one query tile of 128 rows (row m = token * g + head).  One CTA per SM (192 KB of
// shared memory, all 512 tensor-memory columns):
//  * warp 4 loads Q once and streams the 128-key K tiles, warp 5 the V tiles (TMA boxes of 16 or 8
//    slots of the kv head, 64-column quarters, 128-byte swizzle; one lane per box, its page looked
//    up a tile ahead), one stage each (a tile of 128 keys x 256 columns is 64 KB); the K stage is
//    refilled by 64-column quarter as S(j)'s k-steps release them, the V stage by quarter of 32
//    keys as PV(j)'s k-steps release those;
//  * tensor memory holds two S buffers of 128 fp32 columns (P written over each as bf16) and O
//    (256 fp32 columns).  Warp 6 issues S(j) = Q K_j^T (N = 128: both operands in shared memory at
//    the full MMA rate) into buffer j % 2 once PV(j-2), which read P(j-2) from it, completed; warp
//    7 issues O += P(j) V_j (P from tensor memory, N = 256).  With one issuing warp each, S(j+1)
//    runs under the softmax of tile j and PV(j) does not wait behind it;
//  * warps 0-3 run the softmax (thread = query row = TMEM lane); the running maximum moves, and O
//    is rescaled in tensor memory, only when it grows by more than 2^8.
// pv_done is counted per buffer: S(j) waits for PV(j-2) while PV(j-1) may already be done, which a
// single barrier could not tell apart from PV(j-2) by parity.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "prefill_kernel.cuh"

namespace pkv {
namespace dev {

constexpr int kPwKeys = 128;     // keys per K / V tile
constexpr int kPwThreads = 256;  // warps 0-3 softmax, 4 Q and K producer, 5 V producer, 6 S issue, 7 PV issue

struct PwSmem {
    static constexpr int D = 256;
    static constexpr int QUARTERS = D / 64;
    static constexpr uint32_t Q_TILE = 128u * D * 2;                // 64 KB
    static constexpr uint32_t Q_QUARTER = Q_TILE / QUARTERS;        // one 64-column quarter
    static constexpr uint32_t KV_TILE = (uint32_t)kPwKeys * D * 2;  // 64 KB
    static constexpr uint32_t KV_QUARTER = KV_TILE / QUARTERS;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t K_OFF = Q_TILE;
    static constexpr uint32_t V_OFF = K_OFF + KV_TILE;
    static constexpr uint32_t BAR_OFF = V_OFF + KV_TILE;
    static constexpr uint32_t BYTES = BAR_OFF + 256;
};

// A shared-memory descriptor for base + off: the base's plus off >> 4 in the start-address field
// (no carry: every address here is below 256 KB).
__device__ __forceinline__ uint64_t pw_desc(uint64_t d, uint32_t off_bytes) { return d + (off_bytes >> 4); }

template <int G>
__global__ void __launch_bounds__(kPwThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, const PrefillArgs a) {
    using L = PwSmem;
    constexpr int D = L::D;
    constexpr int QUARTERS = L::QUARTERS;
    constexpr int BQ = kPrefillRowsPerTile / G;          // tokens per query tile
    constexpr uint32_t Q_TX = (uint32_t)BQ * G * D * 2;  // rows BQ*G..127 stay unused
    constexpr int PSTEPS = kPwKeys / 16;                 // k-steps of O += P V
    static_assert(PSTEPS == 8, "two PV k-steps per 32-key quarter of V");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    // K / V stages, S / P buffers and PV completions: once per K/V tile (q_full, o_final once)
    // The K stage is filled and released by 64-column quarter: S(j)'s k-steps read the quarters in
    // turn, so quarter q of K(j+1) is requested once the MMAs reading quarter q of K(j) completed.
    // The V stage likewise by quarter of 32 keys: PV(j)'s k-steps read its keys in order.
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;    // [4] a quarter of K(j) landed
    uint64_t *k_empty = bars + 5;   // [4] the S MMAs reading a quarter of K(j) completed
    uint64_t *v_full = bars + 19;   // [4] a quarter (32 keys) of V(j) landed
    uint64_t *v_empty = bars + 23;  // [4] the PV MMAs reading a quarter of V(j) completed
    uint64_t *s_full = bars + 11;   // [2] S(j) in buffer j % 2
    uint64_t *p_full = bars + 13;   // [2] P(j) written over buffer j % 2 (and O rescaled if it had to be)
    uint64_t *pv_done = bars + 15;  // [2] PV(j) completed, counted on buffer j % 2
    uint64_t *o_final = bars + 17;  // the last PV completed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 18);

    if ((int)blockIdx.x >= a.hdr->pf_tiles) return;  // an idle CTA of a launch at the maxima
    const PrefillTile t = a.tiles[blockIdx.x];
    int *const err = &a.hdr->err;
    const int causal = a.hdr->causal;
    const int window_left = a.hdr->window_left;
    const bool dense = a.hdr->dense != 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int P = a.page_size;
    const int kt0 = t.key_begin / kPwKeys;
    const int nt = (t.key_end + kPwKeys - 1) / kPwKeys - kt0;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int q = 0; q < QUARTERS; ++q) {
            mbar_init(&k_full[q], 1);
            mbar_init(&k_empty[q], 1);
        }
        for (int q = 0; q < 4; ++q) {
            mbar_init(&v_full[q], 1);
            mbar_init(&v_empty[q], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4);
            mbar_init(&pv_done[b], 1);
        }
        mbar_init(o_final, 1);
        fence_barrier_init();
    }
    if (warp == 6) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();  // q, the cache (or K / V) may come from the previous kernel
    griddep_launch();
    const uint32_t tmem = *tmem_holder;
    const uint32_t O_col = tmem + 256u;  // S buffers at columns 0 and 128

    if (warp == 4 || warp == 5) {
        // ------------------------------------------------ producers: warp 4 Q and K, warp 5 V
        if (warp == 4) {
            if constexpr (BQ * G < kPrefillRowsPerTile) {
                // a group size that does not divide 128 leaves Q rows BQ*G..127 unloaded: zero
                // them (their S rows are never stored, but must not hold NaN)
                constexpr int ZROWS = kPrefillRowsPerTile - BQ * G;
                for (int i = lane; i < QUARTERS * ZROWS * 8; i += 32) {
                    const int h = i / (ZROWS * 8), r = BQ * G + (i / 8) % ZROWS, c = i % 8;
                    *reinterpret_cast<uint4 *>(sm + L::Q_OFF + h * L::Q_QUARTER + r * 128 + c * 16) =
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
                for (int h = 0; h < QUARTERS; ++h)
                    tma_load_3d(sm + L::Q_OFF + h * L::Q_QUARTER, &tm_q, q_full, h * 64, t.kv_head * G, t.q_begin);
            }
        }
        // A 128-key tile is NB boxes of R = 128 / NB rows (16, or 8 for 8-slot pages); lane b < NB
        // copies box b (its four 64-column quarters) and looks up the box's page one tile ahead.
        const int kv = warp == 5;
        uint8_t *stage = sm + (kv ? L::V_OFF : L::K_OFF);
        const int NB = (dense || a.box_rows == 16) ? 8 : 16;
        const int R = kPwKeys / NB;
        const int npages = (t.length + P - 1) >> a.page_shift;
        const CUtensorMap *map = (kv && dense) ? &tm_v : &tm_kv;
        const int voff = (kv && !dense) ? P : 0;
        // cache row of box `lane` of tile j (a.oob_row past the row's pages: TMA reads zeros;
        // dense: rows past the segment are masked keys with finite V)
        auto box_row = [&](int j) {
            const int kb = (kt0 + j) * kPwKeys + lane * R;
            if (dense) return t.kv_base + kb;
            return (kb >> a.page_shift) < npages
                       ? a.pages[t.kv_base + (kb >> a.page_shift)] * 2 * P + (kb & (P - 1)) + voff
                       : a.oob_row;
        };
        int row = (lane < NB && nt > 0) ? box_row(0) : 0;
        bool ok = true;
        for (int j = 0; j < nt && ok; ++j) {
            if (kv) {
                // key quarter kq (32 keys: boxes kq * NB / 4 .. of NB / 4 lanes), each box with its
                // four 64-column quarters
                for (int kq = 0; kq < 4; ++kq) {
                    // the PV MMAs that read this key quarter of the previous tile must have completed
                    if (j > 0 && !mbar_wait(&v_empty[kq], (j - 1) & 1, err, kErrWaitEmpty)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(&v_full[kq], L::KV_TILE / 4);
                    __syncwarp();
                    if (lane < NB && lane / (NB / 4) == kq) {
#pragma unroll
                        for (int h = 0; h < QUARTERS; ++h)
                            tma_load_3d(stage + h * L::KV_QUARTER + lane * R * 128, map, &v_full[kq], h * 64, row,
                                        t.kv_head);
                    }
                }
            } else {
                for (int h = 0; h < QUARTERS; ++h) {
                    // the S MMAs that read this quarter of the previous tile must have completed
                    if (j > 0 && !mbar_wait(&k_empty[h], (j - 1) & 1, err, kErrWaitEmpty)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(&k_full[h], L::KV_QUARTER);
                    __syncwarp();
                    if (lane < NB)
                        tma_load_3d(stage + h * L::KV_QUARTER + lane * R * 128, map, &k_full[h], h * 64, row,
                                    t.kv_head);
                }
            }
            if (lane < NB && j + 1 < nt) row = box_row(j + 1);  // lands while the stage is awaited
        }
    } else if (warp == 6) {
        // ------------------------------------------------ S(j) = Q K_j^T into buffer j % 2
        constexpr uint32_t ID_S = idesc_bf16_f32(128, kPwKeys, 0, 0);
        // K-major operands: 16-byte leading offset, 8-row groups 1024 bytes apart
        const uint64_t dQ = smem_desc(smem_u32(sm + L::Q_OFF), 16, 1024, kSwizzle128B);
        const uint64_t dK = smem_desc(smem_u32(sm + L::K_OFF), 16, 1024, kSwizzle128B);
        bool ok = mbar_wait(q_full, 0, err, kErrWaitFull);
        for (int j = 0; j < nt && ok; ++j) {
            const int b = j & 1;
#pragma unroll 1
            for (int h = 0; h < QUARTERS && ok; ++h) {
                ok = mbar_wait(&k_full[h], j & 1, err, kErrWaitFull);
                // buffer b holds P(j-2) until PV(j-2) completed (its next phase, PV(j), needs S(j))
                if (ok && h == 0 && j >= 2) ok = mbar_wait(&pv_done[b], ((j - 2) >> 1) & 1, err, kErrWaitFull);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
                    mma_ss_elect(tmem + 128u * (uint32_t)b, pw_desc(dQ, (kk / 4) * L::Q_QUARTER + (kk % 4) * 32),
                                 pw_desc(dK, (kk / 4) * L::KV_QUARTER + (kk % 4) * 32), ID_S, kk > 0 ? 1u : 0u);
                mma_commit_elect(&k_empty[h]);  // this quarter of K_j frees once these MMAs completed
            }
            if (ok) mma_commit_elect(&s_full[b]);
        }
    } else if (warp == 7) {
        // ------------------------------------------------ O += P(j) V_j
        constexpr uint32_t ID_O = idesc_bf16_f32(128, D, 0, 1);
        // V MN-major: its 64-column quarters L::KV_QUARTER apart
        const uint64_t dV = smem_desc(smem_u32(sm + L::V_OFF), L::KV_QUARTER, 1024, kSwizzle128B);
        const int tail_begin = t.length;
        const int tail_end = (t.length + P - 1) & ~(P - 1);
        bool ok = true;
        for (int j = 0; j < nt && ok; ++j) {
            const int b = j & 1;
            ok = mbar_wait(&p_full[b], (j >> 1) & 1, err, kErrWaitFull);
            if (!ok) break;
            const int key0 = (kt0 + j) * kPwKeys;
#pragma unroll 1
            for (int kq = 0; kq < 4 && ok; ++kq) {
                ok = mbar_wait(&v_full[kq], j & 1, err, kErrWaitFull);
                if (!ok) break;
                // V rows of the row's last page past its end (poisoned or stale slots: their P is
                // 0, but 0 * NaN would poison O) are zeroed before the MMAs read them (the last
                // tile: keys never reach past the row's end), quarter by quarter
                const int qb = key0 + kq * (kPwKeys / 4);
                const int zb = max(tail_begin, qb), ze = min(tail_end, qb + kPwKeys / 4);
                if (zb < ze) {
                    uint8_t *vs = sm + L::V_OFF;
                    const int nz = (ze - zb) * (D / 8);
                    for (int e = lane; e < nz; e += 32) {
                        const int k = zb - key0 + e / (D / 8);
                        const int chunk = e % (D / 8);
                        *reinterpret_cast<uint4 *>(vs + (chunk >> 3) * L::KV_QUARTER + swz128(k, chunk & 7)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 2 * kq; kk < 2 * kq + 2; ++kk)  // 16 keys = 16 rows of 128 bytes per k-step
                    mma_ts_elect(O_col, tmem + 128u * (uint32_t)b + kk * 8, pw_desc(dV, kk * 2048), ID_O,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit_elect(&v_empty[kq]);  // this key quarter of V_j frees once these MMAs completed
            }
            if (!ok) {
                // let the MMAs already issued finish before the tensor memory is released
                mma_commit_elect(&pv_done[b]);
                mbar_wait(&pv_done[b], (j >> 1) & 1, err, kErrWaitFull);
                break;
            }
            mma_commit_elect(&pv_done[b]);
            if (j == nt - 1) mma_commit_elect(o_final);
        }
        if (nt == 0 && lane == 0) mma_commit(o_final);  // no MMA: arrives at once
    } else {
        // ------------------------------------------------ softmax + epilogue (warps 0-3)
        const int m = warp * 32 + lane;  // query row = TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const int tok = m / G;  // token within the work tile
        const int hd = t.kv_head * G + m % G;
        const bool live = m < BQ * G && tok < t.n_q;
        const int pos = t.pos0 + tok;
        const int hi = causal == 1 ? pos : t.length - 1;
        const int lo = window_left >= 0 ? max(0, pos - window_left) : 0;
        const float sl = a.hdr->scale_log2;
        const uint32_t Ol = O_col + lane_off;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int b = j & 1;
            const uint32_t Sb = tmem + 128u * (uint32_t)b + lane_off;
            const int key0 = (kt0 + j) * kPwKeys;
            // S(j+2) reuses this buffer only after PV(j), which needs this P(j): this phase is next
            if (!mbar_wait(&s_full[b], (j >> 1) & 1, err, kErrWaitFull)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r0[32], r1[32], r2[32], r3[32];
            tmem_ld32(Sb, r0);
            tmem_ld32(Sb + 32, r1);
            tmem_ld32(Sb + 64, r2);
            tmem_ld32(Sb + 96, r3);
            tmem_wait_ld();
            float sv[kPwKeys];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                sv[c] = __uint_as_float(r0[c]);
                sv[32 + c] = __uint_as_float(r1[c]);
                sv[64 + c] = __uint_as_float(r2[c]);
                sv[96 + c] = __uint_as_float(r3[c]);
            }
            if (key0 < lo || key0 + kPwKeys - 1 > hi || key0 + kPwKeys > t.length) {
#pragma unroll
                for (int c = 0; c < kPwKeys; ++c) {
                    const int k = key0 + c;
                    sv[c] = (k >= lo && k <= hi && k < t.length) ? sv[c] : -INFINITY;
                }
            }
            // the tile's row maximum: eight independent chains of 3-input max
            float m8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) m8[c] = fmaxf(sv[2 * c], sv[2 * c + 1]);
#pragma unroll
            for (int c = 16; c < kPwKeys; c += 16)
#pragma unroll
                for (int q = 0; q < 8; ++q) m8[q] = max3f(m8[q], sv[c + 2 * q], sv[c + 2 * q + 1]);
            const float m_tile =  // -inf when the whole tile is masked for this row
                max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * sl;
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
            // p = 2^(s * sl - mref), two columns per packed FMA; sums in four packed chains; P
            // goes back over the buffer's columns as packed bf16 (64 columns), in two halves
            const float mref = m_run == -INFINITY ? 0.f : m_run;
            const uint64_t sl2 = f2_make(sl, sl), nm2 = f2_make(-mref, -mref);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int e = hlf * 64 + 2 * c;
                    float x0, x1;
                    f2_split(ffma2(f2_make(sv[e], sv[e + 1]), sl2, nm2), x0, x1);
                    const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
                    acc[c & 3] = fadd2(acc[c & 3], f2_make(p0, p1));
                    pk[c] = pack_bf16(p0, p1);
                }
                tmem_st32(Sb + hlf * 32, pk);
            }
            float u0, u1;
            f2_split(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), u0, u1);
            l_run = l_run * alpha + (u0 + u1);
            tmem_wait_st();
            if (warp_grow) {
                // O holds P(0..j-1) V: wait for the last of those MMAs, then scale O rows (PV(j)
                // waits for this p_full, so nothing else touches O now)
                if (!mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, err, kErrWaitFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(Ol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tmem_st32(Ol + c0, o);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[b]);
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
                tmem_ld32(Ol + c0, o);
                tmem_wait_ld();
                uint32_t pkd[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)  // select, not multiply: unwritten O may hold NaN bits
                    pkd[c] = none ? 0u
                                  : pack_bf16(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
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
    if (warp == 6) tmem_dealloc(tmem, 512);
}

}  // namespace dev
}  // namespace pkv

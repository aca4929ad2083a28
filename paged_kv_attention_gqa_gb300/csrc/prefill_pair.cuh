#pragma once
// Ragged paged prefill over a cached prefix (FlashInferPrefillWrapper.run), the prefill pass
// of the mixed step (FlashInferMixedWrapper) and dense varlen attention (DenseAttentionManager),
// for head_dim 64 and 128 with K / V read by TMA: TWO query tiles per CTA.
//
// New token i of row r sits at position p = L_r - n_r + i and sees keys [lo, p] (causal,
// bottom-right aligned: "the cached prefix plus themselves") or [lo, L_r - 1] (non-causal),
// lo = max(0, p - window_left) or 0.
//
// A work tile is up to 2 * BQ consecutive new tokens of one row (BQ = 128 / g) times the g
// query heads of one kv head: two query tiles of 128 rows (row m = token * g + head), Q0 and
// Q1, that share every K/V tile.  One CTA per SM:
//  * warp 8 loads Q0 and Q1 once and streams the 128-key K tiles, warp 11 the V tiles (TMA
//    boxes of 16 or 8 slots of the kv head, 64-column halves, 128-byte swizzle; one lane per
//    box, each looking up its page a tile ahead) through one ring of stages (four of 32 KB at
//    head_dim 128), K_0, V_0, K_1, V_1, ...;
//  * warp 9 owns all 512 tensor-memory columns -- S0, S1 (128 fp32 columns each, P written
//    over them as bf16) and O0, O1 (D columns each).  Warp 9 issues the MMAs of Q0 and warp
//    10 those of Q1, per K/V tile j: S_X = Q_X K_j^T (N = 128: both operands from shared
//    memory at the full MMA rate), then O_X += P_X V_j (P from tensor memory);
//  * warps 0-3 run the softmax of Q0, warps 4-7 that of Q1 (thread = query row = TMEM
//    lane).  The two groups take turns (a token passed through two mbarriers): while one
//    group turns S into P the tensor pipe runs the other tile's MMAs -- PV1_{j-1} and S1_j
//    under the softmax of S0_j, PV0_j and S0_{j+1} under that of S1_j -- and neither group
//    shares the SM sub-partitions with the other during its exp pass.  At head_dim 64 a group
//    passes the turn on once it has loaded S, so the other group's load overlaps its exp pass.
//  * Each S_X overwrites the columns that PV_X of the previous tile read P from, so S_X(j+1)
//    is issued once PV_X(j) has completed; the other tile's MMAs keep the pipe busy meanwhile.
//  * The running maximum moves (and O is rescaled in tensor memory) only when it grows by more
//    than 2^8; the epilogue divides O by the row sum and stores bf16 rows and the lse.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "prefill_kernel.cuh"

namespace pkv {
namespace dev {

constexpr int kPpKeys = 128;     // keys per K / V tile
constexpr int kPpThreads = 384;  // warps 0-3 softmax of Q0, 4-7 of Q1, 8 / 11 producers, 9 / 10 MMA of Q0 / Q1
// Registers: the kernel is launched with 168 per thread (384 x 168 = 64,512 of the SM's 65,536);
// warp group 2 (producer, MMA) gives most of its share to the two softmax groups with
// setmaxnreg: 128 x 96 + 256 x 200 = 63,488.
constexpr int kPpLaunchRegs = 168;
constexpr int kPpSoftmaxRegs = 200;
constexpr int kPpOtherRegs = 96;
static_assert(128 * kPpOtherRegs + 256 * kPpSoftmaxRegs <= kPpThreads * kPpLaunchRegs, "setmaxnreg split fits the launch");

template <int D>
struct PpSmem {
    static constexpr int HALVES = D / 64;
    // ring stages, each one K or one V tile (32 KB at head_dim 128, 16 KB at 64; eight of
    // the smaller ones also keep a second CTA, which could not get tensor memory, off the SM)
    static constexpr int STAGES = D == 64 ? 8 : 4;
    static constexpr uint32_t Q_TILE = 128u * D * 2;                // one query tile
    static constexpr uint32_t Q_HALF = Q_TILE / HALVES;             // its 64-column half
    static constexpr uint32_t KV_TILE = (uint32_t)kPpKeys * D * 2;  // one K or V tile
    static constexpr uint32_t KV_HALF = KV_TILE / HALVES;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t RING_OFF = 2 * Q_TILE;
    static constexpr uint32_t BAR_OFF = RING_OFF + STAGES * KV_TILE;
    static constexpr uint32_t BYTES = BAR_OFF + 256;
};

// Shared-memory descriptors differ only in their start-address field (bits 0..13, in 16-byte
// units), so a descriptor for base + off is the base's plus off >> 4 (no carry: every
// address here is below 256 KB).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off_bytes) { return d + (off_bytes >> 4); }

template <int D, int G>
__global__ void __launch_bounds__(kPpThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q, const PrefillArgs a) {
    using L = PpSmem<D>;
    constexpr int HALVES = L::HALVES;
    constexpr int BQ = kPrefillRowsPerTile / G;          // tokens per query tile
    constexpr uint32_t Q_TX = (uint32_t)BQ * G * D * 2;  // rows BQ*G..127 stay unused
    constexpr int KSTEPS = D / 16;                       // k-steps of S = Q K^T
    constexpr int PSTEPS = kPpKeys / 16;                 // k-steps of O += P V
    constexpr int NS = L::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BAR_OFF);
    // Every barrier below completes once per K/V tile (q_full and o_final once per CTA); a
    // waiter is never two phases behind, because the next phase needs something the waiter
    // itself has yet to provide (see each wait).
    uint64_t *q_full = bars + 0;     // [2] Q_X landed
    uint64_t *kv_full = bars + 2;    // [NS <= 8] ring stage landed
    uint64_t *kv_empty = bars + 10;  // [NS] the MMAs reading a ring stage completed
    uint64_t *s_full = bars + 18;    // [2] S_X(j) in tensor memory
    uint64_t *p_full = bars + 20;    // [2] P_X(j) written (and O_X rescaled if it had to be)
    uint64_t *pv_done = bars + 22;   // [2] PV_X(j) completed
    uint64_t *o_final = bars + 24;   // [2] the last PV_X completed
    uint64_t *v_tail = bars + 26;    // warp 9 zeroed the V tail rows (at most once per CTA)
    // turn[X]: the softmax group of Q_X may start its next tile (the two groups take turns,
    // so neither shares the SM sub-partitions with the other and the pipe runs the other
    // tile's MMAs meanwhile); turn[1] completes a phase when group 0 finished tile j, turn[0]
    // when group 1 did
    uint64_t *turn = bars + 27;      // [2]
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 29);

    if ((int)blockIdx.x >= a.hdr->pf_tiles) return;  // an idle CTA of a launch at the maxima
    const PrefillTile t = a.tiles[blockIdx.x];
    int *const err = &a.hdr->err;
    const int causal = a.hdr->causal;
    const int window_left = a.hdr->window_left;
    const bool dense = a.hdr->dense != 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int P = a.page_size;
    const bool two = t.n_q > BQ;  // the tile's tokens reach into Q1
    const int kt0 = t.key_begin / kPpKeys;
    const int nt = (t.key_end + kPpKeys - 1) / kPpKeys - kt0;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(&q_full[x], 1);
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);
            mbar_init(&pv_done[x], 1);
            mbar_init(&o_final[x], 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], two ? 2 : 1);  // one commit per issuing warp
        }
        mbar_init(v_tail, 1);
        mbar_init(&turn[0], 4);
        mbar_init(&turn[1], 4);
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();  // q, the cache (or K / V) may come from the previous kernel
    griddep_launch();
    const uint32_t tmem = *tmem_holder;
    // S_X at columns 128 X, O_X at 256 + D X (computed, not indexed from an array: an array
    // indexed by X would live in local memory and be reloaded after every MMA, whose inline
    // asm clobbers memory)
    auto S_col = [tmem](int x) { return tmem + 128u * (uint32_t)x; };
    auto O_col = [tmem](int x) { return tmem + 256u + (uint32_t)(D * x); };
    // each warp group changes its register share at the top of its own branch (all four
    // warps of a group execute the same setmaxnreg)
    if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPpOtherRegs));
    if (warp == 8 || warp == 11) {
        // ------------------------------------------------ producers: warp 8 Q and K, warp 11 V
        if (warp == 8) {
            if constexpr (BQ * G < kPrefillRowsPerTile) {
                // a group size that does not divide 128 leaves Q rows BQ*G..127 of both tiles
                // unloaded: zero them (their S rows are never stored, but must not hold NaN)
                constexpr int ZROWS = kPrefillRowsPerTile - BQ * G;
                for (int i = lane; i < 2 * HALVES * ZROWS * 8; i += 32) {
                    const int x = i / (HALVES * ZROWS * 8), rem = i % (HALVES * ZROWS * 8);
                    const int h = rem / (ZROWS * 8), r = BQ * G + (rem / 8) % ZROWS, c = rem % 8;
                    *reinterpret_cast<uint4 *>(sm + L::Q_OFF + x * L::Q_TILE + h * L::Q_HALF + r * 128 + c * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                prefetch_tmap(&tm_kv);
                prefetch_tmap(&tm_v);
                prefetch_tmap(&tm_q);
                for (int x = 0; x < (two ? 2 : 1); ++x) {
                    mbar_arrive_expect_tx(&q_full[x], Q_TX);
#pragma unroll
                    for (int h = 0; h < HALVES; ++h)
                        tma_load_3d(sm + L::Q_OFF + x * L::Q_TILE + h * L::Q_HALF, &tm_q, &q_full[x], h * 64,
                                    t.kv_head * G, t.q_begin + x * BQ);
                }
            }
        }
        // A 128-key tile is NB boxes of R = 128 / NB rows (16, or 8 for 8-slot pages); lane b < NB
        // copies box b (its HALVES 64-column halves) and looks up the box's page one tile ahead.
        const int kv = warp == 11;  // 0: K tiles (ring slots 2j), 1: V tiles (2j + 1)
        const int NB = (dense || a.box_rows == 16) ? 8 : 16;
        const int R = kPpKeys / NB;
        const int npages = (t.length + P - 1) >> a.page_shift;
        const CUtensorMap *map = (kv && dense) ? &tm_v : &tm_kv;
        const int voff = (kv && !dense) ? P : 0;
        // cache row of box `lane` of tile j (a.oob_row past the row's pages: TMA reads zeros;
        // dense: rows past the segment are masked keys with finite V)
        auto box_row = [&](int j) {
            const int kb = (kt0 + j) * kPpKeys + lane * R;
            if (dense) return t.kv_base + kb;
            return (kb >> a.page_shift) < npages
                       ? a.pages[t.kv_base + (kb >> a.page_shift)] * 2 * P + (kb & (P - 1)) + voff
                       : a.oob_row;
        };
        int row = (lane < NB && nt > 0) ? box_row(0) : 0;
        for (int j = 0; j < nt; ++j) {
            const uint32_t i = 2u * j + kv;
            const int s = i % NS;
            const uint32_t use = i / NS;
            // the MMAs that read this stage use-1 rounds ago must have completed
            if (use > 0 && !mbar_wait(&kv_empty[s], (use - 1) & 1, err, kErrWaitEmpty)) break;
            if (lane == 0) mbar_arrive_expect_tx(&kv_full[s], L::KV_TILE);
            __syncwarp();
            uint8_t *dst = sm + L::RING_OFF + s * L::KV_TILE;
            if (lane < NB) {
#pragma unroll
                for (int h = 0; h < HALVES; ++h)
                    tma_load_3d(dst + h * L::KV_HALF + lane * R * 128, map, &kv_full[s], h * 64, row, t.kv_head);
                if (j + 1 < nt) row = box_row(j + 1);  // lands while the next slot is awaited
            }
        }
    } else if (warp == 9 || (warp == 10 && two)) {
        // ------------------------------------------------ MMA issue: warp 9 for Q0, warp 10 for Q1
        // A tcgen05.mma holds its issuing thread until the tensor core takes it (about one MMA
        // deep), so an issuing thread that waits or commits leaves the pipe idle; with one
        // issuing warp per query tile, one of them issues while the other waits.
        const int x = warp - 9;
        constexpr uint32_t ID_S = idesc_bf16_f32(128, kPpKeys, 0, 0);
        constexpr uint32_t ID_O = idesc_bf16_f32(128, D, 0, 1);
        // descriptors of the first k-step of Q_X, of a K tile and of a V tile in ring stage 0
        // (K-major operands: 16-byte leading offset, 8-row groups 1024 bytes apart; V MN-major:
        // its 64-column halves L::KV_HALF apart)
        const uint64_t dQ = smem_desc(smem_u32(sm + L::Q_OFF + x * L::Q_TILE), 16, 1024, kSwizzle128B);
        const uint64_t dK = smem_desc(smem_u32(sm + L::RING_OFF), 16, 1024, kSwizzle128B);
        const uint64_t dV = smem_desc(smem_u32(sm + L::RING_OFF), L::KV_HALF, 1024, kSwizzle128B);
        const uint32_t Sx = S_col(x), Ox = O_col(x);
        const int tail_begin = t.length;
        const int tail_end = (t.length + P - 1) & ~(P - 1);
        bool ok = mbar_wait(&q_full[x], 0, err, kErrWaitFull);
        uint32_t i = 0;  // ring slot sequence, as the producer counts it
        if (ok && nt > 0) ok = mbar_wait(&kv_full[0], 0, err, kErrWaitFull);
        for (int j = 0; j < nt && ok; ++j, i += 2) {
            const int sk = i % NS, sv = (i + 1) % NS;
            // S_X(j) overwrites P_X(j-1), which PV_X(j-1) reads: wait until it completed (PV_X(j)
            // cannot complete before this warp issues it, so the parity is exact)
            if (j > 0) ok = mbar_wait(&pv_done[x], (j - 1) & 1, err, kErrWaitFull);
            if (!ok) break;
            tc_fence_after();
            {
                const uint64_t k = desc_add(dK, sk * L::KV_TILE);
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk)
                    mma_ss_elect(Sx, desc_add(dQ, (kk / 4) * L::Q_HALF + (kk % 4) * 32),
                                 desc_add(k, (kk / 4) * L::KV_HALF + (kk % 4) * 32), ID_S, kk > 0 ? 1u : 0u);
                mma_commit_elect(&s_full[x]);
                mma_commit_elect(&kv_empty[sk]);  // K_j's stage frees once both tiles' S MMAs completed
            }
            ok = mbar_wait(&kv_full[sv], ((i + 1) / NS) & 1, err, kErrWaitFull);
            if (!ok) break;
            // V rows of the row's last page past its end (poisoned or stale slots: their P is 0,
            // but 0 * NaN would poison O) are zeroed by warp 9; warp 10 waits for that on the
            // one tile that has them (the last: keys never reach past the row's end)
            const int key0 = (kt0 + j) * kPpKeys;
            const int zb = max(tail_begin, key0), ze = min(tail_end, key0 + kPpKeys);
            if (zb < ze) {
                if (x == 0) {
                    uint8_t *vs = sm + L::RING_OFF + sv * L::KV_TILE;
                    const int nz = (ze - zb) * (D / 8);
                    for (int e = lane; e < nz; e += 32) {
                        const int k = zb - key0 + e / (D / 8);
                        const int chunk = e % (D / 8);
                        *reinterpret_cast<uint4 *>(vs + (chunk >> 3) * L::KV_HALF + swz128(k, chunk & 7)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && two) mbar_arrive(v_tail);
                } else {
                    ok = mbar_wait(v_tail, 0, err, kErrWaitFull);
                    if (!ok) break;
                }
            }
            // K_{j+1} is awaited here, while the softmax still runs, so that after PV_X(j) only
            // its own completion stands between it and S_X(j+1)
            if (j + 1 < nt) ok = mbar_wait(&kv_full[(i + 2) % NS], ((i + 2) / NS) & 1, err, kErrWaitFull);
            if (ok) ok = mbar_wait(&p_full[x], j & 1, err, kErrWaitFull);
            if (!ok) break;
            tc_fence_after();
            {
                const uint64_t v = desc_add(dV, sv * L::KV_TILE);
#pragma unroll
                for (int kk = 0; kk < PSTEPS; ++kk)  // 16 keys = 16 rows of 128 bytes per k-step
                    mma_ts_elect(Ox, Sx + kk * 8, desc_add(v, kk * 2048), ID_O, (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit_elect(&pv_done[x]);
                mma_commit_elect(&kv_empty[sv]);  // V_j's stage frees once both tiles' PV MMAs completed
                if (j == nt - 1) mma_commit_elect(&o_final[x]);
            }
        }
        if (nt == 0 && lane == 0) mma_commit(&o_final[x]);  // no MMA: arrives at once
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPpSoftmaxRegs));
        // ------------------------------------------------ softmax + epilogue (warps 0-7)
        const int x = warp >> 2;                  // query tile of this warp group
        const int m = (warp & 3) * 32 + lane;     // query row = TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        if (x == 0 || two) {
            const int tok = x * BQ + m / G;  // token within the work tile
            const int hd = t.kv_head * G + m % G;
            const bool live = m < BQ * G && tok < t.n_q;
            const int pos = t.pos0 + tok;
            const int hi = causal == 1 ? pos : t.length - 1;
            const int lo = window_left >= 0 ? max(0, pos - window_left) : 0;
            const float sl = a.hdr->scale_log2;
            const uint32_t Sx = S_col(x) + lane_off, Ox = O_col(x) + lane_off;
            float m_run = -INFINITY, l_run = 0.f;
            bool ok = true;
            for (int j = 0; j < nt; ++j) {
                const int key0 = (kt0 + j) * kPpKeys;
                // take turns with the other group: group 1 starts tile j after group 0 finished
                // it, group 0 starts tile j + 1 after group 1 finished tile j
                if (two && (x == 1 || j > 0) && !mbar_wait(&turn[x], (x ? j : j - 1) & 1, err, kErrWaitFull)) {
                    ok = false;
                    break;
                }
                // S_X(j+1) needs P_X(j) (through PV_X(j)), so this phase is the next one
                if (!mbar_wait(&s_full[x], j & 1, err, kErrWaitFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32(Sx, r0);
                tmem_ld32(Sx + 32, r1);
                tmem_ld32(Sx + 64, r2);
                tmem_ld32(Sx + 96, r3);
                tmem_wait_ld();
                if constexpr (D == 64) {
                    // head_dim 64 (half the MMA work per tile, so the softmax weighs more): the
                    // other group may start as soon as this one holds its S in registers
                    __syncwarp();
                    if (two && lane == 0) mbar_arrive(&turn[1 - x]);
                }
                float sv[kPpKeys];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sv[c] = __uint_as_float(r0[c]);
                    sv[32 + c] = __uint_as_float(r1[c]);
                    sv[64 + c] = __uint_as_float(r2[c]);
                    sv[96 + c] = __uint_as_float(r3[c]);
                }
                if (key0 < lo || key0 + kPpKeys - 1 > hi || key0 + kPpKeys > t.length) {
#pragma unroll
                    for (int c = 0; c < kPpKeys; ++c) {
                        const int k = key0 + c;
                        sv[c] = (k >= lo && k <= hi && k < t.length) ? sv[c] : -INFINITY;
                    }
                }
                // p = 2^(s * sl - mref), two columns per packed FMA; sums in four packed chains;
                // P goes back over the S columns as packed bf16 (64 columns), in two halves
                uint64_t acc[4];
                auto exp_pass = [&](float mref) {
                    const uint64_t sl2 = f2_make(sl, sl), nm2 = f2_make(-mref, -mref);
                    acc[0] = acc[1] = acc[2] = acc[3] = 0;
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
                        tmem_st32(Sx + hlf * 32, pk);
                    }
                };
                // the tile's row maximum: eight independent chains of 3-input max
                auto tile_max = [&]() {
                    float m8[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) m8[c] = fmaxf(sv[2 * c], sv[2 * c + 1]);
#pragma unroll
                    for (int c = 16; c < kPpKeys; c += 16)
#pragma unroll
                        for (int q = 0; q < 8; ++q) m8[q] = max3f(m8[q], sv[c + 2 * q], sv[c + 2 * q + 1]);
                    return max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * sl;
                };
                const float m_tile = tile_max();  // -inf when the whole tile is masked for this row
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
                exp_pass(m_run == -INFINITY ? 0.f : m_run);
                float u0, u1;
                f2_split(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), u0, u1);
                l_run = l_run * alpha + (u0 + u1);
                if constexpr (D != 64) {
                    __syncwarp();
                    if (two && lane == 0) mbar_arrive(&turn[1 - x]);  // the other group's turn
                }
                tmem_wait_st();
                if (warp_grow) {
                    // O holds P_0..P_{j-1} V: wait for the last of those MMAs, then scale O rows
                    // (PV_X(j) waits for this group's p_full, so nothing else touches O now)
                    if (!mbar_wait(&pv_done[x], (j - 1) & 1, err, kErrWaitFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tmem_ld32(Ox + c0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(Ox + c0, o);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[x]);
            }
            // epilogue
            if (ok && mbar_wait(&o_final[x], 0, err, kErrWaitFull)) {
                tc_fence_after();
                const bool none = l_run == 0.f;  // no visible key (empty context): o = 0, lse = -inf
                const float inv = none ? 0.f : 1.f / l_run;
                __nv_bfloat16 *orow = a.out + ((size_t)(t.q_begin + tok) * a.num_qo_heads + hd) * D;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(Ox + c0, o);
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

}  // namespace dev
}  // namespace pkv

// Ragged paged prefill over a cached prefix (FlashInferPrefillWrapper.run), also the
// prefill pass of the mixed step (FlashInferMixedWrapper).
//
// New token i of row r sits at position p = L_r - n_r + i and sees keys
// [lo, p] (causal, bottom-right aligned: "the cached prefix plus themselves") or
// [lo, L_r - 1] (non-causal), lo = max(0, p - window_left) or 0.
//
// A CTA takes one tile: up to BQ = 128 / g consecutive new tokens of one row and all g
// query heads of one kv head, i.e. 128 query rows sharing every K/V tile.  A producer
// thread streams 64-key stages (4 pages of that kv head, K and V, 64-column halves with
// 128-byte swizzle) by TMA; a page past the row's end is fetched at an out-of-range
// coordinate, which TMA fills with zeros.  Eight consumer warps own 16 query rows each
// and run QK^T and PV as 16x8x16 bf16 tensor-core MMAs with an exp2-domain online
// softmax.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "plan.h"
#include "ptx.cuh"

namespace pkv {
namespace dev {

struct PrefillArgs {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    float *lse;
    const PrefillTile *tiles;
    const int32_t *pages;
    int *err;
    int num_qo_heads;
    int page_size;
    int oob_row;       // a row coordinate past the cache: TMA fills it with zeros
    int stages;
    uint32_t stage_bytes;
    int causal;
    int window_left;
    float scale_log2;
};

constexpr int kConsumerWarps = 8;
constexpr float kLn2f = 0.6931471805599453f;

template <int D, int G>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap, const PrefillArgs a) {
    constexpr int HALVES = D / 64;
    constexpr int KEYS = kPrefillKeysPerStage;       // 64 keys per stage
    constexpr int BOX = 16 * 128;                    // one page (16 slots) x 64 columns
    constexpr int BLOCK = KEYS * 128;                // one (K|V, half) block of a stage
    constexpr int BQ = kPrefillRowsPerTile / G;      // query tokens per tile
    constexpr int KS = D / 16;
    constexpr int NT = D / 8;
    static_assert(KEYS == 4 * 16, "a stage is four 16-slot pages");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.stages * a.stage_bytes);
    uint64_t *empty = full + a.stages;

    const PrefillTile t = a.tiles[blockIdx.x];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int P = a.page_size;
    const int kt0 = t.key_begin / KEYS;
    const int kt1 = (t.key_end + KEYS - 1) / KEYS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            prefetch_tmap(&tmap);
            const int npages = (t.length + P - 1) / P;
            uint32_t it = 0;
            for (int kt = kt0; kt < kt1; ++kt, ++it) {
                const int s = it % a.stages;
                const uint32_t use = it / a.stages;
                if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.err, kErrWaitEmpty)) break;
                uint8_t *st = smem + (size_t)s * a.stage_bytes;
                mbar_arrive_expect_tx(&full[s], a.stage_bytes);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int pi = kt * 4 + j;
                    const int row0 = pi < npages ? a.pages[t.kv_base + pi] * 2 * P : a.oob_row;
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv)
#pragma unroll
                        for (int h = 0; h < HALVES; ++h)
                            tma_load_3d(st + (kv * HALVES + h) * BLOCK + j * BOX, &tmap, &full[s], h * 64,
                                        row0 + (pi < npages ? kv * P : 0), t.kv_head);
                }
            }
            const uint32_t issued = it;
            for (uint32_t k = issued > (uint32_t)a.stages ? issued - a.stages : 0; k < issued; ++k)
                if (!mbar_wait(&empty[k % a.stages], (k / a.stages) & 1, a.err, kErrWaitDrain)) break;
        }
        return;
    }

    // ---------------- consumers ----------------
    const int gid = lane >> 2;
    const int tid4 = lane & 3;
    const int Hq = a.num_qo_heads;
    const int m0r = warp * 16 + gid, m1r = m0r + 8;   // this thread's two query rows
    const int tok0 = m0r % BQ, tok1 = m1r % BQ;
    const int hd0 = t.kv_head * G + m0r / BQ, hd1 = t.kv_head * G + m1r / BQ;
    const bool live0 = tok0 < t.n_q, live1 = tok1 < t.n_q;
    const int p0 = t.pos0 + tok0, p1 = t.pos0 + tok1;
    const int hi0 = a.causal ? p0 : t.length - 1, hi1 = a.causal ? p1 : t.length - 1;
    const int lo0 = a.window_left >= 0 ? max(0, p0 - a.window_left) : 0;
    const int lo1 = a.window_left >= 0 ? max(0, p1 - a.window_left) : 0;

    uint32_t qa[KS][4];
    {
        const __nv_bfloat16 *q0 = a.q + ((size_t)(t.q_begin + tok0) * Hq + hd0) * D;
        const __nv_bfloat16 *q1 = a.q + ((size_t)(t.q_begin + tok1) * Hq + hd1) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int c0 = ks * 16 + tid4 * 2;
            qa[ks][0] = live0 ? *reinterpret_cast<const uint32_t *>(q0 + c0) : 0u;
            qa[ks][2] = live0 ? *reinterpret_cast<const uint32_t *>(q0 + c0 + 8) : 0u;
            qa[ks][1] = live1 ? *reinterpret_cast<const uint32_t *>(q1 + c0) : 0u;
            qa[ks][3] = live1 ? *reinterpret_cast<const uint32_t *>(q1 + c0 + 8) : 0u;
        }
    }
    const int k_tok = (lane & 7) + ((lane >> 4) << 3);
    const int k_chk = (lane >> 3) & 1;
    const int v_tok = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int v_chk = lane >> 4;

    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int tail_begin = t.length;                          // first key past the row
    const int tail_end = ((t.length + P - 1) / P) * P;        // end of the row's last page

    uint32_t it = 0;
    for (int kt = kt0; kt < kt1; ++kt, ++it) {
        const int s = it % a.stages;
        if (!mbar_wait(&full[s], (it / a.stages) & 1, a.err, kErrWaitFull)) return;
        uint8_t *st = smem + (size_t)s * a.stage_bytes;
        const uint32_t kb = smem_u32(st);
        const uint32_t vb = kb + HALVES * BLOCK;
        const int key0 = kt * KEYS;
        // zero the V slots of the row's last page past its end (every warp writes the
        // same zeros, then reads only after its own writes)
        const int zb = max(tail_begin, key0), ze = min(tail_end, key0 + KEYS);
        const bool zeroed = zb < ze;
        if (zeroed) {
            const int nz = (ze - zb) * (D / 8);
            for (int i = lane; i < nz; i += 32) {
                const int k = zb - key0 + i / (D / 8);
                const int chunk = i % (D / 8);
                *reinterpret_cast<uint4 *>(st + HALVES * BLOCK + (chunk >> 3) * BLOCK + swz128(k, chunk & 7)) =
                    make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }
        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int chunk = ks * 2 + k_chk;
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const uint32_t addr = kb + (chunk >> 3) * BLOCK + swz128(np * 16 + k_tok, chunk & 7);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(addr, b0, b1, b2, b3);
                mma_bf16_16816(sc[2 * np], qa[ks], b0, b1);
                mma_bf16_16816(sc[2 * np + 1], qa[ks], b2, b3);
            }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kp = key0 + n * 8 + tid4 * 2 + e;
                const bool v0 = kp >= lo0 && kp <= hi0 && kp < t.length;
                const bool v1 = kp >= lo1 && kp <= hi1 && kp < t.length;
                sc[n][e] = v0 ? sc[n][e] * a.scale_log2 : -INFINITY;
                sc[n][e + 2] = v1 ? sc[n][e + 2] * a.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, sc[n][e]);
                mx1 = fmaxf(mx1, sc[n][e + 2]);
            }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float r0 = mn0 == -INFINITY ? 0.f : mn0;
        const float r1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0 - r0), al1 = fast_exp2(m1 - r1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                sc[n][e] = fast_exp2(sc[n][e] - r0);
                sc[n][e + 2] = fast_exp2(sc[n][e + 2] - r1);
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
#pragma unroll
        for (int kk = 0; kk < KEYS / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
            pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
            pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
            for (int dj = 0; dj < D / 16; ++dj) {
                const int chunk = dj * 2 + v_chk;
                const uint32_t addr = vb + (chunk >> 3) * BLOCK + swz128(kk * 16 + v_tok, chunk & 7);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(addr, b0, b1, b2, b3);
                mma_bf16_16816(acc[2 * dj], pa, b0, b1);
                mma_bf16_16816(acc[2 * dj + 1], pa, b2, b3);
            }
        }
        if (zeroed) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    __nv_bfloat16 *o0 = a.out + ((size_t)(t.q_begin + tok0) * Hq + hd0) * D;
    __nv_bfloat16 *o1 = a.out + ((size_t)(t.q_begin + tok1) * Hq + hd1) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int c = n * 8 + tid4 * 2;
        if (live0) *reinterpret_cast<uint32_t *>(o0 + c) = pack_bf16(acc[n][0] * inv0, acc[n][1] * inv0);
        if (live1) *reinterpret_cast<uint32_t *>(o1 + c) = pack_bf16(acc[n][2] * inv1, acc[n][3] * inv1);
    }
    if (a.lse && tid4 == 0) {
        if (live0) a.lse[(size_t)(t.q_begin + tok0) * Hq + hd0] = (m0 + __log2f(l0)) * kLn2f;
        if (live1) a.lse[(size_t)(t.q_begin + tok1) * Hq + hd1] = (m1 + __log2f(l1)) * kLn2f;
    }
}

}  // namespace dev

static uint32_t prefill_stage_bytes(const Shape &s) {
    return (uint32_t)kPrefillKeysPerStage * 2u * (uint32_t)s.head_dim * 2u;
}
static int prefill_stages(const Shape &s) {
    int st = (int)((192u * 1024u) / prefill_stage_bytes(s));
    return st > 6 ? 6 : st;
}
size_t prefill_smem_bytes(const Shape &s) {
    return 1024 + (size_t)prefill_stages(s) * prefill_stage_bytes(s) + 2 * 8 * 8;
}

template <int D, int G>
static cudaError_t launch_prefill_t(const CUtensorMap &tm, const dev::PrefillArgs &a, int grid, size_t smem,
                                    cudaStream_t st) {
    auto fn = dev::prefill_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fn<<<grid, (dev::kConsumerWarps + 1) * 32, smem, st>>>(tm, a);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const Shape &s, const Plan &p, const CUtensorMap &tm, void *ws, const void *q, void *out,
                           float *lse, cudaStream_t st) {
    if (p.pf_tiles == 0) return cudaSuccess;
    uint8_t *w = static_cast<uint8_t *>(ws);
    dev::PrefillArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.tiles = reinterpret_cast<const PrefillTile *>(w + p.lay.pf_tiles);
    a.pages = reinterpret_cast<const int32_t *>(w + p.lay.pf_pages);
    a.err = reinterpret_cast<int *>(w + p.lay.err);
    a.num_qo_heads = s.num_qo_heads;
    a.page_size = s.page_size;
    a.oob_row = s.num_cache_pages * 2 * s.page_size;
    a.stages = prefill_stages(s);
    a.stage_bytes = prefill_stage_bytes(s);
    a.causal = p.causal;
    a.window_left = p.window_left;
    a.scale_log2 = p.sm_scale * 1.4426950408889634f;
    const size_t smem = prefill_smem_bytes(s);
    cudaError_t e = cudaErrorInvalidValue;
    const int g = s.group();
#define PKV_PF(DD, GG) \
    if (s.head_dim == DD && g == GG) e = launch_prefill_t<DD, GG>(tm, a, p.pf_tiles, smem, st);
    PKV_PF(64, 1) PKV_PF(64, 2) PKV_PF(64, 4) PKV_PF(64, 8) PKV_PF(64, 16)
    PKV_PF(128, 1) PKV_PF(128, 2) PKV_PF(128, 4) PKV_PF(128, 8) PKV_PF(128, 16)
#undef PKV_PF
    return e;
}

}  // namespace pkv

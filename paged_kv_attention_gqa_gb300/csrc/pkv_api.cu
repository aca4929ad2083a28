// The C ABI of libpkv (declared in include/pkv.h): handle, plan staging, launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/pkv.h"
#include "launch.h"
#include "plan.h"

using pkv::Plan;
using pkv::Shape;

struct pkv_handle_s {
    Shape shape{};
    std::string err;
    Plan plan;
    // the image buffer of the previous plan, handed to the next one so that building its
    // image reuses memory already mapped (the staged plan keeps no image)
    std::vector<uint8_t> spare_image;
    void *planned_ws = nullptr;
    // Page-locked staging ring (PinnedIndexRing: depth 2; a set is rewritten only after
    // the copy out of it has completed, fenced by an event recorded after that copy).
    void *pinned[2] = {nullptr, nullptr};
    size_t pinned_bytes[2] = {0, 0};
    cudaEvent_t fence[2] = {nullptr, nullptr};
    bool fence_live[2] = {false, false};
    int ring_at = 0;
    // side stream + fork/join events of the mixed step's concurrent passes
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    // last encoded tensor maps (re-encoded when the layer pointer changes)
    const void *tm_dec_ptr = nullptr, *tm_pf_ptr = nullptr, *tm_q_ptr = nullptr;
    int tm_q_rows = -1;
    CUtensorMap tm_dec{}, tm_pf{}, tm_q{};
    bool nvtx = false;  // one NVTX range per call (pkv_config.enable_nvtx)
};

// The NVTX range of one call on a handle with enable_nvtx set: opened here, closed when
// the call returns.
struct NvtxCall {
    bool on;
    NvtxCall(const pkv_handle_s *h, const char *name) : on(h && h->nvtx) {
        if (on) nvtxRangePushA(name);
    }
    ~NvtxCall() {
        if (on) nvtxRangePop();
    }
};

static thread_local std::string g_create_err;

static pkv_status fail(pkv_handle_t h, pkv_status st, const std::string &msg) {
    if (h)
        h->err = msg;
    else
        g_create_err = msg;
    return st;
}

static pkv_status cuda_fail(pkv_handle_t h, cudaError_t e, const char *what) {
    return fail(h, PKV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

extern "C" pkv_status pkv_create(const pkv_config *cfg, pkv_handle_t *out) {
    if (!cfg || !out) return fail(nullptr, PKV_ERR_INVALID, "null argument");
    const pkv_config &c = *cfg;
    if (c.num_qo_heads <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0 || c.page_size <= 0 || c.max_batch <= 0 ||
        c.max_total_tokens < 0 || c.max_num_pages <= 0 || c.num_cache_pages <= 0 || c.max_prefill_rows < 0 ||
        c.sm_count < 0)
        return fail(nullptr, PKV_ERR_INVALID, "configuration sizes must be positive");
    if (c.head_dim != 64 && c.head_dim != 128 && c.head_dim != 256)
        return fail(nullptr, PKV_ERR_UNSUPPORTED,
                    "head_dim " + std::to_string(c.head_dim) + " is not computed (64, 128, 256)");
    if ((c.page_size & (c.page_size - 1)) != 0 || c.page_size > 1024)
        return fail(nullptr, PKV_ERR_UNSUPPORTED,
                    "page_size " + std::to_string(c.page_size) + " is not computed (a power of two up to 1024)");
    if (c.num_qo_heads % c.num_kv_heads != 0)
        return fail(nullptr, PKV_ERR_UNSUPPORTED, "num_qo_heads must be a multiple of num_kv_heads");
    const int g = c.num_qo_heads / c.num_kv_heads;
    if (!((g >= 1 && g <= 8) || g == 16))
        return fail(nullptr, PKV_ERR_UNSUPPORTED, "group size " + std::to_string(g) + " is not computed (1..8, 16)");
    if (c.num_kv_heads > 256) return fail(nullptr, PKV_ERR_UNSUPPORTED, "num_kv_heads above 256 is not computed");
    if (c.sink_page >= c.num_cache_pages)
        return fail(nullptr, PKV_ERR_INVALID, "sink_page outside the cache");
    if (c.graph_static != 0 && c.graph_static != 1) return fail(nullptr, PKV_ERR_INVALID, "graph_static is 0 or 1");
    if (c.enable_nvtx != 0 && c.enable_nvtx != 1) return fail(nullptr, PKV_ERR_INVALID, "enable_nvtx is 0 or 1");
    if ((long long)c.num_cache_pages * 2 * c.page_size >= (1ll << 31))
        return fail(nullptr, PKV_ERR_UNSUPPORTED, "cache has too many pages for 32-bit slot rows");
    int sms = c.sm_count;
    if (sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(nullptr, PKV_ERR_CUDA, std::string("SM count query: ") + cudaGetErrorString(e));
    }
    pkv_handle_t h = new pkv_handle_s();
    h->shape = Shape{c.num_qo_heads, c.num_kv_heads, c.head_dim,       c.page_size, c.max_batch,
                     c.max_total_tokens, c.max_num_pages, c.num_cache_pages, c.max_prefill_rows,
                     sms,             c.sink_page,      c.graph_static};
    h->nvtx = c.enable_nvtx != 0;
    *out = h;
    return PKV_OK;
}

extern "C" void pkv_destroy(pkv_handle_t h) {
    if (!h) return;
    for (int i = 0; i < 2; ++i) {
        if (h->fence[i]) {
            if (h->fence_live[i]) cudaEventSynchronize(h->fence[i]);
            cudaEventDestroy(h->fence[i]);
        }
        if (h->pinned[i]) cudaFreeHost(h->pinned[i]);
    }
    if (h->side) {
        cudaStreamSynchronize(h->side);
        cudaStreamDestroy(h->side);
    }
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    delete h;
}

extern "C" const char *pkv_last_error(pkv_handle_t h) { return h ? h->err.c_str() : g_create_err.c_str(); }

extern "C" pkv_status pkv_workspace_size(pkv_handle_t h, int mode, size_t *bytes) {
    if (!h || !bytes) return fail(h, PKV_ERR_INVALID, "null argument");
    if (mode < PKV_MODE_DECODE || mode > PKV_MODE_DENSE) return fail(h, PKV_ERR_INVALID, "unknown mode");
    *bytes = pkv::workspace_bound(h->shape, mode);
    return PKV_OK;
}

// Copy a plan's integer image into the workspace through the page-locked ring (one
// async H2D) and make it the handle's current plan.
static pkv_status stage_plan(pkv_handle_t h, Plan &plan, void *workspace, size_t workspace_bytes,
                             pkv_stream_t stream) {
    if (plan.lay.total > workspace_bytes)
        return fail(h, PKV_ERR_WORKSPACE,
                    "workspace of " + std::to_string(workspace_bytes) + " bytes is too small: this plan needs " +
                        std::to_string(plan.lay.total) + " bytes (pkv_workspace_size gives the bound at the maxima)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int set = h->ring_at;
    h->ring_at ^= 1;
    cudaError_t e;
    if (!h->fence[set]) {
        e = cudaEventCreateWithFlags(&h->fence[set], cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(h, e, "event create");
    }
    if (h->fence_live[set]) {
        // the copy that last read this set must have completed before we rewrite it
        e = cudaEventSynchronize(h->fence[set]);
        if (e != cudaSuccess) return cuda_fail(h, e, "staging fence");
        h->fence_live[set] = false;
    }
    const size_t nbytes = plan.image.size();
    if (h->pinned_bytes[set] < nbytes) {
        if (h->pinned[set]) cudaFreeHost(h->pinned[set]);
        h->pinned[set] = nullptr;
        h->pinned_bytes[set] = 0;
        const size_t want = pkv::align_up(nbytes > (1u << 20) ? nbytes : (1u << 20), 1u << 20);
        e = cudaHostAlloc(&h->pinned[set], want, cudaHostAllocDefault);
        if (e != cudaSuccess) return cuda_fail(h, e, "pinned staging alloc");
        h->pinned_bytes[set] = want;
    }
    std::memcpy(h->pinned[set], plan.image.data(), nbytes);
    h->spare_image.swap(plan.image);
    e = cudaMemcpyAsync(workspace, h->pinned[set], nbytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "plan H2D");
    e = cudaEventRecord(h->fence[set], st);
    if (e != cudaSuccess) return cuda_fail(h, e, "staging fence record");
    h->fence_live[set] = true;
    h->plan = std::move(plan);
    h->planned_ws = workspace;
    return PKV_OK;
}


extern "C" pkv_status pkv_plan(pkv_handle_t h, int mode, const int32_t *qo_indptr, const int32_t *kv_indptr,
                               const int32_t *kv_indices, const int32_t *last_page_len, int batch, int causal,
                               int window_left, float sm_scale, void *workspace, size_t workspace_bytes,
                               pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_plan");
    if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
    if (!workspace) return fail(h, PKV_ERR_INVALID, "null workspace");
    if (reinterpret_cast<uintptr_t>(workspace) % pkv::kAlign)
        return fail(h, PKV_ERR_INVALID, "workspace must be 256-byte aligned");
    if (!(sm_scale >= 0.f) || std::isinf(sm_scale)) return fail(h, PKV_ERR_INVALID, "sm_scale must be finite and >= 0");
    if (mode == PKV_MODE_MIXED && h->shape.max_prefill_rows < 0) return fail(h, PKV_ERR_INVALID, "no mixed config");
    std::string err;
    Plan plan;
    plan.image.swap(h->spare_image);
    int rc = pkv::make_plan(h->shape, mode, qo_indptr, kv_indptr, kv_indices, last_page_len, batch, causal,
                            window_left, sm_scale, plan, err);
    h->planned_ws = nullptr;
    if (rc) {
        h->spare_image.swap(plan.image);
        return fail(h, (pkv_status)rc, err);
    }
    return stage_plan(h, plan, workspace, workspace_bytes, stream);
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map over one layer slice viewed as [Hkv][pages * 2 * page_size rows][D] with the
// head dimension OUTERMOST, so that a box of (64 columns, box_rows slots, heads) lands
// in shared memory head-major: each head's slots are consecutive 128-byte rows.
static pkv_status encode_rows(pkv_handle_t h, const void *base, long long rows, int box_rows, int box_heads,
                              CUtensorMap *tm);

static pkv_status encode_kv(pkv_handle_t h, const void *kv_layer, int box_rows, int box_heads, CUtensorMap *tm) {
    return encode_rows(h, kv_layer, (long long)h->shape.num_cache_pages * 2 * h->shape.page_size, box_rows, box_heads,
                       tm);
}

// Tensor map over [rows][Hkv][D] bf16 rows of Hkv*D elements (a layer slice viewed as
// pages*2*page_size rows, or a contiguous K or V tensor), boxes of (64 columns, box_rows
// rows, box_heads heads), heads outermost so that one head's rows land contiguously.
static pkv_status encode_rows(pkv_handle_t h, const void *kv_layer, long long rows, int box_rows, int box_heads,
                              CUtensorMap *tm) {
    auto fn = encode_fn();
    if (!fn) return fail(h, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const Shape &s = h->shape;
    if (reinterpret_cast<uintptr_t>(kv_layer) % 16) return fail(h, PKV_ERR_INVALID, "kv_layer must be 16-byte aligned");
    cuuint64_t dims[3] = {(cuuint64_t)s.head_dim, (cuuint64_t)rows, (cuuint64_t)s.num_kv_heads};
    cuuint64_t strides[2] = {(cuuint64_t)s.num_kv_heads * s.head_dim * 2, (cuuint64_t)s.head_dim * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_heads};
    if (rows < 1) return fail(h, PKV_ERR_INVALID, "a K / V tensor needs at least one row");
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(kv_layer), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(h, PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return PKV_OK;
}

// Tensor map over q viewed as [tokens][Hq][D]: a box of (64 columns, g heads, 128 / g
// tokens) lands as 128 query rows (token-major, head-minor) of 128 bytes, 128-byte swizzled.
static pkv_status q_map(pkv_handle_t h, const void *q, int rows) {
    if (h->tm_q_ptr == q && h->tm_q_rows == rows) return PKV_OK;
    auto fn = encode_fn();
    if (!fn) return fail(h, PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const Shape &s = h->shape;
    const int g = s.group();
    cuuint64_t dims[3] = {(cuuint64_t)s.head_dim, (cuuint64_t)s.num_qo_heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)s.head_dim * 2, (cuuint64_t)s.num_qo_heads * s.head_dim * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(pkv::kPrefillRowsPerTile / g)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&h->tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(h, PKV_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (" + std::to_string((int)r) + ")");
    h->tm_q_ptr = q;
    h->tm_q_rows = rows;
    return PKV_OK;
}

// Rows of q the tensor map covers: the plan's tokens, or the maxima in graph mode (a
// captured launch keeps the map it was captured with).
static int q_rows(pkv_handle_t h) {
    return h->shape.graph_static ? h->shape.max_total_tokens : h->plan.num_tokens;
}

static pkv_status check_planned(pkv_handle_t h, void *ws, int mode_a, int mode_b = -1) {
    if (!h) return PKV_ERR_INVALID;
    if (!h->planned_ws || h->planned_ws != ws)
        return fail(h, PKV_ERR_NOT_PLANNED, "no plan was made on this workspace by this handle");
    if (h->plan.mode != mode_a && h->plan.mode != mode_b)
        return fail(h, PKV_ERR_NOT_PLANNED, "the workspace holds a plan of another mode");
    return PKV_OK;
}

static pkv_status dec_map(pkv_handle_t h, const void *kv) {
    if (h->tm_dec_ptr == kv) return PKV_OK;
    pkv_status st = encode_kv(h, kv, h->shape.dec_box_rows(), h->shape.dec_heads(), &h->tm_dec);
    if (st == PKV_OK) h->tm_dec_ptr = kv;
    return st;
}

static pkv_status pf_map(pkv_handle_t h, const void *kv) {
    if (h->tm_pf_ptr == kv) return PKV_OK;
    // pages below 8 slots are gathered by the kernel; the map is then unused
    pkv_status st = encode_kv(h, kv, h->shape.pf_box_rows(), 1, &h->tm_pf);
    if (st == PKV_OK) h->tm_pf_ptr = kv;
    return st;
}

extern "C" pkv_status pkv_kv_append(pkv_handle_t h, const void *k, const void *v, int num_new_tokens, void *kv_layer,
                                    const int32_t *qo_indptr, const int32_t *kv_indptr, const int32_t *kv_indices,
                                    const int32_t *last_page_len, int batch, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_kv_append");
    if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
    if (num_new_tokens < 0 || batch < 0) return fail(h, PKV_ERR_INVALID, "num_new_tokens and batch must be >= 0");
    if (batch > h->shape.max_batch) return fail(h, PKV_ERR_INVALID, "batch above max_batch");
    if (!qo_indptr && num_new_tokens > batch)
        return fail(h, PKV_ERR_INVALID, "without qo_indptr every row has one new token (num_new_tokens <= batch)");
    if (num_new_tokens == 0 || batch == 0) return PKV_OK;
    if (!k || !v || !kv_layer || !kv_indptr || !kv_indices || !last_page_len)
        return fail(h, PKV_ERR_INVALID, "null k, v, kv_layer or index array");
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(kv_layer)) % 16)
        return fail(h, PKV_ERR_INVALID, "k, v and kv_layer must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(qo_indptr) | reinterpret_cast<uintptr_t>(kv_indptr) |
         reinterpret_cast<uintptr_t>(kv_indices) | reinterpret_cast<uintptr_t>(last_page_len)) % 4)
        return fail(h, PKV_ERR_INVALID, "index arrays must be 4-byte aligned");
    cudaError_t e = pkv::launch_append_indexed(h->shape, k, v, num_new_tokens, kv_layer, qo_indptr, kv_indptr,
                                               kv_indices, last_page_len, batch, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "append launch");
}

extern "C" pkv_status pkv_kv_append_planned(pkv_handle_t h, const void *k, const void *v, void *kv_layer,
                                            void *workspace, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_kv_append_planned");
    pkv_status st = check_planned(h, workspace, PKV_MODE_DECODE, PKV_MODE_PREFILL);
    if (st != PKV_OK && h && h->plan.mode == PKV_MODE_MIXED && h->planned_ws == workspace) st = PKV_OK;
    if (st != PKV_OK) return st;
    if (h->plan.num_append && (!k || !v || !kv_layer)) return fail(h, PKV_ERR_INVALID, "null k, v or kv_layer");
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(kv_layer)) % 16)
        return fail(h, PKV_ERR_INVALID, "k, v and kv_layer must be 16-byte aligned");
    cudaError_t e = pkv::launch_append(h->shape, h->plan, workspace, k, v, kv_layer, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "append launch");
}

static pkv_status check_io(pkv_handle_t h, const void *q, const void *kv, void *out) {
    if (!q || !kv || !out) return fail(h, PKV_ERR_INVALID, "null q, kv_layer or out");
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) % 16)
        return fail(h, PKV_ERR_INVALID, "q and out must be 16-byte aligned");
    return PKV_OK;
}

extern "C" pkv_status pkv_run_decode(pkv_handle_t h, const void *q, const void *kv_layer, void *out, float *lse,
                                     void *workspace, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_run_decode");
    pkv_status st = check_planned(h, workspace, PKV_MODE_DECODE);
    if (st != PKV_OK) return st;
    if (h->plan.batch == 0) return PKV_OK;
    if ((st = check_io(h, q, kv_layer, out)) != PKV_OK) return st;
    if ((st = dec_map(h, kv_layer)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_decode(h->shape, h->plan, h->tm_dec, workspace, q, const_cast<void *>(kv_layer), out,
                                       lse, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "decode launch");
}

extern "C" pkv_status pkv_run_decode_append(pkv_handle_t h, const void *q, const void *k, const void *v,
                                            void *kv_layer, void *out, float *lse, void *workspace,
                                            pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_run_decode_append");
    pkv_status st = check_planned(h, workspace, PKV_MODE_DECODE);
    if (st != PKV_OK) return st;
    if (h->plan.batch == 0) return PKV_OK;
    if ((st = check_io(h, q, kv_layer, out)) != PKV_OK) return st;
    if (!k || !v) return fail(h, PKV_ERR_INVALID, "null k or v");
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(kv_layer)) % 16)
        return fail(h, PKV_ERR_INVALID, "k, v and kv_layer must be 16-byte aligned");
    if ((st = dec_map(h, kv_layer)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_decode(h->shape, h->plan, h->tm_dec, workspace, q, kv_layer, out, lse,
                                       static_cast<cudaStream_t>(stream), k, v);
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "decode + append launch");
}

extern "C" pkv_status pkv_run_prefill(pkv_handle_t h, const void *q, const void *kv_layer, void *out, float *lse,
                                      void *workspace, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_run_prefill");
    pkv_status st = check_planned(h, workspace, PKV_MODE_PREFILL);
    if (st != PKV_OK) return st;
    if (h->plan.num_tokens == 0) return PKV_OK;
    if ((st = check_io(h, q, kv_layer, out)) != PKV_OK) return st;
    if ((st = pf_map(h, kv_layer)) != PKV_OK) return st;
    if ((st = q_map(h, q, q_rows(h))) != PKV_OK) return st;
    cudaError_t e = pkv::launch_prefill(h->shape, h->plan, h->tm_pf, h->tm_pf, h->tm_q, kv_layer, workspace, out, lse,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "prefill launch");
}

extern "C" pkv_status pkv_run_mixed(pkv_handle_t h, const void *q, const void *kv_layer, void *out, float *lse,
                                    void *workspace, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_run_mixed");
    pkv_status st = check_planned(h, workspace, PKV_MODE_MIXED);
    if (st != PKV_OK) return st;
    if (h->plan.num_tokens == 0) return PKV_OK;
    if ((st = check_io(h, q, kv_layer, out)) != PKV_OK) return st;
    if ((st = dec_map(h, kv_layer)) != PKV_OK) return st;
    if ((st = pf_map(h, kv_layer)) != PKV_OK) return st;
    if ((st = q_map(h, q, q_rows(h))) != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The two passes write disjoint tokens and only read the cache: the decode pass (HBM-
    // bound, on the SMs the plan gave it) runs on `stream`, the prefill pass (tensor-bound)
    // on a side stream forked from it and joined back.
    cudaError_t e = cudaSuccess;
    if (!h->side) {
        e = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(h, e, "side stream (make the first mixed run outside a capture)");
    }
    e = cudaEventRecord(h->ev_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->ev_fork, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "mixed fork");
    e = pkv::launch_decode(h->shape, h->plan, h->tm_dec, workspace, q, const_cast<void *>(kv_layer), out, lse, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "mixed decode-pass launch");
    e = pkv::launch_prefill(h->shape, h->plan, h->tm_pf, h->tm_pf, h->tm_q, kv_layer, workspace, out, lse, h->side);
    if (e != cudaSuccess) return cuda_fail(h, e, "mixed prefill-pass launch");
    e = cudaEventRecord(h->ev_join, h->side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->ev_join, 0);
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "mixed join");
}

extern "C" pkv_status pkv_check_device_error(pkv_handle_t h, void *workspace, pkv_stream_t stream, int *code) {
    NvtxCall nvtx_range(h, "pkv_check_device_error");
    if (!h || !workspace || !code) return fail(h, PKV_ERR_INVALID, "null argument");
    if (h->planned_ws != workspace) return fail(h, PKV_ERR_NOT_PLANNED, "no plan on this workspace");
    int v = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&v, static_cast<uint8_t *>(workspace) + h->plan.lay.err, sizeof(int),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, e, "error word read");
    *code = v;
    if (v) {
        const int zero = 0;
        e = cudaMemcpyAsync(static_cast<uint8_t *>(workspace) + h->plan.lay.err, &zero, sizeof(int),
                            cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        return fail(h, PKV_ERR_DEVICE, "a kernel gave up waiting (device error " + std::to_string(v) + ")");
    }
    return PKV_OK;
}

extern "C" pkv_status pkv_selftest_wait_timeout(pkv_handle_t h, void *workspace, int polls, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_selftest_wait_timeout");
    if (!h || !workspace) return fail(h, PKV_ERR_INVALID, "null argument");
    if (polls < 1 || polls > (1 << 20)) return fail(h, PKV_ERR_INVALID, "polls must be in [1, 2^20]");
    if (h->planned_ws != workspace) return fail(h, PKV_ERR_NOT_PLANNED, "no plan on this workspace");
    cudaError_t e = pkv::launch_selftest_wait(h->plan, workspace, (uint32_t)polls, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "self-test launch");
}

// ---------------- host-only queries ----------------

extern "C" pkv_status pkv_append_slots(int page_size, const int32_t *qo, const int32_t *kvp, const int32_t *kvi,
                                       const int32_t *lpl, int batch, int32_t *pages, int32_t *slots) {
    if (!kvp || !lpl || !pages || !slots || page_size <= 0 || batch < 0) return PKV_ERR_INVALID;
    std::string err;
    return (pkv_status)pkv::append_slots(page_size, qo, kvp, kvi, lpl, batch, pages, slots, err);
}

extern "C" pkv_status pkv_context_only_views(int page_size, const int32_t *qo, const int32_t *kvp, const int32_t *kvi,
                                             const int32_t *lpl, int batch, int32_t *out_kvp, int32_t *out_kvi,
                                             int32_t *out_lpl, int *out_nnz) {
    if (!qo || !kvp || !lpl || !out_kvp || !out_lpl || !out_nnz || page_size <= 0 || batch < 0) return PKV_ERR_INVALID;
    if (kvp[batch] > 0 && (!kvi || !out_kvi)) return PKV_ERR_INVALID;
    std::string err;
    return (pkv_status)pkv::context_only_views(page_size, qo, kvp, kvi, lpl, batch, out_kvp, out_kvi, out_lpl, out_nnz,
                                               err);
}

extern "C" pkv_status pkv_mixed_layout(const int32_t *qo, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl,
                                       int batch, int max_prefill_rows, int sink_page, int32_t *is_decode,
                                       int32_t *prompt_rows, int32_t *perm, int32_t *pf_qo_indptr,
                                       int32_t *dec_kv_indptr, int32_t *dec_kv_indices, int32_t *dec_last_page_len,
                                       int32_t *dec_q_token, int32_t *dec_out_token, int *dec_nnz) {
    if (!qo || !kvp || !lpl || batch < 0 || max_prefill_rows < 0) return PKV_ERR_INVALID;
    std::string err;
    pkv::MixedLayout m;
    int rc = pkv::mixed_layout(qo, kvp, kvi, lpl, batch, max_prefill_rows, sink_page, m, err);
    if (rc) return (pkv_status)rc;
    auto cp = [](int32_t *dst, const std::vector<int32_t> &src) {
        if (dst && !src.empty()) std::memcpy(dst, src.data(), src.size() * sizeof(int32_t));
    };
    cp(is_decode, m.is_decode);
    cp(prompt_rows, m.prompt_rows);
    cp(perm, m.perm);
    cp(pf_qo_indptr, m.pf_qo_indptr);
    cp(dec_kv_indptr, m.dec_kv_indptr);
    cp(dec_kv_indices, m.dec_kv_indices);
    cp(dec_last_page_len, m.dec_last_page_len);
    cp(dec_q_token, m.dec_q_token);
    cp(dec_out_token, m.dec_out_token);
    if (dec_nnz) *dec_nnz = (int)m.dec_kv_indices.size();
    return PKV_OK;
}

extern "C" pkv_status pkv_decode_split(pkv_handle_t h, const int32_t *kvp, const int32_t *lpl, int batch,
                                       int window_left, int32_t *tiles, int *num_tiles, int *num_ctas) {
    NvtxCall nvtx_range(h, "pkv_decode_split");
    if (!h || !kvp || !lpl || !tiles || !num_tiles || !num_ctas || batch < 0) return PKV_ERR_INVALID;
    std::vector<int32_t> qt(batch), ot(batch);
    for (int r = 0; r < batch; ++r) qt[r] = ot[r] = r;
    std::vector<pkv::DecodeTile> dt;
    std::vector<int32_t> cta;
    std::vector<pkv::MergeRow> mg;
    int parts = 0;
    pkv::decode_split(h->shape, batch, kvp, lpl, qt.data(), ot.data(), window_left, dt, cta, mg, parts);
    if ((int)dt.size() > *num_tiles) return fail(h, PKV_ERR_INVALID, "tile buffer too small");
    int c = 0;
    for (size_t i = 0; i < dt.size(); ++i) {
        while (cta[c + 1] <= (int)i) ++c;
        int32_t *o = tiles + 5 * i;
        o[0] = dt[i].q_token;
        o[1] = dt[i].page_begin;
        o[2] = dt[i].page_count;
        o[3] = dt[i].partial;
        o[4] = c;
    }
    *num_tiles = (int)dt.size();
    *num_ctas = dt.empty() ? 0 : (int)cta.size() - 1;
    return PKV_OK;
}

extern "C" pkv_status pkv_decode_head_rows(pkv_handle_t h, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl,
                                           int batch, int window_left, int32_t *rows, int *num_ctas) {
    NvtxCall nvtx_range(h, "pkv_decode_head_rows");
    if (!h || !kvp || !kvi || !lpl || !rows || !num_ctas || batch < 0) return PKV_ERR_INVALID;
    std::string err;
    const int rc = pkv::validate_rows(h->shape, PKV_MODE_DECODE, nullptr, kvp, kvi, lpl, batch, window_left, err);
    if (rc) return fail(h, (pkv_status)rc, err);
    std::vector<int32_t> qt(batch), ot(batch);
    for (int r = 0; r < batch; ++r) qt[r] = ot[r] = r;
    std::vector<pkv::DecodeTile> dt;
    std::vector<int32_t> cta;
    std::vector<pkv::MergeRow> mg;
    int parts = 0;
    pkv::decode_split(h->shape, batch, kvp, lpl, qt.data(), ot.data(), window_left, dt, cta, mg, parts);
    const int ctas = dt.empty() ? 0 : (int)cta.size() - 1;
    if (ctas > *num_ctas) return fail(h, PKV_ERR_INVALID, "row buffer too small");
    const std::vector<int32_t> hr = pkv::decode_head_rows(h->shape, dt, cta, kvi);
    std::copy(hr.begin(), hr.end(), rows);
    *num_ctas = ctas;
    return PKV_OK;
}

// ---------------- decode without a caller workspace ----------------

extern "C" pkv_status pkv_run_decode_static(pkv_handle_t h, const void *q, const void *kv_layer, void *out,
                                            float *lse, const int32_t *kv_indptr, const int32_t *kv_indices,
                                            const int32_t *last_page_len, int batch, int window_left, float sm_scale,
                                            pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_run_decode_static");
    if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
    if (!(sm_scale >= 0.f) || std::isinf(sm_scale)) return fail(h, PKV_ERR_INVALID, "sm_scale must be finite and >= 0");
    {
        // The plan below is copied from host memory that is freed when this call returns;
        // recorded into a graph, that copy would read freed memory when replayed.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t ce = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs);
        if (ce != cudaSuccess) return cuda_fail(h, ce, "stream capture status");
        if (cs != cudaStreamCaptureStatusNone)
            return fail(h, PKV_ERR_INVALID,
                        "pkv_run_decode_static copies its plan from host memory it frees on return, so it does "
                        "not run on a stream that is capturing");
    }
    std::string err;
    Plan plan;
    int rc = pkv::make_plan(h->shape, PKV_MODE_DECODE, nullptr, kv_indptr, kv_indices, last_page_len, batch, 1,
                            window_left, sm_scale, plan, err);
    if (rc) return fail(h, (pkv_status)rc, err);
    if (plan.lay.total > pkv::static_scratch_bytes())
        return fail(h, PKV_ERR_WORKSPACE,
                    "this decode needs " + std::to_string(plan.lay.total) + " bytes of scratch, above the " +
                        std::to_string(pkv::static_scratch_bytes()) +
                        "-byte static scratch of pkv_run_decode_static; use pkv_plan + pkv_run_decode with a workspace");
    if (batch == 0) return PKV_OK;
    pkv_status st = check_io(h, q, kv_layer, out);
    if (st != PKV_OK) return st;
    void *scratch = nullptr;
    cudaError_t e = pkv::static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail(h, e, "static scratch address");
    if ((st = dec_map(h, kv_layer)) != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The plan image (its error word zeroed) overwrites the previous call's contents.
    e = cudaMemcpyAsync(scratch, plan.image.data(), plan.image.size(), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "static plan H2D");
    e = pkv::launch_decode(h->shape, plan, h->tm_dec, scratch, q, const_cast<void *>(kv_layer), out, lse, s);
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "static decode launch");
}

// ---------------- dense varlen attention ----------------

extern "C" pkv_status pkv_plan_dense(pkv_handle_t h, const int32_t *cu_q, const int32_t *cu_k, int batch, int causal,
                                     int window_left, float sm_scale, void *workspace, size_t workspace_bytes,
                                     pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_plan_dense");
    if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
    if (!workspace) return fail(h, PKV_ERR_INVALID, "null workspace");
    if (reinterpret_cast<uintptr_t>(workspace) % pkv::kAlign)
        return fail(h, PKV_ERR_INVALID, "workspace must be 256-byte aligned");
    if (!(sm_scale >= 0.f) || std::isinf(sm_scale)) return fail(h, PKV_ERR_INVALID, "sm_scale must be finite and >= 0");
    std::string err;
    Plan plan;
    plan.image.swap(h->spare_image);
    int rc = pkv::make_dense_plan(h->shape, cu_q, cu_k, batch, causal, window_left, sm_scale, plan, err);
    h->planned_ws = nullptr;
    if (rc) {
        h->spare_image.swap(plan.image);
        return fail(h, (pkv_status)rc, err);
    }
    return stage_plan(h, plan, workspace, workspace_bytes, stream);
}

extern "C" pkv_status pkv_run_dense(pkv_handle_t h, const void *q, const void *k, const void *v, void *out, float *lse,
                                    void *workspace, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_run_dense");
    pkv_status st = check_planned(h, workspace, PKV_MODE_DENSE);
    if (st != PKV_OK) return st;
    if (h->plan.num_tokens == 0) return PKV_OK;
    if ((st = check_io(h, q, k, out)) != PKV_OK) return st;
    if (!v || (reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16)
        return fail(h, PKV_ERR_INVALID, "k and v must be non-null and 16-byte aligned");
    CUtensorMap tk, tv;
    if ((st = encode_rows(h, k, h->plan.num_keys, 16, 1, &tk)) != PKV_OK) return st;
    if ((st = encode_rows(h, v, h->plan.num_keys, 16, 1, &tv)) != PKV_OK) return st;
    if ((st = q_map(h, q, h->plan.num_tokens)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_prefill(h->shape, h->plan, tk, tv, h->tm_q, nullptr, workspace, out, lse,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "dense launch");
}

extern "C" pkv_status pkv_gather_kv(pkv_handle_t h, const void *kv_layer, const int32_t *pages, int num_tokens,
                                    void *k_out, void *v_out, pkv_stream_t stream) {
    NvtxCall nvtx_range(h, "pkv_gather_kv");
    if (!h) return fail(h, PKV_ERR_INVALID, "null handle");
    if (num_tokens < 0) return fail(h, PKV_ERR_INVALID, "num_tokens must be >= 0");
    if (num_tokens == 0) return PKV_OK;
    if (!kv_layer || !pages || !k_out || !v_out) return fail(h, PKV_ERR_INVALID, "null argument");
    if ((reinterpret_cast<uintptr_t>(kv_layer) | reinterpret_cast<uintptr_t>(k_out) |
         reinterpret_cast<uintptr_t>(v_out)) % 16)
        return fail(h, PKV_ERR_INVALID, "kv_layer, k_out and v_out must be 16-byte aligned");
    cudaError_t e = pkv::launch_gather(h->shape, kv_layer, pages, num_tokens, k_out, v_out,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : cuda_fail(h, e, "gather launch");
}

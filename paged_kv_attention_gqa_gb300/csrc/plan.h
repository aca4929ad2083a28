// Plan structures shared by the host planner and the kernels of libpkv.
//
// A plan is made once per step on the host (mstar.engine.resources.attn.wrappers,
// FlashInfer*Wrapper.plan) and read by every layer's append and run.  Its integer
// part is built in page-locked host memory and copied into the caller's workspace in
// one async H2D; the float part (split-KV partials) follows it in the same workspace
// (mstar.engine.resources.attn.workspace: "the scratch a plan reserves its split-KV
// partials in").
#pragma once
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

namespace pkv {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Query rows of one prefill tile: BQ tokens x all g q-heads of one kv head.
constexpr int kPrefillRowsPerTile = 128;
// Keys per prefill K/V stage.
constexpr int kPrefillKeysPerStage = 64;
// Keys per decode stage (one ring slot): two 8-key n-tiles of the QK^T MMA.
constexpr int kDecodeKeysPerStage = 16;
// Shared memory per SM given to decode rings (split among the SM's decode CTAs).
constexpr uint32_t kDecodeRingBytes = 200u * 1024u;

// First bytes of every plan in the workspace: the per-plan values the kernels read on
// the device, so that launches captured into a CUDA graph stay valid for later plans
// (their arguments are only pointers and static shapes).
struct PlanHeader {
    int32_t err;          // device error word (bounded waits that gave up)
    int32_t num_append;   // new tokens
    int32_t dec_ctas;     // decode CTAs with work
    int32_t num_merge;    // cut rows to merge
    int32_t pf_tiles;     // prefill tiles
    int32_t causal;
    int32_t window_left;
    float scale_log2;     // sm_scale * log2(e)
    int32_t dense;        // prefill tiles read contiguous K / V runs instead of pages
};
static_assert(sizeof(PlanHeader) <= kAlign, "the header fits its aligned slot");

// One piece of a row's visible pages handled by one decode CTA.
struct DecodeTile {
    int32_t q_token;     // token whose query this row uses
    int32_t out_token;   // token the result is written to, -1 = computed and dropped
    int32_t kv_base;     // offset of the row's first page in the plan's page list
    int32_t page_begin;  // first row-local page of this piece
    int32_t page_count;  // pages in this piece (>= 1)
    int32_t length;      // L of the row
    int32_t lo;          // first visible position
    int32_t partial;     // split-KV partial slot, -1 = this piece is the whole row
    int32_t merge_row;   // the row's MergeRow when it is cut, else -1
    int32_t append_token;  // fused append: the row's new token (last piece only), else -1
    int32_t pad[2];
};
static_assert(sizeof(DecodeTile) == 48, "DecodeTile is 12 ints");

#if defined(__CUDACC__)
#define PKV_HOST_DEVICE __host__ __device__ __forceinline__
#else
#define PKV_HOST_DEVICE inline
#endif

// The 16-key chunks of a tile: keys [base + 16 k, base + 16 k + 16) for k in [k0, nk),
// of which positions below `end` belong to the tile (its last page may be cut short by
// the row's end).  The host planner and the decode kernel walk the same chunks.
struct ChunkRange {
    int base, end, k0, nk;
};
PKV_HOST_DEVICE ChunkRange chunk_range(const DecodeTile &t, int P) {
    ChunkRange c;
    c.base = t.page_begin * P;
    const int stop = (t.page_begin + t.page_count) * P;
    c.end = t.length < stop ? t.length : stop;
    c.k0 = ((t.lo > c.base ? t.lo : c.base) - c.base) / kDecodeKeysPerStage;
    c.nk = (c.end - c.base + kDecodeKeysPerStage - 1) / kDecodeKeysPerStage;
    return c;
}

// Chunks of each decode CTA whose cache rows (page id * 2 * page_size + slot) the planner
// stores beside its tile range: the TMA producer issues them as soon as the previous kernel
// allows, without first loading the CTA's tile and then its page id.
constexpr int kDecodeHeadChunks = 4;

// A row whose visible pages were split over several CTAs: its partials
// [first, first + count) are merged into out_token by the merge kernel.
struct MergeRow {
    int32_t out_token;
    int32_t first;
    int32_t count;
    int32_t pad;  // 16 bytes: one vector load
};

// One prefill work tile: up to BQ consecutive new tokens of one row, all q heads of one
// kv head.
struct PrefillTile {
    int32_t q_begin;    // token index (into q / out) of the tile's first query
    int32_t n_q;        // queries in the tile (1..BQ)
    int32_t pos0;       // absolute position p of the tile's first query
    int32_t length;     // L of the row
    int32_t kv_base;    // offset of the row's first page in the plan's page list
    int32_t kv_head;    // kv head of the tile
    int32_t key_begin;  // first key position any query of the tile sees
    int32_t key_end;    // one past the last key position any query of the tile sees
};
static_assert(sizeof(PrefillTile) == 32, "PrefillTile is 8 ints");

// Byte offsets of the plan's arrays inside the workspace.
struct PlanLayout {
    size_t err = 0;            // PlanHeader (its first word is the device error word)
    size_t append_rows = 0;    // int32[num_append]: page * 2 * page_size + slot of each new token
    size_t dec_pages = 0;      // int32[dec_nnz]: page ids the decode pass reads
    size_t pf_pages = 0;       // int32[pf_nnz]:  page ids the prefill pass reads
    size_t dec_tiles = 0;      // DecodeTile[dec_tiles]
    size_t dec_cta_ptr = 0;    // int32[dec_ctas + 1]: tile range of each decode CTA
    size_t dec_cta_rows = 0;   // int32[dec_ctas][kDecodeHeadChunks]: rows of each CTA's first chunks, -1 past its end
    size_t merge_rows = 0;     // MergeRow[num_merge]
    size_t pf_tiles = 0;       // PrefillTile[pf_tiles]
    size_t int_bytes = 0;      // end of the integer part (what the H2D copies)
    size_t part_o = 0;         // float[num_partials, Hq, D]
    size_t part_lse = 0;       // float[num_partials, Hq]
    size_t total = 0;          // workspace bytes this plan needs
};

// Static shape, fixed per handle.
struct Shape {
    int num_qo_heads, num_kv_heads, head_dim, page_size;
    int max_batch, max_total_tokens, max_num_pages, num_cache_pages, max_prefill_rows;
    int sm_count, sink_page;
    int graph_static;  // launch at the maxima with a fixed workspace layout (CUDA-graph mode)
    int group() const { return num_qo_heads / num_kv_heads; }
    // page_size is a power of two: slot = position & (P - 1), page = position >> shift
    int page_shift() const { return __builtin_ctz((unsigned)page_size); }

    // Decode: kv heads one CTA streams (one consumer warp each): the largest divisor of
    // num_kv_heads up to 8 (4 at head_dim 256, whose accumulators take twice the
    // registers); the kv heads are split into dec_head_groups() groups over the grid's y.
    int dec_heads() const {
        const int cap = head_dim > 128 ? 4 : 8;
        for (int d = cap < num_kv_heads ? cap : num_kv_heads; d > 1; --d)
            if (num_kv_heads % d == 0) return d;
        return 1;
    }
    int dec_head_groups() const { return num_kv_heads / dec_heads(); }
    // Decode CTAs per SM: with fewer than 8 kv heads a CTA has few consumer warps, so
    // several CTAs share an SM (and its 200 KB ring budget), up to 8 consumer warps and
    // the warps the registers hold (16 at head_dim 64, 12 at 128, 8 at 256).
    int dec_ctas_per_sm() const {
        const int h = dec_heads();
        const int warp_cap = head_dim <= 64 ? 16 : (head_dim <= 128 ? 12 : 8);
        const int by_warps = warp_cap / (h + dec_producer_warps()), by_heads = 8 / h;
        const int by_smem = (int)(kDecodeRingBytes / (2u * dec_stage_bytes()));  // two stages each
        int k = by_warps < by_heads ? by_warps : by_heads;
        k = k < by_smem ? k : by_smem;
        return k < 1 ? 1 : k;
    }
    // Decode TMA boxes (64 columns x rows x dec_heads() heads, heads outermost): 16 slots of
    // K and the same 16 of V per box pair from page size 16 up, 8 at page size 8.  Pages
    // below 8 slots are gathered by the producer warp with 16-byte cp.async copies into the
    // page-16 layout instead: a box of one such page would be smaller than a swizzle atom,
    // and keys in separate atoms would put an ldmatrix's 8 rows on the same banks.
    bool dec_gather() const { return page_size < 8; }
    // Producer warps of a decode CTA: one thread issues TMA; the cp.async gather takes one
    // warp per two kv heads of the CTA (1 to 4), each copying its share of the heads.
    int dec_producer_warps() const {
        if (!dec_gather()) return 1;
        const int w = dec_heads() / 2;
        return w < 1 ? 1 : (w > 4 ? 4 : w);
    }
    int dec_keys_per_box() const { return page_size == 8 ? 8 : 16; }
    // At page size 16 a chunk is one whole page, whose 16 K rows and 16 V rows are adjacent
    // in the cache: one box of 32 rows takes both (K rows, then V rows), half the boxes.
    bool dec_kv_in_box() const { return page_size == 16; }
    int dec_box_rows() const { return dec_kv_in_box() ? 2 * dec_keys_per_box() : dec_keys_per_box(); }
    // Bytes between boxes in shared memory (a multiple of the 1024-byte swizzle atom).
    int dec_box_stride() const { return dec_box_rows() * dec_heads() * 128; }
    // One ring stage: the K and V boxes of a 16-key chunk, 64-column halves.
    uint32_t dec_stage_bytes() const {
        const uint32_t boxes = kDecodeKeysPerStage / dec_keys_per_box();
        return (dec_kv_in_box() ? 1u : 2u) * (uint32_t)(head_dim / 64) * boxes * (uint32_t)dec_box_stride();
    }
    // Prefill: rows of one paged TMA box (one head); pages smaller than 8 slots are
    // gathered with 16-byte cp.async copies instead (a box would not fill a swizzle atom).
    bool pf_gather() const { return page_size < 8; }
    int pf_box_rows() const { return page_size < 16 ? page_size : 16; }
    // Prefill work tiles of two query tiles (2 x 128 rows sharing every 128-key K/V tile,
    // one CTA per SM): head_dim 64 and 128 with K / V read by TMA (dense plans always are);
    // head_dim 256 and the cp.async gather of small pages keep one query tile per CTA.
    bool pf_pair(bool dense) const { return head_dim <= 128 && (dense || !pf_gather()); }
    int pf_tile_tokens(bool dense) const {
        return (kPrefillRowsPerTile / group()) * (pf_pair(dense) ? 2 : 1);
    }
};

// Worst-case counts at a handle's maxima for one plan mode: the launch grids and the
// workspace layout of graph mode, and the bound pkv_workspace_size reports.
struct StaticCounts {
    int tokens, dec_nnz, pf_nnz, dec_tiles, dec_ctas, num_merge, pf_tiles, partials;
};
StaticCounts static_counts(const Shape &s, int mode);

// Everything a plan produced, host side.  `image` is the integer part exactly as it is
// copied to the workspace.
struct Plan {
    int mode = -1;
    int batch = 0;
    int num_tokens = 0;          // T (decode: batch)
    int num_keys = 0;            // dense plans: rows of the contiguous K / V
    int causal = 1;
    int window_left = -1;
    float sm_scale = 0.f;
    int num_append = 0;
    int dec_rows = 0;            // rows of the decode pass (0 when the mode has none)
    int dec_nnz = 0;
    int pf_nnz = 0;
    int dec_ctas = 0, dec_tiles = 0, num_partials = 0, num_merge = 0;
    int max_pieces = 0;          // pieces of the most-cut row
    int pf_tiles = 0;
    PlanLayout lay;
    std::vector<uint8_t> image;
};

// Host planner entry points (plain C++, no CUDA).  Each returns 0 on success, else a
// pkv_status code with `err` explaining it.
int validate_rows(const Shape &s, int mode, const int32_t *qo, const int32_t *kvp, const int32_t *kvi,
                  const int32_t *lpl, int batch, int window_left, std::string &err, int causal = 1);
// mstar.engine.resources.kv.plan, context_only_views: drop each row's query tokens from
// its view (length shrinks by its query count, pages past the new length dropped).
int context_only_views(int page_size, const int32_t *qo, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl,
                       int batch, int32_t *out_kvp, int32_t *out_kvi, int32_t *out_lpl, int *out_nnz,
                       std::string &err);
int append_slots(int page_size, const int32_t *qo, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl,
                 int batch, int32_t *pages, int32_t *slots, std::string &err);
struct MixedLayout {
    std::vector<int32_t> is_decode, prompt_rows, perm, pf_qo_indptr;
    std::vector<int32_t> dec_kv_indptr, dec_kv_indices, dec_last_page_len, dec_q_token, dec_out_token;
};
int mixed_layout(const int32_t *qo, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl, int batch,
                 int max_prefill_rows, int sink_page, MixedLayout &out, std::string &err);
// Split the visible pages of a decode pass into per-CTA tiles.
// Rows of each decode CTA's first kDecodeHeadChunks chunks (its tiles' chunks in the order the
// kernel walks them), -1 past the CTA's last chunk: int32[ctas][kDecodeHeadChunks].
std::vector<int32_t> decode_head_rows(const Shape &s, const std::vector<DecodeTile> &tiles,
                                      const std::vector<int32_t> &cta_ptr, const int32_t *pages);
void decode_split(const Shape &s, int rows, const int32_t *kvp, const int32_t *lpl, const int32_t *q_token,
                  const int32_t *out_token, int window_left, std::vector<DecodeTile> &tiles,
                  std::vector<int32_t> &cta_ptr, std::vector<MergeRow> &merges, int &num_partials,
                  int max_ctas = 0, bool mark_append = false);
int decode_cta_limit(const Shape &s);
// Dense varlen plan (mstar.engine.resources.attn.dense, DensePlan): segment r's queries are
// q[cu_q[r]..cu_q[r+1]), its keys rows cu_k[r]..cu_k[r+1] of contiguous K / V.
int make_dense_plan(const Shape &s, const int32_t *cu_q, const int32_t *cu_k, int batch, int causal, int window_left,
                    float sm_scale, Plan &plan, std::string &err);
int make_plan(const Shape &s, int mode, const int32_t *qo, const int32_t *kvp, const int32_t *kvi,
              const int32_t *lpl, int batch, int causal, int window_left, float sm_scale, Plan &plan,
              std::string &err);
size_t workspace_bound(const Shape &s, int mode);

}  // namespace pkv

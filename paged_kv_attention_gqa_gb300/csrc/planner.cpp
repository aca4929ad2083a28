// Host planner of libpkv: validation, KV write locations, the decode split-KV work
// split, the mixed step's permutation and sink routing, prefill tiles, and the
// workspace image.  Plain C++: it runs (and is tested) on a machine without a GPU.
//
// Passages restated:
//  * mstar.engine.resources.kv.plan, PagedIndptrs / SequenceView.last_page_len: a row of
//    kv_indptr[r+1]-kv_indptr[r] pages with its last page filled to last_page_len[r]
//    holds L = (pages-1)*page_size + last_page_len tokens.
//  * mstar.engine.resources.attn.wrappers, FlashInferDecodeWrapper.plan: the plan
//    computes the KV write locations; with the post-append arrays a decode token goes to
//    the last page at slot last_page_len-1, and in general position p goes to page
//    kv_indices[kv_indptr[r] + p / page_size], slot p % page_size.
//  * FlashInferPrefillWrapper.plan: window_left preceding positions are visible, -1 = all.
//  * FlashInferMixedWrapper: one-token rows are the decode rows; every row goes through
//    the decode plan (non-decode rows read one token of the sink page, result dropped);
//    at most max_prefill_rows prompt rows go through the prefill plan, their tokens
//    moved to the front by a permutation.
//  * mstar.engine.resources.attn.workspace, Workspace: what a plan needs depends on its
//    rows, heads and the SM count; the split-KV partials live in the workspace.
#include "plan.h"

#include <algorithm>
#include <cmath>
#include <cstring>

#include "../../include/pkv.h"

namespace pkv {

static int row_len(const int32_t *kvp, const int32_t *lpl, int r, int P) {
    int np = kvp[r + 1] - kvp[r];
    return np <= 0 ? 0 : (np - 1) * P + lpl[r];
}

int validate_rows(const Shape &s, int mode, const int32_t *qo, const int32_t *kvp, const int32_t *kvi,
                  const int32_t *lpl, int batch, int window_left, std::string &err, int causal) {
    if (causal < 0 || causal > 2 || (causal == 2 && mode != PKV_MODE_PREFILL)) {
        err = "causal is 0, 1, or 2 (context-only, prefill plans only)";
        return PKV_ERR_INVALID;
    }
    if (batch < 0 || batch > s.max_batch) {
        err = "batch " + std::to_string(batch) + " outside [0, max_batch=" + std::to_string(s.max_batch) + "]";
        return PKV_ERR_INVALID;
    }
    if (window_left < -1) {
        err = "window_left must be -1 (unbounded) or >= 0";
        return PKV_ERR_INVALID;
    }
    if (!kvp || !lpl || (batch > 0 && !kvi && kvp[batch] > 0)) {
        err = "paged_kv_indptr, paged_kv_indices and paged_kv_last_page_len are required";
        return PKV_ERR_INVALID;
    }
    if (mode != PKV_MODE_DECODE && !qo) {
        err = "qo_indptr is required for prefill and mixed plans";
        return PKV_ERR_INVALID;
    }
    if (kvp[0] != 0 || (qo && qo[0] != 0)) {
        err = "indptr arrays must start at 0";
        return PKV_ERR_INVALID;
    }
    for (int r = 0; r < batch; ++r) {
        if (kvp[r + 1] < kvp[r]) {
            err = "paged_kv_indptr decreases at row " + std::to_string(r);
            return PKV_ERR_INVALID;
        }
        if (qo && qo[r + 1] < qo[r]) {
            err = "qo_indptr decreases at row " + std::to_string(r);
            return PKV_ERR_INVALID;
        }
    }
    if (kvp[batch] > s.max_num_pages) {
        err = "paged_kv_indices has " + std::to_string(kvp[batch]) + " entries, above max_num_pages=" +
              std::to_string(s.max_num_pages);
        return PKV_ERR_INVALID;
    }
    int T = qo ? qo[batch] : batch;
    int tok_cap = mode == PKV_MODE_DECODE ? s.max_batch : s.max_total_tokens;
    if (T > tok_cap) {
        err = "step has " + std::to_string(T) + " new tokens, above the handle's maximum " + std::to_string(tok_cap);
        return PKV_ERR_INVALID;
    }
    // every page id in [0, num_cache_pages): one unsigned compare per id, OR-ed together
    // (a loop the compiler vectorises); the offending entry is looked up only on failure
    const uint32_t num_pages = (uint32_t)s.num_cache_pages;
    uint32_t bad = 0;
    for (int i = 0; i < kvp[batch]; ++i) bad |= (uint32_t)kvi[i] >= num_pages;
    if (bad)
        for (int i = 0; i < kvp[batch]; ++i)
            if ((uint32_t)kvi[i] >= num_pages) {
                err = "page id " + std::to_string(kvi[i]) + " at paged_kv_indices[" + std::to_string(i) +
                      "] outside [0, num_cache_pages=" + std::to_string(s.num_cache_pages) + ")";
                return PKV_ERR_INVALID;
            }
    for (int r = 0; r < batch; ++r) {
        int np = kvp[r + 1] - kvp[r];
        int n = qo ? qo[r + 1] - qo[r] : 1;
        if (np > 0 && (lpl[r] < 1 || lpl[r] > s.page_size)) {
            err = "paged_kv_last_page_len[" + std::to_string(r) + "]=" + std::to_string(lpl[r]) +
                  " outside [1, page_size]";
            return PKV_ERR_INVALID;
        }
        int L = row_len(kvp, lpl, r, s.page_size);
        if (mode == PKV_MODE_DECODE && L < 1) {
            err = "decode row " + std::to_string(r) + " has no tokens";
            return PKV_ERR_INVALID;
        }
        if (n > L && causal != 2) {
            err = "row " + std::to_string(r) + " has " + std::to_string(n) + " new tokens but length " +
                  std::to_string(L);
            return PKV_ERR_INVALID;
        }
        if (mode == PKV_MODE_DECODE && n != 1) {
            err = "decode rows have exactly one new token";
            return PKV_ERR_INVALID;
        }
    }
    return PKV_OK;
}

int append_slots(int P, const int32_t *qo, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl, int batch,
                 int32_t *pages, int32_t *slots, std::string &err) {
    for (int r = 0; r < batch; ++r) {
        int L = row_len(kvp, lpl, r, P);
        int t0 = qo ? qo[r] : r;
        int n = qo ? qo[r + 1] - qo[r] : 1;
        if (n > L) {
            err = "row " + std::to_string(r) + " has more new tokens than its length";
            return PKV_ERR_INVALID;
        }
        for (int i = 0; i < n; ++i) {
            int p = L - n + i;
            pages[t0 + i] = kvi[kvp[r] + p / P];
            slots[t0 + i] = p % P;
        }
    }
    return PKV_OK;
}

int context_only_views(int P, const int32_t *qo, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl,
                       int batch, int32_t *out_kvp, int32_t *out_kvi, int32_t *out_lpl, int *out_nnz, std::string &err) {
    int at = 0;
    out_kvp[0] = 0;
    for (int r = 0; r < batch; ++r) {
        const int ctx = row_len(kvp, lpl, r, P) - (qo[r + 1] - qo[r]);
        if (ctx < 0) {
            err = "row " + std::to_string(r) + " appends more tokens than its length";
            return PKV_ERR_INVALID;
        }
        const int keep = (ctx + P - 1) / P;
        for (int i = 0; i < keep; ++i) out_kvi[at++] = kvi[kvp[r] + i];
        out_kvp[r + 1] = at;
        out_lpl[r] = ctx > 0 ? (ctx - 1) % P + 1 : 0;
    }
    *out_nnz = at;
    return PKV_OK;
}

int mixed_layout(const int32_t *qo, const int32_t *kvp, const int32_t *kvi, const int32_t *lpl, int batch,
                 int max_prefill_rows, int sink_page, MixedLayout &m, std::string &err) {
    int T = qo[batch];
    m.is_decode.assign(batch, 0);
    m.prompt_rows.assign(std::max(max_prefill_rows, 0), -1);
    m.perm.clear();
    m.perm.reserve(T);
    m.pf_qo_indptr.assign(1, 0);
    int np = 0;
    for (int r = 0; r < batch; ++r) {
        int n = qo[r + 1] - qo[r];
        m.is_decode[r] = n == 1;
        if (n >= 2) {
            if (np >= max_prefill_rows) {
                err = "mixed step has more than max_prefill_rows=" + std::to_string(max_prefill_rows) +
                      " prompt rows";
                return PKV_ERR_TOO_MANY_PREFILL_ROWS;
            }
            m.prompt_rows[np++] = r;
            for (int t = qo[r]; t < qo[r + 1]; ++t) m.perm.push_back(t);
            m.pf_qo_indptr.push_back((int32_t)m.perm.size());
        }
    }
    while ((int)m.pf_qo_indptr.size() < max_prefill_rows + 1) m.pf_qo_indptr.push_back((int32_t)m.perm.size());
    for (int r = 0; r < batch; ++r)
        if (qo[r + 1] - qo[r] < 2)
            for (int t = qo[r]; t < qo[r + 1]; ++t) m.perm.push_back(t);
    m.dec_kv_indptr.assign(1, 0);
    m.dec_kv_indices.clear();
    m.dec_last_page_len.clear();
    m.dec_q_token.clear();
    m.dec_out_token.clear();
    m.dec_kv_indptr.reserve((size_t)batch + 1);
    m.dec_kv_indices.reserve((size_t)kvp[batch] + (size_t)batch);
    m.dec_last_page_len.reserve(batch);
    m.dec_q_token.reserve(batch);
    m.dec_out_token.reserve(batch);
    for (int r = 0; r < batch; ++r) {
        int n = qo[r + 1] - qo[r];
        if (n == 1) {
            m.dec_kv_indices.insert(m.dec_kv_indices.end(), kvi + kvp[r], kvi + kvp[r + 1]);
            m.dec_last_page_len.push_back(lpl[r]);
            m.dec_out_token.push_back(qo[r]);
        } else {
            if (sink_page < 0) {
                err = "mixed step with a non-decode row needs a sink_page";
                return PKV_ERR_INVALID;
            }
            m.dec_kv_indices.push_back(sink_page);
            m.dec_last_page_len.push_back(1);
            m.dec_out_token.push_back(-1);
        }
        m.dec_kv_indptr.push_back((int32_t)m.dec_kv_indices.size());
        m.dec_q_token.push_back(n >= 1 ? qo[r] : std::max(T - 1, 0));
    }
    return PKV_OK;
}

int decode_cta_limit(const Shape &s) {
    // Persistent decode CTAs, Shape::dec_ctas_per_sm() per SM: each holds a multi-stage
    // ring of 16-key chunks of its kv heads; with several head groups the SMs are shared
    // among them.
    return std::max(1, s.sm_count * s.dec_ctas_per_sm() / s.dec_head_groups());
}

// Keys each decode CTA is given at least (fewer per CTA would only multiply partials
// without shortening the critical path), rounded up to whole pages.
static constexpr int kMinKeysPerCta = 32;

void decode_split(const Shape &s, int rows, const int32_t *kvp, const int32_t *lpl, const int32_t *q_token,
                  const int32_t *out_token, int window_left, std::vector<DecodeTile> &tiles,
                  std::vector<int32_t> &cta_ptr, std::vector<MergeRow> &merges, int &num_partials, int max_ctas,
                  bool mark_append) {
    const int P = s.page_size;
    tiles.clear();
    cta_ptr.assign(1, 0);
    merges.clear();
    num_partials = 0;
    std::vector<int> first(rows), vis(rows), len(rows), lo(rows);
    long long W = 0;
    for (int r = 0; r < rows; ++r) {
        int L = row_len(kvp, lpl, r, P);
        int p = L - 1;
        int l0 = window_left >= 0 ? std::max(0, p - window_left) : 0;
        len[r] = L;
        lo[r] = l0;
        first[r] = l0 / P;
        vis[r] = (L - 1) / P - first[r] + 1;
        W += vis[r];
    }
    if (W == 0) return;
    long long cmax = max_ctas > 0 ? std::min(max_ctas, decode_cta_limit(s)) : decode_cta_limit(s);
    const long long min_pages = (kMinKeysPerCta + P - 1) / P;
    long long per = std::max<long long>((W + cmax - 1) / cmax, min_pages);
    int ctas = (int)((W + per - 1) / per);
    // Walk the rows' visible pages in order, cutting every `per` pages.  The tiles of one row
    // are consecutive: row r's are tiles [row_first[r], row_first[r] + row_count[r]).
    std::vector<int> row_first(rows, 0), row_count(rows, 0);
    tiles.reserve((size_t)rows + (size_t)ctas);
    cta_ptr.reserve((size_t)ctas + 1);
    int r = 0, used = 0;  // pages of row r already assigned
    for (int c = 0; c < ctas; ++c) {
        long long budget = per;
        while (budget > 0 && r < rows) {
            int take = (int)std::min<long long>(budget, vis[r] - used);
            if (take > 0) {
                DecodeTile t;
                t.q_token = q_token[r];
                t.out_token = out_token[r];
                t.kv_base = kvp[r];
                t.page_begin = first[r] + used;
                t.page_count = take;
                t.length = len[r];
                t.lo = lo[r];
                t.partial = -1;
                t.merge_row = -1;
                t.append_token = -1;
                t.pad[0] = t.pad[1] = 0;
                if (row_count[r]++ == 0) row_first[r] = (int)tiles.size();
                tiles.push_back(t);
                used += take;
                budget -= take;
            }
            if (used == vis[r]) {
                ++r;
                used = 0;
            }
        }
        cta_ptr.push_back((int32_t)tiles.size());
    }
    // the piece holding a row's last position also stores its new token (decode plans:
    // the row's only token, the one its query comes from)
    if (mark_append)
        for (int rr = 0; rr < rows; ++rr)
            if (row_count[rr]) tiles[row_first[rr] + row_count[rr] - 1].append_token = q_token[rr];
    for (int rr = 0; rr < rows; ++rr) {
        if (row_count[rr] <= 1) continue;
        MergeRow m;
        m.out_token = out_token[rr];
        m.first = num_partials;
        m.count = row_count[rr];
        m.pad = 0;
        for (int ti = row_first[rr]; ti < row_first[rr] + row_count[rr]; ++ti) {
            tiles[ti].partial = num_partials++;
            tiles[ti].merge_row = (int)merges.size();
        }
        merges.push_back(m);
    }
}

struct PrefillRow {
    int n;        // queries
    int L;        // keys
    int q_begin;  // first query token in q / out
    int kv_base;  // paged: offset of the first page in the page list; dense: first key row
};

// Work tiles of the rows' new tokens into `out` (cleared first), in dispatch order: the q-tiles of
// one (row, kv head) next to each other, so the CTAs in flight together stream the same K/V pages
// and share them in L2; groups longest first (by their longest tile), and longest first inside a
// group, approximating LPT.  Every kv head of a row sees the same key ranges, so the order is
// built directly: rows by their longest tile (ties by page offset, which differs between rows),
// the row's kv heads in turn, and each head's q-tiles longest first (ties in token order).
static void prefill_tiles_rows(const Shape &s, const std::vector<PrefillRow> &rows, int causal, int window_left,
                               std::vector<PrefillTile> &out, bool dense = false) {
    // tokens per work tile: one query tile of 128 / g tokens, or two on the paired kernel
    const int BQ = s.pf_tile_tokens(dense);
    out.clear();
    struct RowTiles {
        int len_max;   // the row's longest key range
        int kv_base;
        int first, n;  // its q-tiles in qtiles
    };
    std::vector<PrefillTile> qtiles;  // one per (row, q-tile), kv head 0
    std::vector<RowTiles> rts;
    for (const PrefillRow &pr : rows) {
        const int n = pr.n, L = pr.L;
        if (n <= 0) continue;
        // causal 2 (context-only): the row's pages hold the context; its queries follow it
        const int c = causal == 2 ? L : L - n;
        RowTiles rt{0, pr.kv_base, (int)qtiles.size(), 0};
        for (int t0 = 0; t0 < n; t0 += BQ) {
            int nq = std::min(BQ, n - t0);
            int p0 = c + t0, p1 = c + t0 + nq - 1;
            int kb = window_left >= 0 ? std::max(0, p0 - window_left) : 0;
            int ke = causal == 1 ? p1 + 1 : L;
            if (ke <= kb) kb = ke = 0;  // no query of the tile sees a key: zeros, lse -inf
            PrefillTile t;
            t.q_begin = pr.q_begin + t0;
            t.n_q = nq;
            t.pos0 = p0;
            t.length = L;
            t.kv_base = pr.kv_base;
            t.kv_head = 0;
            t.key_begin = kb;
            t.key_end = ke;
            qtiles.push_back(t);
            rt.len_max = std::max(rt.len_max, ke - kb);
            ++rt.n;
        }
        rts.push_back(rt);
    }
    std::stable_sort(rts.begin(), rts.end(), [](const RowTiles &a, const RowTiles &b) {
        if (a.len_max != b.len_max) return a.len_max > b.len_max;
        return a.kv_base < b.kv_base;
    });
    out.reserve(qtiles.size() * (size_t)s.num_kv_heads);
    std::vector<int> ord;
    for (const RowTiles &rt : rts) {
        ord.resize(rt.n);
        for (int i = 0; i < rt.n; ++i) ord[i] = rt.first + i;
        std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) {
            return (qtiles[a].key_end - qtiles[a].key_begin) > (qtiles[b].key_end - qtiles[b].key_begin);
        });
        for (int hk = 0; hk < s.num_kv_heads; ++hk)
            for (int i : ord) {
                out.push_back(qtiles[i]);
                out.back().kv_head = hk;
            }
    }
}

static void prefill_tiles(const Shape &s, const std::vector<int> &rows, const int32_t *q_begin_of_row,
                          const int32_t *qo, const int32_t *kvp, const int32_t *lpl, int causal, int window_left,
                          std::vector<PrefillTile> &out) {
    std::vector<PrefillRow> prs;
    for (int r : rows)
        prs.push_back(PrefillRow{qo[r + 1] - qo[r], row_len(kvp, lpl, r, s.page_size), q_begin_of_row[r], kvp[r]});
    prefill_tiles_rows(s, prs, causal, window_left, out);
}

// Time model of one GB300 used to share the SMs between the two passes of a mixed step:
// streaming K/V at ~6.4 TB/s, prefill tiles at 0.7 PFLOP/s (the flops count every query row
// and key of a tile, masked ones included; the rate is the one that gave the shortest step
// when the two passes share the GPU, between 0.3 and 2.5 PFLOP/s on the 96 + 4 row step).
constexpr double kDecodeBytesPerUs = 6.4e6;
constexpr double kPrefillFlopsPerUs = 0.7e9;

static int mixed_decode_ctas(const Shape &s, int rows, const int32_t *kvp, const int32_t *lpl, int window_left,
                             const std::vector<PrefillTile> &ptiles) {
    const int C = decode_cta_limit(s);
    if (ptiles.empty()) return C;
    double bytes = 0.0, flops = 0.0;
    for (int r = 0; r < rows; ++r) {
        const int L = row_len(kvp, lpl, r, s.page_size);
        const int lo = window_left >= 0 ? std::max(0, L - 1 - window_left) : 0;
        bytes += (double)(L - lo) * s.num_kv_heads * s.head_dim * 4.0;
    }
    const double tile_rows = (double)kPrefillRowsPerTile * (s.pf_pair(false) ? 2 : 1);
    for (const PrefillTile &t : ptiles) flops += 4.0 * tile_rows * s.head_dim * (t.key_end - t.key_begin);
    const double t_dec = bytes / kDecodeBytesPerUs, t_pf = flops / kPrefillFlopsPerUs;
    const int pf_sms = (int)(C * t_pf / (t_dec + t_pf) + 0.5);
    return std::max(C / 4, std::min(C, C - pf_sms));
}

static int prefill_tile_bound(const Shape &s, int rows, int tokens) {
    const int BQ = kPrefillRowsPerTile / s.group();
    return (tokens / BQ + rows) * s.num_kv_heads;
}

static PlanLayout layout_for(const Shape &s, int num_append, int dec_nnz, int pf_nnz, int dec_tiles, int dec_ctas,
                             int num_merge, int pf_tiles, int num_partials) {
    PlanLayout L;
    size_t at = 0;
    L.err = at;
    at = align_up(at + 16);
    L.append_rows = at;
    at = align_up(at + sizeof(int32_t) * (size_t)num_append);
    L.dec_pages = at;
    at = align_up(at + sizeof(int32_t) * (size_t)dec_nnz);
    L.pf_pages = at;
    at = align_up(at + sizeof(int32_t) * (size_t)pf_nnz);
    L.dec_tiles = at;
    at = align_up(at + sizeof(DecodeTile) * (size_t)dec_tiles);
    L.dec_cta_ptr = at;
    at = align_up(at + sizeof(int32_t) * (size_t)(dec_ctas + 1));
    L.dec_cta_rows = at;
    at = align_up(at + sizeof(int32_t) * kDecodeHeadChunks * (size_t)dec_ctas);
    L.merge_rows = at;
    at = align_up(at + sizeof(MergeRow) * (size_t)num_merge);
    L.pf_tiles = at;
    at = align_up(at + sizeof(PrefillTile) * (size_t)pf_tiles);
    L.int_bytes = at;
    L.part_o = at;
    at = align_up(at + sizeof(float) * (size_t)num_partials * s.num_qo_heads * s.head_dim);
    L.part_lse = at;
    at = align_up(at + sizeof(float) * (size_t)num_partials * s.num_qo_heads);
    L.total = at;
    return L;
}

StaticCounts static_counts(const Shape &s, int mode) {
    StaticCounts c;
    const int C = decode_cta_limit(s);
    const int rows = s.max_batch;
    if (mode == PKV_MODE_DENSE) {
        c.tokens = s.max_total_tokens;
        c.dec_nnz = c.pf_nnz = c.dec_tiles = c.dec_ctas = c.num_merge = c.partials = 0;
        c.pf_tiles = prefill_tile_bound(s, rows, c.tokens);
        return c;
    }
    const int dec_rows = mode == PKV_MODE_PREFILL ? 0 : rows;
    c.tokens = mode == PKV_MODE_DECODE ? s.max_batch : s.max_total_tokens;
    c.dec_nnz = mode == PKV_MODE_DECODE ? s.max_num_pages : (mode == PKV_MODE_MIXED ? s.max_num_pages + rows : 0);
    c.pf_nnz = mode == PKV_MODE_DECODE ? 0 : s.max_num_pages;
    c.dec_tiles = dec_rows ? dec_rows + C : 0;
    c.dec_ctas = dec_rows ? C : 0;
    c.num_merge = dec_rows ? C : 0;
    const int pf_rows = mode == PKV_MODE_MIXED ? std::min(rows, s.max_prefill_rows) : rows;
    c.pf_tiles = mode == PKV_MODE_DECODE ? 0 : prefill_tile_bound(s, pf_rows, c.tokens);
    c.partials = dec_rows ? dec_rows + C : 0;
    return c;
}

size_t workspace_bound(const Shape &s, int mode) {
    const StaticCounts c = static_counts(s, mode);
    return layout_for(s, c.tokens, c.dec_nnz, c.pf_nnz, c.dec_tiles, c.dec_ctas, c.num_merge, c.pf_tiles, c.partials)
        .total;
}

std::vector<int32_t> decode_head_rows(const Shape &s, const std::vector<DecodeTile> &tiles,
                                      const std::vector<int32_t> &cta_ptr, const int32_t *pages) {
    const int P = s.page_size;
    const int ctas = cta_ptr.empty() ? 0 : (int)cta_ptr.size() - 1;
    std::vector<int32_t> rows((size_t)ctas * kDecodeHeadChunks, -1);
    for (int c = 0; c < ctas; ++c) {
        int n = 0;
        for (int ti = cta_ptr[c]; ti < cta_ptr[c + 1] && n < kDecodeHeadChunks; ++ti) {
            const DecodeTile &t = tiles[ti];
            const ChunkRange cr = chunk_range(t, P);
            for (int k = cr.k0; k < cr.nk && n < kDecodeHeadChunks; ++k) {
                const int pos0 = cr.base + k * kDecodeKeysPerStage;
                rows[(size_t)c * kDecodeHeadChunks + n++] = pages[t.kv_base + (pos0 / P)] * 2 * P + pos0 % P;
            }
        }
    }
    return rows;
}

template <class T>
static void put(std::vector<uint8_t> &img, size_t off, const T *src, size_t n) {
    if (n) std::memcpy(img.data() + off, src, n * sizeof(T));
}

// Reset `plan` to a fresh one, keeping the capacity of its image buffer: a handle hands the
// buffer of its previous plan back in, so that building the image touches memory that is
// already mapped instead of a new ~100 KB allocation per plan.
static void reset_plan(Plan &plan) {
    std::vector<uint8_t> keep;
    keep.swap(plan.image);
    plan = Plan();
    plan.image.swap(keep);
}

// Layout, device header and workspace image of a plan whose pieces are built.
// dec_pages / pf_pages: the page lists of the two passes (dec_nnz / pf_nnz entries), read
// from where they are (the caller's index array or the mixed layout), not copied first.
static void finish_plan(const Shape &s, Plan &plan, int T, int window_left, const std::vector<int32_t> &app,
                        const int32_t *dec_pages, int dec_nnz, const int32_t *pf_pages, int pf_nnz,
                        const std::vector<DecodeTile> &dtiles, std::vector<int32_t> &cta_ptr,
                        const std::vector<MergeRow> &merges, const std::vector<PrefillTile> &ptiles, int partials) {
    const int mode = plan.mode;
    plan.dec_nnz = dec_nnz;
    plan.pf_nnz = pf_nnz;
    plan.dec_tiles = (int)dtiles.size();
    plan.dec_ctas = dtiles.empty() ? 0 : (int)cta_ptr.size() - 1;
    plan.num_merge = (int)merges.size();
    plan.num_partials = partials;
    for (const MergeRow &m : merges) plan.max_pieces = std::max(plan.max_pieces, (int)m.count);
    plan.pf_tiles = (int)ptiles.size();
    if (s.graph_static) {
        // fixed layout at the maxima: captured launches keep pointing at the right arrays;
        // idle decode CTAs get empty tile ranges
        const StaticCounts c = static_counts(s, mode);
        plan.lay = layout_for(s, c.tokens, c.dec_nnz, c.pf_nnz, c.dec_tiles, c.dec_ctas, c.num_merge, c.pf_tiles,
                              c.partials);
        if (c.dec_ctas) {
            if (cta_ptr.empty()) cta_ptr.assign(1, 0);
            while ((int)cta_ptr.size() < c.dec_ctas + 1) cta_ptr.push_back(cta_ptr.back());
        }
    } else {
        plan.lay = layout_for(s, T, plan.dec_nnz, plan.pf_nnz, plan.dec_tiles, plan.dec_ctas, plan.num_merge,
                              plan.pf_tiles, partials);
    }
    plan.image.assign(plan.lay.int_bytes, 0);  // keeps the capacity a reused buffer already has
    PlanHeader hdr;
    hdr.err = 0;
    hdr.num_append = plan.num_append;
    hdr.dec_ctas = plan.dec_ctas;
    hdr.num_merge = plan.num_merge;
    hdr.pf_tiles = plan.pf_tiles;
    hdr.causal = plan.causal;
    hdr.window_left = window_left;
    hdr.scale_log2 = plan.sm_scale * 1.4426950408889634f;
    hdr.dense = mode == PKV_MODE_DENSE ? 1 : 0;
    put(plan.image, plan.lay.err, &hdr, 1);
    put(plan.image, plan.lay.append_rows, app.data(), app.size());
    put(plan.image, plan.lay.dec_pages, dec_pages, (size_t)dec_nnz);
    put(plan.image, plan.lay.pf_pages, pf_pages, (size_t)pf_nnz);
    put(plan.image, plan.lay.dec_tiles, dtiles.data(), dtiles.size());
    if (!cta_ptr.empty() && (plan.dec_ctas || s.graph_static)) {
        put(plan.image, plan.lay.dec_cta_ptr, cta_ptr.data(), cta_ptr.size());
        const std::vector<int32_t> rows = decode_head_rows(s, dtiles, cta_ptr, dec_pages);
        put(plan.image, plan.lay.dec_cta_rows, rows.data(), rows.size());
    }
    put(plan.image, plan.lay.merge_rows, merges.data(), merges.size());
    put(plan.image, plan.lay.pf_tiles, ptiles.data(), ptiles.size());
}

int make_plan(const Shape &s, int mode, const int32_t *qo, const int32_t *kvp, const int32_t *kvi,
              const int32_t *lpl, int batch, int causal, int window_left, float sm_scale, Plan &plan,
              std::string &err) {
    int rc = validate_rows(s, mode, qo, kvp, kvi, lpl, batch, window_left, err, causal);
    if (rc) return rc;
    reset_plan(plan);
    plan.mode = mode;
    plan.batch = batch;
    plan.causal = causal;
    plan.window_left = window_left;
    plan.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt((float)s.head_dim);
    const int T = qo ? qo[batch] : batch;
    plan.num_tokens = T;
    // a context-only plan's arrays describe the context alone: it appends nothing
    plan.num_append = causal == 2 ? 0 : T;
    const int P = s.page_size;

    std::vector<int32_t> pages(T), slots(T), app(plan.num_append);
    if (plan.num_append) {
        rc = append_slots(P, mode == PKV_MODE_DECODE ? nullptr : qo, kvp, kvi, lpl, batch, pages.data(), slots.data(),
                          err);
        if (rc) return rc;
        for (int t = 0; t < T; ++t) app[t] = pages[t] * 2 * P + slots[t];
    }

    std::vector<DecodeTile> dtiles;
    std::vector<int32_t> cta_ptr;
    std::vector<MergeRow> merges;
    std::vector<PrefillTile> ptiles;
    MixedLayout m;  // mixed plans: outlives the branch, finish_plan reads its page list
    const int32_t *dec_pages = nullptr, *pf_pages = nullptr;  // the passes' page lists
    int dec_nnz = 0, pf_nnz = 0;
    int partials = 0;

    if (mode == PKV_MODE_DECODE) {
        std::vector<int32_t> qt(batch), ot(batch);
        for (int r = 0; r < batch; ++r) qt[r] = ot[r] = r;
        decode_split(s, batch, kvp, lpl, qt.data(), ot.data(), window_left, dtiles, cta_ptr, merges, partials, 0,
                     plan.num_append > 0);
        dec_pages = kvi;
        dec_nnz = kvp[batch];
        plan.dec_rows = batch;
    } else if (mode == PKV_MODE_PREFILL) {
        std::vector<int> rows(batch);
        for (int r = 0; r < batch; ++r) rows[r] = r;
        prefill_tiles(s, rows, qo, qo, kvp, lpl, causal, window_left, ptiles);
        pf_pages = kvi;
        pf_nnz = kvp[batch];
    } else if (mode == PKV_MODE_MIXED) {
        rc = mixed_layout(qo, kvp, kvi, lpl, batch, s.max_prefill_rows, s.sink_page, m, err);
        if (rc) return rc;
        if (m.dec_kv_indices.size() > 0 && s.sink_page >= s.num_cache_pages) {
            err = "sink_page outside the cache";
            return PKV_ERR_INVALID;
        }
        // Prefill pass over the prompt rows.  The permutation puts each prompt row's
        // tokens into one contiguous run of the permuted order; the run of prompt row k
        // starts at permuted index pf_qo_indptr[k], i.e. at original token
        // perm[pf_qo_indptr[k]], so the prefill pass reads and writes q / out at those
        // original offsets directly.
        std::vector<int> rows;
        std::vector<int32_t> qbeg(batch, 0);
        for (int k = 0; k < s.max_prefill_rows; ++k) {
            int r = m.prompt_rows[k];
            if (r < 0) continue;
            rows.push_back(r);
            qbeg[r] = m.perm[m.pf_qo_indptr[k]];
        }
        prefill_tiles(s, rows, qbeg.data(), qo, kvp, lpl, causal, window_left, ptiles);
        pf_pages = kvi;
        pf_nnz = kvp[batch];
        // Decode pass over every row: a decode row attends its own pages, any other row
        // one token of the sink page; the latter's result is dropped (out_token -1).  The
        // two passes run concurrently: the decode pass gets the SMs its bytes need, the
        // prefill pass's CTAs fill the others.
        decode_split(s, batch, m.dec_kv_indptr.data(), m.dec_last_page_len.data(), m.dec_q_token.data(),
                     m.dec_out_token.data(), window_left, dtiles, cta_ptr, merges, partials,
                     mixed_decode_ctas(s, batch, m.dec_kv_indptr.data(), m.dec_last_page_len.data(), window_left,
                                       ptiles));
        dec_pages = m.dec_kv_indices.data();
        dec_nnz = (int)m.dec_kv_indices.size();
        plan.dec_rows = batch;
    } else {
        err = "unknown plan mode";
        return PKV_ERR_INVALID;
    }
    finish_plan(s, plan, T, window_left, app, dec_pages, dec_nnz, pf_pages, pf_nnz, dtiles, cta_ptr, merges, ptiles,
                partials);
    return PKV_OK;
}

int make_dense_plan(const Shape &s, const int32_t *cu_q, const int32_t *cu_k, int batch, int causal, int window_left,
                    float sm_scale, Plan &plan, std::string &err) {
    if (!cu_q || !cu_k || batch < 0 || batch > s.max_batch) {
        err = "cu_q and cu_k are required and batch must be in [0, max_batch]";
        return PKV_ERR_INVALID;
    }
    if (causal != 0 && causal != 1) {
        err = "dense plans are causal (1) or non-causal (0)";
        return PKV_ERR_INVALID;
    }
    if (window_left < -1) {
        err = "window_left must be -1 (unbounded) or >= 0";
        return PKV_ERR_INVALID;
    }
    if (cu_q[0] != 0 || cu_k[0] != 0) {
        err = "cu_q and cu_k must start at 0";
        return PKV_ERR_INVALID;
    }
    std::vector<PrefillRow> rows;
    for (int r = 0; r < batch; ++r) {
        const int n = cu_q[r + 1] - cu_q[r], L = cu_k[r + 1] - cu_k[r];
        if (n < 0 || L < 0) {
            err = "cu_q / cu_k decrease at segment " + std::to_string(r);
            return PKV_ERR_INVALID;
        }
        if (n > L) {
            err = "segment " + std::to_string(r) + " has more queries than keys (its fresh tokens are part of its keys)";
            return PKV_ERR_INVALID;
        }
        rows.push_back(PrefillRow{n, L, cu_q[r], cu_k[r]});
    }
    if (cu_q[batch] > s.max_total_tokens) {
        err = "dense plan has " + std::to_string(cu_q[batch]) + " queries, above max_total_tokens";
        return PKV_ERR_INVALID;
    }
    reset_plan(plan);
    plan.mode = PKV_MODE_DENSE;
    plan.batch = batch;
    plan.causal = causal;
    plan.window_left = window_left;
    plan.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt((float)s.head_dim);
    plan.num_tokens = cu_q[batch];
    plan.num_keys = cu_k[batch];
    std::vector<PrefillTile> ptiles;
    prefill_tiles_rows(s, rows, causal, window_left, ptiles, true);
    std::vector<int32_t> none, cta;
    finish_plan(s, plan, plan.num_tokens, window_left, none, nullptr, 0, nullptr, 0, {}, cta, {}, ptiles, 0);
    return PKV_OK;
}

}  // namespace pkv

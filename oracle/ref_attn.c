/*
 * Oracle for batched GQA attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load this file's shared object.  It shares no code, header,
 * table or helper with the CUDA library and is deliberately plain: one thread,
 * fp32 arithmetic, no blocking, no fusion, no reordering beyond the definition.
 *
 * What it computes (written from the pages of the "mstar" engine):
 *
 *   Cache layout (mstar.engine.resources.attn.wrappers, module docstring):
 *     one layer slice is [max_pages, 2, page_size, num_kv_heads, head_dim] bf16;
 *     index 0 of the "2" axis holds K, index 1 holds V.
 *
 *   Index arrays (mstar.engine.resources.kv.plan, PagedIndptrs / SequenceView):
 *     row r owns pages kv_indices[kv_indptr[r] .. kv_indptr[r+1]), its last page
 *     filled to last_page_len[r] slots; its KV length after this step's append is
 *       L_r = (kv_indptr[r+1] - kv_indptr[r] - 1) * page_size + last_page_len[r].
 *     Its new (query) tokens are q[qo_indptr[r] .. qo_indptr[r+1]); with
 *     n_r = qo_indptr[r+1] - qo_indptr[r] the cached prefix is c_r = L_r - n_r and
 *     new token i sits at absolute position p = c_r + i.  Token p lives in page
 *     kv_indices[kv_indptr[r] + p / page_size], slot p % page_size.
 *
 *   Visibility (FlashInferPrefillWrapper.plan, the window_left sentence; causal
 *   alignment "attend to the cached prefix plus themselves"):
 *     causal (1):        keys j with lo <= j <= p
 *     non-causal (0):    keys j with lo <= j <= L_r - 1
 *     context-only (2):  the row's pages hold only the stored context, the queries come
 *                        after it (mstar.engine.resources.kv.plan, context_only_views:
 *                        "length shrinks by to_compute ... to_compute becomes the row's
 *                        query count"): query i sits at p = L_r + i and sees keys
 *                        lo <= j <= L_r - 1; n_r may exceed L_r.
 *     lo = max(0, p - window_left) when window_left >= 0, else 0.
 *     A query that sees no key (an empty context) gets o = 0 and lse = -inf.
 *
 *   Attention (the textbook softmax definition the wrappers compute):
 *     s_j = sm_scale * <q, K_j>;  m = max_j s_j;  l = sum_j exp(s_j - m);
 *     o = sum_j exp(s_j - m) / l * V_j;  lse = m + ln(l)   (natural log).
 *     q head h reads kv head h / (num_qo_heads / num_kv_heads).
 *
 *   Append (FlashInferDecodeWrapper.plan "write location"; the layer writes its
 *   K/V before attention runs, DenseAttentionManager.requires_kv_write):
 *     new token i of row r is stored at position p = c_r + i, i.e. page
 *     kv_indices[kv_indptr[r] + p / page_size], slot p % page_size.
 *
 * Every function returns 0 on success and a negative code on an input it cannot
 * interpret (a row with L_r < n_r, an index outside the pool).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static float bf16_bits_to_float(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Element offset of (page, kv, slot, head, 0) in one layer slice. */
static size_t cache_offset(int64_t page, int kv, int slot, int head,
                           int page_size, int num_kv_heads, int head_dim)
{
    return ((((size_t)page * 2 + (size_t)kv) * (size_t)page_size + (size_t)slot)
                * (size_t)num_kv_heads + (size_t)head) * (size_t)head_dim;
}

static int row_length(const int32_t *kv_indptr, const int32_t *last_page_len,
                      int r, int page_size)
{
    int npages = kv_indptr[r + 1] - kv_indptr[r];
    if (npages <= 0) return 0;
    return (npages - 1) * page_size + last_page_len[r];
}

/*
 * Ragged paged attention.  Decode is the case qo_indptr[r] = r.
 *   q        [T, num_qo_heads, head_dim] bf16 bits, T = qo_indptr[batch]
 *   kv_layer [max_pages, 2, page_size, num_kv_heads, head_dim] bf16 bits
 *   out      [T, num_qo_heads, head_dim] float (unrounded)
 *   lse      [T, num_qo_heads] float
 * Rows listed in row_mask with 0 are skipped (row_mask may be NULL = all rows).
 */
int oracle_attention(const uint16_t *q, const uint16_t *kv_layer, int64_t max_pages,
                     const int32_t *qo_indptr, const int32_t *kv_indptr,
                     const int32_t *kv_indices, const int32_t *last_page_len,
                     int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                     int page_size, int causal, int window_left, float sm_scale,
                     const uint8_t *row_mask, float *out, float *lse)
{
    int group = num_qo_heads / num_kv_heads;
    for (int r = 0; r < batch; ++r) {
        if (row_mask && !row_mask[r]) continue;
        int L = row_length(kv_indptr, last_page_len, r, page_size);
        int n = qo_indptr[r + 1] - qo_indptr[r];
        if (n == 0) continue;
        if (causal != 2 && L < n) return -1;
        int c = causal == 2 ? L : L - n;

        /* Gather the row's pages into contiguous K and V: [L, num_kv_heads, head_dim]. */
        size_t row_elems = (size_t)(L > 0 ? L : 1) * num_kv_heads * head_dim;
        float *K = (float *)malloc(row_elems * sizeof(float));
        float *V = (float *)malloc(row_elems * sizeof(float));
        float *s = (float *)malloc((size_t)(L > 0 ? L : 1) * sizeof(float));
        if (!K || !V || !s) { free(K); free(V); free(s); return -3; }
        for (int p = 0; p < L; ++p) {
            int64_t page = kv_indices[kv_indptr[r] + p / page_size];
            if (page < 0 || page >= max_pages) { free(K); free(V); free(s); return -2; }
            int slot = p % page_size;
            for (int hk = 0; hk < num_kv_heads; ++hk) {
                size_t ko = cache_offset(page, 0, slot, hk, page_size, num_kv_heads, head_dim);
                size_t vo = cache_offset(page, 1, slot, hk, page_size, num_kv_heads, head_dim);
                for (int d = 0; d < head_dim; ++d) {
                    K[((size_t)p * num_kv_heads + hk) * head_dim + d] = bf16_bits_to_float(kv_layer[ko + d]);
                    V[((size_t)p * num_kv_heads + hk) * head_dim + d] = bf16_bits_to_float(kv_layer[vo + d]);
                }
            }
        }

        for (int i = 0; i < n; ++i) {
            int t = qo_indptr[r] + i;
            int p = c + i;
            int hi = causal == 1 ? p : L - 1;
            int lo = 0;
            if (window_left >= 0) lo = p - window_left > 0 ? p - window_left : 0;
            for (int h = 0; h < num_qo_heads; ++h) {
                int hk = h / group;
                const uint16_t *qv = q + ((size_t)t * num_qo_heads + h) * head_dim;
                float *o = out + ((size_t)t * num_qo_heads + h) * head_dim;
                if (hi < lo) {
                    for (int d = 0; d < head_dim; ++d) o[d] = 0.0f;
                    if (lse) lse[(size_t)t * num_qo_heads + h] = -INFINITY;
                    continue;
                }
                float m = -INFINITY;
                for (int j = lo; j <= hi; ++j) {
                    const float *kj = K + ((size_t)j * num_kv_heads + hk) * head_dim;
                    float dot = 0.0f;
                    for (int d = 0; d < head_dim; ++d) dot += bf16_bits_to_float(qv[d]) * kj[d];
                    s[j] = sm_scale * dot;
                    if (s[j] > m) m = s[j];
                }
                float l = 0.0f;
                for (int j = lo; j <= hi; ++j) {
                    s[j] = expf(s[j] - m);
                    l += s[j];
                }
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0f;
                for (int j = lo; j <= hi; ++j) {
                    const float *vj = V + ((size_t)j * num_kv_heads + hk) * head_dim;
                    float w = s[j] / l;
                    for (int d = 0; d < head_dim; ++d) o[d] += w * vj[d];
                }
                if (lse) lse[(size_t)t * num_qo_heads + h] = m + logf(l);
            }
        }
        free(K); free(V); free(s);
    }
    return 0;
}

/*
 * Last-page append: copy this step's new K and V ([T, num_kv_heads, head_dim] bf16
 * bits each) into the layer slice at their positions.  The index arrays describe
 * the cache after the append, as the attention call that follows reads it.
 */
int oracle_kv_append(uint16_t *kv_layer, int64_t max_pages,
                     const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *qo_indptr, const int32_t *kv_indptr,
                     const int32_t *kv_indices, const int32_t *last_page_len,
                     int batch, int num_kv_heads, int head_dim, int page_size)
{
    size_t tok_elems = (size_t)num_kv_heads * head_dim;
    for (int r = 0; r < batch; ++r) {
        int L = row_length(kv_indptr, last_page_len, r, page_size);
        int n = qo_indptr[r + 1] - qo_indptr[r];
        if (L < n) return -1;
        int c = L - n;
        for (int i = 0; i < n; ++i) {
            int t = qo_indptr[r] + i;
            int p = c + i;
            int64_t page = kv_indices[kv_indptr[r] + p / page_size];
            if (page < 0 || page >= max_pages) return -2;
            int slot = p % page_size;
            size_t ko = cache_offset(page, 0, slot, 0, page_size, num_kv_heads, head_dim);
            size_t vo = cache_offset(page, 1, slot, 0, page_size, num_kv_heads, head_dim);
            memcpy(kv_layer + ko, k_new + (size_t)t * tok_elems, tok_elems * sizeof(uint16_t));
            memcpy(kv_layer + vo, v_new + (size_t)t * tok_elems, tok_elems * sizeof(uint16_t));
        }
    }
    return 0;
}

/*
 * Dense varlen attention (mstar.engine.resources.attn.dense, DenseAttentionManager /
 * DensePlan): segment r attends over a contiguous K/V run, rows cu_k[r] .. cu_k[r+1] of
 * k and v ([frozen prefix | fresh tokens], [total_k, num_kv_heads, head_dim] bf16 bits),
 * with its queries q[cu_q[r] .. cu_q[r+1]) being the run's last n_r tokens: query i sits
 * at position p = L_r - n_r + i, L_r = cu_k[r+1] - cu_k[r].  Visibility and arithmetic
 * as in oracle_attention (causal 1 / non-causal 0, window_left).
 */
int oracle_dense_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const int32_t *cu_q, const int32_t *cu_k, int batch,
                           int num_qo_heads, int num_kv_heads, int head_dim,
                           int causal, int window_left, float sm_scale,
                           float *out, float *lse)
{
    int group = num_qo_heads / num_kv_heads;
    for (int r = 0; r < batch; ++r) {
        int L = cu_k[r + 1] - cu_k[r];
        int n = cu_q[r + 1] - cu_q[r];
        if (n == 0) continue;
        if (L < n) return -1;
        float *s = (float *)malloc((size_t)L * sizeof(float));
        if (!s) return -3;
        for (int i = 0; i < n; ++i) {
            int t = cu_q[r] + i;
            int p = L - n + i;
            int hi = causal ? p : L - 1;
            int lo = 0;
            if (window_left >= 0) lo = p - window_left > 0 ? p - window_left : 0;
            for (int h = 0; h < num_qo_heads; ++h) {
                int hk = h / group;
                const uint16_t *qv = q + ((size_t)t * num_qo_heads + h) * head_dim;
                float *o = out + ((size_t)t * num_qo_heads + h) * head_dim;
                float m = -INFINITY;
                for (int j = lo; j <= hi; ++j) {
                    const uint16_t *kj = k + ((size_t)(cu_k[r] + j) * num_kv_heads + hk) * head_dim;
                    float dot = 0.0f;
                    for (int d = 0; d < head_dim; ++d) dot += bf16_bits_to_float(qv[d]) * bf16_bits_to_float(kj[d]);
                    s[j] = sm_scale * dot;
                    if (s[j] > m) m = s[j];
                }
                float l = 0.0f;
                for (int j = lo; j <= hi; ++j) {
                    s[j] = expf(s[j] - m);
                    l += s[j];
                }
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0f;
                for (int j = lo; j <= hi; ++j) {
                    const uint16_t *vj = v + ((size_t)(cu_k[r] + j) * num_kv_heads + hk) * head_dim;
                    float w = s[j] / l;
                    for (int d = 0; d < head_dim; ++d) o[d] += w * bf16_bits_to_float(vj[d]);
                }
                if (lse) lse[(size_t)t * num_qo_heads + h] = m + logf(l);
            }
        }
        free(s);
    }
    return 0;
}

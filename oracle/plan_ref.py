"""Index work of the paged attention path, restated in plain Python.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Integer results here are the
bit-exact expectation for the CUDA library's planner and append kernel.

Passages followed:
  * mstar.engine.resources.kv.plan, SequenceView.last_page_len and PagedIndptrs:
    a row of length L >= 1 spans ceil(L / page_size) pages and fills its last page to
    ((L - 1) mod page_size) + 1 slots.
  * mstar.engine.resources.attn.wrappers, FlashInferDecodeWrapper.plan: the write
    location of a decode token is the row's last page at slot last_page_len - 1
    of the post-append arrays (the garbled sentence there is read this way; the
    arrays the layer's attention reads already include the step's tokens).
  * FlashInferPrefillWrapper.plan: window_left is the number of preceding positions
    a query sees, -1 unbounded.
  * FlashInferMixedWrapper: one-token rows are decode rows and attend their own pages;
    every other row is routed to one token of the sink page in the decode pass and
    its output is dropped; at most max_prefill_rows prompt rows go to the prefill
    pass, their tokens moved to the front by a permutation.
"""
from __future__ import annotations

import numpy as np


def row_lengths(kv_indptr, last_page_len, page_size: int) -> np.ndarray:
    """L_r = (pages_r - 1) * page_size + last_page_len[r]; a row with no pages has L = 0."""
    kvp = np.asarray(kv_indptr, dtype=np.int64)
    lpl = np.asarray(last_page_len, dtype=np.int64)
    out = np.zeros(len(kvp) - 1, dtype=np.int64)
    for r in range(len(kvp) - 1):
        npages = int(kvp[r + 1] - kvp[r])
        out[r] = 0 if npages == 0 else (npages - 1) * page_size + int(lpl[r])
    return out


def last_page_len_of(length: int, page_size: int) -> int:
    """SequenceView.last_page_len: fill of the last page of a length-L stream."""
    assert length >= 1
    return (length - 1) % page_size + 1


def append_slots(qo_indptr, kv_indptr, kv_indices, last_page_len, page_size: int):
    """(page, slot) of every new token, in token order: token i of row r is position
    p = L_r - n_r + i, stored in page kv_indices[kv_indptr[r] + p // page_size] at slot
    p % page_size."""
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kvp = np.asarray(kv_indptr, dtype=np.int64)
    kvi = np.asarray(kv_indices, dtype=np.int64)
    L = row_lengths(kv_indptr, last_page_len, page_size)
    T = int(qo[-1])
    pages = np.zeros(T, dtype=np.int32)
    slots = np.zeros(T, dtype=np.int32)
    for r in range(len(qo) - 1):
        n = int(qo[r + 1] - qo[r])
        c = int(L[r]) - n
        assert c >= 0, "a row cannot have more new tokens than its length"
        for i in range(n):
            p = c + i
            pages[qo[r] + i] = kvi[kvp[r] + p // page_size]
            slots[qo[r] + i] = p % page_size
    return pages, slots


def visible_range(length: int, num_new: int, i: int, causal, window_left: int):
    """Inclusive key range [lo, hi] that new token i of a row sees (empty when hi < lo).
    causal: True / 1 causal, False / 0 non-causal, 2 context-only (the queries follow the
    row's `length` stored tokens)."""
    p = length + i if causal == 2 else length - num_new + i
    hi = p if causal is True or causal == 1 else length - 1
    lo = max(0, p - window_left) if window_left >= 0 else 0
    return lo, hi


def context_only_views(qo_indptr, kv_indptr, kv_indices, last_page_len, page_size: int):
    """mstar.engine.resources.kv.plan, context_only_views: each row's length shrinks by its
    query count (to_compute), the pages past the shorter length are dropped and the last
    page's fill is recomputed.  Returns (kv_indptr, kv_indices, last_page_len); a row left
    with no context has no pages and last_page_len 0."""
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kvp = np.asarray(kv_indptr, dtype=np.int64)
    kvi = np.asarray(kv_indices, dtype=np.int64)
    L = row_lengths(kv_indptr, last_page_len, page_size)
    new_p, new_i, new_l = [0], [], []
    for r in range(len(kvp) - 1):
        ctx = int(L[r]) - int(qo[r + 1] - qo[r])
        assert ctx >= 0, "a row cannot append more tokens than its length"
        keep = -(-ctx // page_size)
        new_i.extend(int(x) for x in kvi[kvp[r]: kvp[r] + keep])
        new_p.append(len(new_i))
        new_l.append(last_page_len_of(ctx, page_size) if ctx > 0 else 0)
    i32 = lambda x: np.asarray(x, dtype=np.int32)
    return i32(new_p), i32(new_i), i32(new_l)


def mixed_layout(qo_indptr, kv_indptr, kv_indices, last_page_len, *, max_prefill_rows: int,
                 sink_page: int):
    """The two plans of a mixed step.

    Returns a dict of int32 arrays:
      is_decode      [B]    1 for a one-token row
      prompt_rows    [max_prefill_rows] prompt row ids in row order, -1 padding
      perm           [T]    perm[k] = original token index of permuted token k:
                            prompt rows' tokens first (row order, token order), then
                            every other token in original order
      pf_qo_indptr   [max_prefill_rows + 1] prefill-pass token offsets in permuted
                            order (padding rows are empty)
      dec_kv_indptr  [B+1], dec_kv_indices, dec_last_page_len [B]: the decode pass over
                            every row: a decode row keeps its pages, any other row reads
                            [sink_page] with last_page_len 1
      dec_q_token    [B]    token whose query the decode pass reads for the row (the
                            row's first token; for a row without tokens, the last token
                            of the batch, or 0 if there is none)
      dec_out_token  [B]    token the decode pass writes for the row, -1 if dropped
    Raises ValueError when more than max_prefill_rows rows have two or more tokens.
    """
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kvp = np.asarray(kv_indptr, dtype=np.int64)
    kvi = np.asarray(kv_indices, dtype=np.int64)
    lpl = np.asarray(last_page_len, dtype=np.int64)
    B = len(qo) - 1
    T = int(qo[-1])
    n = qo[1:] - qo[:-1]
    is_decode = (n == 1).astype(np.int32)
    prompt = [r for r in range(B) if n[r] >= 2]
    if len(prompt) > max_prefill_rows:
        raise ValueError("too many prompt rows for max_prefill_rows")
    prompt_rows = np.full(max_prefill_rows, -1, dtype=np.int32)
    prompt_rows[: len(prompt)] = prompt

    perm = []
    pf_qo = [0]
    for r in prompt:
        perm.extend(range(int(qo[r]), int(qo[r + 1])))
        pf_qo.append(len(perm))
    while len(pf_qo) < max_prefill_rows + 1:
        pf_qo.append(len(perm))
    in_front = set(perm)
    perm.extend(t for t in range(T) if t not in in_front)

    dec_kvp = [0]
    dec_kvi = []
    dec_lpl = []
    dec_q = []
    dec_out = []
    for r in range(B):
        if is_decode[r]:
            dec_kvi.extend(int(x) for x in kvi[kvp[r]: kvp[r + 1]])
            dec_lpl.append(int(lpl[r]))
            dec_out.append(int(qo[r]))
        else:
            dec_kvi.append(int(sink_page))
            dec_lpl.append(1)
            dec_out.append(-1)
        dec_kvp.append(len(dec_kvi))
        if n[r] >= 1:
            dec_q.append(int(qo[r]))
        else:
            dec_q.append(max(T - 1, 0))
    i32 = lambda x: np.asarray(x, dtype=np.int32)
    return dict(is_decode=is_decode, prompt_rows=prompt_rows, perm=i32(perm), pf_qo_indptr=i32(pf_qo),
                dec_kv_indptr=i32(dec_kvp), dec_kv_indices=i32(dec_kvi), dec_last_page_len=i32(dec_lpl),
                dec_q_token=i32(dec_q), dec_out_token=i32(dec_out))

"""libpkv on the host (no GPU): exported symbols, the planner's index work against the
oracle's restatement (bit-exact), the decode work split, and host-side validation."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

from oracle import plan_ref
from paged_kv_attention_gqa_gb300 import binding as B
from paged_kv_attention_gqa_gb300 import build as pkv_build
from paged_kv_attention_gqa_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "mixed_layout.json")))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return B.load()


def test_header_symbols_exported(lib):
    header = open(os.path.join(ROOT, "include", "pkv.h")).read()
    declared = set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", header))
    assert declared == set(B.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def _handle(**kw):
    cfg = dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, max_batch=256, max_total_tokens=65536,
               max_num_pages=200000, num_cache_pages=200000, max_prefill_rows=4, sm_count=152, sink_page=-1)
    cfg.update(kw)
    return B.Handle(**cfg)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), B.ERR_UNSUPPORTED),
    (dict(head_dim=512), B.ERR_UNSUPPORTED),
    (dict(page_size=12), B.ERR_UNSUPPORTED),
    (dict(page_size=24), B.ERR_UNSUPPORTED),
    (dict(page_size=48), B.ERR_UNSUPPORTED),
    (dict(page_size=2048), B.ERR_UNSUPPORTED),
    (dict(num_qo_heads=12), B.ERR_UNSUPPORTED),
    (dict(num_qo_heads=30), B.ERR_UNSUPPORTED),
    (dict(num_kv_heads=2, num_qo_heads=24), B.ERR_UNSUPPORTED),
    (dict(num_kv_heads=1, num_qo_heads=9), B.ERR_UNSUPPORTED),
    (dict(max_batch=0), B.ERR_INVALID),
    (dict(sink_page=200000), B.ERR_INVALID),
    (dict(enable_nvtx=2), B.ERR_INVALID),
])
def test_create_rejects(lib, kw, status):
    with pytest.raises(B.PkvError) as e:
        _handle(**kw)
    assert e.value.status == status


def test_golden_append_slots(lib):
    idx = (GOLD["qo_indptr"], GOLD["kv_indptr"], GOLD["kv_indices"], GOLD["last_page_len"])
    pages, slots = B.append_slots(16, *idx)
    assert pages.tolist() == GOLD["expect"]["append_pages"]
    assert slots.tolist() == GOLD["expect"]["append_slots"]


def test_golden_mixed_layout(lib):
    idx = (GOLD["qo_indptr"], GOLD["kv_indptr"], GOLD["kv_indices"], GOLD["last_page_len"])
    lay = B.mixed_layout(*idx, max_prefill_rows=GOLD["max_prefill_rows"], sink_page=GOLD["sink_page"])
    for key, want in GOLD["expect"].items():
        if key in lay:
            assert lay[key].tolist() == want, key


@pytest.mark.parametrize("name", ["tiny", "batch", "prefill", "mixed", "long"])
def test_planner_matches_oracle_index_work(lib, name):
    pb = wl.WORKLOADS[name]()
    idx = pb.index_arrays()
    a = B.append_slots(pb.page_size, *idx)
    b = plan_ref.append_slots(*idx, pb.page_size)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    if pb.sink_page >= 0:
        got = B.mixed_layout(*idx, max_prefill_rows=pb.max_prefill_rows, sink_page=pb.sink_page)
        want = plan_ref.mixed_layout(*idx, max_prefill_rows=pb.max_prefill_rows, sink_page=pb.sink_page)
        for k in want:
            assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("seed", range(6))
def test_random_mixed_layout_bit_exact(lib, seed):
    rng = np.random.default_rng(1000 + seed)
    Bn = int(rng.integers(1, 64))
    n = rng.choice([0, 1, 1, 1, 1, 2, 9, 40], size=Bn)
    c = rng.integers(0, 90, size=Bn)
    L = np.maximum(c + n, 1)
    maxp = int((n >= 2).sum()) + int(rng.integers(0, 2))
    pb = wl.custom(seed, L, n, num_qo_heads=4, num_kv_heads=2, head_dim=64, page_size=16, reserve_sink=True)
    idx = pb.index_arrays()
    got = B.mixed_layout(*idx, max_prefill_rows=maxp, sink_page=pb.sink_page)
    want = plan_ref.mixed_layout(*idx, max_prefill_rows=maxp, sink_page=pb.sink_page)
    for k in want:
        assert np.array_equal(got[k], want[k]), k
    a = B.append_slots(16, *idx)
    b = plan_ref.append_slots(*idx, 16)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_too_many_prompt_rows_status(lib):
    idx = (GOLD["qo_indptr"], GOLD["kv_indptr"], GOLD["kv_indices"], GOLD["last_page_len"])
    with pytest.raises(B.PkvError) as e:
        B.mixed_layout(*idx, max_prefill_rows=1, sink_page=11)
    assert e.value.status == B.ERR_TOO_MANY_PREFILL_ROWS


def _split_case(name, P):
    if P == 16:
        return wl.WORKLOADS[name]()
    # the same lengths on pages of P slots
    base = wl.WORKLOADS[name]()
    return wl.custom(7, base.kv_lens, base.qo_lens, num_qo_heads=base.num_qo_heads, num_kv_heads=base.num_kv_heads,
                     head_dim=base.head_dim, page_size=P)


@pytest.mark.parametrize("name,window,P", [("batch", -1, 16), ("long", -1, 16), ("long", 4096, 16), ("tiny", -1, 16),
                                           ("tiny", 5, 16), ("batch", -1, 1), ("batch", -1, 8), ("long", 100, 64),
                                           ("tiny", 5, 2)])
@pytest.mark.parametrize("Hkv", [None, 16])
def test_decode_split_covers_each_visible_page_once(lib, name, window, P, Hkv):
    pb = _split_case(name, P)
    Hkv = Hkv or pb.num_kv_heads
    groups = 2 if Hkv == 16 else 1  # 16 kv heads: two groups of 8 share the SMs
    h = _handle(num_qo_heads=Hkv * pb.num_qo_heads // pb.num_kv_heads, num_kv_heads=Hkv, head_dim=pb.head_dim,
                num_cache_pages=pb.max_pages, page_size=P)
    tiles, ctas = h.decode_split(pb.kv_indptr, pb.last_page_len, window)
    assert 1 <= ctas <= 152 // groups
    per_cta = np.bincount(tiles[:, 4], weights=tiles[:, 2], minlength=ctas)
    assert per_cta.max() - per_cta[:-1].min() <= 1 if ctas > 1 else True
    for r in range(pb.batch):
        L = int(pb.kv_lens[r])
        lo, _ = plan_ref.visible_range(L, 1, 0, True, window)
        want = list(range(lo // P, (L - 1) // P + 1))
        mine = tiles[tiles[:, 0] == r]
        got = [p for t in mine for p in range(t[1], t[1] + t[2])]
        assert got == want, r
        if len(mine) == 1:
            assert mine[0, 3] == -1
        else:
            assert np.all(mine[:, 3] >= 0)
    parts = tiles[tiles[:, 3] >= 0, 3]
    assert sorted(parts.tolist()) == list(range(len(parts)))


@pytest.mark.parametrize("name,window,P", [("batch", -1, 16), ("long", 4096, 16), ("tiny", -1, 16), ("tiny", 5, 16),
                                           ("batch", -1, 64), ("long", 100, 64), ("long", 20, 32), ("batch", 0, 16)])
@pytest.mark.parametrize("Hkv", [None, 1])
def test_decode_head_rows_are_the_first_chunks_of_each_cta(lib, name, window, P, Hkv):
    """The rows a decode CTA's first copies are issued from, written into the plan by the
    planner, against the chunks rederived here from the split: CTA c's tiles in order, each
    tile's 16-key chunks from the first one holding a visible key, the row of a chunk being
    its first key's page id * 2P + slot; -1 past the CTA's last chunk."""
    pb = _split_case(name, P)
    Hkv = Hkv or pb.num_kv_heads
    h = _handle(num_qo_heads=Hkv * pb.num_qo_heads // pb.num_kv_heads, num_kv_heads=Hkv, head_dim=pb.head_dim,
                num_cache_pages=pb.max_pages, page_size=P)
    tiles, ctas = h.decode_split(pb.kv_indptr, pb.last_page_len, window)
    rows = h.decode_head_rows(pb.kv_indptr, pb.kv_indices, pb.last_page_len, window)
    assert rows.shape == (ctas, 4)
    want = [[] for _ in range(ctas)]
    for r, page_begin, page_count, _, c in tiles.tolist():
        L = int(pb.kv_lens[r])
        lo = max(0, L - 1 - window) if window >= 0 else 0
        base, end = page_begin * P, min(L, (page_begin + page_count) * P)
        for pos0 in range(base + (max(lo, base) - base) // 16 * 16, end, 16):
            want[c].append(int(pb.kv_indices[pb.kv_indptr[r] + pos0 // P]) * 2 * P + pos0 % P)
    for c in range(ctas):
        first = (want[c] + [-1] * 4)[:4]
        assert rows[c].tolist() == first, c
        assert want[c], c  # every CTA of a split has a chunk to read


def test_decode_head_rows_rejects_invalid_rows(lib):
    """The head-row export validates its index arrays as pkv_plan does (it reads page ids)."""
    h = _handle(num_cache_pages=64)
    for kvp, kvi, lpl in (([0, 2, 1], [0, 1], [1, 1]),       # kv_indptr decreases
                          ([0, 2], [0, 99], [1]),            # a page id past the cache
                          ([0, 1], [0], [17])):              # last_page_len above the page size
        with pytest.raises(B.PkvError) as e:
            h.decode_head_rows(kvp, kvi, lpl)
        assert e.value.status == B.ERR_INVALID


def test_nvtx_ranges_leave_host_results_unchanged(lib):
    """enable_nvtx (the wrappers' constructor flag) only opens a range per call: the split
    and a plan rejected before any copy come out the same, and a range opened by a call
    that returns early is closed (the next calls still work)."""
    pb = _split_case("batch", 16)
    on, off = (_handle(num_cache_pages=pb.max_pages, enable_nvtx=f) for f in (True, False))
    for _ in range(3):
        t_on, c_on = on.decode_split(pb.kv_indptr, pb.last_page_len, -1)
        t_off, c_off = off.decode_split(pb.kv_indptr, pb.last_page_len, -1)
        assert c_on == c_off and np.array_equal(t_on, t_off)
        bad = ([0, 1], [0, 2, 1], [0, 1], [1, 1])  # kv_indptr decreases
        assert _plan_status(on, B.MODE_DECODE, (None,) + bad[1:]) == _plan_status(off, B.MODE_DECODE, (None,) + bad[1:])


def _plan_status(h, mode, idx, **kw):
    ws_bytes = kw.pop("ws_bytes", 1 << 30)
    qo, kvp, kvi, lpl = (None if a is None else np.ascontiguousarray(np.asarray(a, np.int32)) for a in idx)
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    st = h.lib.pkv_plan(h.h, mode, p(qo), p(kvp), p(kvi), p(lpl), len(kvp) - 1, kw.get("causal", 1),
                        kw.get("window_left", -1), kw.get("sm_scale", 0.0), ctypes.c_void_p(1 << 20), ws_bytes, None)
    return st, h.lib.pkv_last_error(h.h).decode()


@pytest.mark.parametrize("case,status", [
    ("indptr_decreases", B.ERR_INVALID),
    ("page_out_of_pool", B.ERR_INVALID),
    ("last_len_zero", B.ERR_INVALID),
    ("last_len_too_big", B.ERR_INVALID),
    ("more_new_than_len", B.ERR_INVALID),
    ("window_below_minus_one", B.ERR_INVALID),
    ("decode_with_two_tokens", B.ERR_INVALID),
    ("too_many_prompt_rows", B.ERR_TOO_MANY_PREFILL_ROWS),
    ("workspace_too_small", B.ERR_WORKSPACE),
])
def test_plan_validation(lib, case, status):
    h = _handle(num_cache_pages=100, max_num_pages=100, max_prefill_rows=1, sink_page=99)
    qo, kvp, kvi, lpl = [0, 1, 4], [0, 1, 3], [5, 6, 7], [3, 16]
    mode, kw = B.MODE_PREFILL, {}
    if case == "indptr_decreases":
        kvp = [0, 2, 1]
    elif case == "page_out_of_pool":
        kvi = [5, 6, 100]
    elif case == "last_len_zero":
        lpl = [0, 16]
    elif case == "last_len_too_big":
        lpl = [17, 16]
    elif case == "more_new_than_len":
        qo, kvp, kvi, lpl = [0, 5], [0, 1], [5], [4]
    elif case == "window_below_minus_one":
        kw["window_left"] = -2
    elif case == "decode_with_two_tokens":
        mode = B.MODE_DECODE
    elif case == "too_many_prompt_rows":
        mode, qo = B.MODE_MIXED, [0, 2, 5]
    elif case == "workspace_too_small":
        kw["ws_bytes"] = 1024
    st, msg = _plan_status(h, mode, (qo, kvp, kvi, lpl), **kw)
    assert st == status, (st, msg)
    assert msg
    if case == "workspace_too_small":
        assert "needs" in msg and re.search(r"\d{4,}", msg)


@pytest.mark.parametrize("bad_at,bad_id", [(0, 100), (17, -1), (33, 2**31 - 1), (5, -2**31)])
def test_plan_names_the_first_page_id_outside_the_cache(lib, bad_at, bad_id):
    """Page ids are range-checked all at once and the offending entry is looked up afterwards:
    the error names the first id outside [0, num_cache_pages) and its index, wherever it sits
    (first, middle or last entry, negative or past the pool), and a second bad id further on
    does not change which one is named."""
    h = _handle(num_cache_pages=100, max_num_pages=100, max_prefill_rows=1, sink_page=99)
    kvi = list(range(40, 74))  # 34 valid ids: rows of 20 and 14 pages
    kvi[bad_at] = bad_id
    if bad_at + 1 < len(kvi):
        kvi[-1] = 1000  # a later bad id
    st, msg = _plan_status(h, B.MODE_PREFILL, ([0, 1, 4], [0, 20, 34], kvi, [3, 16]))
    assert st == B.ERR_INVALID, (st, msg)
    assert f"page id {bad_id} at paged_kv_indices[{bad_at}]" in msg, msg
    ok = list(range(40, 74))
    assert _plan_status(h, B.MODE_PREFILL, ([0, 1, 4], [0, 20, 34], ok, [3, 16]), ws_bytes=1024)[0] == B.ERR_WORKSPACE


def test_workspace_bound_holds(lib):
    for name in ["tiny", "batch", "prefill", "mixed", "long"]:
        pb = wl.WORKLOADS[name]()
        h = _handle(num_qo_heads=pb.num_qo_heads, num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim,
                    max_batch=pb.batch, max_total_tokens=max(pb.num_tokens, pb.batch),
                    max_num_pages=len(pb.kv_indices), num_cache_pages=pb.max_pages,
                    max_prefill_rows=max(pb.max_prefill_rows, 1), sink_page=pb.sink_page)
        mode = {"tiny": 0, "batch": 0, "long": 0, "prefill": 1, "mixed": 2}[name]
        bound = h.workspace_size(mode)
        # a plan whose workspace is exactly the bound must pass the size check (it then
        # fails only at the H2D copy, which needs a GPU)
        st, msg = _plan_status(h, mode, (None if mode == 0 else pb.qo_indptr, pb.kv_indptr, pb.kv_indices,
                                         pb.last_page_len), ws_bytes=bound)
        assert st != B.ERR_WORKSPACE, msg


@pytest.mark.parametrize("seed", range(5))
def test_context_only_views_bit_exact(lib, seed):
    rng = np.random.default_rng(300 + seed)
    Bn = int(rng.integers(1, 30))
    n = rng.integers(0, 40, size=Bn)
    c = rng.integers(0, 70, size=Bn)
    pb = wl.custom(seed, n + c, n, num_qo_heads=8, num_kv_heads=2, head_dim=64, page_size=16)
    got = B.context_only_views(16, *pb.index_arrays())
    want = plan_ref.context_only_views(*pb.index_arrays(), 16)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)
    # the views keep exactly the first L - n positions of every row
    L = plan_ref.row_lengths(got[0], got[2], 16)
    assert np.array_equal(L, c)


def test_context_only_needs_prefill_mode(lib):
    h = _handle(num_cache_pages=100, max_num_pages=100)
    st, msg = _plan_status(h, B.MODE_DECODE, (None, [0, 1], [3], [4]), causal=2)
    assert st == B.ERR_INVALID and "context" in msg


def _dense_status(h, cu_q, cu_k, causal=1):
    cq, ck = (np.ascontiguousarray(np.asarray(a, np.int32)) for a in (cu_q, cu_k))
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = h.lib.pkv_plan_dense(h.h, p(cq), p(ck), len(cq) - 1, causal, -1, 0.0, ctypes.c_void_p(1 << 20), 1024, None)
    return st, h.lib.pkv_last_error(h.h).decode()


def test_dense_plan_validation(lib):
    h = _handle(max_total_tokens=100, max_batch=4)
    assert _dense_status(h, [0, 5], [0, 4])[0] == B.ERR_INVALID          # more queries than keys
    assert _dense_status(h, [0, 3, 2], [0, 4, 9])[0] == B.ERR_INVALID    # decreasing cu_q
    assert _dense_status(h, [0, 101], [0, 200])[0] == B.ERR_INVALID      # above max_total_tokens
    assert _dense_status(h, [0, 3], [0, 4], causal=2)[0] == B.ERR_INVALID
    st, msg = _dense_status(h, [0, 3, 5], [0, 40, 50])                   # valid: too small a workspace
    assert st == B.ERR_WORKSPACE, msg
    assert h.workspace_size(B.MODE_DENSE) > 0

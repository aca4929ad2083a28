"""Shapes beyond page_size 16: page sizes 1 .. 64 and 128 .. 1024, head_dim 256, group sizes that are not
powers of two, and more than 8 kv heads (decode then splits the kv heads over CTA groups),
each through the C ABI against the oracle on the same seeded inputs.

Same bars as the main parity file: the appended layer slice bit-exact, outputs at max-abs
2e-2 and relative L2 1e-2, lse at 1e-3 relative; free pages and page tails hold bf16 NaN,
so a read outside a row's slots shows up.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
from paged_kv_attention_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from paged_kv_attention_gqa_gb300 import build
    build.build()


def _check_step(pb, mode, *, window_left=-1, causal=True, sm_count=0, seed=0, fused=False):
    x = wl.make_inputs(pb, device="cuda", seed=seed, unused="nan", layers=1)
    before = wl.bf16_bits(x["kv_cache"][0])
    out, lse, h, ws = G.gpu_step(pb, x, mode, window_left=window_left, causal=causal, sm_count=sm_count,
                                 fused=fused)
    after = G.oracle_append(pb, before, x)
    assert np.array_equal(wl.bf16_bits(x["kv_cache"][0]), after), "appended cache differs (bit-exact)"
    ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after, causal=causal if mode != "decode" else True,
                                 window_left=window_left)
    return G.compare(out, lse, ref_o, ref_l, what=f"{mode} P{pb.page_size} D{pb.head_dim} "
                                                  f"{pb.num_qo_heads}/{pb.num_kv_heads}")


def _decode_lens(P):
    # page boundaries of this page size, a one-token row, and a few long rows
    return [1, 2, P, P + 1, 2 * P - 1, 3 * P, 17, 100, 257, 1000]


PAGE_SIZES = [1, 2, 4, 8, 32, 64]


# ------------------------------------------------------------------ page sizes

@pytest.mark.parametrize("P", PAGE_SIZES)
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 1, 64), (16, 4, 256), (8, 2, 128)])
def test_decode_page_sizes(P, Hq, Hkv, D):
    lens = _decode_lens(P)
    pb = wl.custom(100 + P, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                   pool_factor=1.3)
    _check_step(pb, "decode", seed=P)


@pytest.mark.parametrize("P", PAGE_SIZES)
@pytest.mark.parametrize("Hq,Hkv,D,sm_count", [(32, 8, 128, 0), (8, 1, 64, 5), (16, 4, 256, 0), (32, 16, 128, 10)])
def test_decode_append_fused_page_sizes(P, Hq, Hkv, D, sm_count):
    """The fused append patches the new token's slot wherever the page layout puts it
    (K and V in separate boxes, or one box per page below 8 slots; head groups)."""
    lens = _decode_lens(P)
    pb = wl.custom(250 + P, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                   pool_factor=1.3)
    _check_step(pb, "decode", sm_count=sm_count, seed=P + 7, fused=True)


@pytest.mark.parametrize("P", PAGE_SIZES)
@pytest.mark.parametrize("sm_count", [1, 3, 40])
def test_decode_page_sizes_forced_splits(P, sm_count):
    """Pieces cut at page boundaries of every page size; 40 CTAs cut the 3000-key row into
    many pieces for the merge kernel, 3 into few."""
    lens = [3000, 5, 64, 1, 333]
    pb = wl.custom(110 + P, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=P)
    _check_step(pb, "decode", sm_count=sm_count, seed=P + 1)


@pytest.mark.parametrize("P", [1, 4, 8, 64])
@pytest.mark.parametrize("window", [0, 3, 16, 100])
def test_decode_page_sizes_window(P, window):
    lens = [1, 5, 16, 17, 40, 300, 1500]
    pb = wl.custom(120 + P, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=P)
    _check_step(pb, "decode", window_left=window, seed=3)


@pytest.mark.parametrize("P", PAGE_SIZES)
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 2, 64), (8, 4, 256)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_page_sizes(P, Hq, Hkv, D, causal):
    n = [1, 7, 33, 130, 64, 2]
    c = [0, 40, 0, 300, 17, 1]
    pb = wl.custom(130 + P, np.add(n, c), n, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P)
    _check_step(pb, "prefill", causal=causal, seed=P + 2)


@pytest.mark.parametrize("P", [1, 2, 8, 64])
@pytest.mark.parametrize("window", [0, 5, 64, 200])
def test_prefill_page_sizes_window(P, window):
    n = [200, 5, 70]
    c = [0, 500, 90]
    pb = wl.custom(140 + P, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=P)
    _check_step(pb, "prefill", window_left=window, seed=4)


@pytest.mark.parametrize("P", [1, 4, 8, 32])
def test_mixed_page_sizes(P):
    n = [1, 1, 40, 1, 3, 1, 0, 1, 100]
    c = [20, 300, 10, 1, 0, 16, 5, 700, 33]
    pb = wl.custom(150 + P, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=P,
                   reserve_sink=True)
    pb.max_prefill_rows = int((np.asarray(n) >= 2).sum()) + 1
    _check_step(pb, "mixed", seed=5)


# ------------------------------------------------------------------ pages of 128 to 1024 slots

LARGE_PAGES = [128, 256, 1024]


@pytest.mark.parametrize("P", LARGE_PAGES)
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 1, 64), (16, 4, 256)])
@pytest.mark.parametrize("fused", [False, True])
def test_decode_large_pages(P, Hq, Hkv, D, fused):
    lens = _decode_lens(P)
    pb = wl.custom(160 + P, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                   pool_factor=1.3)
    _check_step(pb, "decode", seed=P + 11, fused=fused)


@pytest.mark.parametrize("P", LARGE_PAGES)
@pytest.mark.parametrize("sm_count,window", [(1, -1), (3, -1), (40, -1), (40, 100), (0, 0)])
def test_decode_large_pages_splits_and_windows(P, sm_count, window):
    """Pieces cut at the boundaries of long pages (few pages per row) through both merges,
    and windows that start inside a page."""
    lens = [3 * P + 5, 5, P, 1, 2 * P - 3, 7000]
    pb = wl.custom(170 + P, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=P)
    _check_step(pb, "decode", sm_count=sm_count, window_left=window, seed=P + 12, fused=sm_count == 3)


@pytest.mark.parametrize("P", LARGE_PAGES)
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 2, 64), (8, 4, 256)])
@pytest.mark.parametrize("causal,window", [(True, -1), (False, -1), (True, 200)])
def test_prefill_large_pages(P, Hq, Hkv, D, causal, window):
    n = [1, 7, 33, 300, 64, 2]
    c = [0, 40, 0, P + 9, 2 * P, 1]
    pb = wl.custom(180 + P, np.add(n, c), n, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P)
    _check_step(pb, "prefill", causal=causal, window_left=window, seed=P + 13)


@pytest.mark.parametrize("P", LARGE_PAGES)
def test_mixed_large_pages(P):
    n = [1, 1, 40, 1, 3, 1, 0, 1, 100]
    c = [20, 3 * P, 10, 1, 0, P, 5, 700, 33]
    pb = wl.custom(190 + P, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=P,
                   reserve_sink=True)
    pb.max_prefill_rows = int((np.asarray(n) >= 2).sum()) + 1
    _check_step(pb, "mixed", seed=P + 14)


# ------------------------------------------------------------------ head_dim 256

@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (8, 1), (32, 2), (64, 8)])
def test_decode_head_dim_256(Hq, Hkv):
    lens = [1, 15, 16, 17, 100, 1000, 2500]
    pb = wl.custom(160, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=256, page_size=16)
    _check_step(pb, "decode", seed=6)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (8, 1), (32, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_head_dim_256(Hq, Hkv, causal):
    n = [1, 7, 33, 130, 64]
    c = [0, 40, 0, 300, 17]
    pb = wl.custom(161, np.add(n, c), n, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=256, page_size=16)
    _check_step(pb, "prefill", causal=causal, seed=7)


@pytest.mark.parametrize("window", [0, 5, 100, 200])
def test_prefill_head_dim_256_window(window):
    n = [1, 7, 33, 130, 300]
    c = [0, 40, 0, 300, 900]
    pb = wl.custom(162, np.add(n, c), n, num_qo_heads=16, num_kv_heads=8, head_dim=256, page_size=16)
    _check_step(pb, "prefill", window_left=window, seed=8)


# ------------------------------------------------------------------ group sizes 3, 5, 6, 7

@pytest.mark.parametrize("g", [3, 5, 6, 7])
@pytest.mark.parametrize("Hkv,D", [(4, 128), (1, 64), (2, 256)])
def test_decode_odd_groups(g, Hkv, D):
    lens = [1, 16, 17, 100, 1000]
    pb = wl.custom(170 + g, lens, [1] * len(lens), num_qo_heads=g * Hkv, num_kv_heads=Hkv, head_dim=D,
                   page_size=16)
    _check_step(pb, "decode", seed=g)


@pytest.mark.parametrize("g", [3, 5, 6, 7])
@pytest.mark.parametrize("Hkv,D", [(4, 128), (1, 64), (2, 256)])
def test_prefill_odd_groups(g, Hkv, D):
    """128 // g tokens per tile: the tile's last 128 mod g query rows are padding."""
    n = [1, 7, 43, 130, 64]
    c = [0, 40, 0, 300, 17]
    pb = wl.custom(180 + g, np.add(n, c), n, num_qo_heads=g * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=16)
    _check_step(pb, "prefill", seed=g)


@pytest.mark.parametrize("g", [3, 7])
def test_mixed_odd_groups(g):
    n = [1, 40, 1, 3, 1, 100]
    c = [20, 10, 700, 0, 16, 33]
    pb = wl.custom(190 + g, np.add(n, c), n, num_qo_heads=4 * g, num_kv_heads=4, head_dim=128, page_size=8,
                   reserve_sink=True)
    pb.max_prefill_rows = int((np.asarray(n) >= 2).sum()) + 1
    _check_step(pb, "mixed", seed=g)


# ------------------------------------------------------------------ more than 8 kv heads

@pytest.mark.parametrize("Hq,Hkv,D", [(16, 16, 128), (32, 16, 128), (24, 12, 64), (40, 40, 128), (32, 16, 256)])
@pytest.mark.parametrize("sm_count", [0, 10, 60])
def test_decode_many_kv_heads(Hq, Hkv, D, sm_count):
    """Several CTA head groups sharing the SMs, each group cutting the rows at its own piece
    boundaries: 10 SMs cut the long rows into few pieces, 60 into many (the merge kernel
    takes every head group's partials of a row)."""
    lens = [1, 17, 100, 1000, 2048]
    pb = wl.custom(200 + Hkv, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16)
    _check_step(pb, "decode", sm_count=sm_count, seed=Hkv)


@pytest.mark.parametrize("Hq,Hkv", [(16, 16), (32, 16)])
def test_prefill_many_kv_heads(Hq, Hkv):
    n = [1, 33, 130]
    c = [0, 40, 300]
    pb = wl.custom(210 + Hkv, np.add(n, c), n, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=128, page_size=16)
    _check_step(pb, "prefill", seed=Hkv)


# ------------------------------------------------------------------ dense varlen, gather, graph mode

@pytest.mark.parametrize("D,Hq,Hkv,P", [(256, 16, 8, 16), (128, 28, 4, 1), (64, 12, 2, 4)])
def test_dense_shapes(D, Hq, Hkv, P):
    """Dense plans read contiguous K / V in 16-row boxes whatever the handle's page size."""
    import oracle
    from paged_kv_attention_gqa_gb300 import binding as B
    n = [1, 40, 130, 7]
    L = [1, 300, 130, 90]
    gen = torch.Generator(device="cuda").manual_seed(220)
    q = torch.randn(sum(n), Hq, D, generator=gen, device="cuda").to(torch.bfloat16)
    k = torch.randn(sum(L), Hkv, D, generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(sum(L), Hkv, D, generator=gen, device="cuda").to(torch.bfloat16)
    cu_q = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    h = B.Handle(num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P, max_batch=len(n),
                 max_total_tokens=sum(n), max_num_pages=1, num_cache_pages=1)
    ws = torch.empty(h.workspace_size(B.MODE_DENSE), dtype=torch.uint8, device="cuda")
    h.plan_dense(cu_q, cu_k, workspace=ws, causal=True)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    h.run_dense(q, k, v, out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert h.check_device_error(ws) == 0
    ro, rl = oracle.dense_attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), cu_q, cu_k, num_qo_heads=Hq,
                                    num_kv_heads=Hkv, head_dim=D, causal=True)
    G.compare(out, lse, ro, rl, what=f"dense D{D} {Hq}/{Hkv}")


@pytest.mark.parametrize("P", [1, 8, 64])
def test_gather_kv_page_sizes(P):
    """The prefix gather is pure data movement: bit-exact against the logical K / V."""
    pb = wl.custom(230 + P, [200, 3 * P + 1], [1, 1], num_qo_heads=8, num_kv_heads=2, head_dim=128, page_size=P)
    x = wl.make_inputs(pb, device="cuda", seed=9, unused="nan", layers=1)
    h = G.make_handle(pb)
    kv = x["kv_cache"][0]
    for r in range(pb.batch):
        L = int(pb.kv_lens[r]) - 1  # the stored prefix (the step's token is not appended here)
        pages = torch.as_tensor(pb.page_table[r], dtype=torch.int32, device="cuda")
        k = torch.empty(L, 2, 128, dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        h.gather_kv(kv, pages, L, k, v)
        torch.cuda.synchronize()
        rows = wl._flat_slot_rows(pb, r, np.arange(L))
        cache = wl.bf16_bits(kv).reshape(-1, 2, 128)
        assert np.array_equal(wl.bf16_bits(k), cache[rows])
        assert np.array_equal(wl.bf16_bits(v), cache[rows + P])


@pytest.mark.parametrize("P,D,Hq,Hkv", [(4, 128, 32, 8), (16, 256, 16, 8), (1, 64, 24, 12)])
def test_graph_mode_shapes(P, D, Hq, Hkv):
    """Append + decode captured once at the handle's maxima, replayed for a new plan."""
    from paged_kv_attention_gqa_gb300 import binding as B
    lens_a = [5, 40, 300, 17]
    lens_b = [900, 1, 64, 33]
    pbs = [wl.custom(240 + i, L, [1] * 4, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                     pool_pages=2048 // P + 64) for i, L in enumerate((lens_a, lens_b))]
    h = B.Handle(num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P, max_batch=4, max_total_tokens=4,
                 max_num_pages=max(len(pb.kv_indices) for pb in pbs) + 8, num_cache_pages=pbs[0].max_pages,
                 max_prefill_rows=0, graph_static=1)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device="cuda")
    x0 = wl.make_inputs(pbs[0], device="cuda", seed=10, unused="nan", layers=1)
    q = x0["q"].clone()
    k_new, v_new = x0["k_new"].clone(), x0["v_new"].clone()
    kv = x0["kv_cache"][0].clone()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    h.plan(B.MODE_DECODE, None, pbs[0].kv_indptr, pbs[0].kv_indices, pbs[0].last_page_len, workspace=ws)
    h.kv_append_planned(k_new, v_new, kv, workspace=ws)
    h.run_decode(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        h.kv_append_planned(k_new, v_new, kv, workspace=ws)
        h.run_decode(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    for i, pb in enumerate(pbs):
        x = wl.make_inputs(pb, device="cuda", seed=11 + i, unused="nan", layers=1)
        before = wl.bf16_bits(x["kv_cache"][0])
        q.copy_(x["q"])
        k_new.copy_(x["k_new"])
        v_new.copy_(x["v_new"])
        kv.copy_(x["kv_cache"][0])
        out.fill_(float("nan"))
        h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
        graph.replay()
        torch.cuda.synchronize()
        assert h.check_device_error(ws) == 0
        after = G.oracle_append(pb, before, x)
        assert np.array_equal(wl.bf16_bits(kv), after)
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after)
        G.compare(out, lse, ref_o, ref_l, what=f"graph P{P} D{D} plan {i}")


def test_mixed_head_dim_256():
    n = [1, 40, 1, 3, 1, 100]
    c = [20, 10, 700, 0, 16, 33]
    pb = wl.custom(260, np.add(n, c), n, num_qo_heads=16, num_kv_heads=8, head_dim=256, page_size=16,
                   reserve_sink=True)
    pb.max_prefill_rows = int((np.asarray(n) >= 2).sum()) + 1
    _check_step(pb, "mixed", seed=12)


@pytest.mark.parametrize("P", [2, 32])
def test_graph_mode_prefill_page_sizes(P):
    """Prefill (cp.async gather below 8 slots, TMA above) captured once at the maxima,
    replayed for a second plan of another shape of rows."""
    from paged_kv_attention_gqa_gb300 import binding as B
    steps = [([5, 40, 130], [0, 300, 17]), ([64, 1], [900, 3])]
    pbs = [wl.custom(270 + i, np.add(n, c), n, num_qo_heads=16, num_kv_heads=4, head_dim=128, page_size=P,
                     pool_pages=2048 // P + 64) for i, (n, c) in enumerate(steps)]
    T = max(pb.num_tokens for pb in pbs)
    h = B.Handle(num_qo_heads=16, num_kv_heads=4, head_dim=128, page_size=P, max_batch=3, max_total_tokens=T,
                 max_num_pages=max(len(pb.kv_indices) for pb in pbs) + 8, num_cache_pages=pbs[0].max_pages,
                 max_prefill_rows=3, graph_static=1)
    ws = torch.empty(h.workspace_size(B.MODE_PREFILL), dtype=torch.uint8, device="cuda")
    q = torch.zeros(T, 16, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(T, 4, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.zeros_like(q)
    lse = torch.zeros(T, 16, dtype=torch.float32, device="cuda")
    kv = torch.zeros(pbs[0].max_pages, 2, P, 4, 128, dtype=torch.bfloat16, device="cuda")

    def load(pb, seed):
        x = wl.make_inputs(pb, device="cuda", seed=seed, unused="nan", layers=1)
        n = pb.num_tokens
        q[:n].copy_(x["q"])
        k[:n].copy_(x["k_new"])
        v[:n].copy_(x["v_new"])
        kv.copy_(x["kv_cache"][0])
        return x

    def plan(pb):
        h.plan(B.MODE_PREFILL, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)

    load(pbs[0], 20)
    plan(pbs[0])
    h.kv_append_planned(k, v, kv, workspace=ws)
    h.run_prefill(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        h.kv_append_planned(k, v, kv, workspace=ws)
        h.run_prefill(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    for i, pb in enumerate(pbs[::-1]):
        x = load(pb, 21 + i)
        before = wl.bf16_bits(kv)
        out.fill_(float("nan"))
        plan(pb)
        graph.replay()
        torch.cuda.synchronize()
        assert h.check_device_error(ws) == 0
        after = G.oracle_append(pb, before, x)
        assert np.array_equal(wl.bf16_bits(kv), after)
        n = pb.num_tokens
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after)
        G.compare(out[:n], lse[:n], ref_o, ref_l, what=f"graph prefill P{P} plan {i}")

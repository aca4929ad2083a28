"""CUDA path (through the C ABI) against the oracle on the same seeded inputs.

Index and addressing work is compared bit-exactly (the appended cache, every byte of
the layer slice); attention outputs at max-abs 2e-2, relative L2 1e-2, lse 1e-3
relative (|d| <= 1e-3 max(1, |lse|)).  Free pages and page tails hold bf16 NaN unless a
case says otherwise, so any read past a row's end shows up.
"""
import math

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


def _check_step(pb, mode, *, window_left=-1, causal=True, sm_scale=0.0, sm_count=0, seed=0, unused="nan",
                rows=None, fused=False):
    x = wl.make_inputs(pb, device="cuda", seed=seed, unused=unused, layers=1)
    before = wl.bf16_bits(x["kv_cache"][0])
    out, lse, h, ws = G.gpu_step(pb, x, mode, window_left=window_left, causal=causal, sm_scale=sm_scale,
                                 sm_count=sm_count, fused=fused)
    after = G.oracle_append(pb, before, x)
    got = wl.bf16_bits(x["kv_cache"][0])
    assert np.array_equal(got, after), "appended cache differs from the oracle's (bit-exact)"
    ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after, causal=causal if mode != "decode" else True,
                                 window_left=window_left, sm_scale=sm_scale, rows=rows)
    tokens = None if rows is None else G.token_mask(pb, rows)
    return G.compare(out, lse, ref_o, ref_l, tokens=tokens, what=f"{pb.name}/{mode}")


# ------------------------------------------------------------------ decode

def test_tiny_decode_config():
    pb = wl.config_tiny()
    _check_step(pb, "decode")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (8, 2), (16, 2), (32, 2)])
def test_decode_groups_and_dims(D, Hq, Hkv):
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 100, 257, 1000]
    pb = wl.custom(3, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16,
                   pool_factor=1.3)
    _check_step(pb, "decode", seed=1)


@pytest.mark.parametrize("window", [0, 1, 5, 15, 16, 17, 100])
def test_decode_window(window):
    lens = [1, 5, 16, 17, 40, 300, 1500]
    pb = wl.custom(4, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    _check_step(pb, "decode", window_left=window, seed=2)


@pytest.mark.parametrize("sm_count", [1, 2, 3, 7, 152, 300])
def test_decode_forced_splits(sm_count):
    lens = [700, 33, 1, 2048, 129, 16, 4000]
    pb = wl.custom(5, lens, [1] * len(lens), num_qo_heads=64, num_kv_heads=8, head_dim=128, page_size=16)
    _check_step(pb, "decode", sm_count=sm_count, seed=3)


@pytest.mark.parametrize("D,Hq,Hkv", [(64, 16, 4), (256, 16, 4)])
@pytest.mark.parametrize("sm_count", [10, 40, 152, 300])
def test_decode_merge_piece_counts(D, Hq, Hkv, sm_count):
    """Rows cut into 3 to ~130 pieces at head_dim 64 and 256: the merge kernel's small and large
    instances, one or several batches of pieces, and more than 32 pieces per row (lse values
    past a lane each)."""
    lens = [4000, 1200, 33, 1]
    pb = wl.custom(6, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16)
    _check_step(pb, "decode", sm_count=sm_count, seed=4)


# (head_dim, Hq, Hkv, row length, SM count, pieces of the long row): each merge-kernel instance
# at the end of its batch of pieces and one past it (B = 32 / 16 / 8 small, 32 / 32 / 16 large at
# head_dim 64 / 128 / 256), and 32 / 33 pieces (the lse values past one per lane)
MERGE_EDGES = [(64, 16, 4, 3000, 16, 32), (64, 16, 4, 4100, 17, 33), (128, 32, 8, 3000, 16, 16),
               (128, 32, 8, 3500, 18, 17), (128, 32, 8, 3000, 32, 32), (128, 32, 8, 4100, 33, 33),
               (256, 16, 4, 3000, 8, 8), (256, 16, 4, 3000, 9, 9), (256, 16, 4, 3000, 16, 16),
               (256, 16, 4, 3500, 18, 17), (256, 16, 4, 4100, 33, 33)]


@pytest.mark.parametrize("D,Hq,Hkv,L,sm_count,pieces", MERGE_EDGES)
def test_decode_merge_batch_edges(D, Hq, Hkv, L, sm_count, pieces):
    pb = wl.custom(8, [L, 40], [1, 1], num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16)
    h = G.make_handle(pb, sm_count=sm_count)
    tiles, _ = h.decode_split(pb.kv_indptr, pb.last_page_len)
    assert np.bincount(tiles[:, 0]).max() == pieces, "the split no longer cuts the row into this many pieces"
    _check_step(pb, "decode", sm_count=sm_count, seed=9)


# ------------------------------------------------------------------ append fused into the decode launch

@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 8, 2), (128, 16, 1)])
@pytest.mark.parametrize("sm_count", [0, 1, 3, 7, 300])
def test_decode_append_fused(D, Hq, Hkv, sm_count):
    """pkv_run_decode_append: the appended slice bit-exact and the outputs at tolerance,
    with the row's new token taken from the stage patched in shared memory (poisoned
    slots would show otherwise: the slot holds NaN until the append)."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 100, 257, 1000, 4000]
    pb = wl.custom(20, lens, [1] * len(lens), num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16)
    _check_step(pb, "decode", sm_count=sm_count, seed=21, fused=True)


@pytest.mark.parametrize("window", [0, 1, 16, 100])
def test_decode_append_fused_window(window):
    lens = [1, 5, 16, 17, 40, 300, 1500]
    pb = wl.custom(22, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    _check_step(pb, "decode", window_left=window, seed=23, fused=True)


def test_decode_append_fused_equals_separate_calls():
    """Same plan, same inputs: the fused launch gives the same bits as append + decode."""
    lens = [700, 33, 1, 2048, 129, 16, 4000]
    pb = wl.custom(24, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    res = []
    for fused in (False, True):
        x = wl.make_inputs(pb, device="cuda", seed=25, unused="nan", layers=1)
        out, lse, _, _ = G.gpu_step(pb, x, "decode", fused=fused)
        res.append((wl.bf16_bits(out), lse.cpu().numpy(), wl.bf16_bits(x["kv_cache"][0])))
    for a, b in zip(*res):
        assert np.array_equal(a, b)


def test_decode_sm_scale():
    pb = wl.custom(6, [90, 400], [1, 1], num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    _check_step(pb, "decode", sm_scale=0.3, seed=4)


def test_decode_page_pool_permutation_is_bit_identical():
    import oracle_pins
    pb = wl.custom(7, [300, 17, 1000, 64], [1, 1, 1, 1], num_qo_heads=32, num_kv_heads=8, head_dim=128,
                   page_size=16, pool_factor=1.5)
    x = wl.make_inputs(pb, device="cuda", seed=5, unused="nan", layers=1)
    out1, lse1, _, _ = G.gpu_step(pb, x, "decode")
    pb2, kv2 = oracle_pins.relabel_pool(pb, x["kv_cache"][0], seed=9)
    x2 = dict(x, kv_cache=kv2.unsqueeze(0))
    out2, lse2, _, _ = G.gpu_step(pb2, x2, "decode", append=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


@pytest.mark.parametrize("heads", [(32, 8, 128), (16, 8, 256)])
def test_prefill_page_pool_permutation_is_bit_identical(heads):
    """The plan depends only on the lengths, so relabelling and moving the pool's pages leaves
    every output bit unchanged (the two-query-tile kernel at head_dim 128, the head_dim-256
    kernel)."""
    import oracle_pins
    pb = wl.custom(17, [300, 17, 1000, 64, 200], [40, 17, 300, 1, 129], num_qo_heads=heads[0],
                   num_kv_heads=heads[1], head_dim=heads[2], page_size=16, pool_factor=1.5)
    x = wl.make_inputs(pb, device="cuda", seed=15, unused="nan", layers=1)
    out1, lse1, _, _ = G.gpu_step(pb, x, "prefill")
    pb2, kv2 = oracle_pins.relabel_pool(pb, x["kv_cache"][0], seed=19)
    x2 = dict(x, kv_cache=kv2.unsqueeze(0))
    out2, lse2, _, _ = G.gpu_step(pb2, x2, "prefill", append=False)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_empty_batch_is_a_no_op():
    pb = wl.custom(8, [5], [1], num_qo_heads=8, num_kv_heads=2, head_dim=64, page_size=16)
    h = G.make_handle(pb)
    ws = torch.empty(h.workspace_size(0), dtype=torch.uint8, device="cuda")
    h.plan(0, None, [0], [], [], workspace=ws)
    q = torch.zeros(0, 8, 64, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(pb.max_pages, 2, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    h.run_decode(q, kv, q, None, workspace=ws)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 8, 8), (128, 16, 2), (64, 32, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_ragged(D, Hq, Hkv, causal):
    n = [1, 7, 33, 130, 64, 2]
    c = [0, 40, 0, 300, 17, 1]
    pb = wl.custom(10, np.add(n, c), n, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16)
    _check_step(pb, "prefill", causal=causal, seed=6)


@pytest.mark.parametrize("window", [0, 3, 16, 63, 64, 200])
def test_prefill_window(window):
    n = [200, 5, 70]
    c = [0, 500, 90]
    pb = wl.custom(11, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    _check_step(pb, "prefill", window_left=window, seed=7)


def test_prefill_rows_without_tokens():
    n = [0, 20, 0, 3]
    c = [50, 10, 1, 0]
    pb = wl.custom(12, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    _check_step(pb, "prefill", seed=8)


# ------------------------------------------------------------------ mixed

def _mixed_batch(seed, n, c, **kw):
    pb = wl.custom(seed, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                   reserve_sink=True, **kw)
    pb.max_prefill_rows = int((np.asarray(n) >= 2).sum()) + 1
    return pb


def test_mixed_small():
    n = [1, 1, 40, 1, 3, 1, 0, 1, 100]
    c = [20, 300, 10, 1, 0, 16, 5, 700, 33]
    pb = _mixed_batch(13, n, c)
    _check_step(pb, "mixed", seed=9)


def test_mixed_matches_separate_passes():
    n = [1, 70, 1, 1, 9]
    c = [33, 0, 500, 1, 60]
    pb = _mixed_batch(14, n, c)
    x = wl.make_inputs(pb, device="cuda", seed=10, unused="nan", layers=1)
    out_m, lse_m, _, _ = G.gpu_step(pb, x, "mixed")
    # the same rows through the plain prefill plan (no append: the cache already holds them)
    out_p, lse_p, _, _ = G.gpu_step(pb, x, "prefill", append=False)
    G.compare(out_m, lse_m, out_p.float().cpu().numpy(), lse_p.cpu().numpy(), what="mixed vs prefill")


def test_mixed_poisoned_sink_rows_do_not_leak():
    """Every prompt row's decode-pass result is dropped: poisoning q of prompt tokens'
    decode-pass reads cannot reach out (the sink page holds finite values)."""
    n = [1, 12, 1]
    c = [5, 3, 40]
    pb = _mixed_batch(15, n, c)
    _check_step(pb, "mixed", seed=11)


# ------------------------------------------------------------------ full-size workloads (launch configuration of bench.py)

def test_batch_decode_full_size():
    """The bench's step: one plan, then one fused append + decode launch per layer over the
    32-layer cache.  Layers 0 and 31: the whole appended slice bit-exact and every row
    against the oracle.  Every other layer: a seeded 8-row sample against the oracle and
    its appended slots bit-exact."""
    pb = wl.config_batch_decode()
    x = wl.make_inputs(pb, device="cuda", seed=0, unused="randn")
    h = G.make_handle(pb)
    ws = torch.empty(h.workspace_size(0), dtype=torch.uint8, device="cuda")
    h.plan(0, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    rng = np.random.default_rng(2024)
    check_layers = {l: None if l in (0, pb.num_layers - 1) else sorted(rng.choice(pb.batch, 8, replace=False))
                    for l in range(pb.num_layers)}
    befores = {l: wl.bf16_bits(x["kv_cache"][l]) for l, rows in check_layers.items() if rows is None}
    outs = {}
    for l in range(pb.num_layers):  # as bench.py runs the step: one fused launch per layer
        kv = x["kv_cache"][l]
        out = torch.empty_like(x["q"])
        lse = torch.empty(pb.batch, pb.num_qo_heads, dtype=torch.float32, device="cuda")
        h.run_decode_append(x["q"], x["k_new"], x["v_new"], kv, out, lse, workspace=ws)
        outs[l] = (out, lse)
    torch.cuda.synchronize()
    assert h.check_device_error(ws) == 0
    k_bits, v_bits = wl.bf16_bits(x["k_new"]), wl.bf16_bits(x["v_new"])
    P = pb.page_size
    for l, rows in check_layers.items():
        after = wl.bf16_bits(x["kv_cache"][l])
        if rows is None:
            assert np.array_equal(after, G.oracle_append(pb, befores[l], x)), l
        else:
            for r in rows:  # the row's new token at (last page, last slot)
                page, slot = int(pb.page_table[r][(int(pb.kv_lens[r]) - 1) // P]), (int(pb.kv_lens[r]) - 1) % P
                assert np.array_equal(after[page, 0, slot], k_bits[r]), (l, r)
                assert np.array_equal(after[page, 1, slot], v_bits[r]), (l, r)
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after, rows=rows, threads=16)
        G.compare(*outs[l], ref_o, ref_l, tokens=None if rows is None else G.token_mask(pb, rows), what=f"layer {l}")


def test_ragged_prefill_full_size():
    """Every token of every row of the timed prefill workload against the oracle (its rows
    cut into causal runs so the oracle spreads them over 16 threads)."""
    pb = wl.config_prefill()
    x = wl.make_inputs(pb, device="cuda", seed=0, unused="randn", layers=1)
    before = wl.bf16_bits(x["kv_cache"][0])
    out, lse, h, ws = G.gpu_step(pb, x, "prefill")
    after = G.oracle_append(pb, before, x)
    assert np.array_equal(wl.bf16_bits(x["kv_cache"][0]), after), "appended cache differs from the oracle's"
    ref_o, ref_l = G.oracle_attn_causal_split(pb, wl.bf16_bits(x["q"]), after)
    G.compare(out, lse, ref_o, ref_l, what="ragged prefill, all 16 rows")


def test_mixed_full_size():
    pb = wl.config_mixed()
    _check_step(pb, "mixed", unused="nan")


@pytest.mark.parametrize("window", [-1, 4096])
def test_long_decode_full_size(window):
    pb = wl.config_long(window_left=window)
    _check_step(pb, "decode", window_left=window, unused="randn")


# ------------------------------------------------------------------ determinism (races show up here)

@pytest.mark.parametrize("mode", ["decode", "prefill", "mixed"])
def test_repeated_runs_are_bit_identical(mode):
    if mode == "decode":
        lens = list(np.random.default_rng(40).integers(1, 3000, size=60))
        pb = wl.custom(40, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    elif mode == "prefill":
        n = list(np.random.default_rng(41).integers(1, 400, size=12))
        c = list(np.random.default_rng(42).integers(0, 700, size=12))
        pb = wl.custom(41, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    else:
        n = [1, 1, 300, 1, 1, 77, 1]
        c = [900, 40, 20, 1, 2000, 300, 5]
        pb = _mixed_batch(43, n, c)
    x = wl.make_inputs(pb, device="cuda", seed=13, unused="nan", layers=1)
    out0, lse0, h, ws = G.gpu_step(pb, x, mode)
    for _ in range(4):
        out = torch.full_like(out0, float("nan"))
        lse = torch.full_like(lse0, float("nan"))
        getattr(h, "run_" + mode)(x["q"], x["kv_cache"][0], out, lse, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse, lse0)


@pytest.mark.parametrize("mode", ["decode", "prefill", "mixed"])
def test_nvtx_handle_gives_bit_identical_results(mode):
    """A handle made with enable_nvtx (one NVTX range per call) computes exactly what a
    handle without it computes: plan, append and run on copies of the same inputs."""
    n = [1, 1, 300, 1, 77] if mode == "mixed" else ([1] * 5 if mode == "decode" else [40, 3, 300, 9, 77])
    c = [900, 40, 20, 2000, 300]
    pb = _mixed_batch(44, n, c) if mode == "mixed" else wl.custom(44, np.add(n, c), n, num_qo_heads=32,
                                                                  num_kv_heads=8, head_dim=128, page_size=16)
    res = []
    for nvtx in (False, True):
        x = wl.make_inputs(pb, device="cuda", seed=14, unused="nan", layers=1)
        h = G.make_handle(pb, enable_nvtx=nvtx)
        out, lse, _, _ = G.gpu_step(pb, x, mode, handle=h)
        res.append((out.view(torch.int16).clone(), lse.clone(), x["kv_cache"][0].view(torch.int16).clone()))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])


# ------------------------------------------------------------------ context-only attention (causal = 2)

@pytest.mark.parametrize("heads", [(32, 8, 128), (16, 8, 256)])
@pytest.mark.parametrize("window", [-1, 0, 5, 100])
def test_prefill_context_only(window, heads):
    import oracle_pins
    from paged_kv_attention_gqa_gb300 import binding as B
    L = [0, 37, 16, 300, 5, 129, 64]
    n = [3, 10, 40, 64, 70, 1, 130]
    pb = wl.custom(60, L, n, num_qo_heads=heads[0], num_kv_heads=heads[1], head_dim=heads[2], page_size=16)
    q, kv = oracle_pins.context_step(pb, seed=3)
    x = dict(q=q.cuda(), k_new=None, v_new=None, kv_cache=kv.unsqueeze(0).cuda())
    out, lse, h, ws = G.gpu_step(pb, x, "prefill", causal=B.CONTEXT_ONLY, window_left=window, append=False)
    ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(q), wl.bf16_bits(kv), causal=2, window_left=window)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    empty = ~np.isfinite(ref_l)
    assert np.array_equal(~np.isfinite(l), empty)
    assert np.all(o[np.broadcast_to(empty[..., None], o.shape)] == 0)
    ref_l = np.where(empty, 0, ref_l)
    l_cmp = torch.from_numpy(np.where(empty, 0, l))
    G.compare(out, l_cmp, ref_o, ref_l, what=f"context-only window {window} D{heads[2]}")


def test_context_only_views_then_prefill_matches_full_rows_without_their_queries():
    """A step's rows through pkv_context_only_views: the context-only pass over the shrunk
    views equals the oracle's context-only attention over the same context."""
    import oracle_pins
    from paged_kv_attention_gqa_gb300 import binding as B
    n = [5, 1, 33, 70]
    c = [40, 0, 100, 7]
    full = wl.custom(61, np.add(n, c), n, num_qo_heads=16, num_kv_heads=2, head_dim=64, page_size=16)
    kvp, kvi, lpl = B.context_only_views(16, *full.index_arrays())
    table = [kvi[kvp[r]: kvp[r + 1]] for r in range(full.batch)]
    ctx = wl.PagedBatch("ctx", 16, 2, 64, 16, np.asarray(c), np.asarray(n), table, full.max_pages)
    assert np.array_equal(ctx.kv_indptr, kvp) and np.array_equal(ctx.last_page_len, lpl)
    q, kv = oracle_pins.context_step(ctx, seed=4)
    x = dict(q=q.cuda(), k_new=None, v_new=None, kv_cache=kv.unsqueeze(0).cuda())
    out, lse, _, _ = G.gpu_step(ctx, x, "prefill", causal=B.CONTEXT_ONLY, append=False)
    ref_o, ref_l = G.oracle_attn(ctx, wl.bf16_bits(q), wl.bf16_bits(kv), causal=2)
    G.compare(out, lse, ref_o, ref_l, what="context-only views")


# ------------------------------------------------------------------ dense varlen (DenseAttentionManager)

def _dense_inputs(seed, n, L, Hq, Hkv, D):
    g = torch.Generator(device="cuda").manual_seed(seed)
    Tq, Tk = int(np.sum(n)), int(np.sum(L))
    q = torch.randn(Tq, Hq, D, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(Tk, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(Tk, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    cu_q = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    return q, k, v, cu_q, cu_k


def _dense_handle(Hq, Hkv, D, batch, tokens):
    from paged_kv_attention_gqa_gb300 import binding as B
    return B.Handle(num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=16, max_batch=batch,
                    max_total_tokens=tokens, max_num_pages=1, num_cache_pages=1)


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 16, 2)])
@pytest.mark.parametrize("causal,window", [(True, -1), (False, -1), (True, 33)])
def test_dense_matches_oracle(D, Hq, Hkv, causal, window):
    import oracle
    from paged_kv_attention_gqa_gb300 import binding as B
    n = [1, 40, 130, 7, 64]
    L = [1, 300, 130, 90, 1000]
    q, k, v, cu_q, cu_k = _dense_inputs(70, n, L, Hq, Hkv, D)
    h = _dense_handle(Hq, Hkv, D, len(n), int(np.sum(n)))
    ws = torch.empty(h.workspace_size(B.MODE_DENSE), dtype=torch.uint8, device="cuda")
    h.plan_dense(cu_q, cu_k, workspace=ws, causal=causal, window_left=window)
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    h.run_dense(q, k, v, out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert h.check_device_error(ws) == 0
    ro, rl = oracle.dense_attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), cu_q, cu_k, num_qo_heads=Hq,
                                    num_kv_heads=Hkv, head_dim=D, causal=causal, window_left=window)
    G.compare(out, lse, ro, rl, what="dense")


def test_dense_over_gathered_prefix_is_bit_identical_to_paged_prefill():
    """Gather each row's frozen prefix from the pages (bit-exact), append the fresh K/V
    after it, run the dense pass: the result equals the paged prefill over the same
    cache bit for bit (same kernel, same key order)."""
    from paged_kv_attention_gqa_gb300 import binding as B
    n = [20, 1, 130, 64]
    c = [100, 0, 33, 900]
    pb = wl.custom(71, np.add(n, c), n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    x = wl.make_inputs(pb, device="cuda", seed=14, unused="nan", layers=1)
    out_p, lse_p, h, ws = G.gpu_step(pb, x, "prefill")
    kv = x["kv_cache"][0]
    cu_k = np.concatenate([[0], np.cumsum(pb.kv_lens)]).astype(np.int32)
    k = torch.empty(int(cu_k[-1]), 8, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    qo = pb.qo_indptr
    for r in range(pb.batch):
        pages = torch.as_tensor(pb.page_table[r], dtype=torch.int32, device="cuda")
        h.gather_kv(kv, pages, c[r], k[cu_k[r]:], v[cu_k[r]:])
        k[cu_k[r] + c[r]: cu_k[r + 1]] = x["k_new"][qo[r]: qo[r + 1]]
        v[cu_k[r] + c[r]: cu_k[r + 1]] = x["v_new"][qo[r]: qo[r + 1]]
    torch.cuda.synchronize()
    for r in range(pb.batch):
        K, V = wl.logical_kv(pb, kv, r)
        assert torch.equal(k[cu_k[r]: cu_k[r + 1]].view(torch.int16), K.view(torch.int16))
        assert torch.equal(v[cu_k[r]: cu_k[r + 1]].view(torch.int16), V.view(torch.int16))
    hd = _dense_handle(32, 8, 128, pb.batch, pb.num_tokens)
    wsd = torch.empty(hd.workspace_size(B.MODE_DENSE), dtype=torch.uint8, device="cuda")
    hd.plan_dense(pb.qo_indptr, cu_k, workspace=wsd)
    out_d = torch.full_like(out_p, float("nan"))
    lse_d = torch.full_like(lse_p, float("nan"))
    hd.run_dense(x["q"], k, v, out_d, lse_d, workspace=wsd)
    torch.cuda.synchronize()
    assert torch.equal(out_d.view(torch.int16), out_p.view(torch.int16))
    assert torch.equal(lse_d, lse_p)

"""CUDA-graph mode (the wrappers' accelerator_graph): append + run captured once at static
shapes, then replayed after each new plan of a different step.

FlashInfer*Wrapper (mstar.engine.resources.attn.wrappers): "plan() updates values via
.copy_() without reallocating; the same wrapper object must be used during both capture
and replay".  Here pkv_plan rewrites the plan inside the same workspace and the captured
kernels read it from there.  Every replay is checked against the oracle: the appended
cache bit-exactly, outputs at the parity tolerances.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
from paged_kv_attention_gqa_gb300 import binding as B
from paged_kv_attention_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

POOL = 600
HQ, HKV, D = 32, 8, 128


def _steps(mode):
    rng = np.random.default_rng({"decode": 1, "prefill": 2, "mixed": 3}[mode])
    out = []
    for s in range(3):
        B_ = int(rng.integers(3, 9))
        if mode == "decode":
            n = np.ones(B_, np.int64)
            c = rng.integers(0, 900, B_)
        elif mode == "prefill":
            n = rng.integers(1, 150, B_)
            c = rng.integers(0, 400, B_)
        else:
            n = np.where(rng.random(B_) < 0.7, 1, rng.integers(2, 120, B_))
            n[: 2] = [1, 40]
            c = rng.integers(0, 500, B_)
        pb = wl.custom(50 + s, np.maximum(n + c, 1), n, num_qo_heads=HQ, num_kv_heads=HKV, head_dim=D, page_size=16,
                       pool_pages=POOL, reserve_sink=(mode == "mixed"))
        pb.max_prefill_rows = 8
        out.append(pb)
    return out


@pytest.mark.parametrize("mode", ["decode", "prefill", "mixed"])
def test_captured_step_replays_after_replanning(mode):
    from paged_kv_attention_gqa_gb300 import build
    build.build()
    steps = _steps(mode)
    max_batch, max_tokens = 8, 1200
    n_pages = steps[0].max_pages
    sink = steps[0].sink_page
    h = B.Handle(num_qo_heads=HQ, num_kv_heads=HKV, head_dim=D, page_size=16, max_batch=max_batch,
                 max_total_tokens=max_tokens, max_num_pages=POOL, num_cache_pages=n_pages, max_prefill_rows=8,
                 sink_page=sink, graph_static=1)
    m = G.MODES[mode]
    rows = max_batch if mode == "decode" else max_tokens
    ws = torch.empty(h.workspace_size(m), dtype=torch.uint8, device="cuda")
    q = torch.zeros(rows, HQ, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(rows, HKV, D, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.zeros_like(q)
    lse = torch.zeros(rows, HQ, dtype=torch.float32, device="cuda")
    kv = torch.zeros(n_pages, 2, 16, HKV, D, dtype=torch.bfloat16, device="cuda")
    run = getattr(h, "run_" + mode)

    def load(pb, seed):
        x = wl.make_inputs(pb, device="cuda", seed=seed, unused="nan", layers=1)
        T = pb.num_tokens
        q[:T].copy_(x["q"])
        k[:T].copy_(x["k_new"])
        v[:T].copy_(x["v_new"])
        kv.copy_(x["kv_cache"][0])
        return x

    def plan(pb):
        h.plan(m, None if mode == "decode" else pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len,
               workspace=ws)

    # one uncaptured call of each kind, then the capture
    load(steps[0], 0)
    plan(steps[0])
    h.kv_append_planned(k, v, kv, workspace=ws)
    run(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        h.kv_append_planned(k, v, kv, workspace=ws)
        run(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()

    for i, pb in enumerate(steps[::-1] + steps[:1]):
        x = load(pb, 10 + i)
        before = wl.bf16_bits(kv)
        out.fill_(float("nan"))
        plan(pb)
        graph.replay()
        torch.cuda.synchronize()
        assert h.check_device_error(ws) == 0
        after = G.oracle_append(pb, before, x)
        assert np.array_equal(wl.bf16_bits(kv), after), f"replay {i}: appended cache differs"
        T = pb.num_tokens
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after)
        G.compare(out[:T], lse[:T], ref_o, ref_l, what=f"{mode} replay {i}")


def test_captured_fused_decode_append_replays_after_replanning():
    """pkv_run_decode_append (one launch) captured once, replayed after new decode plans."""
    from paged_kv_attention_gqa_gb300 import build
    build.build()
    steps = _steps("decode")
    max_batch = 8
    n_pages = steps[0].max_pages
    h = B.Handle(num_qo_heads=HQ, num_kv_heads=HKV, head_dim=D, page_size=16, max_batch=max_batch,
                 max_total_tokens=max_batch, max_num_pages=POOL, num_cache_pages=n_pages, max_prefill_rows=0,
                 graph_static=1)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device="cuda")
    q = torch.zeros(max_batch, HQ, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(max_batch, HKV, D, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.zeros_like(q)
    lse = torch.zeros(max_batch, HQ, dtype=torch.float32, device="cuda")
    kv = torch.zeros(n_pages, 2, 16, HKV, D, dtype=torch.bfloat16, device="cuda")

    def load(pb, seed):
        x = wl.make_inputs(pb, device="cuda", seed=seed, unused="nan", layers=1)
        T = pb.num_tokens
        q[:T].copy_(x["q"])
        k[:T].copy_(x["k_new"])
        v[:T].copy_(x["v_new"])
        kv.copy_(x["kv_cache"][0])
        return x

    def plan(pb):
        h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)

    load(steps[0], 0)
    plan(steps[0])
    h.run_decode_append(q, k, v, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        h.run_decode_append(q, k, v, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    for i, pb in enumerate(steps[::-1] + steps[:1]):
        x = load(pb, 30 + i)
        before = wl.bf16_bits(kv)
        out.fill_(float("nan"))
        plan(pb)
        graph.replay()
        torch.cuda.synchronize()
        assert h.check_device_error(ws) == 0
        after = G.oracle_append(pb, before, x)
        assert np.array_equal(wl.bf16_bits(kv), after), f"replay {i}: appended cache differs"
        T = pb.num_tokens
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after)
        G.compare(out[:T], lse[:T], ref_o, ref_l, what=f"fused replay {i}")

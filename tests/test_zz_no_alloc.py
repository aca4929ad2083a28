"""pkv_run_decode_static: decode for callers that may not allocate device memory.

Some callers only receive their inputs, outputs and a stream -- an inference runtime's
plugin hook whose host owns every allocation, or a latency-critical path that must not
enter an allocator that can synchronise the device or fail -- and cannot hand the
library a workspace.  For them the library keeps the plan and the split-KV partials of
one decode in a fixed 16 MiB device array of its own.  These tests call that entry point
through the C ABI twice in a row per case and check each result against the oracle and
against the workspace-based pkv_run_decode, at the tolerances of the other parity tests:
once with rows cut into many pieces (the large merge-kernel instance, several batches),
once with every cut row in at most four pieces (one batch of the small instance), once
with a window.
The file is collected last, and its tests pass alone or after the others.
"""
import ctypes

import numpy as np
import pytest
import torch

import gpu_util as G
from paged_kv_attention_gqa_gb300 import binding as B
from paged_kv_attention_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from paged_kv_attention_gqa_gb300 import build
    build.build()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _host(a):
    a = np.ascontiguousarray(np.asarray(a, np.int32))
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _static_decode(h, pb, q, kv, out, lse, window_left=-1, stream=None):
    kvp, kvp_p = _host(pb.kv_indptr)
    kvi, kvi_p = _host(pb.kv_indices)
    lpl, lpl_p = _host(pb.last_page_len)
    s = stream if stream is not None else torch.cuda.current_stream()
    return h.lib.pkv_run_decode_static(h.h, _ptr(q), _ptr(kv), _ptr(out), _ptr(lse), kvp_p, kvi_p, lpl_p,
                                       pb.batch, window_left, 0.0, ctypes.c_void_p(s.cuda_stream))


def _pieces_per_cut_row(tiles):
    rows = tiles[tiles[:, 3] >= 0, 0]
    return np.bincount(rows) if rows.size else np.zeros(0, np.int64)


CASES = {
    # long rows over 152 CTAs: rows are cut into many pieces (several batches of the merge kernel)
    "many_pieces": dict(lens=[4000, 2500, 17, 1, 3100, 900, 6000, 33], window=-1),
    # 96 rows of 1-3k tokens: every cut row has at most four pieces
    "few_pieces": dict(lens=list(np.random.default_rng(5).integers(1000, 3000, size=96)), window=-1),
    # a window: the split covers only the visible pages, still cut into partials
    "window": dict(lens=[30000, 20000, 17, 9000, 4097, 12000], window=2000),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_static_scratch_decode_matches_oracle_and_workspace_decode(case):
    lens, window = CASES[case]["lens"], CASES[case]["window"]
    pb = wl.custom(31, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    x = wl.make_inputs(pb, device="cuda", seed=12, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    h = G.make_handle(pb)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device="cuda")
    h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws, window_left=window)
    h.kv_append_planned(x["k_new"], x["v_new"], kv, workspace=ws)
    torch.cuda.synchronize()
    kv_bits = wl.bf16_bits(kv)

    tiles, _ = h.decode_split(pb.kv_indptr, pb.last_page_len, window_left=window)
    pieces = _pieces_per_cut_row(tiles)
    assert pieces.size and pieces.max() >= 2, "the case must exercise split-KV partials"
    if case == "few_pieces":
        assert pieces.max() <= 4, "every cut row has few pieces (one batch of the merge kernel)"
    else:
        assert pieces.max() > 16, "some cut row has more pieces than one batch of the small merge kernel"

    queries = [x["q"], (x["q"].float() * -0.75 + 0.1).to(torch.bfloat16)]
    for call, q in enumerate(queries):
        out_s = torch.full_like(q, float("nan"))
        lse_s = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        st = _static_decode(h, pb, q, kv, out_s, lse_s, window_left=window)
        assert st == B.OK, h.lib.pkv_last_error(h.h).decode()
        out_w = torch.full_like(q, float("nan"))
        lse_w = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        h.run_decode(q, kv, out_w, lse_w, workspace=ws)
        torch.cuda.synchronize()
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(q), kv_bits, window_left=window, threads=16)
        G.compare(out_s, lse_s, ref_o, ref_l, what=f"{case}: static call {call} vs oracle")
        G.compare(out_s, lse_s, out_w.float().cpu().numpy(), lse_w.cpu().numpy(),
                  what=f"{case}: static call {call} vs workspace decode")


def test_static_scratch_rejects_oversized_decode():
    # 64 rows of 4096 tokens over a 5000-CTA split: every row is cut into 64 pieces, and
    # 4096 fp32 partials of 32 heads x 129 floats need 67 MB, above the 16 MiB scratch
    n = 64
    pb = wl.custom(32, [4096] * n, [1] * n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    h = G.make_handle(pb, sm_count=5000)
    q = torch.zeros(n, 32, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(16, 2, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    st = _static_decode(h, pb, q, kv, out, None)
    assert st == B.ERR_WORKSPACE
    assert "static scratch" in h.lib.pkv_last_error(h.h).decode()


def test_static_scratch_refuses_a_capturing_stream():
    """The call copies its plan from host memory it frees on return, so on a stream that
    is capturing it returns PKV_ERR_INVALID before it queues anything."""
    lens = [40, 300]
    pb = wl.custom(33, lens, [1, 1], num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    x = wl.make_inputs(pb, device="cuda", seed=13, unused="randn", layers=1)
    h = G.make_handle(pb)
    out = torch.zeros_like(x["q"])
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    marker = torch.zeros(1, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        marker.add_(1.0)  # something for the capture to hold
        st = _static_decode(h, pb, x["q"], x["kv_cache"][0], out, None, stream=side)
    torch.cuda.synchronize()
    assert st == B.ERR_INVALID
    assert "capturing" in h.lib.pkv_last_error(h.h).decode()
    assert torch.count_nonzero(out).item() == 0

"""pkv_run_decode_static: decode for callers that may not allocate device memory.

Some callers only receive their inputs, outputs and a stream (a graph being captured,
an inference runtime's plugin hook, a path that must not enter an allocator) and cannot
hand the library a workspace.  For them the library keeps the plan and the split-KV
partials of one decode in a fixed 16 MiB device array of its own.  This test calls that
entry point through the C ABI twice in a row and checks each result against the
workspace-based pkv_run_decode at the tolerances of the other parity tests.  It lives in
a file of its own that pytest collects last, and passes alone or after the others.
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


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _host(a):
    a = np.ascontiguousarray(np.asarray(a, np.int32))
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _static_decode(h, pb, q, kv, out, lse, window_left=-1):
    kvp, kvp_p = _host(pb.kv_indptr)
    kvi, kvi_p = _host(pb.kv_indices)
    lpl, lpl_p = _host(pb.last_page_len)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return h.lib.pkv_run_decode_static(h.h, _ptr(q), _ptr(kv), _ptr(out), _ptr(lse), kvp_p, kvi_p, lpl_p,
                                       pb.batch, window_left, 0.0, stream)


def test_static_scratch_decode_matches_workspace_decode():
    from paged_kv_attention_gqa_gb300 import build
    build.build()
    # long rows over 152 CTAs: rows are cut, so split-KV partials land in the scratch
    lens = [4000, 2500, 17, 1, 3100, 900, 6000, 33]
    pb = wl.custom(31, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    x = wl.make_inputs(pb, device="cuda", seed=12, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    h = G.make_handle(pb)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device="cuda")
    h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    h.kv_append(x["k_new"], x["v_new"], kv, workspace=ws)
    tiles, _ = h.decode_split(pb.kv_indptr, pb.last_page_len)
    assert (tiles[:, 3] >= 0).any(), "the case must exercise split-KV partials"

    queries = [x["q"], (x["q"].float() * -0.75 + 0.1).to(torch.bfloat16)]
    for call, q in enumerate(queries):
        out_s = torch.full_like(q, float("nan"))
        lse_s = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        st = _static_decode(h, pb, q, kv, out_s, lse_s)
        assert st == B.OK, h.lib.pkv_last_error(h.h).decode()
        out_w = torch.full_like(q, float("nan"))
        lse_w = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        h.run_decode(q, kv, out_w, lse_w, workspace=ws)
        torch.cuda.synchronize()
        G.compare(out_s, lse_s, out_w.float().cpu().numpy(), lse_w.cpu().numpy(), what=f"static call {call}")


def test_static_scratch_rejects_oversized_decode():
    from paged_kv_attention_gqa_gb300 import build
    build.build()
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

"""Plan staging while the host runs ahead of the GPU (PinnedIndexRing; the race that
DenseAttentionManager's force_double_buffer describes: a later plan overwriting a staging
buffer before an earlier step's copy out of it has run).

One stream, one handle, one workspace.  A long GPU backlog is queued first, so the plans
that follow are made while the GPU is still busy: each pkv_plan copies its arrays from
the handle's page-locked ring into the workspace on the stream, and the ring must not
hand a set out again before the copy that read it has executed.  Six different decode
and mixed steps (disjoint rows of one cache, different lengths and row counts) are issued
back to back, each plan followed by its append and run into its own output buffer, with
no host synchronisation in between.  Every step's output and the appended cache are
then checked against the oracle.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
from paged_kv_attention_gqa_gb300 import binding as B
from paged_kv_attention_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from paged_kv_attention_gqa_gb300 import build
    build.build()


def _sub(base, rows):
    rows = np.asarray(rows)
    return wl.PagedBatch(base.name + "-sub", base.num_qo_heads, base.num_kv_heads, base.head_dim, base.page_size,
                         base.kv_lens[rows], base.qo_lens[rows], [base.page_table[r] for r in rows], base.max_pages,
                         sink_page=base.sink_page, max_prefill_rows=base.max_prefill_rows)


def test_plans_issued_ahead_of_the_gpu_each_step_matches_the_oracle():
    rng = np.random.default_rng(17)
    n_dec, n_pf = 36, 6
    dec_L = rng.integers(100, 3000, size=n_dec)
    pf_n = rng.integers(40, 300, size=n_pf)
    pf_L = pf_n + rng.integers(0, 600, size=n_pf)
    L = np.concatenate([dec_L, pf_L])
    n = np.concatenate([np.ones(n_dec, np.int64), pf_n])
    base = wl.custom(51, L, n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, reserve_sink=True)
    base.max_prefill_rows = 2
    x = wl.make_inputs(base, device="cuda", seed=52, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    before = wl.bf16_bits(kv)

    # disjoint rows per step; prompt rows are base rows n_dec.. (two per mixed step)
    steps = [
        ("decode", list(range(0, 12))),
        ("mixed", list(range(12, 16)) + [n_dec + 0, n_dec + 1]),
        ("decode", list(range(16, 19))),
        ("mixed", [19, n_dec + 2, 20, n_dec + 3, 21]),
        ("decode", list(range(22, 34))),
        ("mixed", [n_dec + 4, 34, 35, n_dec + 5]),
    ]
    subs = [(mode, _sub(base, rows), rows) for mode, rows in steps]
    h = G.make_handle(base)
    ws_bytes = max(h.workspace_size(B.MODE_DECODE), h.workspace_size(B.MODE_MIXED))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(53)
    ins = []
    for mode, pb, rows in subs:
        T = pb.num_tokens
        q = torch.randn(T, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
        k = torch.randn(T, 8, 128, generator=g, device="cuda").to(torch.bfloat16)
        v = torch.randn(T, 8, 128, generator=g, device="cuda").to(torch.bfloat16)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((T, 32), float("nan"), dtype=torch.float32, device="cuda")
        ins.append((q, k, v, out, lse))
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    backlog_done = torch.cuda.Event()
    torch.cuda._sleep(200_000_000)  # ~0.1 s of GPU time queued ahead of the first plan
    backlog_done.record(stream)
    ahead = []
    for (mode, pb, rows), (q, k, v, out, lse) in zip(subs, ins):
        m = G.MODES[mode]
        qo = None if mode == "decode" else pb.qo_indptr
        h.plan(m, qo, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
        ahead.append(not backlog_done.query())  # this plan was made while the GPU was still busy
        h.kv_append_planned(k, v, kv, workspace=ws)
        if mode == "decode":
            h.run_decode(q, kv, out, lse, workspace=ws)
        else:
            h.run_mixed(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert h.check_device_error(ws) == 0
    assert ahead[0] and ahead[1], "the first two plans must be made while the backlog still runs"

    # the appended cache: every step's new tokens at their slots, nothing else touched
    want = before
    for (mode, pb, rows), (q, k, v, out, lse) in zip(subs, ins):
        want = G.oracle_append(pb, want, dict(k_new=k, v_new=v))
    got = wl.bf16_bits(kv)
    assert np.array_equal(got, want), "appended cache differs from the oracle's"
    for i, ((mode, pb, rows), (q, k, v, out, lse)) in enumerate(zip(subs, ins)):
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(q), got, threads=16)
        G.compare(out, lse, ref_o, ref_l, what=f"step {i} ({mode}, {pb.batch} rows)")

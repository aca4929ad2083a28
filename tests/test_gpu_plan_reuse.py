"""One handle, one workspace, plans of every mode in turn, the plan image growing and shrinking.

pkv_plan builds each plan's image in the buffer the previous plan on the handle used (the
handle keeps it, so that a plan touches memory that is already mapped); a plan smaller than
the one before must still start from zeros where it has no data, and a switch between the
paged modes and the dense mode must leave nothing of the other layout behind.  Six steps
on disjoint rows of one cache (the prompt rows' cache is written again, with new values, by
the last step) and one dense step in the middle are each planned, appended and run on the
same handle and workspace, and each is checked against the oracle right after it ran.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
import oracle
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


def test_plans_of_every_mode_in_turn_on_one_handle_match_the_oracle():
    rng = np.random.default_rng(81)
    n_dec, n_pf = 34, 6
    dec_L = rng.integers(50, 2500, size=n_dec)
    pf_n = rng.integers(30, 260, size=n_pf)
    pf_L = pf_n + rng.integers(0, 700, size=n_pf)
    L = np.concatenate([dec_L, pf_L])
    n = np.concatenate([np.ones(n_dec, np.int64), pf_n])
    base = wl.custom(82, L, n, num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, reserve_sink=True)
    base.max_prefill_rows = 2
    x = wl.make_inputs(base, device="cuda", seed=83, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    P = n_dec  # first prompt row
    steps = [
        ("prefill", [P + 0, P + 1, P + 2, P + 3, P + 4, P + 5]),
        ("decode", [0, 1, 2]),
        ("mixed", [3, P + 0, 4, P + 1]),
        ("dense", None),
        ("decode", list(range(5, 34))),
        ("prefill", [P + 4, P + 5]),
        ("mixed", [P + 2, P + 3]),
    ]
    h = G.make_handle(base)
    modes = (B.MODE_DECODE, B.MODE_PREFILL, B.MODE_MIXED, B.MODE_DENSE)
    ws = torch.empty(max(h.workspace_size(m) for m in modes), dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(84)
    for i, (mode, rows) in enumerate(steps):
        if mode == "dense":
            # segments of fresh queries at the end of their keys, K / V contiguous
            nq, nk = [40, 1, 130], [300, 1, 400]
            cu_q = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
            cu_k = np.concatenate([[0], np.cumsum(nk)]).astype(np.int32)
            q = torch.randn(int(cu_q[-1]), 32, 128, generator=g, device="cuda").to(torch.bfloat16)
            k = torch.randn(int(cu_k[-1]), 8, 128, generator=g, device="cuda").to(torch.bfloat16)
            v = torch.randn(int(cu_k[-1]), 8, 128, generator=g, device="cuda").to(torch.bfloat16)
            out = torch.full_like(q, float("nan"))
            lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
            h.plan_dense(cu_q, cu_k, workspace=ws)
            h.run_dense(q, k, v, out, lse, workspace=ws)
            torch.cuda.synchronize()
            assert h.check_device_error(ws) == 0
            ro, rl = oracle.dense_attention(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), cu_q, cu_k,
                                            num_qo_heads=32, num_kv_heads=8, head_dim=128, causal=True,
                                            window_left=-1)
            G.compare(out, lse, ro, rl, what=f"step {i} (dense)")
            continue
        pb = _sub(base, rows)
        T = pb.num_tokens
        q = torch.randn(T, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
        k_new = torch.randn(T, 8, 128, generator=g, device="cuda").to(torch.bfloat16)
        v_new = torch.randn(T, 8, 128, generator=g, device="cuda").to(torch.bfloat16)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((T, 32), float("nan"), dtype=torch.float32, device="cuda")
        before = wl.bf16_bits(kv)
        qo = None if mode == "decode" else pb.qo_indptr
        h.plan(G.MODES[mode], qo, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
        h.kv_append_planned(k_new, v_new, kv, workspace=ws)
        getattr(h, "run_" + mode)(q, kv, out, lse, workspace=ws)
        torch.cuda.synchronize()
        assert h.check_device_error(ws) == 0
        got = wl.bf16_bits(kv)
        want = G.oracle_append(pb, before, dict(k_new=k_new, v_new=v_new))
        assert np.array_equal(got, want), f"step {i} ({mode}): appended cache differs from the oracle's"
        ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(q), got, threads=16)
        G.compare(out, lse, ref_o, ref_l, what=f"step {i} ({mode}, {pb.batch} rows)")

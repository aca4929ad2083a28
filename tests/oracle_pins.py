"""Pins that tie the oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (the ctypes library
``lib``, default: the real one) disagrees with
  * hand-worked closed forms (tests/golden/hand_worked.json),
  * torch's scaled_dot_product_attention / logsumexp in float64 on unpaged K/V
    (a library routine the oracle does not call),
  * invariants the paging must satisfy (page-pool relabelling, page_size 1 vs 16),
  * special cases (all-ones V channel, single visible key, decode == 1-token prefill),
  * the append's placement, read back through the generator's own page table.
The mutation test runs these same functions against broken copies of the oracle.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from oracle import plan_ref
from paged_kv_attention_gqa_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
_ENV = {"e": math.e, "log": math.log, "exp": math.exp, "inf": math.inf}


def closed_form(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, _ENV))


def to_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return wl.bf16_bits(t)


def golden_case_arrays(case):
    """Paged arrays for a hand-worked case: tokens placed at page pages[p // P], slot p % P."""
    P, Hkv, D = case["page_size"], case["num_kv_heads"], case["head_dim"]
    Hq = case["num_qo_heads"]
    cache = np.full((case["max_pages"], 2, P, Hkv, D), np.nan, dtype=np.float32)
    qo, kvp, kvi, lpl, qs = [0], [0], [], [], []
    for row in case["rows"]:
        L = len(row["k"])
        assert len(row["pages"]) == math.ceil(L / P)
        for p in range(L):
            page, slot = row["pages"][p // P], p % P
            cache[page, 0, slot] = np.asarray(row["k"][p], np.float32)
            cache[page, 1, slot] = np.asarray(row["v"][p], np.float32)
        qs.extend(row["q"])
        qo.append(qo[-1] + row["n_new"])
        kvi.extend(row["pages"])
        kvp.append(len(kvi))
        lpl.append((L - 1) % P + 1 if L else 0)
    q = np.asarray(qs, np.float32).reshape(-1, Hq, D)
    return to_bits(q), to_bits(cache), (np.array(qo), np.array(kvp), np.array(kvi), np.array(lpl))


def pin_golden(lib=None, tol=2e-6):
    cases = json.load(open(os.path.join(GOLDEN, "hand_worked.json")))["cases"]
    for case in cases:
        q, cache, idx = golden_case_arrays(case)
        out, lse = oracle.attention(q, cache, *idx, num_qo_heads=case["num_qo_heads"],
                                    num_kv_heads=case["num_kv_heads"], head_dim=case["head_dim"],
                                    page_size=case["page_size"], causal=case["causal"],
                                    window_left=case["window_left"],
                                    sm_scale=closed_form(case["sm_scale"]), lib=lib)
        for ex in case["expect"]:
            t, h = ex["token"], ex["head"]
            want = np.array([closed_form(e) for e in ex["out"]])
            got = out[t, h].astype(np.float64)
            assert np.all(np.abs(got - want) <= tol * np.maximum(1, np.abs(want))), (case["name"], t, h, got, want)
            wl_ = closed_form(ex["lse"])
            if math.isinf(wl_):
                assert float(lse[t, h]) == wl_, (case["name"], t, h, lse[t, h], wl_)
            else:
                assert abs(float(lse[t, h]) - wl_) <= tol * max(1, abs(wl_)), (case["name"], t, h, lse[t, h], wl_)


def build_step(pb, seed=0):
    """Inputs with the step's new K/V already appended by the generator's page table (so
    the attention pins do not depend on the oracle's own append)."""
    x = wl.make_inputs(pb, seed=seed, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    flat = kv.view(pb.max_pages * 2 * pb.page_size, pb.num_kv_heads, pb.head_dim)
    qo = pb.qo_indptr
    for r in range(pb.batch):
        n, L = int(pb.qo_lens[r]), int(pb.kv_lens[r])
        if n == 0:
            continue
        rows = torch.as_tensor(wl._flat_slot_rows(pb, r, range(L - n, L)))
        flat[rows] = x["k_new"][qo[r]: qo[r + 1]]
        flat[rows + pb.page_size] = x["v_new"][qo[r]: qo[r + 1]]
    return x["q"], kv, x


def sdpa_reference(pb, q, kv_layer, *, causal, window_left, sm_scale):
    """float64 attention on unpaged K/V through torch's SDPA (the masks follow the
    visibility rule; softmax, scaling and the weighted sum are the library's).  A query
    with no visible key is given o = 0, lse = -inf."""
    T, Hq, D = q.shape
    g = pb.num_qo_heads // pb.num_kv_heads
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.float64)
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float64)
    qo = pb.qo_indptr
    for r in range(pb.batch):
        n, L = int(pb.qo_lens[r]), int(pb.kv_lens[r])
        if n == 0:
            continue
        if L == 0:
            out[qo[r]: qo[r + 1]] = 0.0
            lse[qo[r]: qo[r + 1]] = float("-inf")
            continue
        K, V = wl.logical_kv(pb, kv_layer, r)
        K = K.double().repeat_interleave(g, dim=1).transpose(0, 1)   # [Hq, L, D]
        V = V.double().repeat_interleave(g, dim=1).transpose(0, 1)
        Q = q[qo[r]: qo[r + 1]].double().transpose(0, 1)             # [Hq, n, D]
        mask = torch.zeros(n, L, dtype=torch.bool)
        for i in range(n):
            lo, hi = plan_ref.visible_range(L, n, i, causal, window_left)
            mask[i, lo: hi + 1] = True
        empty = ~mask.any(dim=1)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask | empty[:, None], scale=sm_scale)
        s = torch.matmul(Q, K.transpose(1, 2)) * sm_scale
        s = s.masked_fill(~mask, float("-inf"))
        o[:, empty] = 0.0
        out[qo[r]: qo[r + 1]] = o.transpose(0, 1)
        lse[qo[r]: qo[r + 1]] = torch.logsumexp(s, dim=-1).transpose(0, 1)
    return out, lse


def run_oracle(pb, q, kv_layer, *, causal=True, window_left=-1, sm_scale=None, lib=None, page_table=None):
    return oracle.attention(wl.bf16_bits(q), wl.bf16_bits(kv_layer), *pb.index_arrays(),
                            num_qo_heads=pb.num_qo_heads, num_kv_heads=pb.num_kv_heads,
                            head_dim=pb.head_dim, page_size=pb.page_size, causal=causal,
                            window_left=window_left, sm_scale=sm_scale, lib=lib)


SDPA_CASES = [
    # (kv_lens, qo_lens, Hq, Hkv, D, P, causal, window_left)
    ([37, 5, 16, 1], [1, 1, 1, 1], 8, 2, 64, 16, True, -1),
    ([37, 50, 16, 33], [1, 7, 16, 33], 4, 1, 32, 16, True, -1),
    ([40, 21, 64], [9, 21, 3], 8, 8, 16, 4, True, 5),
    ([40, 21, 64], [9, 21, 3], 16, 2, 16, 16, False, -1),
    ([70, 3], [70, 2], 8, 1, 8, 8, True, 17),
    ([29, 31], [1, 1], 4, 4, 16, 1, True, 0),
    ([130, 9], [3, 1], 14, 2, 256, 2, True, -1),       # head_dim 256, group 7, 2-slot pages
    ([200, 65], [65, 1], 6, 2, 128, 64, False, -1),    # group 3, 64-slot pages, non-causal
    ([100, 40], [1, 40], 40, 40, 32, 32, True, 10),    # 40 kv heads, window
]


def pin_sdpa(lib=None, tol=2e-5):
    for k, (Ls, ns, Hq, Hkv, D, P, causal, wleft) in enumerate(SDPA_CASES):
        pb = wl.custom(100 + k, Ls, ns, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P)
        q, kv, _ = build_step(pb, seed=k)
        scale = 1.0 / math.sqrt(D) * (1.5 if k % 2 else 1.0)
        out, lse = run_oracle(pb, q, kv, causal=causal, window_left=wleft, sm_scale=scale, lib=lib)
        ref_o, ref_l = sdpa_reference(pb, q, kv, causal=causal, window_left=wleft, sm_scale=scale)
        d_o = np.abs(out - ref_o.numpy()).max()
        d_l = np.abs(lse - ref_l.numpy()).max()
        assert d_o <= tol and d_l <= tol, (k, d_o, d_l)


def relabel_pool(pb, kv_layer, seed):
    """Move every page p to page pi[p] and rewrite the indices accordingly."""
    rng = np.random.default_rng(seed)
    pi = rng.permutation(pb.max_pages)
    new = torch.empty_like(kv_layer)
    new[torch.as_tensor(pi)] = kv_layer
    pb2 = wl.PagedBatch(pb.name, pb.num_qo_heads, pb.num_kv_heads, pb.head_dim, pb.page_size,
                        pb.kv_lens, pb.qo_lens, [pi[t] for t in pb.page_table], pb.max_pages)
    return pb2, new


def pin_pool_permutation(lib=None):
    pb = wl.custom(7, [45, 17, 80, 3], [1, 17, 20, 2], num_qo_heads=8, num_kv_heads=2, head_dim=32,
                   page_size=16, pool_factor=2.0)
    q, kv, _ = build_step(pb, seed=3)
    for causal, wl_ in [(True, -1), (False, -1), (True, 9)]:
        a = run_oracle(pb, q, kv, causal=causal, window_left=wl_, lib=lib)
        pb2, kv2 = relabel_pool(pb, kv, seed=11)
        b = run_oracle(pb2, q, kv2, causal=causal, window_left=wl_, lib=lib)
        assert np.array_equal(a[0], b[0], equal_nan=True) and np.array_equal(a[1], b[1], equal_nan=True)


def repage(pb, kv_layer, page_size, seed):
    """The same logical K/V stored with another page size (pages drawn afresh)."""
    pb2 = wl.custom(seed, pb.kv_lens, pb.qo_lens, num_qo_heads=pb.num_qo_heads,
                    num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim, page_size=page_size)
    kv2 = torch.full((pb2.max_pages, 2, page_size, pb.num_kv_heads, pb.head_dim), float("nan"),
                     dtype=kv_layer.dtype)
    flat2 = kv2.view(-1, pb.num_kv_heads, pb.head_dim)
    for r in range(pb.batch):
        K, V = wl.logical_kv(pb, kv_layer, r)
        rows = torch.as_tensor(wl._flat_slot_rows(pb2, r, range(int(pb.kv_lens[r]))))
        flat2[rows] = K
        flat2[rows + page_size] = V
    return pb2, kv2


def pin_page_size_invariance(lib=None):
    pb = wl.custom(8, [45, 17, 80, 3], [1, 17, 20, 2], num_qo_heads=8, num_kv_heads=2, head_dim=32,
                   page_size=16)
    q, kv, _ = build_step(pb, seed=4)
    base = run_oracle(pb, q, kv, window_left=6, lib=lib)
    for P in (1, 3):
        pb2, kv2 = repage(pb, kv, P, seed=20 + P)
        other = run_oracle(pb2, q, kv2, window_left=6, lib=lib)
        assert np.array_equal(base[0], other[0]) and np.array_equal(base[1], other[1]), P


def pin_rows_sum_to_one(lib=None):
    """With V = 1 in channel 0 for every token, o[..., 0] = sum of the softmax row = 1."""
    pb = wl.custom(9, [300, 77, 1], [1, 40, 1], num_qo_heads=8, num_kv_heads=4, head_dim=16, page_size=16)
    q, kv, _ = build_step(pb, seed=5)
    kv = kv.clone()
    kv[:, 1, :, :, 0] = 1.0
    for causal, w in [(True, -1), (False, 13)]:
        out, _ = run_oracle(pb, q, kv, causal=causal, window_left=w, lib=lib)
        assert np.abs(out[..., 0] - 1.0).max() <= 1e-6


def pin_single_key_cases(lib=None):
    """window_left = 0 and a length-1 row both return the visible V row exactly, with
    lse equal to that key's score."""
    pb = wl.custom(10, [33, 1, 64], [5, 1, 64], num_qo_heads=4, num_kv_heads=2, head_dim=16, page_size=16)
    q, kv, _ = build_step(pb, seed=6)
    scale = 0.25
    out, lse = run_oracle(pb, q, kv, window_left=0, sm_scale=scale, lib=lib)
    qo = pb.qo_indptr
    g = pb.num_qo_heads // pb.num_kv_heads
    for r in range(pb.batch):
        K, V = wl.logical_kv(pb, kv, r)
        n, L = int(pb.qo_lens[r]), int(pb.kv_lens[r])
        for i in range(n):
            p = L - n + i
            for h in range(pb.num_qo_heads):
                assert np.array_equal(out[qo[r] + i, h], V[p, h // g].float().numpy())
                s = scale * float(np.dot(q[qo[r] + i, h].float().numpy().astype(np.float64),
                                         K[p, h // g].float().numpy().astype(np.float64)))
                assert abs(lse[qo[r] + i, h] - s) <= 1e-5 * max(1, abs(s))


def pin_decode_is_one_token_prefill(lib=None):
    """A decode batch equals the same rows planned as 1-token causal prefill rows, and
    non-causal, since the only new token is the last position."""
    pb = wl.custom(12, [90, 16, 17, 5], [1, 1, 1, 1], num_qo_heads=8, num_kv_heads=2, head_dim=32, page_size=16)
    q, kv, _ = build_step(pb, seed=7)
    a = run_oracle(pb, q, kv, causal=True, lib=lib)
    b = run_oracle(pb, q, kv, causal=False, lib=lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_append(lib=None):
    """The oracle's append puts token i of row r where the generator's page table says
    position L_r - n_r + i lives, touches nothing else, and attention after it matches
    SDPA on the unpaged [prefix | new] sequence."""
    pb = wl.custom(13, [45, 16, 17, 80, 2, 33], [1, 16, 2, 30, 2, 1], num_qo_heads=8, num_kv_heads=2,
                   head_dim=32, page_size=16, pool_factor=1.5)
    x = wl.make_inputs(pb, seed=8, unused="nan", layers=1)
    kv0 = x["kv_cache"][0]
    bits = oracle.kv_append(wl.bf16_bits(kv0), wl.bf16_bits(x["k_new"]), wl.bf16_bits(x["v_new"]),
                            *pb.index_arrays(), num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim,
                            page_size=pb.page_size, lib=lib)
    kv1 = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    qo = pb.qo_indptr
    written = torch.zeros(pb.max_pages * 2 * pb.page_size, dtype=torch.bool)
    for r in range(pb.batch):
        n, L = int(pb.qo_lens[r]), int(pb.kv_lens[r])
        K, V = wl.logical_kv(pb, kv1, r)
        K0, V0 = wl.logical_kv(pb, kv0, r)
        assert torch.equal(K[: L - n].view(torch.int16), K0[: L - n].view(torch.int16))
        assert torch.equal(K[L - n:].view(torch.int16), x["k_new"][qo[r]: qo[r + 1]].view(torch.int16))
        assert torch.equal(V[L - n:].view(torch.int16), x["v_new"][qo[r]: qo[r + 1]].view(torch.int16))
        rows = torch.as_tensor(wl._flat_slot_rows(pb, r, range(L - n, L)))
        written[rows] = True
        written[rows + pb.page_size] = True
    f0 = kv0.reshape(-1, pb.num_kv_heads * pb.head_dim).view(torch.int16)
    f1 = kv1.reshape(-1, pb.num_kv_heads * pb.head_dim).view(torch.int16)
    assert torch.equal(f0[~written], f1[~written])
    pages, slots = plan_ref.append_slots(*pb.index_arrays(), pb.page_size)
    out, lse = run_oracle(pb, x["q"], kv1, lib=lib)
    ro, rl = sdpa_reference(pb, x["q"], kv1, causal=True, window_left=-1, sm_scale=1 / math.sqrt(pb.head_dim))
    assert np.abs(out - ro.numpy()).max() <= 2e-5 and np.abs(lse - rl.numpy()).max() <= 2e-5


def context_step(pb, seed=0):
    """Inputs for context-only attention: every stored position of each row holds K/V
    (the context) and the rows' queries are drawn separately."""
    ctx = wl.PagedBatch(pb.name, pb.num_qo_heads, pb.num_kv_heads, pb.head_dim, pb.page_size, pb.kv_lens,
                        np.zeros_like(pb.qo_lens), pb.page_table, pb.max_pages)
    x = wl.make_inputs(ctx, seed=seed, unused="nan", layers=1)
    g = torch.Generator().manual_seed(seed + 1000)
    q = torch.randn(pb.num_tokens, pb.num_qo_heads, pb.head_dim, generator=g).to(torch.bfloat16)
    return q, x["kv_cache"][0]


def pin_sdpa_context_only(lib=None, tol=2e-5):
    cases = [([37, 0, 16, 5], [3, 2, 40, 1], 8, 2, 64, 16, -1),
             ([70, 33, 1], [9, 1, 4], 4, 1, 32, 8, 10),
             ([64, 3], [64, 70], 8, 8, 16, 4, 0),
             ([64, 3], [64, 70], 8, 8, 16, 4, 40)]
    for k, (Ls, ns, Hq, Hkv, D, P, wleft) in enumerate(cases):
        pb = wl.custom(200 + k, Ls, ns, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P)
        q, kv = context_step(pb, seed=k)
        out, lse = run_oracle(pb, q, kv, causal=2, window_left=wleft, sm_scale=0.2, lib=lib)
        ro, rl = sdpa_reference(pb, q, kv, causal=2, window_left=wleft, sm_scale=0.2)
        assert np.abs(out - ro.numpy()).max() <= tol, k
        fin = np.isfinite(rl.numpy())
        assert np.array_equal(fin, np.isfinite(lse)), k
        assert not fin.any() or np.abs(lse[fin] - rl.numpy()[fin]).max() <= tol, k


def dense_from_paged(pb, kv_layer):
    """Contiguous per-row K/V runs ([prefix | new] = the row's L tokens) and cu arrays."""
    ks, vs = [], []
    for r in range(pb.batch):
        K, V = wl.logical_kv(pb, kv_layer, r)
        ks.append(K)
        vs.append(V)
    cu_k = np.concatenate([[0], np.cumsum(pb.kv_lens)]).astype(np.int32)
    return torch.cat(ks), torch.cat(vs), pb.qo_indptr, cu_k


def pin_dense(lib=None, tol=2e-5):
    """Dense varlen over the rows' contiguous K/V equals the paged oracle on the same
    logical K/V bit for bit (same definition, same order), and SDPA in float64."""
    for k, (Ls, ns, Hq, Hkv, D, P, causal, wleft) in enumerate(SDPA_CASES[:5]):
        pb = wl.custom(300 + k, Ls, ns, num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P)
        q, kv, _ = build_step(pb, seed=k)
        K, V, cu_q, cu_k = dense_from_paged(pb, kv)
        d_o, d_l = oracle.dense_attention(wl.bf16_bits(q), wl.bf16_bits(K), wl.bf16_bits(V), cu_q, cu_k,
                                          num_qo_heads=Hq, num_kv_heads=Hkv, head_dim=D, causal=causal,
                                          window_left=wleft, sm_scale=0.3, lib=lib)
        p_o, p_l = run_oracle(pb, q, kv, causal=causal, window_left=wleft, sm_scale=0.3, lib=lib)
        assert np.array_equal(d_o, p_o) and np.array_equal(d_l, p_l), k
        ro, rl = sdpa_reference(pb, q, kv, causal=causal, window_left=wleft, sm_scale=0.3)
        assert np.abs(d_o - ro.numpy()).max() <= tol and np.abs(d_l - rl.numpy()).max() <= tol, k


ALL_PINS = [pin_golden, pin_sdpa, pin_pool_permutation, pin_page_size_invariance, pin_rows_sum_to_one,
            pin_single_key_cases, pin_decode_is_one_token_prefill, pin_append, pin_sdpa_context_only,
            pin_dense]

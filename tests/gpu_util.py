"""Helpers for the GPU parity tests: run a step through the C ABI, run the oracle on the
same seeded inputs, compare at the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from paged_kv_attention_gqa_gb300 import binding as B
from paged_kv_attention_gqa_gb300 import workloads as wl

# bf16 output: max-abs 2e-2 and relative L2 1e-2; lse: |d| <= 1e-3 * max(1, |lse|)
MAX_ABS = 2e-2
REL_L2 = 1e-2
LSE_REL = 1e-3

MODES = {"decode": B.MODE_DECODE, "prefill": B.MODE_PREFILL, "mixed": B.MODE_MIXED}


def make_handle(pb, *, sm_count=0, max_prefill_rows=None, enable_nvtx=False):
    mpr = pb.max_prefill_rows if max_prefill_rows is None else max_prefill_rows
    return B.Handle(num_qo_heads=pb.num_qo_heads, num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim,
                    page_size=pb.page_size, max_batch=max(pb.batch, 1), max_total_tokens=max(pb.num_tokens, 1),
                    max_num_pages=max(len(pb.kv_indices), 1), num_cache_pages=pb.max_pages,
                    max_prefill_rows=mpr, sm_count=sm_count, sink_page=pb.sink_page, enable_nvtx=enable_nvtx)


def gpu_step(pb, x, mode, *, layer=0, window_left=-1, causal=True, sm_scale=0.0, sm_count=0, append=True,
             handle=None, workspace=None, fused=False):
    """plan -> append -> run for one layer; returns (out, lse, handle, workspace).  fused:
    decode plans append inside the decode launch (pkv_run_decode_append)."""
    h = handle or make_handle(pb, sm_count=sm_count)
    m = MODES[mode]
    ws = workspace if workspace is not None else torch.empty(h.workspace_size(m), dtype=torch.uint8, device="cuda")
    qo = None if mode == "decode" else pb.qo_indptr
    h.plan(m, qo, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws, causal=causal,
           window_left=window_left, sm_scale=sm_scale)
    kv = x["kv_cache"][layer]
    q = x["q"]
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    if fused:
        assert mode == "decode" and append
        h.run_decode_append(q, x["k_new"], x["v_new"], kv, out, lse, workspace=ws)
    else:
        if append and x.get("k_new") is not None:
            h.kv_append_planned(x["k_new"], x["v_new"], kv, workspace=ws)
        getattr(h, "run_" + mode)(q, kv, out, lse, workspace=ws)
    torch.cuda.synchronize()
    assert h.check_device_error(ws) == 0
    return out, lse, h, ws


def oracle_append(pb, kv_before_bits, x):
    return oracle.kv_append(kv_before_bits, wl.bf16_bits(x["k_new"]), wl.bf16_bits(x["v_new"]), *pb.index_arrays(),
                            num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim, page_size=pb.page_size)


def oracle_attn(pb, q_bits, kv_bits, *, causal=True, window_left=-1, sm_scale=None, rows=None, threads=8):
    return oracle.attention(q_bits, kv_bits, *pb.index_arrays(), num_qo_heads=pb.num_qo_heads,
                            num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim, page_size=pb.page_size,
                            causal=causal, window_left=window_left, sm_scale=sm_scale or None, rows=rows,
                            threads=threads)


def token_mask(pb, rows):
    m = np.zeros(pb.num_tokens, bool)
    qo = pb.qo_indptr
    for r in rows:
        m[qo[r]: qo[r + 1]] = True
    return m


def compare(out, lse, ref_out, ref_lse, tokens=None, what=""):
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    if tokens is not None:
        o, l, ref_out, ref_lse = o[tokens], l[tokens], ref_out[tokens], ref_lse[tokens]
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert np.isfinite(ref_out).all(), f"{what}: oracle produced non-finite output"
    d = np.abs(o - ref_out)
    max_abs = float(d.max()) if d.size else 0.0
    rel = float(np.linalg.norm(o - ref_out) / max(np.linalg.norm(ref_out), 1e-30)) if d.size else 0.0
    both_empty = np.isneginf(l) & np.isneginf(ref_lse)  # queries that see no key: lse = -inf on both sides
    with np.errstate(invalid="ignore"):
        dl = np.where(both_empty, 0.0, np.abs(l - ref_lse))
    lse_ok = bool(np.all(dl <= LSE_REL * np.maximum(1.0, np.where(both_empty, 1.0, np.abs(ref_lse)))))
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs {max_abs:.3e} rel_l2 {rel:.3e}"
    assert lse_ok, f"{what}: lse max diff {float(dl.max()):.3e}"
    return max_abs, rel


def compact_rows(pb, kv_bits, rows, extra_pages=()):
    """A smaller pool holding only `rows`' pages (and `extra_pages`), with the index
    arrays of that sub-batch: the oracle sees identical attention inputs."""
    pages = sorted({int(p) for r in rows for p in pb.page_table[r]} | {int(p) for p in extra_pages})
    remap = {p: i for i, p in enumerate(pages)}
    sub = wl.PagedBatch(pb.name, pb.num_qo_heads, pb.num_kv_heads, pb.head_dim, pb.page_size,
                        pb.kv_lens[rows], pb.qo_lens[rows], [np.array([remap[int(p)] for p in pb.page_table[r]])
                                                             for r in rows], len(pages))
    return sub, kv_bits[np.asarray(pages, np.int64)], remap


def causal_subrows(pb, max_tokens=256):
    """The same causal attention as smaller independent rows: each row's new tokens are cut
    into runs of at most `max_tokens`, and a run ending at position e (exclusive) becomes a
    row of length e over the parent's first ceil(e / P) pages.  A causal query at position
    p sees keys 0..p only, so the run's queries see exactly the keys they see in the parent
    row; the runs keep the parent's token order, so the result lines up with q / out of
    the parent batch.  Lets the oracle spread one long row over several threads."""
    P = pb.page_size
    qo, kvp, kvi, _ = pb.index_arrays()
    n_qo, n_kvp, n_kvi, n_lpl = [0], [0], [], []
    for r in range(pb.batch):
        L, n = int(pb.kv_lens[r]), int(pb.qo_lens[r])
        c = L - n
        starts = list(range(0, n, max_tokens)) if n else [0]
        for a in starts:
            b = min(n, a + max_tokens)
            e = c + b  # length of the sub-row: up to its last query
            if e == 0:
                n_qo.append(n_qo[-1])
                n_kvp.append(n_kvp[-1])
                n_lpl.append(0)
                continue
            pages = -(-e // P)
            n_kvi.extend(int(p) for p in kvi[kvp[r]: kvp[r] + pages])
            n_kvp.append(len(n_kvi))
            n_qo.append(n_qo[-1] + (b - a))
            n_lpl.append((e - 1) % P + 1)
    i32 = lambda a: np.asarray(a, np.int32)
    assert n_qo[-1] == pb.num_tokens
    return i32(n_qo), i32(n_kvp), i32(n_kvi), i32(n_lpl)


def oracle_attn_causal_split(pb, q_bits, kv_bits, *, window_left=-1, threads=16, max_tokens=256):
    """oracle.attention over causal_subrows(pb): identical per-token definition, rows
    small enough to balance over the threads."""
    qo, kvp, kvi, lpl = causal_subrows(pb, max_tokens)
    return oracle.attention(q_bits, kv_bits, qo, kvp, kvi, lpl, num_qo_heads=pb.num_qo_heads,
                            num_kv_heads=pb.num_kv_heads, head_dim=pb.head_dim, page_size=pb.page_size,
                            causal=True, window_left=window_left, threads=threads)

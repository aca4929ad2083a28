"""Pins of the oracle's index work (oracle/plan_ref.py), each callable on a module so that
tests/test_oracle_mutations.py can run them against a deliberately broken copy.

Every pin fixes the oracle against something other than itself: a hand-worked layout
stored under tests/golden/ (with the passage it follows in its "about" field), or a
property that the pages' definitions force at any size.
"""
from __future__ import annotations

import json
import os

import numpy as np

from oracle import plan_ref as _plan_ref

_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
MIXED = json.load(open(os.path.join(_GOLDEN, "mixed_layout.json")))
CTX = json.load(open(os.path.join(_GOLDEN, "context_only_views.json")))


def _idx(g):
    return g["qo_indptr"], g["kv_indptr"], g["kv_indices"], g["last_page_len"]


def pin_append_slots_golden(mod=_plan_ref):
    """FlashInferDecodeWrapper.plan's write location, worked by hand for a ragged step."""
    ex = MIXED["expect"]
    assert mod.row_lengths(MIXED["kv_indptr"], MIXED["last_page_len"], 16).tolist() == ex["row_lengths"]
    pages, slots = mod.append_slots(*_idx(MIXED), 16)
    assert pages.tolist() == ex["append_pages"]
    assert slots.tolist() == ex["append_slots"]


def pin_mixed_layout_golden(mod=_plan_ref):
    """FlashInferMixedWrapper's two plans, worked by hand."""
    lay = mod.mixed_layout(*_idx(MIXED), max_prefill_rows=MIXED["max_prefill_rows"], sink_page=MIXED["sink_page"])
    for key, want in MIXED["expect"].items():
        if key in lay:
            assert lay[key].tolist() == want, key


def pin_context_only_golden(mod=_plan_ref):
    """context_only_views worked by hand: first pages kept, zero-context row, a context
    ending on a page boundary, a row without queries."""
    P = CTX["page_size"]
    ex = CTX["expect"]
    assert mod.row_lengths(CTX["kv_indptr"], CTX["last_page_len"], P).tolist() == ex["row_lengths"]
    kvp, kvi, lpl = mod.context_only_views(*_idx(CTX), P)
    assert kvp.tolist() == ex["kv_indptr"]
    assert kvi.tolist() == ex["kv_indices"]
    assert lpl.tolist() == ex["last_page_len"]


def _slot(kvp, kvi, r, p, P):
    return int(kvi[kvp[r] + p // P]), p % P


def pin_context_only_positions(mod=_plan_ref, seeds=range(6)):
    """At any size: the shrunk view addresses every context position 0..ctx-1 at the same
    (page, slot) as the full view (so the tokens it holds are the stored context, in
    order), it has exactly ceil(ctx / P) pages and its own length is ctx."""
    for seed in seeds:
        rng = np.random.default_rng(100 + seed)
        P = int(rng.choice([1, 2, 4, 16]))
        B = int(rng.integers(1, 12))
        L = rng.integers(1, 70, size=B)
        n = np.array([int(rng.integers(0, l + 1)) for l in L])
        pages = [int(-(-l // P)) for l in L]
        pool = rng.permutation(sum(pages) + 7)
        kvp = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
        kvi = pool[: kvp[-1]].astype(np.int32)
        lpl = np.array([(l - 1) % P + 1 for l in L], np.int32)
        qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        okvp, okvi, olpl = mod.context_only_views(qo, kvp, kvi, lpl, P)
        ctx = L - n
        assert mod.row_lengths(okvp, olpl, P).tolist() == ctx.tolist()
        for r in range(B):
            assert okvp[r + 1] - okvp[r] == -(-int(ctx[r]) // P), f"row {r}: page count"
            for p in range(int(ctx[r])):
                assert _slot(okvp, okvi, r, p, P) == _slot(kvp, kvi, r, p, P), f"row {r} position {p}"


def pin_append_slots_fill_order(mod=_plan_ref, seeds=range(4)):
    """Brute force: replaying a row's positions 0..L-1 into its pages in order puts the
    last n_r of them at exactly the slots append_slots reports."""
    for seed in seeds:
        rng = np.random.default_rng(200 + seed)
        P = int(rng.choice([1, 3, 8, 16]))
        B = int(rng.integers(1, 10))
        L = rng.integers(1, 60, size=B)
        n = np.array([int(rng.integers(0, l + 1)) for l in L])
        pages = [int(-(-l // P)) for l in L]
        kvp = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
        kvi = rng.permutation(kvp[-1] + 3)[: kvp[-1]].astype(np.int32)
        lpl = np.array([(l - 1) % P + 1 for l in L], np.int32)
        qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        got_p, got_s = mod.append_slots(qo, kvp, kvi, lpl, P)
        t = 0
        for r in range(B):
            filled = []  # (page, slot) of positions 0, 1, ... walking page by page
            for k in range(pages[r]):
                for s in range(P):
                    filled.append((int(kvi[kvp[r] + k]), s))
            for p in range(int(L[r]) - int(n[r]), int(L[r])):
                assert (int(got_p[t]), int(got_s[t])) == filled[p], f"row {r} position {p}"
                t += 1


ALL_PLAN_PINS = [pin_append_slots_golden, pin_mixed_layout_golden, pin_context_only_golden,
                 pin_context_only_positions, pin_append_slots_fill_order]

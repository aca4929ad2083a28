"""The oracle's index work against a hand-worked layout and against brute-force
properties (CPU only)."""
import numpy as np
import pytest

from oracle import plan_ref
import plan_pins
from paged_kv_attention_gqa_gb300 import workloads as wl

GOLD = plan_pins.MIXED


def _idx(g):
    return g["qo_indptr"], g["kv_indptr"], g["kv_indices"], g["last_page_len"]


@pytest.mark.parametrize("pin", plan_pins.ALL_PLAN_PINS, ids=lambda f: f.__name__)
def test_plan_pin(pin):
    pin()


def test_too_many_prompt_rows():
    with pytest.raises(ValueError):
        plan_ref.mixed_layout(*_idx(GOLD), max_prefill_rows=1, sink_page=11)


def test_last_page_len_formula():
    # brute force: fill a length-L stream one token at a time into pages of size P
    for P in (1, 2, 3, 16):
        for L in range(1, 70):
            fill, pages = 0, 0
            for _ in range(L):
                if fill == 0 or fill == P:
                    pages, fill = pages + 1, 0
                fill += 1
            assert plan_ref.last_page_len_of(L, P) == fill
            assert pages == -(-L // P)


@pytest.mark.parametrize("seed", range(5))
def test_mixed_layout_properties(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    n = rng.choice([0, 1, 1, 1, 2, 5, 17], size=B)
    c = rng.integers(0, 50, size=B)
    L = np.maximum(c + n, 1)
    maxp = int((n >= 2).sum()) + int(rng.integers(0, 3))
    pb = wl.custom(seed, L, n, num_qo_heads=4, num_kv_heads=2, head_dim=8, page_size=16, reserve_sink=True)
    lay = plan_ref.mixed_layout(*pb.index_arrays(), max_prefill_rows=maxp, sink_page=pb.sink_page)
    T = int(n.sum())
    perm = lay["perm"]
    assert sorted(perm.tolist()) == list(range(T))
    qo = pb.qo_indptr
    front = [t for r in range(B) if n[r] >= 2 for t in range(qo[r], qo[r + 1])]
    assert perm[: len(front)].tolist() == front
    rest = perm[len(front):]
    assert np.all(np.diff(rest) > 0)
    dec = lay["is_decode"].astype(bool)
    assert np.array_equal(dec, n == 1)
    for r in range(B):
        a, b = lay["dec_kv_indptr"][r], lay["dec_kv_indptr"][r + 1]
        if dec[r]:
            assert lay["dec_kv_indices"][a:b].tolist() == pb.page_table[r].tolist()
            assert lay["dec_last_page_len"][r] == pb.last_page_len[r]
            assert lay["dec_out_token"][r] == qo[r]
        else:
            assert lay["dec_kv_indices"][a:b].tolist() == [pb.sink_page]
            assert lay["dec_last_page_len"][r] == 1 and lay["dec_out_token"][r] == -1
    pf = lay["pf_qo_indptr"]
    assert len(pf) == maxp + 1 and pf[-1] == len(front)

"""The causal-run split the full-size prefill parity test feeds the oracle computes the
same thing as the oracle on the original rows, bit for bit (CPU only)."""
import numpy as np
import pytest

import gpu_util as G
import oracle
from paged_kv_attention_gqa_gb300 import workloads as wl


@pytest.mark.parametrize("P,window", [(16, -1), (4, -1), (16, 7), (1, 30)])
def test_causal_subrows_match_whole_rows(P, window):
    rng = np.random.default_rng(P + 3 * window)
    n = rng.integers(0, 40, size=6)
    n[0] = 37
    c = rng.integers(0, 50, size=6)
    L = np.maximum(n + c, 1)
    pb = wl.custom(61, L, n, num_qo_heads=4, num_kv_heads=2, head_dim=16, page_size=P)
    x = wl.make_inputs(pb, device="cpu", seed=62, unused="nan", layers=1)
    kv = G.oracle_append(pb, wl.bf16_bits(x["kv_cache"][0]), x)
    q = wl.bf16_bits(x["q"])
    o1, l1 = oracle.attention(q, kv, *pb.index_arrays(), num_qo_heads=4, num_kv_heads=2, head_dim=16, page_size=P,
                              causal=True, window_left=window)
    o2, l2 = G.oracle_attn_causal_split(pb, q, kv, window_left=window, threads=3, max_tokens=5)
    assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))
    assert np.array_equal(l1.view(np.uint32), l2.view(np.uint32))

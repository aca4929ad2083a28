"""Rows near the largest sizes a serving step meets: a million-token decode row (65,537 pages
of 16, positions and slot rows far past 16 bits, the row cut over every CTA of the grid and
merged by the separate merge kernel) and a prefill row of 9 new tokens after a million-token
prefix (16,385 key tiles in its query tile).  One kv head keeps the cache at ~0.6 GB and the
oracle at seconds."""
import numpy as np
import pytest
import torch

import gpu_util as G
from paged_kv_attention_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

MILLION = (1 << 20) + 17


@pytest.fixture(scope="module", autouse=True)
def _build():
    from paged_kv_attention_gqa_gb300 import build
    build.build()


def _check(pb, mode, fused=False, seed=0):
    x = wl.make_inputs(pb, device="cuda", seed=seed, unused="nan", layers=1)
    before = wl.bf16_bits(x["kv_cache"][0])
    out, lse, _, _ = G.gpu_step(pb, x, mode, fused=fused)
    after = G.oracle_append(pb, before, x)
    assert np.array_equal(wl.bf16_bits(x["kv_cache"][0]), after)
    ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after, threads=16)
    G.compare(out, lse, ref_o, ref_l, what=f"{mode} at {int(pb.kv_lens.max())} keys")


@pytest.mark.parametrize("fused", [False, True])
def test_million_token_decode_row(fused):
    pb = wl.custom(300, [MILLION, 5, 33], [1, 1, 1], num_qo_heads=8, num_kv_heads=1, head_dim=128, page_size=16)
    _check(pb, "decode", fused=fused, seed=1)


def test_prefill_after_a_million_token_prefix():
    n = [9, 3]
    c = [MILLION, 40]
    pb = wl.custom(301, np.add(n, c), n, num_qo_heads=8, num_kv_heads=1, head_dim=128, page_size=16)
    _check(pb, "prefill", seed=2)

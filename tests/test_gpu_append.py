"""pkv_kv_append straight from device index arrays (no plan), through the C ABI.

The appended layer slice is compared bit for bit with the oracle's append (every byte of
the slice: the new tokens' K and V rows at their (page, slot), nothing else touched) on
the tiny decode, one layer of the batch decode, the ragged prefill and the mixed-step
workloads, and against the planned append (pkv_kv_append_planned) on the same arrays.
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


def _dev(a):
    return torch.as_tensor(np.asarray(a, np.int32), device="cuda")


def _indexed_append(h, pb, x, kv, *, with_qo=True):
    qo, kvp, kvi, lpl = (_dev(a) for a in pb.index_arrays())
    h.kv_append(x["k_new"], x["v_new"], pb.num_tokens, kv, qo if with_qo else None, kvp, kvi, lpl, pb.batch)
    torch.cuda.synchronize()


WORKLOADS = {
    "tiny_decode": lambda: wl.config_tiny(),
    "batch_decode_layer": lambda: wl.config_batch_decode(num_layers=1),
    "ragged_prefill": lambda: wl.config_prefill(),
    "mixed": lambda: wl.config_mixed(),
    "page_size_1": lambda: wl.custom(41, [1, 7, 30, 2], [1, 3, 30, 0], num_qo_heads=8, num_kv_heads=2, head_dim=64,
                                     page_size=1),
    "page_size_128": lambda: wl.custom(42, [1, 127, 128, 129, 400], [1, 5, 128, 2, 200], num_qo_heads=8,
                                       num_kv_heads=4, head_dim=128, page_size=128),
}


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_indexed_append_bit_exact(name):
    pb = WORKLOADS[name]()
    x = wl.make_inputs(pb, device="cuda", seed=3, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    before = wl.bf16_bits(kv)
    h = G.make_handle(pb)
    _indexed_append(h, pb, x, kv)
    want = G.oracle_append(pb, before, x)
    assert np.array_equal(wl.bf16_bits(kv), want), "appended slice differs from the oracle's"


def test_indexed_append_equals_planned_append():
    pb = wl.config_prefill()
    x = wl.make_inputs(pb, device="cuda", seed=4, unused="nan", layers=1)
    kv_a = x["kv_cache"][0].clone()
    kv_b = x["kv_cache"][0].clone()
    h = G.make_handle(pb)
    _indexed_append(h, pb, x, kv_a)
    ws = torch.empty(h.workspace_size(B.MODE_PREFILL), dtype=torch.uint8, device="cuda")
    h.plan(B.MODE_PREFILL, pb.qo_indptr, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    h.kv_append_planned(x["k_new"], x["v_new"], kv_b, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(wl.bf16_bits(kv_a), wl.bf16_bits(kv_b))


def test_indexed_append_decode_without_qo_indptr():
    lens = [1, 2, 15, 16, 17, 100, 1000]
    pb = wl.custom(43, lens, [1] * len(lens), num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    x = wl.make_inputs(pb, device="cuda", seed=5, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    before = wl.bf16_bits(kv)
    h = G.make_handle(pb)
    _indexed_append(h, pb, x, kv, with_qo=False)
    assert np.array_equal(wl.bf16_bits(kv), G.oracle_append(pb, before, x))


def test_indexed_append_leaves_inconsistent_rows_unwritten():
    """A row whose page id lies outside the cache is skipped by the kernel's own checks;
    the other rows are appended exactly."""
    lens = [5, 40, 17]
    pb = wl.custom(44, lens, [2, 3, 1], num_qo_heads=8, num_kv_heads=2, head_dim=64, page_size=16)
    x = wl.make_inputs(pb, device="cuda", seed=6, unused="nan", layers=1)
    kv = x["kv_cache"][0]
    before = wl.bf16_bits(kv)
    h = G.make_handle(pb)
    qo, kvp, kvi, lpl = (np.array(a) for a in pb.index_arrays())
    bad = kvi.copy()
    bad[kvp[1] + 2] = pb.max_pages + 1000  # row 1's last page (positions 32..39) now points outside the cache
    h.kv_append(x["k_new"], x["v_new"], pb.num_tokens, kv, _dev(qo), _dev(kvp), _dev(bad), _dev(lpl), pb.batch)
    torch.cuda.synchronize()
    want = G.oracle_append(pb, before, x)
    # expected: the oracle's append with row 1's tokens not written
    keep = before.copy().reshape(want.shape)
    rows_ok = [0, 2]
    sub_mask = np.zeros(pb.num_tokens, bool)
    for r in rows_ok:
        sub_mask[qo[r]: qo[r + 1]] = True
    P = pb.page_size
    for t in np.nonzero(sub_mask)[0]:
        r = int(np.searchsorted(qo, t, side="right") - 1)
        p = int(pb.kv_lens[r] - pb.qo_lens[r] + (t - qo[r]))
        page, slot = int(kvi[kvp[r] + p // P]), p % P
        keep[page, :, slot] = want[page, :, slot]
    assert np.array_equal(wl.bf16_bits(kv), keep)

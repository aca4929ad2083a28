"""The device error path, made to fire without a fault: a wait that no barrier phase ever
satisfies gives up after its poll limit and records a code in the workspace's error word;
the host reads it through pkv_check_device_error, which clears it, and the same handle,
workspace and context then run a normal step whose results match the oracle."""
import numpy as np
import pytest
import torch

import gpu_util as G
from paged_kv_attention_gqa_gb300 import binding as B
from paged_kv_attention_gqa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from paged_kv_attention_gqa_gb300 import build
    build.build()


def test_wait_timeout_is_reported_and_cleared_then_the_context_still_works():
    pb = wl.config_tiny()
    x = wl.make_inputs(pb, device="cuda", seed=0, unused="nan", layers=1)
    before = wl.bf16_bits(x["kv_cache"][0])
    h = G.make_handle(pb)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device="cuda")
    h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    assert h.check_device_error(ws) == 0
    h.selftest_wait_timeout(ws, polls=1000)
    assert h.check_device_error(ws) == 4  # kErrWaitSelfTest, reported once ...
    assert h.check_device_error(ws) == 0  # ... and cleared
    # the same handle and workspace (plan still in place) run a normal step
    out, lse, _, _ = G.gpu_step(pb, x, "decode", handle=h, workspace=ws)
    after = G.oracle_append(pb, before, x)
    assert np.array_equal(wl.bf16_bits(x["kv_cache"][0]), after)
    ref_o, ref_l = G.oracle_attn(pb, wl.bf16_bits(x["q"]), after)
    G.compare(out, lse, ref_o, ref_l, what="decode after a reported wait timeout")


def test_selftest_rejects_bad_arguments():
    pb = wl.config_tiny()
    h = G.make_handle(pb)
    ws = torch.empty(h.workspace_size(B.MODE_DECODE), dtype=torch.uint8, device="cuda")
    with pytest.raises(B.PkvError) as e:
        h.selftest_wait_timeout(ws, polls=1000)  # no plan on the workspace yet
    assert e.value.status == B.ERR_NOT_PLANNED
    h.plan(B.MODE_DECODE, None, pb.kv_indptr, pb.kv_indices, pb.last_page_len, workspace=ws)
    for polls in (0, (1 << 20) + 1):
        with pytest.raises(B.PkvError) as e:
            h.selftest_wait_timeout(ws, polls=polls)
        assert e.value.status == B.ERR_INVALID

"""Device-detected failures, provoked without faulting, trapping or hanging the GPU:
a malformed cu_seqlens (the plan marks it, every sequence is treated as empty, nothing is
read) and an expiring bounded wait (the GDN_DEBUG_WAIT_TIMEOUT hook: the tensor-core
kernels wait on a barrier nothing arrives at, record the expiry and return before any
copy or product).  Each leaves the context usable: the next clean call is correct."""
import pytest
import torch

import gated_deltanet_linear_15_gb300 as g
from gated_deltanet_linear_15_gb300 import _lib
from gdn_inputs import make_inputs
from tests.gpu_util import TOL, compare, run_oracle

pytestmark = pytest.mark.gpu


def _fwd(x, shape):
    o = torch.empty_like(x["v"])
    ST = torch.empty(x["N"], x["H"], x["D"], x["D"], dtype=torch.float32, device="cuda")
    ws = torch.empty(g.gdn_fwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    rc = g.gdn_chunk_fwd(shape, x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], o, ST, ws)
    return rc, o, ST, ws


def _clean_call_is_correct(x):
    shape = g.make_shape(x["q"], x["v"], cu_seqlens=x["cu_seqlens"], scale=x["scale"], l2norm=x["l2norm"])
    rc, o, ST, ws = _fwd(x, shape)
    assert rc == 0
    assert g.gdn_get_device_status(shape, ws) == 0
    compare(dict(o=o, S_T=ST), run_oracle(x, bwd=False), TOL[x["dtype"]])


@pytest.mark.parametrize("lens", [[100, -30, 200], [0, 100, 250]], ids=["decreasing", "wrong_total"])
def test_malformed_cu_seqlens_sets_status(lens):
    x = make_inputs("varlen_n16_h32", "cuda", seqlens=[100, 70, 130], H=2, seed=21)
    cu = torch.tensor([0] + lens, dtype=torch.int32, device="cuda")  # total stays 300 or ends at 250
    shape = g.make_shape(x["q"], x["v"], cu_seqlens=cu, scale=x["scale"], l2norm=x["l2norm"])
    rc, _, _, ws = _fwd(x, shape)
    assert rc == 0  # detected on the device, not on the host
    assert g.gdn_get_device_status(shape, ws) & 2
    _clean_call_is_correct(x)


def test_forced_wait_expiry_sets_status_and_returns():
    x = make_inputs("prefill_h32_t8192", "cuda", T=200, H=2, seed=22)
    shape = g.make_shape(x["q"], x["v"], scale=x["scale"], l2norm=x["l2norm"])
    shape.flags |= _lib.GDN_DEBUG_WAIT_TIMEOUT
    rc, _, _, ws = _fwd(x, shape)
    assert rc == 0
    torch.cuda.synchronize()  # the kernels returned: no hang
    assert g.gdn_get_device_status(shape, ws) & 4
    _clean_call_is_correct(x)

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


@pytest.mark.parametrize("D", [128, 64])
def test_numeric_guard_forward(D):
    """A value beyond fp16's range in v (|v| ~ 1e5, fine in bf16) cannot become an fp16 tensor-core
    operand: the forward sets status bit 0 (GDN_ERR_NUMERIC) instead of returning silent infinities."""
    x = make_inputs("prefill_h32_t8192", "cuda", T=130, H=2, D=D, seed=23)
    x["v"][0, 70, 1, 5] = 1e5
    shape = g.make_shape(x["q"], x["v"], scale=x["scale"], l2norm=x["l2norm"])
    rc, _, _, ws = _fwd(x, shape)
    assert rc == 0
    word = g.gdn_get_device_status(shape, ws)
    assert word & 1
    assert g.gdn_device_status_code(word) == _lib.GDN_ERR_NUMERIC
    _clean_call_is_correct(make_inputs("prefill_h32_t8192", "cuda", T=130, H=2, D=D, seed=23))


def test_numeric_guard_backward():
    """The same guard on dO in the backward (widened where the reverse chain converts it)."""
    x = make_inputs("train_b4_h16_t4096", "cuda", B=1, T=130, H=2, seed=24)
    x["dO"][0, 100, 0, 3] = -1e5
    shape = g.make_shape(x["q"], x["v"], scale=x["scale"], l2norm=x["l2norm"])
    ws = torch.empty(g.gdn_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    g.chunk_gated_delta_rule_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dO"], x["S0"], None, None,
                                 x["scale"], x["l2norm"], workspace=ws)
    assert g.gdn_get_device_status(shape, ws) & 1


@pytest.mark.parametrize("direction", ["forward", "backward"])
def test_forced_peer_wait_expiry_sets_status_and_returns(direction):
    """The single-launch sequence parallelism's (GDN_SP_SINGLE_LAUNCH) bounded wait between CTAs: with the
    GDN_DEBUG_PEER_TIMEOUT hook every fixed-up segment waits for a fix-up block that never
    comes; the wait expires, the kernel records status value 16 and the call ends (no hang).
    A clean call afterwards is correct."""
    x = make_inputs("long_h8_t65536", "cuda", T=64 * 7 + 9, H=8, seed=25, with_S0=True)
    shape = g.make_shape(x["q"], x["v"], scale=x["scale"], l2norm=x["l2norm"], seg_chunks=1, window=False,
                         single_launch=True)
    shape.flags |= _lib.GDN_DEBUG_PEER_TIMEOUT
    if direction == "forward":
        rc, _, _, ws = _fwd(x, shape)
        assert rc == 0
    else:
        ws = torch.empty(g.gdn_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
        grads = [torch.empty_like(x[k]) for k in ("q", "k", "v", "g", "beta", "S0")]
        rc = g.gdn_chunk_bwd(shape, x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["dO"], None, *grads, ws)
        assert rc == 0
    torch.cuda.synchronize()  # the kernels returned: no hang
    word = g.gdn_get_device_status(shape, ws)
    assert word & 16
    assert g.gdn_device_status_code(word) == _lib.GDN_ERR_TIMEOUT
    _clean_call_is_correct(x)

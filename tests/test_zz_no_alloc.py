"""The allocation-free forward entry point, gdn_chunk_fwd_static.

Some callers cannot call cudaMalloc at all (code running where device
allocation is forbidden or the memory pool is fully reserved); for them the
library keeps its forward scratch in a fixed device array.  These tests call
that entry point through the C ABI and check that it computes exactly what
gdn_chunk_fwd computes with a caller-provided workspace (bit for bit: the same
kernels on the same inputs), and that both match the fp64 oracle:

* two calls in a row with different shapes, a larger packed batch first and a
  smaller uniform batch after it, so the second call runs over the first one's
  leftovers in the shared array;
* a shape whose sequence-parallel scratch does not fit the array, which the
  entry point runs with one segment per sequence;
* the device status word of a static call, read with a NULL workspace, for a
  clean call and for one whose bounded waits are made to expire.

The file is collected last and passes alone in a fresh process or after the
other tests.
"""
import ctypes

import pytest
import torch

from gdn_inputs import make_inputs
from tests.gpu_util import TOL, compare, run_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _call_static(lib, shape, x, o, ST):
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda t: None if t is None else t.data_ptr()
    return lib.gdn_chunk_fwd_static(ctypes.byref(shape), p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                                    p(x["S0"]), p(o), p(ST), stream)


def _shape(x, sp=True):
    import gated_deltanet_linear_15_gb300 as g
    return g.make_shape(x["q"], x["v"], cu_seqlens=x["cu_seqlens"], scale=x["scale"], l2norm=x["l2norm"], sp=sp)


def _static_equals_workspace_call(x):
    """One static call; its o and S_T equal gdn_chunk_fwd's and the oracle's.  The reference call uses the
    segment plan the static entry point runs: sequence parallelism unless its scratch exceeds the array."""
    import gated_deltanet_linear_15_gb300 as g
    from gated_deltanet_linear_15_gb300 import _lib
    lib = _lib.load()
    sp_ref = g.gdn_fwd_workspace_size(_shape(x)) <= _lib.GDN_STATIC_SCRATCH_BYTES
    o_ref, S_ref = g.chunk_gated_delta_rule_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], True,
                                                x["cu_seqlens"], x["scale"], x["l2norm"], sp=sp_ref)
    o = torch.full_like(x["v"], float("nan"))
    ST = torch.full_like(S_ref, float("nan"))
    shape = _shape(x)
    rc = _call_static(lib, shape, x, o, ST)
    assert rc == 0, lib.gdn_last_error_string()
    assert g.gdn_get_device_status(shape, None) == 0   # the static call's status word (synchronises)
    assert torch.equal(o, o_ref)
    assert torch.equal(ST, S_ref)
    compare(dict(o=o, S_T=ST), run_oracle(x, bwd=False), TOL["bf16"])


def test_static_scratch_two_calls_different_shapes():
    big = make_inputs("varlen_n16_h32", DEV, seqlens=[700, 64, 1200, 5, 333], H=3, seed=11)
    small = make_inputs("train_b4_h16_t4096", DEV, B=2, T=333, H=3, seed=12)
    _static_equals_workspace_call(big)
    _static_equals_workspace_call(small)


def test_static_scratch_drops_sequence_parallelism_when_it_does_not_fit():
    import gated_deltanet_linear_15_gb300 as g
    from gated_deltanet_linear_15_gb300 import _lib
    x = make_inputs("prefill_h32_t8192", DEV, T=8192, H=1, seed=13)
    # this shape's sequence-parallel scratch exceeds the array, its one-segment scratch fits
    assert g.gdn_fwd_workspace_size(_shape(x)) > _lib.GDN_STATIC_SCRATCH_BYTES
    assert g.gdn_fwd_workspace_size(_shape(x, sp=False)) <= _lib.GDN_STATIC_SCRATCH_BYTES
    _static_equals_workspace_call(x)


def test_static_status_word_reports_an_expired_wait():
    import gated_deltanet_linear_15_gb300 as g
    from gated_deltanet_linear_15_gb300 import _lib
    lib = _lib.load()
    x = make_inputs("prefill_h32_t8192", DEV, T=200, H=2, seed=14)
    shape = _shape(x)
    shape.flags |= _lib.GDN_DEBUG_WAIT_TIMEOUT
    o = torch.empty_like(x["v"])
    ST = torch.empty(1, 2, 128, 128, dtype=torch.float32, device=DEV)
    assert _call_static(lib, shape, x, o, ST) == 0
    word = g.gdn_get_device_status(shape, None)
    assert word & 4
    assert g.gdn_device_status_code(word) == _lib.GDN_ERR_TIMEOUT
    _static_equals_workspace_call(x)   # the next clean call is correct and its status is 0


def test_static_scratch_rejects_oversized_shape():
    import gated_deltanet_linear_15_gb300 as g
    from gated_deltanet_linear_15_gb300 import _lib
    lib = _lib.load()
    s = g.GdnShape()
    s.B, s.T, s.H, s.Dk, s.Dv = 1, 1 << 20, 64, 128, 128   # the forward's chunk-context region alone exceeds the array
    s.dtype, s.scale = _lib.GDN_BF16, 0.1
    p = 1 << 20
    rc = lib.gdn_chunk_fwd_static(ctypes.byref(s), p, p, p, p, p, None, p, None, None)
    assert rc == _lib.GDN_ERR_WORKSPACE
    assert b"static scratch" in lib.gdn_last_error_string()

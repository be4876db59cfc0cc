"""The allocation-free forward entry point, gdn_chunk_fwd_static.

Some callers cannot call cudaMalloc at all (code running where device
allocation is forbidden or the memory pool is fully reserved); for them the
library keeps its forward scratch in a fixed device array.  This test calls that
entry point through the C ABI twice in a row, with different inputs, and checks
each result against gdn_chunk_fwd on the same inputs.  It lives in its own file,
collected last, and passes alone in a fresh process or after the other tests.
"""
import ctypes

import pytest
import torch

from gdn_inputs import make_inputs
from tests.gpu_util import TOL, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build_library()


def _call_static(lib, shape, x, o, ST):
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda t: None if t is None else t.data_ptr()
    return lib.gdn_chunk_fwd_static(ctypes.byref(shape), p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                                    p(x["S0"]), p(o), p(ST), stream)


def test_static_scratch_matches_workspace_entry_point_twice():
    import gated_deltanet_linear_15_gb300 as g
    from gated_deltanet_linear_15_gb300 import _lib
    lib = _lib.load()
    for seed in (11, 12):   # two calls in a row; the second sees the first one's leftovers
        x = make_inputs("train_b4_h16_t4096", DEV, B=2, T=333, H=3, seed=seed)
        shape = g.make_shape(x["q"], x["v"], scale=x["scale"], l2norm=x["l2norm"])
        o_ref, S_ref = g.chunk_gated_delta_rule_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], True, None,
                                                    x["scale"], x["l2norm"])
        o = torch.empty_like(x["v"])
        ST = torch.empty_like(S_ref)
        rc = _call_static(lib, shape, x, o, ST)
        assert rc == 0, lib.gdn_last_error_string()
        torch.cuda.synchronize()
        assert rel_err(o, o_ref.double().cpu().numpy()) <= TOL["bf16"]
        assert rel_err(ST, S_ref.double().cpu().numpy()) <= TOL["bf16"]


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

"""Saved-context training pair (gdn_chunk_fwd_save + gdn_chunk_bwd_saved) against the fp64
oracle: the forward's outputs are those of the plain forward bit for bit, and the backward that
reads the saved chunk-start states and WY tiles meets the same tolerance as the recomputing
one, in every segment-plan mode and with a different plan in the backward."""
import pytest
import torch

import gated_deltanet_linear_15_gb300 as g
from gdn_inputs import make_inputs
from tests.gpu_util import TOL, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("T", [1, 64, 65, 320])
@pytest.mark.parametrize("D", [64, 128])
def test_saved_bf16_lengths(T, D):
    x = make_inputs("train_b4_h16_t4096", DEV, B=2, T=T, H=2, D=D, with_S0=True, with_dST=True)
    got = run_gpu(x, saved=True)
    compare(got, run_oracle(x), TOL["bf16"])
    plain = run_gpu(x, bwd=False)
    assert torch.equal(got["o"], plain["o"]) and torch.equal(got["S_T"], plain["S_T"])


def test_saved_fp32():
    x = make_inputs("tiny_fp32", DEV, B=2, T=200, H=3, with_S0=True, with_dST=True, seed=5)
    compare(run_gpu(x, saved=True), run_oracle(x), TOL["fp32"])


@pytest.mark.parametrize("seg_chunks", [1, 3])
@pytest.mark.parametrize("window", [True, False])
def test_saved_sequence_parallel(seg_chunks, window):
    x = make_inputs("long_h8_t65536", DEV, T=64 * 7 + 9, H=8, with_S0=True, with_dST=True)
    compare(run_gpu(x, seg_chunks=seg_chunks, window=window, saved=True), run_oracle(x), TOL["bf16"])


def test_saved_other_plan_in_backward():
    """The saved context is indexed by chunk: a backward with another segment plan reads it as well."""
    x = make_inputs("long_h8_t65536", DEV, T=64 * 9 + 3, H=8, with_S0=True, with_dST=True)
    ref = run_oracle(x)
    compare(run_gpu(x, seg_chunks=2, window=False, saved=True, bwd_plan=dict(sp=False)), ref, TOL["bf16"])
    compare(run_gpu(x, sp=False, saved=True, bwd_plan=dict(sp=True, seg_chunks=3)), ref, TOL["bf16"])


def test_saved_varlen():
    x = make_inputs("varlen_n16_h32", DEV, seqlens=[1, 64, 100, 0, 257, 63, 65], H=3, with_dST=True)
    ref = run_oracle(x)
    compare(run_gpu(x, saved=True), ref, TOL["bf16"])
    compare(run_gpu(x, seg_chunks=1, saved=True), ref, TOL["bf16"])


def test_saved_deterministic():
    x = make_inputs("train_b4_h16_t4096", DEV, B=1, T=333, H=2, with_dST=True)
    a, b = run_gpu(x, saved=True), run_gpu(x, saved=True)
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("save_context", [True, False])
def test_autograd_save_context(save_context):
    x = make_inputs("train_b4_h16_t4096", DEV, B=1, T=130, H=2)
    leaves = [x[k].clone().requires_grad_(True) for k in ("q", "k", "v", "g", "beta", "S0")]
    o, S = g.chunk_gated_delta_rule(*leaves, scale=x["scale"], use_qk_l2norm_in_kernel=True,
                                    save_context=save_context)
    (o.float() * x["dO"].float()).sum().backward()
    ref = run_oracle(x)
    from tests.gpu_util import rel_err
    for leaf, key in zip(leaves, ("dq", "dk", "dv", "dg", "dbeta", "dS0")):
        assert rel_err(leaf.grad, ref[key]) <= TOL["bf16"], key

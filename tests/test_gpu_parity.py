"""CUDA path vs the fp64 CPU oracle, element by element, on seeded inputs.

Sizes here are ones the oracle finishes in seconds and that still span several
chunks and a ragged tail; every sequence-parallel mode is forced at least once
(one segment, several segments with the exact fix-up, window skip)."""
import pytest
import torch

from gdn_inputs import make_inputs
from tests.gpu_util import TOL, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_tiny_fp32_workload():
    """B=1 H=1 T=256 d=64 fp32, explicit zero S0, random dS_T: tolerance 1e-4."""
    x = make_inputs("tiny_fp32", DEV, with_dST=True)
    compare(run_gpu(x), run_oracle(x), TOL["fp32"])


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 320])
@pytest.mark.parametrize("D", [64, 128])
def test_bf16_lengths(T, D):
    x = make_inputs("train_b4_h16_t4096", DEV, B=2, T=T, H=2, D=D, with_dST=True)
    compare(run_gpu(x), run_oracle(x), TOL["bf16"])


@pytest.mark.parametrize("T", [70, 200])
def test_fp32_lengths(T):
    x = make_inputs("tiny_fp32", DEV, B=2, T=T, H=3, with_S0=True, with_dST=True, seed=5)
    compare(run_gpu(x), run_oracle(x), TOL["fp32"])


def test_no_initial_state_no_norm():
    x = make_inputs("prefill_h32_t8192", DEV, T=300, H=2, unit_keys=True, with_dST=False)
    compare(run_gpu(x), run_oracle(x), TOL["bf16"])


@pytest.mark.parametrize("single_launch", [False, True], ids=["three_launches", "single_launch"])
@pytest.mark.parametrize("seg_chunks", [1, 2, 3])
@pytest.mark.parametrize("window", [True, False])
def test_sequence_parallel_exact_and_window(seg_chunks, window, single_launch):
    """Forced segmentation: slow decay (alpha ~ 1) exercises pass A + fix-up; with the
    window on, fast-decay heads take the warm-up path instead.  Both the three-launch form and
    the single launch whose CTAs wait for each other's work items (GDN_SP_SINGLE_LAUNCH)."""
    x = make_inputs("long_h8_t65536", DEV, T=64 * 7 + 9, H=8, with_S0=True, with_dST=True)
    for saved in (False, True):
        compare(run_gpu(x, seg_chunks=seg_chunks, window=window, single_launch=single_launch, saved=saved),
                run_oracle(x), TOL["bf16"])


@pytest.mark.parametrize("seg_chunks,seg_first", [(3, 1), (2, 4), (1, 2)])
@pytest.mark.parametrize("window", [True, False])
def test_first_segment_length(seg_chunks, seg_first, window):
    """Segments of two lengths (each sequence's first segment seg_first chunks, the later ones seg_chunks):
    the passes, the fix-up and the mode scan take the same boundaries; slow decay (alpha ~ 1) with the
    window off exercises pass A + fix-up on them, the window on the warm-up path; both pairs."""
    x = make_inputs("long_h8_t65536", DEV, T=64 * 7 + 9, H=8, with_S0=True, with_dST=True)
    ref = run_oracle(x)
    for saved in (False, True):
        compare(run_gpu(x, seg_chunks=seg_chunks, seg_first=seg_first, window=window, saved=saved), ref,
                TOL["bf16"])


def test_balanced_recurrent_grid():
    """More (segment, head) items than SMs while the later segments fit the SMs one each: the recurrent
    passes and the reverse chain run on one CTA per SM, the later segments one per CTA and the one-chunk
    first segments several to a CTA in turn (9 chunks: 1 + 4 x 2, 32 heads); window on and off, both
    pairs, a ragged last chunk."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H, ns = 32, 5
    if not H * (ns - 1) < sms < H * ns:
        pytest.skip(f"{sms} SMs: this plan would not take the balanced grid")
    x = make_inputs("prefill_h32_t8192", DEV, T=64 * 8 + 40, H=H, with_S0=True, with_dST=True)
    ref = run_oracle(x)
    for window in (True, False):
        for saved in (False, True):
            compare(run_gpu(x, seg_chunks=2, seg_first=1, window=window, saved=saved), ref, TOL["bf16"])
    # two sequences of 16 heads: the same 32 (sequence, head) pairs, segment indices across sequences
    x = make_inputs("train_b4_h16_t4096", DEV, B=2, T=64 * 8 + 40, H=H // 2, with_S0=True, with_dST=True, seed=7)
    compare(run_gpu(x, seg_chunks=2, seg_first=1, saved=True), run_oracle(x), TOL["bf16"])


def test_sp_on_off_agree():
    x = make_inputs("long_h8_t65536", DEV, T=64 * 9, H=8, with_dST=True)
    a = run_gpu(x, sp=False)
    b = run_gpu(x, seg_chunks=2, window=False)
    ref = run_oracle(x)
    compare(a, ref, TOL["bf16"])
    compare(b, ref, TOL["bf16"])


def test_varlen_packed():
    x = make_inputs("varlen_n16_h32", DEV, seqlens=[1, 64, 100, 0, 257, 63, 65], H=3, with_dST=True)
    compare(run_gpu(x), run_oracle(x), TOL["bf16"])
    compare(run_gpu(x, seg_chunks=1), run_oracle(x), TOL["bf16"])


def test_empty_sequence_passes_state():
    x = make_inputs("varlen_n16_h32", DEV, seqlens=[0, 5], H=2, with_dST=True)
    got = run_gpu(x)
    torch.testing.assert_close(got["S_T"][0], x["S0"][0], rtol=0, atol=0)
    torch.testing.assert_close(got["dS0"][0], x["dST"][0], rtol=0, atol=0)


def test_deterministic():
    x = make_inputs("train_b4_h16_t4096", DEV, B=1, T=333, H=2, with_dST=True)
    a, b = run_gpu(x), run_gpu(x)
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key


def test_continuation_two_calls():
    """fwd(x[:t]) -> S_t, then fwd(x[t:], S0 = S_t) equals fwd(x)."""
    import gated_deltanet_linear_15_gb300 as g
    x = make_inputs("train_b4_h16_t4096", DEV, B=1, T=448, H=2)
    o, S = g.chunk_gated_delta_rule_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], True, None, x["scale"],
                                        True)
    t = 192
    sl = lambda a: a[:, :t].contiguous()
    sr = lambda a: a[:, t:].contiguous()
    o1, S1 = g.chunk_gated_delta_rule_fwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(x["beta"]), x["S0"],
                                          True, None, x["scale"], True)
    o2, S2 = g.chunk_gated_delta_rule_fwd(sr(x["q"]), sr(x["k"]), sr(x["v"]), sr(x["g"]), sr(x["beta"]), S1, True,
                                          None, x["scale"], True)
    torch.testing.assert_close(torch.cat([o1, o2], 1).float(), o.float(), atol=2e-2, rtol=0)
    torch.testing.assert_close(S2, S, atol=1e-2, rtol=1e-2)


def test_autograd_function():
    import gated_deltanet_linear_15_gb300 as g
    x = make_inputs("train_b4_h16_t4096", DEV, B=1, T=130, H=2)
    leaves = [x[k].clone().requires_grad_(True) for k in ("q", "k", "v", "g", "beta", "S0")]
    o, S = g.chunk_gated_delta_rule(*leaves, scale=x["scale"], use_qk_l2norm_in_kernel=True)
    (o.float() * x["dO"].float()).sum().backward()
    ref = run_oracle(x)
    import numpy as np
    from tests.gpu_util import rel_err
    for leaf, key in zip(leaves, ("dq", "dk", "dv", "dg", "dbeta", "dS0")):
        assert rel_err(leaf.grad, ref[key]) <= TOL["bf16"], key

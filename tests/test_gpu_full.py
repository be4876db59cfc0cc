"""Full-size workloads in the launch configuration the bench times (automatic
segment plan), both training pairs, compared with the oracle element by element
over every (sequence, head) of the prefill, training and long-context
workloads, and over every sequence of four heads of the packed varlen batch
(whose fp64 copies of all 32 heads would take tens of GB of host memory); plus
the Euler-homogeneity identities of the backward over every element.  The raw
and adjusted margins of each output are printed at the end of the session."""
import pytest
import torch

from gdn_inputs import make_inputs
from tests.gpu_util import TOL, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (workload, heads compared; None = all)
CASES = [
    ("prefill_h32_t8192", None),
    ("train_b4_h16_t4096", None),
    ("long_h8_t65536", None),
    ("varlen_n16_h32", [0, 7, 20, 31]),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _heads(t, heads, state=False):
    """Select heads of a [B, T, H, ...] tensor (or a [N, H, D, D] state) on the CPU."""
    if t is None:
        return None
    t = t.detach().cpu()
    return t[:, heads].contiguous() if state else t[:, :, heads].contiguous()


@pytest.mark.parametrize("name,heads", CASES, ids=[c[0] for c in CASES])
def test_full_size_every_sequence_and_head(name, heads):
    x = make_inputs(name, DEV)
    runs = {"recompute": run_gpu(x), "saved": run_gpu(x, saved=True)}
    heads = list(range(x["H"])) if heads is None else heads
    xs = {k: _heads(x[k], heads) for k in ("q", "k", "v", "g", "beta", "dO")}
    xs.update(S0=_heads(x["S0"], heads, True), dST=None, cu_seqlens=x["cu_seqlens"], scale=x["scale"],
              l2norm=x["l2norm"])
    ref = run_oracle(xs)
    for mode, got in runs.items():
        sel = {k: _heads(got[k], heads, k in ("S_T", "dS0")) for k in got if got[k] is not None}
        compare(sel, ref, TOL["bf16"], label=f"full {name} ({mode})")


def test_homogeneity_full_prefill():
    """With normalisation off, O is linear in q and (O, S_T) jointly linear in (v, S0):
    <q, dq> = <dO, O>, <v, dv> + <S0, dS0> = <dO, O> + <dS_T, S_T>, over all elements."""
    x = make_inputs("train_b4_h16_t4096", DEV, unit_keys=True, with_dST=True)
    got = run_gpu(x)
    f = lambda t: t.double()
    dOO = (f(x["dO"]) * f(got["o"])).sum().item()
    lhs_q = (f(x["q"]) * f(got["dq"])).sum().item()
    lhs_v = (f(x["v"]) * f(got["dv"])).sum().item() + (f(x["S0"]) * f(got["dS0"])).sum().item()
    rhs_v = dOO + (f(x["dST"]) * f(got["S_T"])).sum().item()
    assert abs(lhs_q - dOO) <= 1e-2 * abs(dOO) + 1e-3
    assert abs(lhs_v - rhs_v) <= 1e-2 * abs(rhs_v) + 1e-3

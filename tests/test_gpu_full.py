"""Full-size workloads in the launch configuration the bench times (automatic
segment plan), checked against the oracle on sampled (sequence, head) pairs,
plus the Euler-homogeneity identities of the backward over every element."""
import numpy as np
import pytest
import torch

import oracle
from gdn_inputs import make_inputs
from tests.gpu_util import TOL, rel_err, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (workload, sampled (sequence, head) pairs)
CASES = [
    ("prefill_h32_t8192", [(0, 0), (0, 31)]),
    ("train_b4_h16_t4096", [(0, 0), (3, 15)]),
    ("long_h8_t65536", [(0, 2), (0, 7)]),        # a decaying head and an alpha ~ 1 head
    ("varlen_n16_h32", None),                      # shortest and longest sequence
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _slice(x, n, h):
    cu = x["cu_seqlens"]
    if cu is None:
        sl = lambda t: t[n:n + 1, :, h:h + 1]
    else:
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda t: t[:, a:b, h:h + 1]
    return sl


@pytest.mark.parametrize("name,pairs", CASES, ids=[c[0] for c in CASES])
def test_full_size_sampled(name, pairs):
    x = make_inputs(name, DEV)
    runs = {"recompute": run_gpu(x), "saved": run_gpu(x, saved=True)}
    if pairs is None:
        lens = np.array(x["seqlens"])
        pairs = [(int(lens.argmin()), 3), (int(lens.argmax()), 20)]
    for n, h in pairs:
        sl = _slice(x, n, h)
        S0 = None if x["S0"] is None else x["S0"][n:n + 1, h:h + 1]
        ro, rS = oracle.fwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(x["beta"]), S0, scale=x["scale"],
                            l2norm=x["l2norm"])
        rg = oracle.bwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(x["beta"]), sl(x["dO"]), S0, None,
                        scale=x["scale"], l2norm=x["l2norm"])
        for mode, got in runs.items():
            errs = {"o": rel_err(sl(got["o"]), ro), "S_T": rel_err(got["S_T"][n:n + 1, h:h + 1], rS)}
            for key in ("dq", "dk", "dv", "dg", "dbeta"):
                errs[key] = rel_err(sl(got[key]), rg[key])
            if S0 is not None:
                errs["dS0"] = rel_err(got["dS0"][n:n + 1, h:h + 1], rg["dS0"])
            bad = {k: v for k, v in errs.items() if not v <= TOL["bf16"]}
            assert not bad, f"{name} ({mode}) seq {n} head {h}: {bad} (all {errs})"


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

"""Context parallelism on the real kernels, with the ranks emulated in one process:
a sequence split into three contiguous shards, each summarised (end state from zero and
transition), the summaries composed into every shard's exact start state (and, backward,
end gradient), each shard rerun — against the fp64 oracle over the whole sequence."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_15_gb300 import cp
from gdn_inputs import make_inputs
from tests.gpu_util import TOL, compare, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,with_S0", [("prefill_h32_t8192", False), ("train_b4_h16_t4096", True)])
def test_three_shards_match_whole_sequence(name, with_S0):
    T, cuts = 448, [0, 128, 320, 448]  # shards of 128, 192 and 128 tokens (chunk-aligned and not)
    x = make_inputs(name, "cuda", T=T, B=2, H=3, with_S0=with_S0, with_dST=True, seed=31)
    fns = cp.library_fns(x["scale"], x["l2norm"])
    sh = lambda t, r: t[:, cuts[r]:cuts[r + 1]].contiguous()
    keys = ("q", "k", "v", "g", "beta", "dO")
    shards = [{kk: sh(x[kk], r) for kk in keys} for r in range(3)]
    summaries = [cp.shard_summary(fns, *(s[kk] for kk in keys[:5])) for s in shards]
    starts = [cp.compose_forward(x["S0"], summaries, r) for r in range(3)]
    outs = [fns.fwd(*(s[kk] for kk in keys[:5]), starts[r]) for r, s in enumerate(shards)]
    F = [fns.bwd(*(s[kk] for kk in keys), starts[r], torch.zeros_like(starts[r]))[5] for r, s in enumerate(shards)]
    Ms = [m for _, m in summaries]
    ends = [cp.compose_backward(x["dST"], F, Ms, r) for r in range(3)]
    grads = [fns.bwd(*(s[kk] for kk in keys), starts[r], ends[r]) for r, s in enumerate(shards)]
    torch.cuda.synchronize()
    got = dict(o=torch.cat([o for o, _ in outs], 1), S_T=outs[2][1],
               dq=torch.cat([gr[0] for gr in grads], 1), dk=torch.cat([gr[1] for gr in grads], 1),
               dv=torch.cat([gr[2] for gr in grads], 1), dg=torch.cat([gr[3] for gr in grads], 1),
               dbeta=torch.cat([gr[4] for gr in grads], 1))
    if with_S0:
        got["dS0"] = grads[0][5]
    compare(got, run_oracle(x), TOL[x["dtype"]])

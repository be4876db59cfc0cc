"""GPU parity of the token-by-token (decode) entry point gdn_recurrent_fwd against
the fp64 oracle: output o and final state for B sequences of T tokens, in bf16
and fp32, d = 64 and 128, with and without an initial state and the in-kernel
L2 norm; gates at the extremes (strong decay, alpha = 0, alpha ~ 1 runs); the
in-place state update; T = 0; and a chunked prefill continued by recurrent decode
steps, against the oracle run over the whole sequence."""
import pytest
import torch

import gated_deltanet_linear_15_gb300 as g
import oracle
from gdn_inputs import make_inputs
from tests.gpu_util import TOL, rel_err

pytestmark = pytest.mark.gpu


def _oracle(x, S0):
    return oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, None, scale=x["scale"], l2norm=x["l2norm"])


def _check(o, S, ref_o, ref_S, dtype):
    tol = TOL[dtype]
    eo, es = rel_err(o, ref_o), rel_err(S, ref_S)
    assert eo <= tol and es <= tol, (eo, es)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("fp32", 64), ("fp32", 128)])
@pytest.mark.parametrize("T", [1, 5, 37])  # 37: tokens staged in blocks of 16 with a ragged last block
@pytest.mark.parametrize("with_S0", [True, False])
@pytest.mark.parametrize("unit_keys", [False, True])
def test_recurrent_matches_oracle(dtype, D, T, with_S0, unit_keys):
    x = make_inputs("train_b4_h16_t4096", "cuda", T=T, B=3, H=4, D=D, dtype=dtype, with_S0=with_S0,
                    unit_keys=unit_keys, seed=11 + T)
    o, S = g.recurrent_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["scale"],
                                        x["l2norm"])
    torch.cuda.synchronize()
    ref_o, ref_S = _oracle(x, x["S0"])
    _check(o, S, ref_o, ref_S, dtype)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("fp32", 128)])
@pytest.mark.parametrize("gate", ["uniform_8_2", "alpha0_heads", "runs_0_6"])
def test_recurrent_gate_extremes(dtype, D, gate):
    """Strong decay (g ~ U[-8, -2]: the running gate product leaves fp32's normal range within a few
    tokens), alpha = 0 in even heads, and runs of alpha ~ 1 broken by g = -6, over 70 tokens (five staged
    blocks, the last one ragged), with an initial state."""
    x = make_inputs("train_b4_h16_t4096", "cuda", T=70, B=2, H=4, D=D, dtype=dtype, with_S0=True, gate=gate,
                    seed=23)
    o, S = g.recurrent_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["scale"],
                                        x["l2norm"])
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(S).all()
    ref_o, ref_S = _oracle(x, x["S0"])
    _check(o, S, ref_o, ref_S, dtype)


def test_recurrent_in_place_state():
    x = make_inputs("train_b4_h16_t4096", "cuda", T=3, B=2, H=3, D=128, with_S0=True, seed=5)
    S = x["S0"].clone()
    o, S_out = g.recurrent_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], S, x["scale"],
                                            x["l2norm"], inplace=True)
    torch.cuda.synchronize()
    assert S_out.data_ptr() == S.data_ptr()
    ref_o, ref_S = _oracle(x, x["S0"])
    _check(o, S, ref_o, ref_S, "bf16")


def test_recurrent_zero_tokens_copies_state():
    x = make_inputs("train_b4_h16_t4096", "cuda", T=0, B=2, H=3, D=64, with_S0=True, seed=6)
    o, S = g.recurrent_gated_delta_rule(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], x["scale"],
                                        x["l2norm"])
    torch.cuda.synchronize()
    assert torch.equal(S, x["S0"])


def test_prefill_then_decode_matches_whole_sequence():
    """Chunked forward over 200 tokens, then 3 decode calls of 2 tokens each, carrying the state."""
    T1, steps, T2 = 200, 3, 2
    x = make_inputs("prefill_h32_t8192", "cuda", T=T1 + steps * T2, B=2, H=3, seed=7)
    ref_o, ref_S = _oracle(x, None)
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o1, S = g.chunk_gated_delta_rule_fwd(sl(x["q"], 0, T1), sl(x["k"], 0, T1), sl(x["v"], 0, T1),
                                         sl(x["g"], 0, T1), sl(x["beta"], 0, T1), None, True, None, x["scale"],
                                         x["l2norm"])
    outs = [o1]
    for i in range(steps):
        a, b = T1 + i * T2, T1 + (i + 1) * T2
        o, S = g.recurrent_gated_delta_rule(sl(x["q"], a, b), sl(x["k"], a, b), sl(x["v"], a, b),
                                            sl(x["g"], a, b), sl(x["beta"], a, b), S, x["scale"], x["l2norm"])
        outs.append(o)
    torch.cuda.synchronize()
    _check(torch.cat(outs, dim=1), S, ref_o, ref_S, "bf16")

"""Shared helpers of the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import gated_deltanet_linear_15_gb300 as g
import oracle

# max |x - ref| / rms(ref), per output tensor: bf16 inputs with fp32 accumulation, and fp32 mode
TOL = {"bf16": 2e-2, "fp32": 1e-4}
# Outputs stored in bf16 (o, dq, dk, dv) carry their own rounding, up to 2^-8 |x|
# (half an ulp of an 8-bit significand); that much is allowed on top of the
# tolerance, which bounds the computation's error.
BF16_HALF_ULP = 2.0 ** -8


def rel_err(x, ref):
    ref = np.asarray(ref, dtype=np.float64)
    out_bf16 = hasattr(x, "dtype") and x.dtype == torch.bfloat16
    x = x.detach().float().cpu().numpy().astype(np.float64) if hasattr(x, "detach") else np.asarray(x, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    dev = np.abs(x - ref)
    if out_bf16:
        dev = np.maximum(dev - BF16_HALF_ULP * np.abs(ref), 0.0)
    if rms == 0.0:
        return float(np.max(dev))
    return float(np.max(dev)) / rms


def run_gpu(x, *, bwd=True, sp=True, window=True, seg_chunks=0, with_final=True, saved=False, bwd_plan=None):
    """Forward (+ backward) through the library.  saved=True: the forward keeps its per-chunk states
    and WY tiles and the backward reads them; bwd_plan = dict(sp=, window=, seg_chunks=) gives the
    backward another segment plan than the forward."""
    res = g.chunk_gated_delta_rule_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], with_final,
                                       x["cu_seqlens"], x["scale"], x["l2norm"], sp=sp, window=window,
                                       seg_chunks=seg_chunks, save_context=saved)
    o, ST = res[0], res[1]
    ctx = res[2] if saved else None
    out = dict(o=o, S_T=ST)
    if bwd:
        plan = dict(sp=sp, window=window, seg_chunks=seg_chunks)
        plan.update(bwd_plan or {})
        dq, dk, dv, dg, db, dS0 = g.chunk_gated_delta_rule_bwd(
            x["q"], x["k"], x["v"], x["g"], x["beta"], x["dO"], x["S0"], x["dST"], x["cu_seqlens"], x["scale"],
            x["l2norm"], saved=ctx, **plan)
        out.update(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=db, dS0=dS0)
    torch.cuda.synchronize()
    return out


def run_oracle(x, *, bwd=True):
    cu = x["cu_seqlens"]
    o, ST = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], cu, scale=x["scale"],
                       l2norm=x["l2norm"])
    out = dict(o=o, S_T=ST)
    if bwd:
        out.update(oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dO"], x["S0"], x["dST"], cu,
                              scale=x["scale"], l2norm=x["l2norm"]))
    return out


def compare(got, ref, tol, keys=None):
    errs = {}
    for key in keys or ref.keys():
        if got.get(key) is None or ref.get(key) is None:
            continue
        errs[key] = rel_err(got[key], ref[key])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"errors above {tol}: {bad} (all: {errs})"
    return errs

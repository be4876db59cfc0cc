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


def rel_errs(x, ref):
    """(raw, adjusted): raw = max |x - ref| / rms(ref); adjusted allows, for outputs stored in
    bf16, the output's own rounding 2^-8 |ref| on top (equal to raw for other outputs)."""
    ref = np.asarray(ref, dtype=np.float64)
    out_bf16 = hasattr(x, "dtype") and x.dtype == torch.bfloat16
    x = x.detach().float().cpu().numpy().astype(np.float64) if hasattr(x, "detach") else np.asarray(x, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    dev = np.abs(x - ref)
    raw = float(np.max(dev)) if dev.size else 0.0
    adj = float(np.max(np.maximum(dev - BF16_HALF_ULP * np.abs(ref), 0.0))) if (out_bf16 and dev.size) else raw
    if rms == 0.0:
        return raw, adj
    return raw / rms, adj / rms


def rel_err(x, ref):
    return rel_errs(x, ref)[1]


# (label, output, raw, adjusted) of every comparison made with a label; tests/conftest.py prints them
# at the end of the session, so the margin against the tolerance is visible in the test log
MARGINS = []


def run_gpu(x, *, bwd=True, sp=True, window=True, seg_chunks=0, with_final=True, saved=False, bwd_plan=None,
            check_status=True, single_launch=False, seg_first=0):
    """Forward (+ backward) through the library.  saved=True: the forward keeps its per-chunk states
    and WY tiles and the backward reads them; bwd_plan = dict(sp=, window=, seg_chunks=, seg_first=) gives the
    backward another segment plan than the forward.  The device status word of each call must be 0
    (no numeric-guard hit, no expired wait, no malformed plan) unless check_status is False."""
    def shape_of(plan):
        return g.make_shape(x["q"], x["v"], cu_seqlens=x["cu_seqlens"], scale=x["scale"], l2norm=x["l2norm"], **plan)

    fplan = dict(sp=sp, window=window, seg_chunks=seg_chunks, single_launch=single_launch, seg_first=seg_first)
    fshape = shape_of(fplan)
    fws = torch.empty(max(g.gdn_fwd_workspace_size(fshape), 256), dtype=torch.uint8, device=x["q"].device)
    res = g.chunk_gated_delta_rule_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], with_final,
                                       x["cu_seqlens"], x["scale"], x["l2norm"], save_context=saved, workspace=fws,
                                       **fplan)
    o, ST = res[0], res[1]
    ctx = res[2] if saved else None
    out = dict(o=o, S_T=ST)
    status = {"fwd": g.gdn_get_device_status(fshape, fws)}
    if bwd:
        plan = dict(fplan)
        plan.update(bwd_plan or {})
        bshape = shape_of(plan)
        need = g.gdn_bwd_workspace_size(bshape) if ctx is None else g.gdn_bwd_saved_workspace_size(bshape)
        bws = torch.empty(max(need, 256), dtype=torch.uint8, device=x["q"].device)
        dq, dk, dv, dg, db, dS0 = g.chunk_gated_delta_rule_bwd(
            x["q"], x["k"], x["v"], x["g"], x["beta"], x["dO"], x["S0"], x["dST"], x["cu_seqlens"], x["scale"],
            x["l2norm"], saved=ctx, workspace=bws, **plan)
        out.update(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=db, dS0=dS0)
        status["bwd"] = g.gdn_get_device_status(bshape, bws)
    torch.cuda.synchronize()
    if check_status:
        assert all(v == 0 for v in status.values()), f"device status words {status}"
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


def compare(got, ref, tol, keys=None, label=None):
    """Every output within tol (adjusted error, see rel_errs); with a label, (raw, adjusted) of each
    output is recorded for the session's margin report."""
    errs, raws = {}, {}
    for key in keys or ref.keys():
        if got.get(key) is None or ref.get(key) is None:
            continue
        raws[key], errs[key] = rel_errs(got[key], ref[key])
        if label:
            MARGINS.append((label, key, raws[key], errs[key]))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"errors above {tol}: {bad} (all: {errs}; raw {raws})"
    return errs

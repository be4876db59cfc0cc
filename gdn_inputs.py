"""Seeded synthetic inputs for the gated delta-rule workloads.

This module only draws random tensors with the distributions and shapes of the
five workloads below; it contains none of the recurrence's arithmetic.  Both the
CPU oracle (``oracle/``) and the CUDA library are fed from here, so that they see
exactly the same values.

Distributions (drawn with a seeded ``torch.Generator`` on the requested device,
so GPU runs generate on the GPU and CPU tests on the CPU):

* q, k ~ N(0, 1) per element, *raw* (not normalised).  The workloads run with
  in-kernel L2 normalisation of q and k (``l2norm=True``) and ``scale =
  1/sqrt(d_k)``, which is how the talk summary describes the keys ("K is
  L2-normalised", onedev.kr FlashQLA talk summary, paragraph on the effective
  sliding window).  ``unit_keys=True`` instead draws q and k uniformly on the
  unit sphere (a Gaussian divided by its norm), for runs with normalisation
  off.
* v ~ N(0, 1); beta = sigmoid(N(0, 1)); dO ~ N(0, 1).
* log-gate g: per-workload law (uniform, or -softplus(N(0,1) - 2)).  Extra laws
  for strong decay, which the pages allow (alpha in (0, 1) with no lower bound):
  ``uniform_8_2`` g ~ U[-8, -2]; ``alpha0_heads`` g = -1e4 (alpha = 0 in any
  float format) in even heads and -softplus(N(0,1) - 2) in odd ones;
  ``runs_0_6`` per head, runs of 17 tokens with g ~ U[-1e-3, 0] (alpha ~ 1)
  alternating with runs of 17 tokens at g = -6, the phase shifted per head.
* ``beta_one=True`` sets beta = 1; ``repeat_keys=m`` makes token t's key (and
  query) the one drawn for token t mod m of the same sequence and head, so
  the same key recurs (the overwrite case of the delta rule).
* S0 ~ N(0, 0.02^2) where a workload carries an initial state.
* varlen lengths: integers uniform on [512, 16384], inclusive.

Every tensor is drawn in fp32 and then cast to the workload dtype (bf16 or
fp32) for q, k, v, dO; g, beta and states stay fp32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int                      # tokens per sequence (uniform batches) or total (varlen)
    D: int
    dtype: str                  # "bf16" or "fp32"
    gate: str                   # gate law
    has_S0: bool
    seed: int
    nseq_varlen: int = 0        # >0: packed varlen batch with this many sequences
    description: str = ""

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# The five workloads of the method's evaluation plan (tiny fp32 check, H=32
# prefill, B=4 training, long low-head-count context, varlen packed batch).
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", B=1, H=1, T=256, D=64, dtype="fp32",
                          gate="uniform_0.1_0.001", has_S0=True, seed=0,
                          description="B=1 H=1 T=256 d=64 fp32, zero initial state passed explicitly"),
    "prefill_h32_t8192": Workload("prefill_h32_t8192", B=1, H=32, T=8192, D=128, dtype="bf16",
                                  gate="neg_softplus", has_S0=False, seed=1,
                                  description="B=1 H=32 T=8192 d=128 bf16, no initial state"),
    "train_b4_h16_t4096": Workload("train_b4_h16_t4096", B=4, H=16, T=4096, D=128, dtype="bf16",
                                   gate="uniform_0.1_0.001", has_S0=True, seed=2,
                                   description="B=4 H=16 T=4096 d=128 bf16, S0 ~ N(0,0.02^2)"),
    "long_h8_t65536": Workload("long_h8_t65536", B=1, H=8, T=65536, D=128, dtype="bf16",
                               gate="long_mixed", has_S0=False, seed=3,
                               description="B=1 H=8 T=65536 d=128 bf16; heads 0-5 decaying, 6-7 alpha~1"),
    "varlen_n16_h32": Workload("varlen_n16_h32", B=1, H=32, T=0, D=128, dtype="bf16",
                               gate="neg_softplus", has_S0=True, seed=4, nseq_varlen=16,
                               description="16 packed sequences, lengths U{512..16384}, H=32 d=128 bf16"),
}


def _gate(law: str, shape, H: int, gen: torch.Generator, device) -> torch.Tensor:
    """Draw the log-gate g (fp32) of shape [..., H] according to ``law``."""
    if law == "uniform_0.1_0.001":
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        return -0.1 + (0.1 - 0.001) * u
    if law == "neg_softplus":
        z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        return -torch.nn.functional.softplus(z - 2.0)
    if law == "long_mixed":
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        fast = -0.2 + (0.2 - 0.02) * u          # heads 0-5: U[-0.2, -0.02]
        slow = -1e-4 + 1e-4 * u                 # heads 6-7: U[-1e-4, 0]
        head = torch.arange(H, device=device).view(*([1] * (len(shape) - 1)), H)
        return torch.where(head < 6, fast, slow)
    if law == "zero":
        return torch.zeros(shape, device=device, dtype=torch.float32)
    if law == "uniform_8_2":
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        return -8.0 + 6.0 * u
    if law == "alpha0_heads":
        z = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        head = torch.arange(H, device=device).view(*([1] * (len(shape) - 1)), H)
        return torch.where(head % 2 == 0, torch.full_like(z, -1e4), -torch.nn.functional.softplus(z - 2.0))
    if law == "runs_0_6":
        u = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        t = torch.arange(shape[-2], device=device).view(*([1] * (len(shape) - 2)), shape[-2], 1)
        head = torch.arange(H, device=device).view(*([1] * (len(shape) - 1)), H)
        fast = ((t + 7 * head) // 17) % 2 == 1
        return torch.where(fast, torch.full_like(u, -6.0), -1e-3 * u)
    raise ValueError(f"unknown gate law {law}")


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_inputs(w: Workload | str, device="cpu", *, T: Optional[int] = None, H: Optional[int] = None,
                B: Optional[int] = None, seqlens: Optional[list[int]] = None, seed: Optional[int] = None,
                unit_keys: bool = False, with_dST: bool = False, gate: Optional[str] = None,
                dtype: Optional[str] = None, D: Optional[int] = None, with_S0: Optional[bool] = None,
                beta_one: bool = False, repeat_keys: int = 0):
    """Return a dict of tensors for workload ``w`` (optionally with overridden sizes).

    Keys: q, k, v [B, T, H, D] (or [1, sum(L), H, D] for varlen), g, beta
    [B, T, H] fp32, S0 [N, H, D, D] fp32 or None, dO like v, dST or None,
    cu_seqlens (int32, device) or None, and the scalar settings ``scale``,
    ``l2norm``.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    B = w.B if B is None else B
    H = w.H if H is None else H
    D = w.D if D is None else D
    seed = w.seed if seed is None else seed
    law = w.gate if gate is None else gate
    tdt = w.torch_dtype if dtype is None else (torch.bfloat16 if dtype == "bf16" else torch.float32)
    has_S0 = w.has_S0 if with_S0 is None else with_S0
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    cu = None
    if w.nseq_varlen or seqlens is not None:
        if seqlens is None:
            lens = torch.randint(512, 16385, (w.nseq_varlen,), generator=gen, device=device)
            seqlens = [int(x) for x in lens.tolist()]
        N = len(seqlens)
        Ttot = int(sum(seqlens))
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(seqlens, dtype=torch.int64), 0).to(torch.int32)
        cu = cu.to(device)
        B, Tdim = 1, Ttot
    else:
        Tdim = w.T if T is None else T
        N = B

    shp = (B, Tdim, H, D)

    def randn(shape):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)

    q = randn(shp)
    k = randn(shp)
    if repeat_keys:
        idx = torch.arange(Tdim, device=device) % repeat_keys
        if cu is not None:   # within each packed sequence
            starts = torch.repeat_interleave(cu[:-1].long(), torch.tensor(seqlens, device=device))
            idx = starts + (torch.arange(Tdim, device=device) - starts) % repeat_keys
        q, k = q[:, idx], k[:, idx]
    if unit_keys:
        q, k = _unit(q), _unit(k)
    v = randn(shp)
    beta = torch.sigmoid(randn((B, Tdim, H)))
    if beta_one:
        beta = torch.ones_like(beta)
    g = _gate(law, (B, Tdim, H), H, gen, device)
    S0 = 0.02 * randn((N, H, D, D)) if has_S0 else None
    if has_S0 and w.name == "tiny_fp32" and T is None:
        S0 = torch.zeros((N, H, D, D), device=device, dtype=torch.float32)
    dO = randn(shp)
    dST = randn((N, H, D, D)) if with_dST else None
    return dict(q=q.to(tdt), k=k.to(tdt), v=v.to(tdt), g=g, beta=beta, S0=S0,
                dO=dO.to(tdt), dST=dST, cu_seqlens=cu, seqlens=seqlens,
                scale=1.0 / math.sqrt(D), l2norm=not unit_keys, N=N, H=H, D=D,
                dtype="bf16" if tdt == torch.bfloat16 else "fp32")

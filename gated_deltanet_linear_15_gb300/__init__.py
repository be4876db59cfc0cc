"""GB300 (sm_103a) chunked Gated DeltaNet: Python binding of the C ABI in include/gdn.h.

Every step of the forward and backward runs in the library's CUDA kernels;
this module only marshals arguments (tensor pointers, the current stream,
workspace tensors from PyTorch's allocator).  If the library is not built the
calls raise: there is no CPU or PyTorch fallback.

Low-level (same names as the C entry points): ``gdn_chunk_fwd``,
``gdn_chunk_fwd_static``, ``gdn_chunk_bwd``, ``gdn_chunk_fwd_save``,
``gdn_chunk_bwd_saved``, ``gdn_recurrent_fwd``, ``gdn_fwd_workspace_size``,
``gdn_bwd_workspace_size``, ``gdn_saved_size``, ``gdn_bwd_saved_workspace_size``,
``gdn_plan_query``, ``gdn_get_device_status``.
High-level: ``chunk_gated_delta_rule_fwd/_bwd`` (allocate outputs; optionally
the forward keeps the per-chunk states and WY tiles for the backward),
``chunk_gated_delta_rule`` (autograd), ``recurrent_gated_delta_rule`` (decode);
``cp`` splits sequences across ranks.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _lib
from ._lib import (GDN_BF16, GDN_FP32, GDN_L2NORM_QK, GDN_SP_OFF, GDN_WINDOW_OFF, GdnShape)

__all__ = ["GdnShape", "make_shape", "gdn_chunk_fwd", "gdn_chunk_fwd_static", "gdn_chunk_bwd", "gdn_fwd_workspace_size",
           "gdn_bwd_workspace_size", "gdn_saved_size", "gdn_bwd_saved_workspace_size", "gdn_chunk_fwd_save",
           "gdn_chunk_bwd_saved", "gdn_plan_query", "gdn_plan_estimate", "gdn_get_device_status", "gdn_device_status_code",
           "gdn_profile_enable", "gdn_profile_only", "gdn_profile_report",
           "chunk_gated_delta_rule_fwd", "chunk_gated_delta_rule_bwd", "chunk_gated_delta_rule",
           "GDN_L2NORM_QK", "GDN_SP_OFF", "GDN_WINDOW_OFF"]


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != 0:
        lib = _lib.load()
        raise RuntimeError(f"{what}: {lib.gdn_status_string(rc).decode()} ({_lib.last_error()})")


def make_shape(q: torch.Tensor, v: torch.Tensor, *, cu_seqlens: Optional[torch.Tensor] = None,
               scale: Optional[float] = None, l2norm: bool = False, sp: bool = True, window: bool = True,
               seg_chunks: int = 0, single_launch: bool = False, seg_first: int = 0) -> GdnShape:
    B, T, H, Dk = q.shape
    s = GdnShape()
    s.B, s.T, s.H, s.Dk, s.Dv = B, T, H, Dk, v.shape[-1]
    if cu_seqlens is not None:
        s.cu_seqlens = cu_seqlens.data_ptr()
        s.num_seqs = cu_seqlens.numel() - 1
    s.dtype = GDN_BF16 if q.dtype == torch.bfloat16 else GDN_FP32
    s.scale = 1.0 / math.sqrt(Dk) if scale is None else float(scale)
    s.flags = (GDN_L2NORM_QK if l2norm else 0) | (0 if sp else GDN_SP_OFF) | (0 if window else GDN_WINDOW_OFF) | \
        (_lib.GDN_SP_SINGLE_LAUNCH if single_launch else 0)
    s.seg_chunks = int(seg_chunks)
    s.seg_first = int(seg_first)
    return s


# ------------------------------------------------------------------ C entry points
def gdn_fwd_workspace_size(shape: GdnShape) -> int:
    return int(_lib.load().gdn_fwd_workspace_size(ctypes.byref(shape)))


def gdn_bwd_workspace_size(shape: GdnShape) -> int:
    return int(_lib.load().gdn_bwd_workspace_size(ctypes.byref(shape)))


def gdn_plan_query(shape: GdnShape):
    a, b, c, f = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(_lib.load().gdn_plan_query(ctypes.byref(shape), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                      ctypes.byref(f)), "gdn_plan_query")
    return dict(seg_chunks=a.value, max_segments=b.value, max_chunks=c.value, seg_first=f.value)


def gdn_plan_estimate(shape: GdnShape):
    """The library's modelled time (µs) of the forward state pass and the backward reverse chain."""
    f, b = ctypes.c_double(), ctypes.c_double()
    _check(_lib.load().gdn_plan_estimate(ctypes.byref(shape), ctypes.byref(f), ctypes.byref(b)), "gdn_plan_estimate")
    return dict(fwd_us=round(f.value, 2), bwd_us=round(b.value, 2))


def gdn_chunk_fwd(shape: GdnShape, q, k, v, g, beta, S0, o, S_T, workspace, workspace_bytes: int = None,
                  stream=None) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return _lib.load().gdn_chunk_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(S0), _ptr(o), _ptr(S_T), _ptr(workspace), int(workspace_bytes),
                                     _stream(stream))


def gdn_chunk_fwd_static(shape: GdnShape, q, k, v, g, beta, S0, o, S_T, stream=None) -> int:
    """Forward whose scratch is the library's fixed device array (no allocation
    anywhere); for callers that cannot allocate device memory.  See gdn.h."""
    return _lib.load().gdn_chunk_fwd_static(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                            _ptr(S0), _ptr(o), _ptr(S_T), _stream(stream))


def gdn_chunk_bwd(shape: GdnShape, q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, workspace,
                  workspace_bytes: int = None, stream=None) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    return _lib.load().gdn_chunk_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(S0), _ptr(dO), _ptr(dS_T), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                                     _ptr(dbeta), _ptr(dS0), _ptr(workspace), int(workspace_bytes),
                                     _stream(stream))


def gdn_saved_size(shape: GdnShape) -> int:
    return int(_lib.load().gdn_saved_size(ctypes.byref(shape)))


def gdn_bwd_saved_workspace_size(shape: GdnShape) -> int:
    return int(_lib.load().gdn_bwd_saved_workspace_size(ctypes.byref(shape)))


def _nbytes(t, given):
    return int(given) if given is not None else t.numel() * t.element_size()


def gdn_chunk_fwd_save(shape: GdnShape, q, k, v, g, beta, S0, o, S_T, saved, workspace, saved_bytes: int = None,
                       workspace_bytes: int = None, stream=None) -> int:
    """gdn_chunk_fwd that also leaves the per-chunk states and WY tiles in `saved`.  See gdn.h."""
    return _lib.load().gdn_chunk_fwd_save(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                          _ptr(S0), _ptr(o), _ptr(S_T), _ptr(saved), _nbytes(saved, saved_bytes),
                                          _ptr(workspace), _nbytes(workspace, workspace_bytes), _stream(stream))


def gdn_chunk_bwd_saved(shape: GdnShape, q, k, v, g, beta, S0, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, saved,
                        workspace, saved_bytes: int = None, workspace_bytes: int = None, stream=None) -> int:
    """gdn_chunk_bwd reading the forward's saved context instead of recomputing it.  See gdn.h."""
    return _lib.load().gdn_chunk_bwd_saved(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                           _ptr(S0), _ptr(dO), _ptr(dS_T), _ptr(dq), _ptr(dk), _ptr(dv),
                                           _ptr(dg), _ptr(dbeta), _ptr(dS0), _ptr(saved),
                                           _nbytes(saved, saved_bytes), _ptr(workspace),
                                           _nbytes(workspace, workspace_bytes), _stream(stream))


def gdn_recurrent_fwd(shape: GdnShape, q, k, v, g, beta, S_in, o, S_out, stream=None) -> int:
    """Token-by-token forward (decoding); S_out may be S_in.  See gdn.h."""
    return _lib.load().gdn_recurrent_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                         _ptr(S_in), _ptr(o), _ptr(S_out), _stream(stream))


def gdn_profile_enable(on: bool) -> None:
    _check(_lib.load().gdn_profile_enable(int(bool(on))), "gdn_profile_enable")


def gdn_profile_only(name: Optional[str]) -> None:
    """Bracket only launches of kernel `name` (None: every launch) while profiling is on."""
    _check(_lib.load().gdn_profile_only(name.encode() if name else None), "gdn_profile_only")


def gdn_profile_report(reset: bool = True) -> dict:
    """{kernel: (launches, total_ms)} since the last reset."""
    lib = _lib.load()
    n = lib.gdn_profile_report(None, 0, 0)
    buf = ctypes.create_string_buffer(n + 1)
    lib.gdn_profile_report(buf, n + 1, int(bool(reset)))
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out


def gdn_get_device_status(shape: GdnShape, workspace, stream=None) -> int:
    """The device status word of the last call (workspace None: of gdn_chunk_fwd_static)."""
    return int(_lib.load().gdn_get_device_status(ctypes.byref(shape), _ptr(workspace), _stream(stream)))


def gdn_device_status_code(word: int) -> int:
    return int(_lib.load().gdn_device_status_code(int(word)))


# ------------------------------------------------------------------ allocation helpers
def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, initial_state=None, output_final_state=True, cu_seqlens=None,
                               scale=None, use_qk_l2norm_in_kernel=False, sp=True, window=True, seg_chunks=0,
                               workspace=None, save_context=False, single_launch=False, seg_first=0):
    """o, S_T (S_T None unless output_final_state); with save_context=True also the saved
    context (a uint8 tensor) to pass to chunk_gated_delta_rule_bwd(saved=...)."""
    _contig(q, k, v, g, beta, initial_state)
    shape = make_shape(q, v, cu_seqlens=cu_seqlens, scale=scale, l2norm=use_qk_l2norm_in_kernel, sp=sp,
                       window=window, seg_chunks=seg_chunks, single_launch=single_launch, seg_first=seg_first)
    N = shape.num_seqs if cu_seqlens is not None else q.shape[0]
    o = torch.empty_like(v)
    S_T = torch.empty(N, q.shape[2], v.shape[-1], q.shape[-1], dtype=torch.float32, device=q.device) \
        if output_final_state else None
    need = gdn_fwd_workspace_size(shape)
    if need == 0:
        _check(_lib.GDN_ERR_INVALID_ARG, "gdn_fwd_workspace_size")
    ws = workspace if workspace is not None and workspace.numel() >= need else _workspace(need, q.device)
    if not save_context:
        _check(gdn_chunk_fwd(shape, q, k, v, g, beta, initial_state, o, S_T, ws), "gdn_chunk_fwd")
        return o, S_T
    saved = _workspace(gdn_saved_size(shape), q.device)
    _check(gdn_chunk_fwd_save(shape, q, k, v, g, beta, initial_state, o, S_T, saved, ws), "gdn_chunk_fwd_save")
    return o, S_T, saved


def recurrent_gated_delta_rule(q, k, v, g, beta, initial_state=None, scale=None, use_qk_l2norm_in_kernel=False,
                               inplace=False):
    """Decode T tokens per sequence: returns (o, S_out).  q, k, v [B, T, H, d]; g, beta [B, T, H];
    initial_state fp32 [B, H, d, d] or None.  With inplace=True the state is updated in
    initial_state's own buffer (which is then returned as S_out)."""
    _contig(q, k, v, g, beta, initial_state)
    shape = make_shape(q, v, scale=scale, l2norm=use_qk_l2norm_in_kernel)
    o = torch.empty_like(v)
    B, _, H, D = q.shape
    if inplace:
        if initial_state is None:
            raise ValueError("inplace=True needs an initial_state buffer")
        S_out = initial_state
    else:
        S_out = torch.empty(B, H, v.shape[-1], D, dtype=torch.float32, device=q.device)
    _check(gdn_recurrent_fwd(shape, q, k, v, g, beta, initial_state, o, S_out), "gdn_recurrent_fwd")
    return o, S_out


def chunk_gated_delta_rule_bwd(q, k, v, g, beta, dO, initial_state=None, dS_T=None, cu_seqlens=None, scale=None,
                               use_qk_l2norm_in_kernel=False, sp=True, window=True, seg_chunks=0, workspace=None,
                               saved=None, single_launch=False, seg_first=0):
    """dq, dk, dv, dg, dbeta, dS0 (dS0 None without an initial state).  `saved`: the context
    that chunk_gated_delta_rule_fwd(save_context=True) returned for these same inputs."""
    _contig(q, k, v, g, beta, dO, initial_state, dS_T)
    shape = make_shape(q, v, cu_seqlens=cu_seqlens, scale=scale, l2norm=use_qk_l2norm_in_kernel, sp=sp,
                       window=window, seg_chunks=seg_chunks, single_launch=single_launch, seg_first=seg_first)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg, db = torch.empty_like(g), torch.empty_like(beta)
    dS0 = torch.empty_like(initial_state) if initial_state is not None else None
    need = gdn_bwd_workspace_size(shape) if saved is None else gdn_bwd_saved_workspace_size(shape)
    if need == 0:
        _check(_lib.GDN_ERR_INVALID_ARG, "gdn_bwd_workspace_size")
    ws = workspace if workspace is not None and workspace.numel() >= need else _workspace(need, q.device)
    if saved is None:
        _check(gdn_chunk_bwd(shape, q, k, v, g, beta, initial_state, dO, dS_T, dq, dk, dv, dg, db, dS0, ws),
               "gdn_chunk_bwd")
    else:
        _check(gdn_chunk_bwd_saved(shape, q, k, v, g, beta, initial_state, dO, dS_T, dq, dk, dv, dg, db, dS0,
                                   saved, ws), "gdn_chunk_bwd_saved")
    return dq, dk, dv, dg, db, dS0


class ChunkGatedDeltaRuleFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, cu_seqlens, scale, l2norm, save_context):
        if save_context:
            o, S_T, saved = chunk_gated_delta_rule_fwd(q, k, v, g, beta, initial_state, True, cu_seqlens, scale,
                                                       l2norm, save_context=True)
        else:
            (o, S_T), saved = chunk_gated_delta_rule_fwd(q, k, v, g, beta, initial_state, True, cu_seqlens, scale,
                                                         l2norm), None
        ctx.save_for_backward(q, k, v, g, beta, initial_state, cu_seqlens, saved)
        ctx.scale, ctx.l2norm = scale, l2norm
        return o, S_T

    @staticmethod
    def backward(ctx, dO, dS_T):
        q, k, v, g, beta, S0, cu, saved = ctx.saved_tensors
        dq, dk, dv, dg, db, dS0 = chunk_gated_delta_rule_bwd(
            q, k, v, g, beta, dO.contiguous(), S0, None if dS_T is None else dS_T.contiguous(), cu, ctx.scale,
            ctx.l2norm, saved=saved)
        return dq, dk, dv, dg, db, dS0, None, None, None, None


def chunk_gated_delta_rule(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None,
                           use_qk_l2norm_in_kernel=False, save_context=True):
    """Autograd entry: returns (o, final_state).  save_context=True keeps the per-chunk states
    and chunk context from the forward until the backward (gdn_saved_size bytes: about 152.5 KB per chunk
    and head at d = 128, bf16) instead of recomputing them there."""
    return ChunkGatedDeltaRuleFunction.apply(q, k, v, g, beta, initial_state, cu_seqlens, scale,
                                             use_qk_l2norm_in_kernel, save_context)

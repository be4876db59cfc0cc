"""CPU checks of the C ABI: the library loads, exports every declared symbol, and
rejects bad arguments on the host with the documented status codes (these
paths return before any CUDA launch, so no GPU is needed)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from gated_deltanet_linear_15_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build_library()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert _declared() == sorted(_lib.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def _shape(**kw):
    s = _lib.GdnShape()
    s.B, s.T, s.H, s.Dk, s.Dv = 1, 128, 2, 128, 128
    s.dtype, s.scale, s.flags = _lib.GDN_BF16, 1.0, 0
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def _fwd(lib, s, ptr=0x10000, ws_bytes=1 << 40, q=None):
    p = ptr if q is None else q
    return lib.gdn_chunk_fwd(ctypes.byref(s), p, ptr, ptr, ptr, ptr, None, ptr, None, ptr, ws_bytes, None)


def test_status_strings(lib):
    assert lib.gdn_status_string(0) == b"ok"
    assert lib.gdn_status_string(2) == b"unsupported configuration"
    assert b"wait" in lib.gdn_status_string(_lib.GDN_ERR_TIMEOUT)
    assert b"fp16" in lib.gdn_status_string(_lib.GDN_ERR_NUMERIC)


@pytest.mark.parametrize("word,code", [
    (0, _lib.GDN_OK), (1, _lib.GDN_ERR_NUMERIC), (2, _lib.GDN_ERR_INVALID_ARG), (3, _lib.GDN_ERR_INVALID_ARG),
    (4, _lib.GDN_ERR_TIMEOUT), (8, _lib.GDN_ERR_TIMEOUT), (16, _lib.GDN_ERR_TIMEOUT), (5, _lib.GDN_ERR_TIMEOUT),
    (-1, _lib.GDN_ERR_CUDA),
])
def test_device_status_code(lib, word, code):
    """Status words map to one code: malformed cu_seqlens first, then an expired wait, then the numeric guard."""
    assert lib.gdn_device_status_code(word) == code


@pytest.mark.parametrize("kw,code", [
    (dict(Dk=96, Dv=96), _lib.GDN_ERR_UNSUPPORTED),
    (dict(Dk=128, Dv=64), _lib.GDN_ERR_UNSUPPORTED),
    (dict(dtype=_lib.GDN_FP32), _lib.GDN_ERR_UNSUPPORTED),      # fp32 needs d = 64
    (dict(H=0), _lib.GDN_ERR_INVALID_ARG),
    (dict(B=0), _lib.GDN_ERR_INVALID_ARG),
    (dict(T=-1), _lib.GDN_ERR_INVALID_ARG),
    (dict(dtype=7), _lib.GDN_ERR_INVALID_ARG),
    (dict(seg_chunks=-2), _lib.GDN_ERR_INVALID_ARG),
    (dict(seg_chunks=2, seg_first=-1), _lib.GDN_ERR_INVALID_ARG),
    (dict(seg_first=3), _lib.GDN_ERR_INVALID_ARG),              # seg_first needs seg_chunks
])
def test_bad_shapes_rejected(lib, kw, code):
    s = _shape(**kw)
    assert _fwd(lib, s) == code
    assert lib.gdn_last_error_string() != b""
    assert lib.gdn_fwd_workspace_size(ctypes.byref(s)) == 0


def test_reserved_must_be_zero(lib):
    s = _shape()
    s.reserved[1] = 3
    assert _fwd(lib, s) == _lib.GDN_ERR_INVALID_ARG


def test_automatic_plan_balances_the_prefill_shape(lib):
    """H=32, T=8192 (128 chunks per head) on a GPU of 129-159 SMs: four segments per head leave SMs
    idle and five do not fit one wave, so the automatic plan gives each sequence a shorter first segment
    (at least 8 chunks, so the next segment's warm-up is never cut short) and four later ones that fill
    the rest, 5 segments in all; the model's estimate is finite and positive."""
    import torch
    if torch.cuda.is_available():  # without a GPU the library plans for 148 SMs
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        if not 128 < sms < 160:
            pytest.skip(f"{sms} SMs: another plan is the right one")
    s = _shape(T=8192, H=32)
    L, S, C, F = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert lib.gdn_plan_query(ctypes.byref(s), ctypes.byref(L), ctypes.byref(S), ctypes.byref(C), ctypes.byref(F)) == 0
    assert S.value == 5 and 8 <= F.value < L.value and F.value + 4 * L.value >= 128 > F.value + 3 * L.value
    f, b = ctypes.c_double(), ctypes.c_double()
    assert lib.gdn_plan_estimate(ctypes.byref(s), ctypes.byref(f), ctypes.byref(b)) == 0
    assert 0 < f.value < 1e4 and 0 < b.value < 1e4
    # the d = 64 / fp32 kernels keep one segment length
    s = _shape(T=8192, H=32, Dk=64, Dv=64, dtype=_lib.GDN_FP32)
    assert lib.gdn_plan_query(ctypes.byref(s), ctypes.byref(L), ctypes.byref(S), ctypes.byref(C), ctypes.byref(F)) == 0
    assert F.value == L.value


def test_first_segment_length_in_plan(lib):
    """seg_first sets the first segment of every sequence, seg_chunks the later ones: 130 chunks as
    3 + 127 / 8 -> 1 + 16 segments per sequence (the sequence-parallel buffers grow with the count)."""
    base = _shape(T=130 * 64, H=2, seg_chunks=8)
    first = _shape(T=130 * 64, H=2, seg_chunks=8, seg_first=3)
    a, b = ctypes.c_int(), ctypes.c_int()
    c = ctypes.c_int()
    assert lib.gdn_plan_query(ctypes.byref(base), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None) == 0
    assert (a.value, b.value) == (8, 17)
    assert lib.gdn_plan_query(ctypes.byref(first), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None) == 0
    assert (a.value, b.value) == (8, 17)
    assert lib.gdn_fwd_workspace_size(ctypes.byref(first)) > 0
    first.seg_first = 2     # 2 + 128 / 8: 17 segments
    assert lib.gdn_plan_query(ctypes.byref(first), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None) == 0
    assert b.value == 17
    first.seg_first = 10    # 10 + 120 / 8: 16 segments
    assert lib.gdn_plan_query(ctypes.byref(first), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None) == 0
    assert b.value == 16


def test_null_and_misaligned_pointers(lib):
    s = _shape()
    assert _fwd(lib, s, q=0) == _lib.GDN_ERR_INVALID_ARG
    assert b"q is NULL" in lib.gdn_last_error_string()
    assert _fwd(lib, s, q=0x10008) == _lib.GDN_ERR_INVALID_ARG
    assert b"aligned" in lib.gdn_last_error_string()


def test_workspace_checks(lib):
    s = _shape()
    need = lib.gdn_fwd_workspace_size(ctypes.byref(s))
    assert need > 0
    assert _fwd(lib, s, ws_bytes=need - 1) == _lib.GDN_ERR_WORKSPACE
    assert lib.gdn_bwd_workspace_size(ctypes.byref(s)) > need   # per-chunk states for the backward


def test_saved_context_sizes(lib):
    """Saved context = fp16 chunk-start states + five fp16 64 x 64 tiles (X1, X2, Ahat, P, N) + two
    fp16 128 x 64 tiles (scaled W^T, Ut^T) + three fp16 64 x 128 operand tiles (K, Q, V) + 2 x 64 fp32
    reciprocal norms per (chunk, head) at bf16, d = 128, then the fp32 gate sum of every (chunk, head)
    (a 256-byte aligned region); the saved-context backward needs the recompute workspace minus
    exactly the states and tiles (the gate sums replace no workspace region)."""
    s = _shape(T=1000, H=3)
    chunks = (1000 + 63) // 64
    gsum = (chunks * 3 * 4 + 255) // 256 * 256
    states = chunks * 3 * 128 * 128 * 2
    tiles = chunks * 3 * ((5 * 64 * 64 + 2 * 128 * 64 + 3 * 64 * 128) * 2 + 2 * 64 * 4)
    assert lib.gdn_saved_size(ctypes.byref(s)) == states + tiles + gsum
    full = lib.gdn_bwd_workspace_size(ctypes.byref(s))
    assert lib.gdn_bwd_saved_workspace_size(ctypes.byref(s)) == full - states - tiles
    # fp32, d = 64: fp32 states, no WY tiles
    s = _shape(T=1000, H=3, Dk=64, Dv=64, dtype=_lib.GDN_FP32)
    assert lib.gdn_saved_size(ctypes.byref(s)) == chunks * 3 * 64 * 64 * 4 + gsum
    assert lib.gdn_saved_size(ctypes.byref(_shape(Dk=96, Dv=96))) == 0


def test_forward_context_region(lib):
    """bf16, d = 128: the forward workspace carries the chunk-local half's tiles for the recurrent half
    (five fp16 64 x 64 tiles and three fp16 64 x 128 operand tiles per (chunk, head)); the backward's
    buffers start where that region starts.  With one segment per sequence (no sequence-parallel
    buffers) the forward and the saved-context backward share the same core, so the difference of
    their workspaces is exactly that region minus the backward's fp16 per-chunk dS (128 x 128) and the
    reverse chain's fp16 per-chunk dUt^T and dO tiles (2 x 128 x 64), which the local-gradient kernel reads."""
    chunks, H = (1000 + 63) // 64, 3
    s = _shape(T=1000, H=H, flags=_lib.GDN_SP_OFF)
    ctx = chunks * H * (5 * 64 * 64 + 3 * 64 * 128) * 2
    dstates = chunks * H * 128 * 128 * 2
    dut = chunks * H * 2 * 128 * 64 * 2
    fwd = lib.gdn_fwd_workspace_size(ctypes.byref(s))
    assert fwd - lib.gdn_bwd_saved_workspace_size(ctypes.byref(s)) == ctx - dstates - dut
    # fp32, d = 64 runs the mma.sync kernels: no context region, fp32 per-chunk dS
    s = _shape(T=1000, H=H, Dk=64, Dv=64, dtype=_lib.GDN_FP32, flags=_lib.GDN_SP_OFF)
    fwd = lib.gdn_fwd_workspace_size(ctypes.byref(s))
    assert fwd - lib.gdn_bwd_saved_workspace_size(ctypes.byref(s)) == -chunks * H * 64 * 64 * 4


def test_context_tile_coordinates_bound(lib):
    """The context tiles are addressed by 32-bit TMA row coordinates (320 rows per (chunk, head) in
    the largest map): a bf16, d = 128 shape beyond that is refused before any launch; fp32, d = 64
    (no context tiles) is not limited by it."""
    s = _shape(T=(1 << 30) // 2 - 64, H=64)   # 8.4 M chunks x 64 heads
    assert lib.gdn_fwd_workspace_size(ctypes.byref(s)) == 0
    assert _fwd(lib, s) == _lib.GDN_ERR_UNSUPPORTED
    assert b"context tiles" in lib.gdn_last_error_string()
    s = _shape(T=1 << 16, H=64)               # 1024 chunks x 64 heads: fine
    assert lib.gdn_fwd_workspace_size(ctypes.byref(s)) > 0


def test_saved_context_checks(lib):
    s = _shape()
    p, big = 0x10000, 1 << 40
    need = lib.gdn_saved_size(ctypes.byref(s))

    def fwd(saved, nbytes):
        return lib.gdn_chunk_fwd_save(ctypes.byref(s), p, p, p, p, p, None, p, None, saved, nbytes, p, big, None)

    def bwd(saved, nbytes, ws_bytes=big):
        return lib.gdn_chunk_bwd_saved(ctypes.byref(s), p, p, p, p, p, None, p, None, p, p, p, p, p, None, saved,
                                       nbytes, p, ws_bytes, None)

    assert fwd(None, need) == _lib.GDN_ERR_INVALID_ARG
    assert b"saved" in lib.gdn_last_error_string()
    assert fwd(p, need - 1) == _lib.GDN_ERR_WORKSPACE
    assert fwd(p + 8, need) == _lib.GDN_ERR_INVALID_ARG
    assert bwd(None, need) == _lib.GDN_ERR_INVALID_ARG
    assert bwd(p, need - 1) == _lib.GDN_ERR_WORKSPACE
    assert bwd(p + 4, need) == _lib.GDN_ERR_INVALID_ARG
    ws = lib.gdn_bwd_saved_workspace_size(ctypes.byref(s))
    assert bwd(p, need, ws - 1) == _lib.GDN_ERR_WORKSPACE
    assert b"workspace" in lib.gdn_last_error_string()


def test_cu_seqlens_requires_B1(lib):
    s = _shape(B=2, cu_seqlens=0x10000, num_seqs=2)
    assert _fwd(lib, s) == _lib.GDN_ERR_INVALID_ARG


def test_bwd_requires_dS0_with_S0(lib):
    s = _shape()
    p = 0x10000
    rc = lib.gdn_chunk_bwd(ctypes.byref(s), p, p, p, p, p, p, p, None, p, p, p, p, p, None, p, 1 << 40, None)
    assert rc == _lib.GDN_ERR_INVALID_ARG
    assert b"dS0" in lib.gdn_last_error_string()


def test_plan_query_sp_policy(lib):
    """The segment plan: SP off gives one segment per sequence; forced segment length is honoured;
    with many (sequence, head) pairs no split happens."""
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    s = _shape(T=8192, H=32, flags=_lib.GDN_SP_OFF)
    assert lib.gdn_plan_query(ctypes.byref(s), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None) == 0
    assert (a.value, b.value, c.value) == (128, 1, 128)
    s = _shape(T=8192, H=32, seg_chunks=10)
    lib.gdn_plan_query(ctypes.byref(s), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None)
    assert (a.value, b.value) == (10, 13)
    s = _shape(B=64, T=4096, H=32)
    lib.gdn_plan_query(ctypes.byref(s), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None)
    assert a.value == 64 and b.value == 64
    s = _shape(T=65536, H=8)           # long context, few heads: split
    lib.gdn_plan_query(ctypes.byref(s), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None)
    assert 1 < a.value < 1024 and b.value * 8 >= 100


def _rec(lib, s, **ptrs):
    p = dict(q=0x10000, k=0x10000, v=0x10000, g=0x10000, beta=0x10000, S_in=0, o=0x10000, S_out=0x10000)
    p.update(ptrs)
    return lib.gdn_recurrent_fwd(ctypes.byref(s), p["q"], p["k"], p["v"], p["g"], p["beta"], p["S_in"], p["o"],
                                 p["S_out"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(Dk=96, Dv=96), _lib.GDN_ERR_UNSUPPORTED),
    (dict(Dk=128, Dv=64), _lib.GDN_ERR_UNSUPPORTED),
    (dict(cu_seqlens=0x10000, num_seqs=1, B=1), _lib.GDN_ERR_UNSUPPORTED),  # B sequences of T tokens only
    (dict(H=0), _lib.GDN_ERR_INVALID_ARG),
    (dict(T=-1), _lib.GDN_ERR_INVALID_ARG),
    (dict(dtype=7), _lib.GDN_ERR_INVALID_ARG),
])
def test_recurrent_bad_shapes_rejected(lib, kw, code):
    assert _rec(lib, _shape(**kw)) == code
    assert lib.gdn_last_error_string() != b""


def test_recurrent_pointer_checks(lib):
    s = _shape()
    assert _rec(lib, s, S_out=0) == _lib.GDN_ERR_INVALID_ARG
    assert b"S_out is NULL" in lib.gdn_last_error_string()
    assert _rec(lib, s, k=0) == _lib.GDN_ERR_INVALID_ARG
    assert _rec(lib, s, S_in=0x10004) == _lib.GDN_ERR_INVALID_ARG
    assert b"aligned" in lib.gdn_last_error_string()

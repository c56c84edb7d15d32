"""Thin Python binding of the C ABI in include/qw.h (argument marshalling only).

Every function here has the name of the C entry point it calls and takes torch
tensors (device memory) or plain Python values; it passes ``data_ptr()`` and the
current CUDA stream and raises :class:`QwError` on a non-OK status.  No arithmetic of
the method happens in Python: every step runs in the library's CUDA kernels.  If the
shared library is missing the import of this module fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

QW_OK = 0
QW_ERR_INVALID_ARG = 1
QW_ERR_UNSUPPORTED = 2
QW_ERR_ALIGNMENT = 3
QW_ERR_VALUE = 4
QW_ERR_WORKSPACE = 5
QW_ERR_TIMEOUT = 6
QW_ERR_CUDA = 7

QW_W_INT4_G128_BF16 = 0
QW_W_INT3_G128_BF16 = 1
QW_W_MXFP4_G32 = 2
QW_W_MXFP8_G32 = 3
QW_W_NVFP4_G16 = 4
QW_W_UINT4ZP_G128_BF16 = 5
QW_W_INT2_G128_BF16 = 6
QW_W_FP8E4M3_G128_BF16 = 7
QW_W_INT1_G128_BF16 = 8
QW_W_FP4E2M1_G128_BF16 = 9
QW_W_SCALE2 = 0x100  # flag: second-level FP32 scale per output channel (and expert)
QW_A_BF16 = 0
QW_A_MXFP8_G32 = 1
QW_A_NVFP4_G16 = 2

EXPORTS = (
    "qw_status_str", "qw_version", "qw_repack_query", "qw_repack", "qw_unpack",
    "qw_repack_scale2", "qw_unpack_scale2",
    "qgemm_workspace_size", "qgemm_dense", "qgemm_moe_route_workspace_size", "qgemm_moe_route",
    "qgemm_moe_permute", "qgemm_moe_grouped", "qgemm_moe_grouped_indexed", "qw_read_error",
    "qw_test_wait_timeout",
    "qgemm_moe_route_noalloc", "qw_quantize_mxfp8", "qw_silu_mul",
    "qgemm_moe_combine_workspace_size", "qgemm_moe_combine", "qw_stream_read",
    "qw_mma_rate_probe",
)


class PackedDesc(ctypes.Structure):
    _fields_ = [
        ("wfmt", ctypes.c_int32), ("E", ctypes.c_int32), ("N", ctypes.c_int32),
        ("K", ctypes.c_int32), ("N_pad", ctypes.c_int32), ("K_pad", ctypes.c_int32),
        ("group", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("w_bytes", ctypes.c_uint64), ("s_bytes", ctypes.c_uint64),
        ("w_expert_stride", ctypes.c_uint64), ("s_expert_stride", ctypes.c_uint64),
    ]


class QwError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_str(status)} (status {status})")


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_DESC = ctypes.POINTER(PackedDesc)

_SIGS = {
    "qw_status_str": (ctypes.c_char_p, [_I32]),
    "qw_version": (_I32, []),
    "qw_repack_query": (_I32, [_I32, _I32, _I32, _I32, _DESC]),
    "qw_repack": (_I32, [_DESC, _P, _P, _P, _P, _P, _P]),
    "qw_unpack": (_I32, [_DESC, _P, _P, _P, _P, _P, _P]),
    "qw_repack_scale2": (_I32, [_DESC, _P, _P, _P, _P]),
    "qw_unpack_scale2": (_I32, [_DESC, _P, _P, _P]),
    "qgemm_workspace_size": (_I32, [_DESC, _I32, _I64, ctypes.POINTER(_U64)]),
    "qgemm_dense": (_I32, [_DESC, _P, _P, _I32, _P, _P, _P, _P, _I64, _P, _U64, _P, _P]),
    "qgemm_moe_route_workspace_size": (_I32, [_I32, _I32, _I32, ctypes.POINTER(_U64)]),
    "qgemm_moe_route": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _U64, _P, _P]),
    "qgemm_moe_permute": (_I32, [_I32, _P, _P, _I32, _P, _I64, _I32, _P, _P, _P]),
    "qgemm_moe_grouped": (_I32, [_DESC, _P, _P, _I32, _P, _P, _P, _I64, _P, _P, _P, _U64, _P, _P]),
    "qgemm_moe_grouped_indexed": (_I32, [_DESC, _P, _P, _I32, _P, _P, _I64, _P, _I32, _P, _I64,
                                         _P, _P, _P, _U64, _P, _P]),
    "qw_read_error": (_I32, [_P, _P, ctypes.POINTER(_I32)]),
    "qw_test_wait_timeout": (_I32, [_P, _I64, _P]),
    "qgemm_moe_route_noalloc": (_I32, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "qw_quantize_mxfp8": (_I32, [_P, _I64, _I32, _P, _P, _P, _P]),
    "qw_silu_mul": (_I32, [_P, _I64, _I32, _P, _P]),
    "qgemm_moe_combine_workspace_size": (_I32, [_I32, _I32, ctypes.POINTER(_U64)]),
    "qgemm_moe_combine": (_I32, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _U64, _P, _P]),
    "qw_stream_read": (_I32, [_P, _U64, _P, _I32, _P]),
    "qw_mma_rate_probe": (_I32, [_I32, _I32, _I32, _P, _P, _P]),
}


def lib_path() -> str:
    return _build.LIB


def _load():
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"libqw is not built ({path} missing): run `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


LIB = _load()


# ----------------------------------------------------------------------------- helpers
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, status):
    if status != QW_OK:
        raise QwError(fn, status)


def status_str(status: int) -> str:
    return LIB.qw_status_str(status).decode()


def qw_version() -> int:
    return LIB.qw_version()


# ----------------------------------------------------------------------------- entry points
def qw_repack_query(wfmt: int, E: int, N: int, K: int) -> PackedDesc:
    d = PackedDesc()
    _check("qw_repack_query", LIB.qw_repack_query(wfmt, E, N, K, ctypes.byref(d)))
    return d


def qw_repack(desc, w_canon, s_canon, w_packed, s_packed, d_err=None, stream=None):
    _check("qw_repack", LIB.qw_repack(ctypes.byref(desc), _ptr(w_canon), _ptr(s_canon),
                                      _ptr(w_packed), _ptr(s_packed), _ptr(d_err),
                                      _stream(stream)))


def qw_unpack(desc, w_packed, s_packed, w_canon, s_canon, d_err=None, stream=None):
    _check("qw_unpack", LIB.qw_unpack(ctypes.byref(desc), _ptr(w_packed), _ptr(s_packed),
                                      _ptr(w_canon), _ptr(s_canon), _ptr(d_err),
                                      _stream(stream)))


def qw_repack_scale2(desc, t_canon, s_packed, d_err=None, stream=None):
    _check("qw_repack_scale2", LIB.qw_repack_scale2(ctypes.byref(desc), _ptr(t_canon),
                                                    _ptr(s_packed), _ptr(d_err),
                                                    _stream(stream)))


def qw_unpack_scale2(desc, s_packed, t_canon, stream=None):
    _check("qw_unpack_scale2", LIB.qw_unpack_scale2(ctypes.byref(desc), _ptr(s_packed),
                                                    _ptr(t_canon), _stream(stream)))


def qgemm_workspace_size(desc, afmt: int, max_rows: int) -> int:
    n = _U64(0)
    _check("qgemm_workspace_size",
           LIB.qgemm_workspace_size(ctypes.byref(desc), afmt, max_rows, ctypes.byref(n)))
    return n.value


def qgemm_dense(desc, w_packed, s_packed, afmt, A, A_sf, bias, C, M, workspace=None,
                ws_bytes=0, d_err=None, stream=None):
    _check("qgemm_dense", LIB.qgemm_dense(
        ctypes.byref(desc), _ptr(w_packed), _ptr(s_packed), afmt, _ptr(A), _ptr(A_sf),
        _ptr(bias), _ptr(C), M, _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)))


def qgemm_moe_route_workspace_size(T: int, E: int, topk: int) -> int:
    n = _U64(0)
    _check("qgemm_moe_route_workspace_size",
           LIB.qgemm_moe_route_workspace_size(T, E, topk, ctypes.byref(n)))
    return n.value


def qgemm_moe_route(logits, T, E, topk, topk_ids, sorted_pairs, expert_offsets, workspace,
                    ws_bytes, d_err=None, stream=None):
    _check("qgemm_moe_route", LIB.qgemm_moe_route(
        _ptr(logits), T, E, topk, _ptr(topk_ids), _ptr(sorted_pairs), _ptr(expert_offsets),
        _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)))


def qgemm_moe_route_noalloc(logits, T, E, topk, topk_ids, sorted_pairs, expert_offsets,
                            d_err=None, stream=None):
    """Routing without a workspace argument, for callers that cannot allocate device
    memory: the library's static device scratch is used (see include/qw.h for its size
    limit and the rule that overlapping calls race)."""
    _check("qgemm_moe_route_noalloc", LIB.qgemm_moe_route_noalloc(
        _ptr(logits), T, E, topk, _ptr(topk_ids), _ptr(sorted_pairs), _ptr(expert_offsets),
        _ptr(d_err), _stream(stream)))


def qgemm_moe_permute(afmt, A, A_sf, K, sorted_pairs, P, topk, A_sorted, A_sf_sorted,
                      stream=None):
    _check("qgemm_moe_permute", LIB.qgemm_moe_permute(
        afmt, _ptr(A), _ptr(A_sf), K, _ptr(sorted_pairs), P, topk, _ptr(A_sorted),
        _ptr(A_sf_sorted), _stream(stream)))


def qgemm_moe_grouped(desc, w_packed, s_packed, afmt, A_sorted, A_sf_sorted, expert_offsets,
                      total_rows, bias, C, workspace=None, ws_bytes=0, d_err=None, stream=None):
    _check("qgemm_moe_grouped", LIB.qgemm_moe_grouped(
        ctypes.byref(desc), _ptr(w_packed), _ptr(s_packed), afmt, _ptr(A_sorted),
        _ptr(A_sf_sorted), _ptr(expert_offsets), total_rows, _ptr(bias), _ptr(C),
        _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)))


def qgemm_moe_grouped_indexed(desc, w_packed, s_packed, afmt, A, A_sf, T, sorted_pairs, topk,
                              expert_offsets, total_rows, bias, C, workspace=None, ws_bytes=0,
                              d_err=None, stream=None):
    _check("qgemm_moe_grouped_indexed", LIB.qgemm_moe_grouped_indexed(
        ctypes.byref(desc), _ptr(w_packed), _ptr(s_packed), afmt, _ptr(A), _ptr(A_sf), T,
        _ptr(sorted_pairs), topk, _ptr(expert_offsets), total_rows, _ptr(bias), _ptr(C),
        _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)))


def qw_quantize_mxfp8(A, rows, K, A_q, A_sf, d_err=None, stream=None):
    _check("qw_quantize_mxfp8", LIB.qw_quantize_mxfp8(_ptr(A), rows, K, _ptr(A_q), _ptr(A_sf),
                                                      _ptr(d_err), _stream(stream)))


def qw_silu_mul(GU, rows, I, Y, stream=None):
    _check("qw_silu_mul", LIB.qw_silu_mul(_ptr(GU), rows, I, _ptr(Y), _stream(stream)))


def qgemm_moe_combine_workspace_size(T: int, topk: int) -> int:
    n = _U64(0)
    _check("qgemm_moe_combine_workspace_size",
           LIB.qgemm_moe_combine_workspace_size(T, topk, ctypes.byref(n)))
    return n.value


def qgemm_moe_combine(Y, sorted_pairs, topk_ids, logits, T, E, topk, N, out, workspace,
                      ws_bytes, d_err=None, stream=None):
    _check("qgemm_moe_combine", LIB.qgemm_moe_combine(
        _ptr(Y), _ptr(sorted_pairs), _ptr(topk_ids), _ptr(logits), T, E, topk, N, _ptr(out),
        _ptr(workspace), ws_bytes, _ptr(d_err), _stream(stream)))


def qw_read_error(d_err, stream=None) -> int:
    code = _I32(0)
    LIB.qw_read_error(_ptr(d_err), _stream(stream), ctypes.byref(code))
    return code.value


def qw_test_wait_timeout(d_err, limit_ns: int, stream=None):
    _check("qw_test_wait_timeout", LIB.qw_test_wait_timeout(_ptr(d_err), limit_ns,
                                                            _stream(stream)))


QW_STREAM_READ_SINK_WORDS = 4096


def qw_stream_read(src, nbytes: int, sink, chained: bool = False, stream=None):
    _check("qw_stream_read", LIB.qw_stream_read(_ptr(src), nbytes, _ptr(sink), int(chained),
                                                _stream(stream)))


QW_MMA_PROBE_F16_TMEM_A = 0
QW_MMA_PROBE_F16_SMEM = 1
QW_MMA_PROBE_MXF8F6F4 = 2
QW_MMA_PROBE_MXF8F6F4_CP = 3
QW_MMA_PROBE_MXF8F6F4_CP_AHEAD = 4
QW_MMA_PROBE_MXF8F6F4_CP_WIDE = 5
QW_MMA_PROBE_MXF4NVF4 = 6
QW_MMA_PROBE_MXF4NVF4_CP = 7
QW_MMA_PROBE_RANDOM = 8
QW_MMA_PROBE_MAX_CTAS = 1024


def qw_mma_rate_probe(mode: int, n: int, iters: int, out, d_err, stream=None):
    """out: device uint64 (int64 tensor) of 2 * QW_MMA_PROBE_MAX_CTAS entries."""
    _check("qw_mma_rate_probe", LIB.qw_mma_rate_probe(mode, n, iters, _ptr(out), _ptr(d_err),
                                                      _stream(stream)))


def mma_rate(mode: int, n: int, iters: int = 4096):
    """Runs the probe once and returns (cycles per MMA, ns per MMA) for each CTA that ran
    (one per SM), as float64 arrays."""
    import numpy as np
    out = torch.zeros(2 * QW_MMA_PROBE_MAX_CTAS, dtype=torch.int64, device="cuda")
    err = new_error_flag()
    qw_mma_rate_probe(mode, n, iters, out, err)
    if qw_read_error(err) != 0:
        raise QwError("qw_mma_rate_probe", qw_read_error(err))
    v = out.cpu().numpy().astype(np.float64).reshape(-1, 2)
    v = v[v[:, 0] > 0]
    return v[:, 0] / iters, v[:, 1] / iters


# ----------------------------------------------------------------------------- conveniences
def empty_packed(desc, device="cuda"):
    """Allocate packed weight / scale buffers for ``desc`` (torch's allocator returns
    blocks aligned to at least 256 bytes)."""
    w = torch.empty(int(desc.w_bytes), dtype=torch.uint8, device=device)
    s = torch.empty(int(desc.s_bytes), dtype=torch.uint8, device=device)
    return w, s


def new_error_flag(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)

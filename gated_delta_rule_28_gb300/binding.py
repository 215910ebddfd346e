"""Thin ctypes binding of ``libgdn.so`` (declared in ``include/gdn.h``).

Every function has the C name and argument order; the binding only turns
tensors into device pointers, fills the ``gdn_problem`` struct, picks the
current CUDA stream and raises ``GdnError`` on a nonzero status. All work runs
in the library's CUDA kernels. When the library has not been built the first
call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

GDN_OK = 0
GDN_ERR_INVALID_ARGUMENT = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_WORKSPACE = 3
GDN_ERR_CUDA = 4
GDN_ERR_TIMEOUT = 5
GDN_ERR_DEVICE_CHECK = 6

GDN_LAYOUT_BSND, GDN_LAYOUT_TND = 0, 1
GDN_GATE_SCALAR, GDN_GATE_PER_KEY = 0, 1
GDN_DTYPE_F32, GDN_DTYPE_BF16 = 0, 1

# every symbol the public header declares
EXPORTS = ("gdn_last_error", "gdn_device_status", "gdn_prepare_varlen", "gdn_chunk_fwd_workspace",
           "gdn_chunk_fwd", "gdn_chunk_bwd_workspace", "gdn_chunk_bwd", "gdn_chunk_bwd_noalloc",
           "kda_segment_summary_workspace", "kda_segment_summary", "kda_segment_merge",
           "kda_segment_summary_bwd_workspace", "kda_segment_summary_bwd", "kda_segment_merge_bwd",
           "gdn_selftest_wait_timeout", "frame_scan_workspace", "frame_scan_fwd",
           "gdn_chunk_fwd_split_workspace", "gdn_chunk_fwd_split")
# bytes of the library's built-in scratch array used by gdn_chunk_bwd_noalloc
GDN_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"gdn status {status}: {message}")
        self.status = status


class gdn_problem(ctypes.Structure):  # noqa: N801  (C name)
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
        ("K", ctypes.c_int32), ("V", ctypes.c_int32),
        ("layout", ctypes.c_int32), ("gate_kind", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("use_exp2", ctypes.c_int32), ("scale", ctypes.c_float), ("chunk_size", ctypes.c_int32),
        ("use_qk_l2norm", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
        ("chunk_indices", ctypes.c_void_p), ("num_chunks", ctypes.c_int32),
        ("segment_len", ctypes.c_int32), ("use_beta_sigmoid", ctypes.c_int32),
    ]


class frame_scan_problem(ctypes.Structure):  # noqa: N801  (C name)
    _fields_ = [("BH", ctypes.c_int32), ("T", ctypes.c_int32), ("D", ctypes.c_int32),
                ("active", ctypes.c_int32), ("segment_len", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load ``libgdn.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libgdn.so is not built ({path}); run "
                                   "gated_delta_rule_28_gb300.build.build() first")
            lib = ctypes.CDLL(path)
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            P = ctypes.POINTER(gdn_problem)
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.gdn_last_error.restype = ctypes.c_char_p
            lib.gdn_last_error.argtypes = []
            lib.gdn_device_status.argtypes = [vp]
            lib.gdn_prepare_varlen.argtypes = [i32p, ctypes.c_int32, ctypes.c_int64, i32p, i32p]
            lib.gdn_chunk_fwd_workspace.argtypes = [P, ctypes.POINTER(sz)]
            lib.gdn_chunk_fwd.argtypes = [P] + [vp] * 11 + [vp, sz, vp]
            lib.gdn_chunk_bwd_workspace.argtypes = [P, ctypes.POINTER(sz)]
            lib.gdn_chunk_bwd.argtypes = [P] + [vp] * 15 + [vp, sz, vp]
            lib.gdn_chunk_bwd_noalloc.argtypes = [P] + [vp] * 15 + [vp]
            lib.kda_segment_summary_workspace.argtypes = [P, ctypes.c_int32, ctypes.POINTER(sz)]
            lib.kda_segment_summary.argtypes = [P, vp, vp, vp, vp, ctypes.c_int32, vp, vp, vp, sz, vp]
            lib.kda_segment_merge.argtypes = [P, vp, vp, ctypes.c_int32, vp, vp, vp, vp]
            lib.gdn_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
            lib.kda_segment_summary_bwd_workspace.argtypes = [P, ctypes.c_int32, ctypes.POINTER(sz)]
            lib.kda_segment_summary_bwd.argtypes = [P] + [vp] * 6 + [ctypes.c_int32, vp, vp, sz, vp]
            lib.kda_segment_merge_bwd.argtypes = [P, vp, vp, ctypes.c_int32, vp, vp, vp, vp]
            lib.gdn_chunk_fwd_split_workspace.argtypes = [P, ctypes.c_int32, ctypes.POINTER(sz)]
            lib.gdn_chunk_fwd_split.argtypes = [P] + [vp] * 6 + [ctypes.c_int32] + [vp] * 8 + [vp, sz, vp]
            FP = ctypes.POINTER(frame_scan_problem)
            lib.frame_scan_workspace.argtypes = [FP, ctypes.POINTER(sz)]
            lib.frame_scan_fwd.argtypes = [FP] + [vp] * 10 + [vp, sz, vp]
            for name in EXPORTS[1:]:
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(status: int):
    if status != GDN_OK:
        raise GdnError(status, load().gdn_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def make_problem(B, T, H, K=128, V=128, *, layout=GDN_LAYOUT_BSND, gate_kind=GDN_GATE_SCALAR,
                 dtype=GDN_DTYPE_BF16, use_exp2=False, scale=0.0, chunk_size=64,
                 use_qk_l2norm=False, cu_seqlens=None, num_seqs=0, chunk_indices=None,
                 num_chunks=0, segment_len=0, use_beta_sigmoid=False) -> gdn_problem:
    """Fill a ``gdn_problem``; cu_seqlens / chunk_indices are device tensors (or None)."""
    p = gdn_problem()
    p.B, p.T, p.H, p.K, p.V = int(B), int(T), int(H), int(K), int(V)
    p.layout, p.gate_kind, p.dtype = int(layout), int(gate_kind), int(dtype)
    p.use_exp2, p.scale, p.chunk_size = int(use_exp2), float(scale), int(chunk_size)
    p.use_qk_l2norm = int(use_qk_l2norm)
    p.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    p.num_seqs = int(num_seqs)
    p.chunk_indices = None if chunk_indices is None else chunk_indices.data_ptr()
    p.num_chunks = int(num_chunks)
    p.segment_len = int(segment_len)
    p.use_beta_sigmoid = int(use_beta_sigmoid)
    return p


def gdn_last_error() -> str:
    return load().gdn_last_error().decode()


def gdn_device_status(stream=None) -> int:
    """Status of the device-side error flag (synchronises the stream); raises on error."""
    _check(load().gdn_device_status(_stream(stream)))
    return GDN_OK


def gdn_selftest_wait_timeout(polls, stream=None):
    """Launch the bounded-wait self-test (its wait always runs out; see gdn.h)."""
    _check(load().gdn_selftest_wait_timeout(int(polls), _stream(stream)))


def gdn_prepare_varlen(cu_seqlens, total_tokens):
    """Host-only metadata: returns (chunk_indices int32 [num_chunks, 2], num_chunks)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    if np.any(cu != cu.astype(np.int32)):
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens values exceed int32")
    cu = cu.astype(np.int32)
    i32p = ctypes.POINTER(ctypes.c_int32)
    n = ctypes.c_int32(0)
    lib = load()
    _check(lib.gdn_prepare_varlen(cu.ctypes.data_as(i32p), int(cu.shape[0]), int(total_tokens),
                                  None, ctypes.byref(n)))
    out = np.zeros((max(n.value, 1), 2), np.int32)
    cap = ctypes.c_int32(n.value)
    _check(lib.gdn_prepare_varlen(cu.ctypes.data_as(i32p), int(cu.shape[0]), int(total_tokens),
                                  out.ctypes.data_as(i32p), ctypes.byref(cap)))
    return out[:n.value], n.value


def gdn_chunk_fwd_workspace(p: gdn_problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gdn_chunk_fwd_workspace(ctypes.byref(p), ctypes.byref(n)))
    return n.value


def gdn_chunk_fwd(p: gdn_problem, q, k, v, g, beta, h0, o, ht=None, g_cumsum=None, A=None,
                  h_chunks=None, ws=None, ws_bytes=0, stream=None):
    _check(load().gdn_chunk_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                _ptr(h0), _ptr(o), _ptr(ht), _ptr(g_cumsum), _ptr(A),
                                _ptr(h_chunks), _ptr(ws), int(ws_bytes), _stream(stream)))


def gdn_chunk_bwd_workspace(p: gdn_problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gdn_chunk_bwd_workspace(ctypes.byref(p), ctypes.byref(n)))
    return n.value


def gdn_chunk_bwd(p: gdn_problem, q, k, v, g_cumsum, beta, A, dO, h0, dht, dq, dk, dv, dg,
                  dbeta, dh0, ws, ws_bytes, stream=None):
    _check(load().gdn_chunk_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g_cumsum),
                                _ptr(beta), _ptr(A), _ptr(dO), _ptr(h0), _ptr(dht), _ptr(dq),
                                _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), _ptr(ws),
                                int(ws_bytes), _stream(stream)))


def gdn_chunk_bwd_noalloc(p: gdn_problem, q, k, v, g_cumsum, beta, A, dO, h0, dht, dq, dk, dv, dg,
                          dbeta, dh0, stream=None):
    """Backward with the library's built-in scratch instead of a workspace (see gdn.h)."""
    _check(load().gdn_chunk_bwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g_cumsum),
                                        _ptr(beta), _ptr(A), _ptr(dO), _ptr(h0), _ptr(dht),
                                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                                        _ptr(dh0), _stream(stream)))


def kda_segment_summary_workspace(p: gdn_problem, segment_len) -> int:
    n = ctypes.c_size_t(0)
    _check(load().kda_segment_summary_workspace(ctypes.byref(p), int(segment_len), ctypes.byref(n)))
    return n.value


def kda_segment_summary(p: gdn_problem, k, v, g, beta, segment_len, S_ext, M, ws=None, ws_bytes=0,
                        stream=None):
    _check(load().kda_segment_summary(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                      int(segment_len), _ptr(S_ext), _ptr(M), _ptr(ws),
                                      int(ws_bytes), _stream(stream)))


def gdn_chunk_fwd_split_workspace(p: gdn_problem, segment_len) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gdn_chunk_fwd_split_workspace(ctypes.byref(p), int(segment_len), ctypes.byref(n)))
    return n.value


def gdn_chunk_fwd_split(p: gdn_problem, q, k, v, g, beta, h0, segment_len, o, ht, S_ext, M, S_init,
                        g_cumsum=None, A=None, h_chunks=None, ws=None, ws_bytes=0, stream=None):
    _check(load().gdn_chunk_fwd_split(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                      _ptr(h0), int(segment_len), _ptr(o), _ptr(ht), _ptr(S_ext), _ptr(M),
                                      _ptr(S_init), _ptr(g_cumsum), _ptr(A), _ptr(h_chunks), _ptr(ws),
                                      int(ws_bytes), _stream(stream)))


def kda_segment_summary_bwd_workspace(p: gdn_problem, segment_len) -> int:
    n = ctypes.c_size_t(0)
    _check(load().kda_segment_summary_bwd_workspace(ctypes.byref(p), int(segment_len), ctypes.byref(n)))
    return n.value


def kda_segment_summary_bwd(p: gdn_problem, q, k, g_cumsum, beta, A, dO, segment_len, dS_ext, ws,
                            ws_bytes, stream=None):
    _check(load().kda_segment_summary_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(g_cumsum), _ptr(beta),
                                          _ptr(A), _ptr(dO), int(segment_len), _ptr(dS_ext), _ptr(ws),
                                          int(ws_bytes), _stream(stream)))


def kda_segment_merge_bwd(p: gdn_problem, dS_ext, M, nseg, dht, dS_exit, dh0=None, stream=None):
    _check(load().kda_segment_merge_bwd(ctypes.byref(p), _ptr(dS_ext), _ptr(M), int(nseg), _ptr(dht),
                                        _ptr(dS_exit), _ptr(dh0), _stream(stream)))


def kda_segment_merge(p: gdn_problem, S_ext, M, nseg, h0, S_init, ht=None, stream=None):
    _check(load().kda_segment_merge(ctypes.byref(p), _ptr(S_ext), _ptr(M), int(nseg), _ptr(h0),
                                    _ptr(S_init), _ptr(ht), _stream(stream)))


def make_frame_problem(BH, T, D, *, active=0, segment_len=0) -> frame_scan_problem:
    return frame_scan_problem(int(BH), int(T), int(D), int(active), int(segment_len))


def frame_scan_workspace(p: frame_scan_problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load().frame_scan_workspace(ctypes.byref(p), ctypes.byref(n)))
    return n.value


def frame_scan_fwd(p: frame_scan_problem, W_kv, U_kv, W_z, u_z, S0_kv, s0_z, S_kv_all, s_z_all,
                   S_kv_last=None, s_z_last=None, ws=None, ws_bytes=0, stream=None):
    _check(load().frame_scan_fwd(ctypes.byref(p), _ptr(W_kv), _ptr(U_kv), _ptr(W_z), _ptr(u_z),
                                 _ptr(S0_kv), _ptr(s0_z), _ptr(S_kv_all), _ptr(s_z_all),
                                 _ptr(S_kv_last), _ptr(s_z_last), _ptr(ws), int(ws_bytes),
                                 _stream(stream)))

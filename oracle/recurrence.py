"""ctypes front end of the fp64 token-by-token oracle in ``gdn_oracle.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring). Every array is float64
in the padded layout [B, T, H, D] or the packed layout [T, H, D] (B == 1) with
document offsets ``cu``; states are [N, H, K, V].

Definitions followed (restated in ``gdn_oracle.c``):
  * the recurrence S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T,
    o_t = scale S_t^T q_t, a_t = exp(g_t) or 2^(g_t) -- the gated delta
    rule, decay-first for the per-key gate as in
    "state_summary.py" kda_split_state_summary_kernel;
  * the segment summary (S_ext, M) and merge S_{s+1} = M_s S_s + S_ext_s of
    apply_kda_state_summary (coverage-diff page) and SANA's
    _exclusive_prefix_compose;
  * the optional in-kernel input maps of the KDA adapter (coverage-diff page,
    _prepare_kda: use_qk_l2norm_in_kernel with epsilon=1e-6, and
    use_beta_sigmoid_in_kernel; its backward finalize takes q_rstd / k_rstd and
    the beta-sigmoid backward helper): q, k <- x / sqrt(sum_d x_d^2 + 1e-6) and
    beta <- 1 / (1 + exp(-beta)) before the recurrence, and the chain rule of
    those two maps after its reverse mode.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
        ("K", ctypes.c_int64), ("V", ctypes.c_int64),
        ("per_key", ctypes.c_int32), ("use_exp2", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("n_seq", ctypes.c_int64), ("cu", ctypes.POINTER(ctypes.c_int64)),
        ("n_threads", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` with gcc (plain -O2, no arch flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC,
                           "-lm", "-lpthread"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            D = ctypes.POINTER(ctypes.c_double)
            lib.orc_forward.argtypes = [P] + [D] * 8
            lib.orc_backward.argtypes = [P] + [D] * 14
            lib.orc_segment_summary.argtypes = [P, D, D, D, D, ctypes.c_int64, D, D]
            lib.orc_segment_merge.argtypes = [P, D, D, ctypes.c_int64, D, D, D]
            for f in (lib.orc_forward, lib.orc_backward, lib.orc_segment_summary,
                      lib.orc_segment_merge):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


L2_EPS = 1e-6  # the KDA adapter's epsilon for the in-kernel q/k norm


def l2norm(x):
    """x / sqrt(sum_d x_d^2 + 1e-6) along the last axis, and 1 / sqrt(sum_d x_d^2 + 1e-6)."""
    x = np.asarray(x, np.float64)
    rstd = 1.0 / np.sqrt((x * x).sum(-1, keepdims=True) + L2_EPS)
    return x * rstd, rstd


def l2norm_backward(x, dxn):
    """Gradient w.r.t. x of <x / sqrt(|x|^2 + eps), dxn>: rstd (dxn - xn <xn, dxn>)."""
    xn, rstd = l2norm(x)
    return rstd * (dxn - xn * (xn * dxn).sum(-1, keepdims=True))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, np.float64)))


def default_threads() -> int:
    return os.cpu_count() or 1


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _problem(q, v, per_key, use_exp2, scale, cu, n_threads):
    if q.ndim == 3:  # packed [T, H, K]
        if cu is None:
            raise ValueError("packed inputs need document offsets")
        B, T, H, K = 1, q.shape[0], q.shape[1], q.shape[2]
    else:
        B, T, H, K = q.shape
    V = v.shape[-1]
    p = _Problem()
    p.B, p.T, p.H, p.K, p.V = B, T, H, K, V
    p.per_key, p.use_exp2 = int(per_key), int(use_exp2)
    p.scale = float(K ** -0.5 if scale is None else scale)
    p.n_threads = int(n_threads or default_threads())
    keep = None
    if cu is not None:
        keep = np.ascontiguousarray(cu, dtype=np.int64)
        p.n_seq = keep.shape[0] - 1
        p.cu = keep.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    else:
        p.n_seq = B
        p.cu = None
    n_state = p.n_seq if cu is not None else B
    return p, keep, n_state


def forward(q, k, v, g, beta, h0=None, *, scale=None, per_key=False, use_exp2=False,
            cu=None, n_threads=None, want_o=True, want_ht=True, use_qk_l2norm=False,
            beta_sigmoid=False):
    """Return (o, ht). ``g`` is [.., H] (scalar gate) or [.., H, K] (per key).
    ``use_qk_l2norm`` / ``beta_sigmoid``: q, k and beta are raw and mapped first."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    if use_qk_l2norm:
        q, k = l2norm(q)[0], l2norm(k)[0]
    if beta_sigmoid:
        beta = sigmoid(beta)
    p, keep, n_state = _problem(q, v, per_key, use_exp2, scale, cu, n_threads)
    o = np.zeros(v.shape, np.float64) if want_o else None
    ht = np.zeros((n_state, p.H, p.K, p.V), np.float64) if want_ht else None
    rc = _load().orc_forward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                             _ptr(h0), _ptr(o), _ptr(ht))
    assert rc == 0
    del keep
    return o, ht


def backward(q, k, v, g, beta, h0=None, dO=None, dht=None, *, scale=None, per_key=False,
             use_exp2=False, cu=None, n_threads=None, use_qk_l2norm=False, beta_sigmoid=False):
    """Reverse mode of ``forward`` for the loss <o, dO> + <ht, dht>.

    Returns dict(dq, dk, dv, dg, dbeta, dh0); dg is w.r.t. the raw per-token gate; with
    ``use_qk_l2norm`` / ``beta_sigmoid`` dq, dk and dbeta are w.r.t. the raw inputs.
    """
    q, k, v, g, beta, h0, dO, dht = map(_f64, (q, k, v, g, beta, h0, dO, dht))
    q_raw, k_raw, beta_raw = q, k, beta
    if use_qk_l2norm:
        q, k = l2norm(q)[0], l2norm(k)[0]
    if beta_sigmoid:
        beta = sigmoid(beta)
    p, keep, n_state = _problem(q, v, per_key, use_exp2, scale, cu, n_threads)
    out = dict(dq=np.zeros(q.shape), dk=np.zeros(k.shape), dv=np.zeros(v.shape),
               dg=np.zeros(g.shape), dbeta=np.zeros(beta.shape),
               dh0=np.zeros((n_state, p.H, p.K, p.V)))
    rc = _load().orc_backward(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              _ptr(h0), _ptr(dO), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]),
                              _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
                              _ptr(out["dh0"]))
    assert rc == 0
    del keep
    if use_qk_l2norm:
        out["dq"] = l2norm_backward(q_raw, out["dq"])
        out["dk"] = l2norm_backward(k_raw, out["dk"])
    if beta_sigmoid:
        sb = sigmoid(beta_raw)
        out["dbeta"] = out["dbeta"] * sb * (1.0 - sb)
    return out


def segment_summary(k, v, g, beta, seg_len, *, per_key=False, use_exp2=False, n_threads=None):
    """Per segment of ``seg_len`` tokens: S_ext [B,H,nseg,K,V] and M [B,H,nseg,K,K]."""
    k, v, g, beta = map(_f64, (k, v, g, beta))
    p, keep, _ = _problem(k, v, per_key, use_exp2, 1.0, None, n_threads)
    nseg = -(-p.T // seg_len)
    S = np.zeros((p.B, p.H, nseg, p.K, p.V))
    M = np.zeros((p.B, p.H, nseg, p.K, p.K))
    rc = _load().orc_segment_summary(ctypes.byref(p), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     int(seg_len), _ptr(S), _ptr(M))
    assert rc == 0
    return S, M


def segment_merge(S_ext, M, h0=None):
    """S_init [B,H,nseg,K,V] (entry state of each segment) and the final state."""
    S_ext, M, h0 = map(_f64, (S_ext, M, h0))
    B, H, nseg, K, V = S_ext.shape
    p = _Problem()
    p.B, p.T, p.H, p.K, p.V = B, 0, H, K, V
    p.scale, p.n_threads = 1.0, 1
    S_init = np.zeros_like(S_ext)
    ht = np.zeros((B, H, K, V))
    rc = _load().orc_segment_merge(ctypes.byref(p), _ptr(S_ext), _ptr(M), int(nseg), _ptr(h0),
                                   _ptr(S_init), _ptr(ht))
    assert rc == 0
    return S_init, ht


def segment_summary_bwd(q, k, v, g, beta, dO, seg_len, *, scale=None, per_key=False, use_exp2=False,
                        n_threads=None):
    """Backward segment summary: per segment of ``seg_len`` tokens, the gradient of the
    segment's entry state from its own outputs alone (the reverse recurrence started from
    a zero gradient at the segment's exit; "state_summary.py" kda_state_grad_ext_kernel).
    It does not depend on the state, so it is the segment run's dh0 for any entry state.
    Returns dS_ext [B, H, nseg, K, V]."""
    q, k, v, g, beta, dO = map(_f64, (q, k, v, g, beta, dO))
    B, T, H, K = q.shape
    nseg = -(-T // seg_len)
    out = np.zeros((B, H, nseg, K, v.shape[-1]))
    for s in range(nseg):
        sl = lambda x: x[:, s * seg_len:(s + 1) * seg_len]  # noqa: E731
        r = backward(sl(q), sl(k), sl(v), sl(g), sl(beta), None, sl(dO), None, scale=scale,
                     per_key=per_key, use_exp2=use_exp2, n_threads=n_threads)
        out[:, :, s] = r["dh0"]
    return out


def segment_merge_bwd(dS_ext, M, dht=None):
    """Adjoint of the ordered merge: the state gradient flows from the last segment to the
    first through the transposed transfer maps (SANA distributed_scan.py,
    _CPAllGatherMerge.backward; the coverage-diff page's state-summary apply helpers):
        dS_exit[nseg-1] = dht (or 0),  dS_entry[s] = M_s^T dS_exit[s] + dS_ext[s],
        dS_exit[s-1] = dS_entry[s].
    Returns (dS_exit [B,H,nseg,K,V]: the gradient at every segment's exit, dh0 = dS_entry[0])."""
    dS_ext, M, dht = map(_f64, (dS_ext, M, dht))
    B, H, nseg, K, V = dS_ext.shape
    dS_exit = np.zeros_like(dS_ext)
    cur = np.zeros((B, H, K, V)) if dht is None else dht.copy()
    for s in range(nseg - 1, -1, -1):
        dS_exit[:, :, s] = cur
        cur = np.einsum("bhji,bhjv->bhiv", M[:, :, s], cur) + dS_ext[:, :, s]
    return dS_exit, cur

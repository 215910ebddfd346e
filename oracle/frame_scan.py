"""fp64 oracle of the dense per-token transition scan (SANA, distributed_scan.py page).

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain numpy; every array
is float64.

What it computes (the page's local scan and its context-parallel correction,
cp_frame_gdn_scan): for each of BH independent sequences of T positions with
D x D transitions,

  KV state, right multiply:  S_kv[t] = S_kv[t-1] @ W_kv[t] + U_kv[t]
  Z state, left multiply:    s_z[t]  = W_z[t] @ s_z[t-1] + u_z[t]

from S_kv[-1] = S0_kv (or 0) and s_z[-1] = s0_z (or 0). With ``active`` set
(the page's truncate_to_active), positions t >= active take W = I and U = 0,
so the state stops changing after position active-1, and the terminal state
is the state at position active-1.

``scan`` runs that recurrence position by position. ``split_scan`` follows the
page's five steps over segments of one sequence (the page's ranks): a local
scan of every segment from zero, the cumulative transition products of every
segment (right-multiplied for KV, left-multiplied for Z), the composites
(h_ext = the local scan's last state, M = the last cumulative product), the
exclusive prefix composition of the composites (``exclusive_compose``), and the
additive correction S[t] = S_local[t] + S_init @ W_cum[t] (KV),
s[t] = s_local[t] + W_cum[t] @ s_init (Z).
"""
from __future__ import annotations

import numpy as np


def _mask(W_kv, U_kv, W_z, u_z, active):
    """The page's truncate_to_active: W -> I, U -> 0 at positions >= active."""
    if active is None:
        return W_kv, U_kv, W_z, u_z
    T, D = W_kv.shape[1], W_kv.shape[-1]
    if not 1 <= active <= T:
        raise ValueError("active must satisfy 1 <= active <= T")
    W_kv, U_kv, W_z, u_z = (np.array(x, dtype=np.float64, copy=True) for x in (W_kv, U_kv, W_z, u_z))
    eye = np.eye(D)
    W_kv[:, active:] = eye
    U_kv[:, active:] = 0.0
    W_z[:, active:] = eye
    u_z[:, active:] = 0.0
    return W_kv, U_kv, W_z, u_z


def scan(W_kv, U_kv, W_z, u_z, S0_kv=None, s0_z=None, active=None):
    """Position-by-position scan. Shapes: W_kv, U_kv, W_z [BH, T, D, D]; u_z [BH, T, D];
    S0_kv [BH, D, D]; s0_z [BH, D]. Returns (S_kv_all [BH, T, D, D], s_z_all [BH, T, D],
    terminal S_kv [BH, D, D], terminal s_z [BH, D])."""
    W_kv, U_kv, W_z, u_z = (np.asarray(x, dtype=np.float64) for x in (W_kv, U_kv, W_z, u_z))
    W_kv, U_kv, W_z, u_z = _mask(W_kv, U_kv, W_z, u_z, active)
    BH, T, D, _ = W_kv.shape
    S = np.zeros((BH, D, D)) if S0_kv is None else np.array(S0_kv, dtype=np.float64)
    s = np.zeros((BH, D)) if s0_z is None else np.array(s0_z, dtype=np.float64)
    S_all = np.empty((BH, T, D, D))
    s_all = np.empty((BH, T, D))
    for t in range(T):
        S = S @ W_kv[:, t] + U_kv[:, t]
        s = np.einsum("bij,bj->bi", W_z[:, t], s) + u_z[:, t]
        S_all[:, t] = S
        s_all[:, t] = s
    last = T - 1 if active is None else active - 1
    return S_all, s_all, S_all[:, last].copy(), s_all[:, last].copy()


def cumulative_products(W_kv, W_z):
    """W_kv_cum[t] = W_kv[0] @ ... @ W_kv[t] (right); W_z_cum[t] = W_z[t] @ ... @ W_z[0] (left)."""
    BH, T, D, _ = W_kv.shape
    ckv = np.empty_like(W_kv, dtype=np.float64)
    cz = np.empty_like(W_z, dtype=np.float64)
    ckv[:, 0] = W_kv[:, 0]
    cz[:, 0] = W_z[:, 0]
    for t in range(1, T):
        ckv[:, t] = ckv[:, t - 1] @ W_kv[:, t]
        cz[:, t] = W_z[:, t] @ cz[:, t - 1]
    return ckv, cz


def exclusive_compose(h_kv, M_kv, h_z, M_z, S0_kv=None, s0_z=None):
    """Entry state of every segment: S_init_0 = S0 (or 0), then
    S_init_{j+1} = S_init_j @ M_kv_j + h_kv_j (KV) and s_init_{j+1} = M_z_j @ s_init_j + h_z_j (Z).
    h_kv, M_kv, M_z: [nseg, BH, D, D]; h_z: [nseg, BH, D]. Returns the entry states of all
    segments ([nseg, BH, D, D], [nseg, BH, D]) and the state after the last segment."""
    nseg, BH, D, _ = h_kv.shape
    S = np.zeros((BH, D, D)) if S0_kv is None else np.array(S0_kv, dtype=np.float64)
    s = np.zeros((BH, D)) if s0_z is None else np.array(s0_z, dtype=np.float64)
    S_init = np.empty((nseg, BH, D, D))
    s_init = np.empty((nseg, BH, D))
    for j in range(nseg):
        S_init[j] = S
        s_init[j] = s
        S = S @ M_kv[j] + h_kv[j]
        s = np.einsum("bij,bj->bi", M_z[j], s) + h_z[j]
    return S_init, s_init, S, s


def split_scan(W_kv, U_kv, W_z, u_z, segment_len, S0_kv=None, s0_z=None, active=None):
    """The page's context-parallel scan over segments of ``segment_len`` positions of one
    sequence (its ranks), same outputs as ``scan``."""
    W_kv, U_kv, W_z, u_z = (np.asarray(x, dtype=np.float64) for x in (W_kv, U_kv, W_z, u_z))
    W_kv, U_kv, W_z, u_z = _mask(W_kv, U_kv, W_z, u_z, active)
    BH, T, D, _ = W_kv.shape
    bounds = [(a, min(a + segment_len, T)) for a in range(0, T, segment_len)]
    local, cums, comps = [], [], []
    for a, b in bounds:
        # 1. local scan from zero; 2. cumulative products; 3. composites
        S_loc, s_loc, _, _ = scan(W_kv[:, a:b], U_kv[:, a:b], W_z[:, a:b], u_z[:, a:b])
        ckv, cz = cumulative_products(W_kv[:, a:b], W_z[:, a:b])
        local.append((S_loc, s_loc))
        cums.append((ckv, cz))
        comps.append((S_loc[:, -1], ckv[:, -1], s_loc[:, -1], cz[:, -1]))
    # 4. exclusive prefix composition of the composites
    h_kv = np.stack([c[0] for c in comps])
    M_kv = np.stack([c[1] for c in comps])
    h_z = np.stack([c[2] for c in comps])
    M_z = np.stack([c[3] for c in comps])
    S_init, s_init, _, _ = exclusive_compose(h_kv, M_kv, h_z, M_z, S0_kv, s0_z)
    # 5. additive correction
    S_all = np.empty((BH, T, D, D))
    s_all = np.empty((BH, T, D))
    for j, (a, b) in enumerate(bounds):
        S_loc, s_loc = local[j]
        ckv, cz = cums[j]
        S_all[:, a:b] = S_loc + np.einsum("bij,btjk->btik", S_init[j], ckv)
        s_all[:, a:b] = s_loc + np.einsum("btij,bj->bti", cz, s_init[j])
    last = T - 1 if active is None else active - 1
    return S_all, s_all, S_all[:, last].copy(), s_all[:, last].copy()

"""fp64 numpy statement of the 64-token chunk algorithm and its reverse mode.

TEST INFRASTRUCTURE ONLY (see the package docstring).

It takes the steps the pages name, in their order, one chunk at a time:

  1. cumulative log-gate G inside the chunk, restarting at every chunk and
     document start ("per-chunk cumulative log2-gate", state_summary.py
     kda_split_state_summary_kernel argument list; the GDN adapter's forward
     returns it as the g_cumsum slot);
  2. L = strictly-lower(diag(beta) (K K^T (.) Gamma)), Gamma_ij = base^(G_i - G_j)
     (per key channel for the per-key gate), and A = (I + L)^-1 (the UT/WY
     transform; the GDN forward's "A" slot holds this inverse and
     beta stays separate in the "beta_eff" slot);
  3. w = A diag(beta) (K (.) base^G),  u = A diag(beta) V;
  4. state recurrence over chunks: v_new = u - w h;
     h <- Diag(base^G_last) h + (K (.) base^(G_last - G))^T v_new
     (state_summary.py kda_split_state_summary_kernel loop body: residual
     against the entry state, decay of the state by the last cumulative gate,
     then the gated-key update; the KDA stage chunk_fwd_h returns the entry
     states and v_new);
  5. output o = scale ((Q (.) base^G) h + A_qk v_new),
     A_qk = lower-incl(Q K^T (.) Gamma) (chunk_kda_fwd_finalize(qg_scaled,
     aqk, v_new, hidden) on the coverage-diff page).

A partial last chunk uses only its valid rows; G_last is the cumulative gate
at its last valid token ("last_idx = min((chunk+1)*BT, T) - 1" in the
summary kernel). Everything is fp64; matrix products and the triangular
inverse are numpy library calls.
"""
from __future__ import annotations

import math

import numpy as np

CHUNK = 64


def _docs(rows_shape, cu, T):
    """List of (batch, row0, row1) token ranges (rows index the flat layout)."""
    if cu is None:
        B = rows_shape
        return [(b, b * T, b * T + T) for b in range(B)]
    cu = [int(x) for x in cu]
    return [(n, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def _gates(g, per_key, K):
    """[n] or [n, K] -> [n, K] (the scalar gate broadcast over key channels)."""
    return g if per_key else np.repeat(g[:, None], K, axis=1)


def chunk_intermediates(qc, kc, vc, gc, bc, h, scale, per_key, use_exp2):
    """One chunk of n <= 64 valid rows for one head: every intermediate."""
    n, K = kc.shape
    base = 2.0 if use_exp2 else math.e
    G = np.cumsum(gc, axis=0)                      # [n] or [n,K]
    Gk = _gates(G, per_key, K)                     # [n,K]
    Glast = Gk[n - 1]                              # [K]
    diff = Gk[:, None, :] - Gk[None, :, :]         # [i,j,d] = G_id - G_jd
    gam = np.power(base, diff)
    P = np.einsum("id,jd,ijd->ij", kc, kc, gam)    # K K^T (.) Gamma
    L = np.tril(bc[:, None] * P, -1)
    A = np.linalg.inv(np.eye(n) + L)
    Kg = kc * np.power(base, Gk)
    W = A @ (bc[:, None] * Kg)
    U = A @ (bc[:, None] * vc)
    Delta = U - W @ h
    Aqk = np.tril(np.einsum("id,jd,ijd->ij", qc, kc, gam))
    Qg = qc * np.power(base, Gk)
    O = scale * (Qg @ h + Aqk @ Delta)
    kgl = kc * np.power(base, Glast[None, :] - Gk)
    h_next = np.power(base, Glast)[:, None] * h + kgl.T @ Delta
    return dict(G=G, L=L, P=P, A=A, W=W, U=U, Delta=Delta, Aqk=Aqk, Qg=Qg, Kg=Kg, kgl=kgl,
                O=O, h_next=h_next, gam=gam, Glast=Glast)


def forward(q, k, v, g, beta, h0=None, *, scale=None, per_key=False, use_exp2=False, cu=None):
    """Chunk-form forward. Layout [B,T,H,D] or packed [T,H,D] with offsets ``cu``.

    Returns dict with o, ht [N,H,K,V], g_cumsum (shape of g), A [rows..,H,64],
    w, u, v_new (token layout), h_chunks [N,H,NT,K,V] (padded batch) or
    [num_chunks,H,K,V] (packed, chunks in document order).
    """
    packed = q.ndim == 3
    H, K, V = q.shape[-2], q.shape[-1], v.shape[-1]
    T = q.shape[0] if packed else q.shape[1]
    B = 1 if packed else q.shape[0]
    scale = K ** -0.5 if scale is None else scale
    f = lambda x, d: np.asarray(x, np.float64).reshape((-1, H) + ((d,) if d else ()))  # noqa: E731
    qf, kf, vf = f(q, K), f(k, K), f(v, V)
    gf = f(g, K if per_key else 0)
    bf = f(beta, 0)
    rows = qf.shape[0]
    o = np.zeros((rows, H, V))
    gcs = np.zeros_like(gf)
    Aout = np.zeros((rows, H, CHUNK))
    w = np.zeros((rows, H, K))
    u = np.zeros((rows, H, V))
    vnew = np.zeros((rows, H, V))
    docs = _docs(B, cu if packed else None, T)
    N = len(docs)
    NT = -(-T // CHUNK)
    ht = np.zeros((N, H, K, V))
    hch = []
    for n, r0, r1 in docs:
        for hh in range(H):
            h = np.zeros((K, V)) if h0 is None else np.asarray(h0, np.float64)[n, hh].copy()
            chunks = []
            for c0 in range(r0, r1, CHUNK):
                c1 = min(c0 + CHUNK, r1)
                sl = slice(c0, c1)
                chunks.append(h.copy())
                R = chunk_intermediates(qf[sl, hh], kf[sl, hh], vf[sl, hh], gf[sl, hh],
                                        bf[sl, hh], h, scale, per_key, use_exp2)
                o[sl, hh] = R["O"]
                gcs[sl, hh] = R["G"]
                Aout[sl, hh, :c1 - c0] = R["A"]
                w[sl, hh], u[sl, hh], vnew[sl, hh] = R["W"], R["U"], R["Delta"]
                h = R["h_next"]
            ht[n, hh] = h
            hch.append(chunks)
    if packed:
        # document order: all chunks of document 0, then 1, ... ; per head
        per_doc = [hch[n * H:(n + 1) * H] for n in range(N)]
        flat = []
        for n in range(N):
            for c in range(len(per_doc[n][0])):
                flat.append(np.stack([per_doc[n][hh][c] for hh in range(H)]))
        h_chunks = np.stack(flat) if flat else np.zeros((0, H, K, V))
    else:
        h_chunks = np.zeros((N, H, NT, K, V))
        for n in range(N):
            for hh in range(H):
                for c, hc in enumerate(hch[n * H + hh]):
                    h_chunks[n, hh, c] = hc
    shp = lambda x, d: x.reshape(q.shape[:-2] + (H,) + ((d,) if d else ()))  # noqa: E731
    return dict(o=shp(o, V), ht=ht, g_cumsum=gcs.reshape(np.shape(g)), A=shp(Aout, CHUNK),
                w=shp(w, K), u=shp(u, V), v_new=shp(vnew, V), h_chunks=h_chunks)


def backward(q, k, v, g, beta, h0=None, dO=None, dht=None, *, scale=None, per_key=False,
             use_exp2=False, cu=None):
    """Chunk-form reverse mode of ``forward`` for the loss <o,dO> + <ht,dht>.

    The reverse state recurrence per chunk is
        dv_c = kgl_c dh_{c+1} + scale A_qk^T dO_c,
        dh_c = Diag(base^G_last) dh_{c+1} + scale Qg^T dO_c - w_c^T dv_c
    (the dhu stage of the KDA backward on the coverage-diff page, and the
    reverse loop of state_summary.py kda_state_grad_ext_kernel), followed by
    the local adjoint of steps 1-3 and 5 of ``forward``. dg is w.r.t. the raw
    per-token gate (reverse cumulative sum inside the chunk).
    """
    packed = q.ndim == 3
    H, K, V = q.shape[-2], q.shape[-1], v.shape[-1]
    T = q.shape[0] if packed else q.shape[1]
    B = 1 if packed else q.shape[0]
    scale = K ** -0.5 if scale is None else scale
    lnb = math.log(2.0) if use_exp2 else 1.0
    f = lambda x, d: np.asarray(x, np.float64).reshape((-1, H) + ((d,) if d else ()))  # noqa: E731
    qf, kf, vf = f(q, K), f(k, K), f(v, V)
    gf = f(g, K if per_key else 0)
    bf = f(beta, 0)
    dOf = np.zeros_like(vf) if dO is None else f(dO, V)
    rows = qf.shape[0]
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    dgf, dbf = np.zeros_like(gf), np.zeros_like(bf)
    docs = _docs(B, cu if packed else None, T)
    N = len(docs)
    dh0 = np.zeros((N, H, K, V))
    for n, r0, r1 in docs:
        for hh in range(H):
            h = np.zeros((K, V)) if h0 is None else np.asarray(h0, np.float64)[n, hh].copy()
            starts = list(range(r0, r1, CHUNK))
            entry = []
            for c0 in starts:
                c1 = min(c0 + CHUNK, r1)
                entry.append(h.copy())
                R = chunk_intermediates(qf[c0:c1, hh], kf[c0:c1, hh], vf[c0:c1, hh],
                                        gf[c0:c1, hh], bf[c0:c1, hh], h, scale, per_key, use_exp2)
                h = R["h_next"]
            dh = np.zeros((K, V)) if dht is None else np.asarray(dht, np.float64)[n, hh].copy()
            for ci in range(len(starts) - 1, -1, -1):
                c0 = starts[ci]
                c1 = min(c0 + CHUNK, r1)
                sl = slice(c0, c1)
                qc, kc, vc, bc = qf[sl, hh], kf[sl, hh], vf[sl, hh], bf[sl, hh]
                h = entry[ci]
                R = chunk_intermediates(qc, kc, vc, gf[sl, hh], bc, h, scale, per_key, use_exp2)
                do = dOf[sl, hh]
                nrow = c1 - c0
                Gk = _gates(R["G"], per_key, K)
                base = 2.0 if use_exp2 else math.e
                E = np.power(base, R["Glast"])                     # [K]
                dG = np.zeros((nrow, K))
                dGlast = np.zeros(K)
                # h' = E h + kgl^T Delta
                dDelta = R["kgl"] @ dh
                dkgl = R["Delta"] @ dh.T
                dGlast += lnb * np.sum(dh * (E[:, None] * h), axis=1)
                # O = scale (Qg h + Aqk Delta)
                dQg = scale * do @ h.T
                dh_new = E[:, None] * dh + scale * R["Qg"].T @ do
                dAqk = np.tril(scale * do @ R["Delta"].T)
                dDelta += scale * R["Aqk"].T @ do
                # Delta = U - W h
                dU = dDelta
                dW = -dDelta @ h.T
                dh_new -= R["W"].T @ dDelta
                # U = A (b V), W = A (b Kg)
                Y = bc[:, None] * vc
                Z = bc[:, None] * R["Kg"]
                dA = dU @ Y.T + dW @ Z.T
                dY = R["A"].T @ dU
                dZ = R["A"].T @ dW
                dvc = bc[:, None] * dY
                dbc = np.sum(dY * vc, axis=1) + np.sum(dZ * R["Kg"], axis=1)
                dKg = bc[:, None] * dZ
                # A = (I + L)^-1, L = strictly-lower(b P)
                dL = np.tril(-R["A"].T @ dA @ R["A"].T, -1)
                dbc += np.sum(dL * R["P"], axis=1)
                dP = bc[:, None] * dL
                gam = R["gam"]
                # P_ij = sum_d k_id k_jd gam_ijd ; Aqk_ij = sum_d q_id k_jd gam_ijd
                dkc = np.einsum("ij,jd,ijd->id", dP, kc, gam) + np.einsum("ij,id,ijd->jd", dP, kc, gam)
                tP = np.einsum("ij,id,jd,ijd->ijd", dP, kc, kc, gam)
                dqc = np.einsum("ij,jd,ijd->id", dAqk, kc, gam)
                dkc += np.einsum("ij,id,ijd->jd", dAqk, qc, gam)
                tA = np.einsum("ij,id,jd,ijd->ijd", dAqk, qc, kc, gam)
                dG += lnb * (tP.sum(axis=1) - tP.sum(axis=0) + tA.sum(axis=1) - tA.sum(axis=0))
                # Kg = K base^G ; Qg = Q base^G ; kgl = K base^(Glast - G)
                eG = np.power(base, Gk)
                dkc += dKg * eG
                dG += lnb * dKg * R["Kg"]
                dqc += dQg * eG
                dG += lnb * dQg * R["Qg"]
                egl = np.power(base, R["Glast"][None, :] - Gk)
                dkc += dkgl * egl
                t = lnb * dkgl * R["kgl"]
                dGlast += t.sum(axis=0)
                dG -= t
                dG[nrow - 1] += dGlast
                dGc = dG if per_key else dG.sum(axis=1)
                dgc = np.flip(np.cumsum(np.flip(dGc, axis=0), axis=0), axis=0)
                dq[sl, hh], dk[sl, hh], dv[sl, hh] = dqc, dkc, dvc
                dgf[sl, hh], dbf[sl, hh] = dgc, dbc
                dh = dh_new
            dh0[n, hh] = dh
    shp = lambda x, d: x.reshape(q.shape[:-2] + (H,) + ((d,) if d else ()))  # noqa: E731
    return dict(dq=shp(dq, K), dk=shp(dk, K), dv=shp(dv, V),
                dg=dgf.reshape(np.shape(g)), dbeta=dbf.reshape(np.shape(beta)), dh0=dh0)


def transfer_chunks(k, g, beta, *, per_key=False, use_exp2=False):
    """Chunk transfer M_c = Diag(base^G_last) - kgl^T w for one head's chunk list.

    ``k`` [n,K], ``g`` [n] or [n,K], ``beta`` [n] for one chunk; the segment
    transfer is the ordered product of these (kda_state_transition_kernel:
    "diagonal - interaction" composed from the identity).
    """
    n, K = k.shape
    R = chunk_intermediates(np.zeros_like(k), k, np.zeros((n, 1)), g, beta, np.zeros((K, 1)),
                            1.0, per_key, use_exp2)
    base = 2.0 if use_exp2 else math.e
    return np.diag(np.power(base, R["Glast"])) - R["kgl"].T @ R["W"]

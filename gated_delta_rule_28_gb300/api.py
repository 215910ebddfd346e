"""Tensor-level entry points over the C ABI.

These allocate outputs and workspace with PyTorch (device memory and the
current stream are the only things PyTorch provides here), derive the packed
metadata with ``gdn_prepare_varlen`` and call the library. Every arithmetic
step runs in the library's CUDA kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return B.GDN_DTYPE_BF16
    if t.dtype == torch.float32:
        return B.GDN_DTYPE_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


class Varlen:
    """Validated packed-document metadata on the device (int32 offsets and chunk pairs)."""

    def __init__(self, cu_seqlens, total_tokens: int, device):
        cu = np.asarray(cu_seqlens.cpu() if isinstance(cu_seqlens, torch.Tensor) else cu_seqlens,
                        dtype=np.int64)
        idx, n = B.gdn_prepare_varlen(cu, total_tokens)
        self.num_seqs = len(cu) - 1
        self.num_chunks = n
        self.cu = torch.from_numpy(cu.astype(np.int32)).to(device)
        self.chunk_indices = torch.from_numpy(np.ascontiguousarray(idx)).to(device)
        self.chunk_indices_host = idx


def problem_for(q, v, g, *, scale=None, use_exp2=False, varlen: Varlen | None = None,
                use_qk_l2norm=False, segment_len=0, use_beta_sigmoid=False):
    packed = varlen is not None
    if packed:
        if q.ndim != 3:
            raise ValueError("packed inputs must be [T, H, K]")
        Bsz, T, H, K = 1, q.shape[0], q.shape[1], q.shape[2]
    else:
        if q.ndim != 4:
            raise ValueError("inputs must be [B, T, H, K]")
        Bsz, T, H, K = q.shape
    per_key = g.ndim == q.ndim
    return B.make_problem(
        Bsz, T, H, K, v.shape[-1], layout=B.GDN_LAYOUT_TND if packed else B.GDN_LAYOUT_BSND,
        gate_kind=B.GDN_GATE_PER_KEY if per_key else B.GDN_GATE_SCALAR, dtype=_dtype_code(q),
        use_exp2=use_exp2, scale=0.0 if scale is None else scale, use_qk_l2norm=use_qk_l2norm,
        cu_seqlens=varlen.cu if packed else None, num_seqs=varlen.num_seqs if packed else 0,
        chunk_indices=varlen.chunk_indices if packed else None,
        num_chunks=varlen.num_chunks if packed else 0, segment_len=segment_len,
        use_beta_sigmoid=use_beta_sigmoid)


def chunk_gated_delta_rule_fwd(q, k, v, g, beta, *, h0=None, scale=None, use_exp2=False,
                               cu_seqlens=None, varlen=None, output_final_state=True,
                               return_g_cumsum=False, return_A=False, return_h_chunks=False,
                               use_qk_l2norm=False, use_beta_sigmoid=False, segment_len=0, stream=None):
    """Chunked forward; returns a dict with o and, as requested, ht, g_cumsum, A, h_chunks."""
    if cu_seqlens is not None and varlen is None:
        varlen = Varlen(cu_seqlens, q.shape[0], q.device)
    p = problem_for(q, v, g, scale=scale, use_exp2=use_exp2, varlen=varlen,
                    use_qk_l2norm=use_qk_l2norm, segment_len=segment_len,
                    use_beta_sigmoid=use_beta_sigmoid)
    dev = q.device
    out = {"o": torch.empty_like(v)}
    nstate = varlen.num_seqs if varlen is not None else p.B
    if output_final_state:
        out["ht"] = torch.empty((nstate, p.H, p.K, p.V), device=dev, dtype=torch.float32)
    if return_g_cumsum:
        out["g_cumsum"] = torch.empty_like(g, dtype=torch.float32)
    if return_A:
        out["A"] = torch.empty(q.shape[:-1] + (64,), device=dev, dtype=torch.float32)
    if return_h_chunks:
        if varlen is not None:
            shape = (varlen.num_chunks, p.H, p.K, p.V)
        else:
            shape = (p.B, p.H, -(-p.T // 64), p.K, p.V)
        out["h_chunks"] = torch.empty(shape, device=dev, dtype=torch.float32)
    nws = B.gdn_chunk_fwd_workspace(p)
    ws = torch.empty(nws, device=dev, dtype=torch.uint8) if nws else None
    B.gdn_chunk_fwd(p, q, k, v, g, beta, h0, out["o"], out.get("ht"), out.get("g_cumsum"),
                    out.get("A"), out.get("h_chunks"), ws, nws, stream)
    return out


class HostPipeline:
    """Forward calls on inputs that live in pinned host memory, pipelined.

    Each ``submit`` enqueues one call: the host-to-device copies of its inputs (spread over
    ``h2d_streams`` streams, each taking a contiguous share of every tensor), the forward on
    the compute stream, and the device-to-host copies of o and ht on a third stream. Calls
    rotate over ``depth`` device buffer sets, so the copies of one call overlap the kernels
    and copies of its neighbours; a set is refilled only after the kernels that read it and
    the copies out of it have finished (stream events, no host waits). ``synchronize`` waits
    for every call submitted so far. BSND layout, bf16 q/k/v/beta, fp32 scalar gate.
    """

    def __init__(self, Bsz, T, H, K, V, device, *, depth=2, h2d_streams=2, use_exp2=False, scale=None):
        self.p = B.make_problem(Bsz, T, H, K, V, dtype=B.GDN_DTYPE_BF16, use_exp2=use_exp2,
                                scale=0.0 if scale is None else scale)
        self.nws = B.gdn_chunk_fwd_workspace(self.p)
        self.ws = torch.empty(max(self.nws, 1), device=device, dtype=torch.uint8)
        bf, f32 = torch.bfloat16, torch.float32
        self.sets = [dict(q=torch.empty((Bsz, T, H, K), device=device, dtype=bf),
                          k=torch.empty((Bsz, T, H, K), device=device, dtype=bf),
                          v=torch.empty((Bsz, T, H, V), device=device, dtype=bf),
                          g=torch.empty((Bsz, T, H), device=device, dtype=f32),
                          beta=torch.empty((Bsz, T, H), device=device, dtype=bf),
                          o=torch.empty((Bsz, T, H, V), device=device, dtype=bf),
                          ht=torch.empty((Bsz, H, K, V), device=device, dtype=f32)) for _ in range(depth)]
        self.depth = depth
        self.s_in = [torch.cuda.Stream(device=device) for _ in range(h2d_streams)]
        self.s_comp = torch.cuda.Stream(device=device)
        self.s_out = torch.cuda.Stream(device=device)
        self.ev_in = [[torch.cuda.Event() for _ in range(h2d_streams)] for _ in range(depth)]
        self.ev_comp = [torch.cuda.Event() for _ in range(depth)]
        self.ev_out = [torch.cuda.Event() for _ in range(depth)]
        self.n = 0

    def streams(self):
        return self.s_in + [self.s_comp, self.s_out]

    def submit(self, hq, hk, hv, hg, hbeta, ho, hht):
        i = self.n % self.depth
        s = self.sets[i]
        reuse = self.n >= self.depth
        pairs = [(s["q"], hq), (s["k"], hk), (s["v"], hv), (s["g"], hg), (s["beta"], hbeta)]
        ns = len(self.s_in)
        for j, st in enumerate(self.s_in):
            if reuse:
                st.wait_event(self.ev_comp[i])  # the kernels that read this set have finished
            with torch.cuda.stream(st):
                for dst, src in pairs:
                    n = dst.numel()
                    a, b = n * j // ns, n * (j + 1) // ns
                    dst.view(-1)[a:b].copy_(src.view(-1)[a:b], non_blocking=True)
            self.ev_in[i][j].record(st)
        for j in range(ns):
            self.s_comp.wait_event(self.ev_in[i][j])
        if reuse:
            self.s_comp.wait_event(self.ev_out[i])  # the outputs of this set have been copied out
        B.gdn_chunk_fwd(self.p, s["q"], s["k"], s["v"], s["g"], s["beta"], None, s["o"], s["ht"],
                        None, None, None, self.ws, self.nws, self.s_comp.cuda_stream)
        self.ev_comp[i].record(self.s_comp)
        self.s_out.wait_event(self.ev_comp[i])
        with torch.cuda.stream(self.s_out):
            ho.copy_(s["o"], non_blocking=True)
            hht.copy_(s["ht"], non_blocking=True)
        self.ev_out[i].record(self.s_out)
        self.n += 1

    def synchronize(self):
        for st in self.streams():
            st.synchronize()


def chunk_gated_delta_rule_bwd(q, k, v, g_cumsum, beta, A, dO, *, h0=None, dht=None, scale=None,
                               use_exp2=False, cu_seqlens=None, varlen=None, use_qk_l2norm=False,
                               use_beta_sigmoid=False, segment_len=0, stream=None):
    """Chunked backward; returns dq, dk, dv, dbeta, dg (raw gate) and dh0. With the input
    maps on, q, k, beta are the forward's raw inputs and dq, dk, dbeta are w.r.t. them."""
    if cu_seqlens is not None and varlen is None:
        varlen = Varlen(cu_seqlens, q.shape[0], q.device)
    p = problem_for(q, v, g_cumsum, scale=scale, use_exp2=use_exp2, varlen=varlen,
                    use_qk_l2norm=use_qk_l2norm, use_beta_sigmoid=use_beta_sigmoid,
                    segment_len=segment_len)
    nstate = varlen.num_seqs if varlen is not None else p.B
    sshape = ((p.B, p.H, -(-p.T // segment_len), p.K, p.V) if segment_len
              else (nstate, p.H, p.K, p.V))
    out = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
               dbeta=torch.empty_like(beta), dg=torch.empty_like(g_cumsum),
               dh0=torch.empty(sshape, device=q.device, dtype=torch.float32))
    nws = B.gdn_chunk_bwd_workspace(p)
    ws = torch.empty(nws, device=q.device, dtype=torch.uint8) if nws else None
    B.gdn_chunk_bwd(p, q, k, v, g_cumsum, beta, A, dO, h0, dht, out["dq"], out["dk"], out["dv"],
                    out["dg"], out["dbeta"], out["dh0"], ws, nws, stream)
    return out


def segment_summary(k, v, g, beta, segment_len, *, use_exp2=False, use_qk_l2norm=False,
                    use_beta_sigmoid=False, stream=None):
    """(S_ext [B,H,nseg,K,V], M [B,H,nseg,K,K]) for every segment of ``segment_len`` tokens."""
    p = problem_for(k, v, g, use_exp2=use_exp2, use_qk_l2norm=use_qk_l2norm,
                    use_beta_sigmoid=use_beta_sigmoid)
    nseg = -(-p.T // segment_len)
    S = torch.empty((p.B, p.H, nseg, p.K, p.V), device=k.device, dtype=torch.float32)
    M = torch.empty((p.B, p.H, nseg, p.K, p.K), device=k.device, dtype=torch.float32)
    nws = B.kda_segment_summary_workspace(p, segment_len)
    ws = torch.empty(nws, device=k.device, dtype=torch.uint8) if nws else None
    B.kda_segment_summary(p, k, v, g, beta, segment_len, S, M, ws, nws, stream)
    return S, M


def segment_merge(S_ext, M, h0=None, stream=None):
    """(S_init [B,H,nseg,K,V], ht [B,H,K,V]): ordered composition of the summaries."""
    Bsz, H, nseg, K, V = S_ext.shape
    p = B.make_problem(Bsz, nseg * 64, H, K, V, dtype=B.GDN_DTYPE_F32)
    S_init = torch.empty_like(S_ext)
    ht = torch.empty((Bsz, H, K, V), device=S_ext.device, dtype=torch.float32)
    B.kda_segment_merge(p, S_ext, M, nseg, h0, S_init, ht, stream)
    return S_init, ht


def split_forward(q, k, v, g, beta, segment_len, *, h0=None, scale=None, use_exp2=False,
                  use_qk_l2norm=False, use_beta_sigmoid=False, return_h_chunks=False,
                  return_g_cumsum=False, return_A=False, stream=None):
    """Long-sequence forward split across SMs: summaries, merge, corrected run (bf16 with a
    per-key gate: one ``gdn_chunk_fwd_split`` call, whose chunk preparation serves both passes)."""
    maps = dict(use_qk_l2norm=use_qk_l2norm, use_beta_sigmoid=use_beta_sigmoid)
    p = problem_for(q, v, g, scale=scale, use_exp2=use_exp2, **maps)
    if p.dtype == B.GDN_DTYPE_BF16 and p.gate_kind == B.GDN_GATE_PER_KEY:
        dev = q.device
        nseg = -(-p.T // segment_len)
        out = {"o": torch.empty_like(v),
               "ht": torch.empty((p.B, p.H, p.K, p.V), device=dev, dtype=torch.float32),
               "S_ext": torch.empty((p.B, p.H, nseg, p.K, p.V), device=dev, dtype=torch.float32),
               "M": torch.empty((p.B, p.H, nseg, p.K, p.K), device=dev, dtype=torch.float32)}
        out["S_init"] = torch.empty_like(out["S_ext"])
        if return_g_cumsum:
            out["g_cumsum"] = torch.empty_like(g, dtype=torch.float32)
        if return_A:
            out["A"] = torch.empty(q.shape[:-1] + (64,), device=dev, dtype=torch.float32)
        if return_h_chunks:
            out["h_chunks"] = torch.empty((p.B, p.H, -(-p.T // 64), p.K, p.V), device=dev,
                                          dtype=torch.float32)
        nws = B.gdn_chunk_fwd_split_workspace(p, segment_len)
        ws = torch.empty(nws, device=dev, dtype=torch.uint8) if nws else None
        B.gdn_chunk_fwd_split(p, q, k, v, g, beta, h0, segment_len, out["o"], out["ht"], out["S_ext"],
                              out["M"], out["S_init"], out.get("g_cumsum"), out.get("A"),
                              out.get("h_chunks"), ws, nws, stream)
        return out
    S, M = segment_summary(k, v, g, beta, segment_len, use_exp2=use_exp2, stream=stream, **maps)
    S_init, _ = segment_merge(S, M, h0, stream=stream)
    out = chunk_gated_delta_rule_fwd(q, k, v, g, beta, h0=S_init, scale=scale, use_exp2=use_exp2,
                                     segment_len=segment_len, return_h_chunks=return_h_chunks,
                                     return_g_cumsum=return_g_cumsum, return_A=return_A,
                                     stream=stream, **maps)
    out.update(S_ext=S, M=M, S_init=S_init)
    return out


def split_backward(q, k, v, g_cumsum, beta, A, dO, segment_len, S_init, M, *, dht=None, scale=None,
                   use_exp2=False, use_qk_l2norm=False, use_beta_sigmoid=False, stream=None):
    """Backward of ``split_forward``: backward segment summaries (all segments at once), their
    adjoint merge through M^T, then every segment's backward seeded with its exit gradient.
    ``S_init`` and ``M`` are the forward split's. Returns the gradients with dh0 [B,H,K,V]."""
    maps = dict(use_qk_l2norm=use_qk_l2norm, use_beta_sigmoid=use_beta_sigmoid)
    p = problem_for(q, v, g_cumsum, scale=scale, use_exp2=use_exp2, **maps)
    nseg = -(-p.T // segment_len)
    dS_ext = torch.empty((p.B, p.H, nseg, p.K, p.V), device=q.device, dtype=torch.float32)
    nws = B.kda_segment_summary_bwd_workspace(p, segment_len)
    ws = torch.empty(max(nws, 1), device=q.device, dtype=torch.uint8)
    B.kda_segment_summary_bwd(p, q, k, g_cumsum, beta, A, dO, segment_len, dS_ext, ws, nws, stream)
    dS_exit = torch.empty_like(dS_ext)
    dh0 = torch.empty((p.B, p.H, p.K, p.V), device=q.device, dtype=torch.float32)
    mp = B.make_problem(p.B, nseg * 64, p.H, p.K, p.V, dtype=B.GDN_DTYPE_F32)
    B.kda_segment_merge_bwd(mp, dS_ext, M, nseg, dht, dS_exit, dh0, stream)
    out = chunk_gated_delta_rule_bwd(q, k, v, g_cumsum, beta, A, dO, h0=S_init, dht=dS_exit,
                                     scale=scale, use_exp2=use_exp2, segment_len=segment_len,
                                     stream=stream, **maps)
    out.update(dh0=dh0, dS_ext=dS_ext, dS_exit=dS_exit)
    return out


def frame_scan(W_kv, U_kv, W_z, u_z, *, S0_kv=None, s0_z=None, active=0, segment_len=0, stream=None):
    """Dense per-token transition scan (SANA's cp_frame_gdn_scan and its local scan) through
    ``frame_scan_fwd``: S_kv[t] = S_kv[t-1] @ W_kv[t] + U_kv[t], s_z[t] = W_z[t] @ s_z[t-1] + u_z[t],
    fp32 [BH, T, D, D] / [BH, T, D] on the device; ``active`` is truncate_to_active (0: off);
    ``segment_len`` > 0 splits each sequence over the SMs. Returns (S_kv_all, s_z_all,
    S_kv_last, s_z_last)."""
    BH, T, D, _ = W_kv.shape
    p = B.make_frame_problem(BH, T, D, active=active, segment_len=segment_len)
    S_all = torch.empty_like(U_kv)
    z_all = torch.empty_like(u_z)
    S_last = torch.empty((BH, D, D), device=W_kv.device, dtype=torch.float32)
    z_last = torch.empty((BH, D), device=W_kv.device, dtype=torch.float32)
    nbytes = B.frame_scan_workspace(p)
    ws = torch.empty(max(nbytes, 16), device=W_kv.device, dtype=torch.uint8) if nbytes else None
    B.frame_scan_fwd(p, W_kv, U_kv, W_z, u_z, S0_kv, s0_z, S_all, z_all, S_last, z_last,
                     ws, nbytes, stream)
    return S_all, z_all, S_last, z_last

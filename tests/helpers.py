"""Shared helpers for the GPU parity tests: device upload, oracle runs, error measure."""
from __future__ import annotations

import numpy as np

from oracle import chunk_form as CF, recurrence as R

# relative Frobenius bounds: bf16 inputs with fp32 accumulation,
# and fp32 inputs
TOL = {"bf16": 1e-2, "f32": 1e-4}


def rel_frob(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def to_dev(inp, device="cuda"):
    """Upload workload arrays as torch tensors in the kernel dtype."""
    import torch
    dt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32
    t = lambda x, d=dt: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=d)  # noqa: E731
    return dict(q=t(inp.q), k=t(inp.k), v=t(inp.v), beta=t(inp.beta), g=t(inp.g, torch.float32),
                h0=t(inp.h0, torch.float32), dO=t(inp.dO))


def host(x):
    return x.detach().float().cpu().numpy()


def oracle_fwd(inp, scale=None, h0="inp"):
    h0 = inp.h0 if isinstance(h0, str) else h0
    if inp.layout == "TND":
        return R.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, h0, scale=scale, per_key=inp.per_key,
                         use_exp2=inp.use_exp2, cu=inp.cu)
    return R.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, h0, scale=scale, per_key=inp.per_key,
                     use_exp2=inp.use_exp2)


def chunk_ref(inp, scale=None, h0="inp"):
    h0 = inp.h0 if isinstance(h0, str) else h0
    return CF.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, h0, scale=scale, per_key=inp.per_key,
                      use_exp2=inp.use_exp2, cu=inp.cu if inp.layout == "TND" else None)

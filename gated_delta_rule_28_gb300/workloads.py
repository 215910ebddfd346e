"""Seeded synthetic inputs shaped like the pages' workloads.

Input recipe only: random draws, the per-token L2 normalisation of q and k,
sigmoid for beta and -softplus for the log-gate that the workload statements
prescribe, and rounding to the kernel's element type. None of the method's
arithmetic lives here; both the CUDA path and the oracle read these arrays.

Workloads (one numpy generator per workload, ``default_rng(seed)``, seed =
workload number - 1; draws in the fixed order q, k, v, beta, g, h0, dO):

1 ``gdn_tiny_f32``      fp32, B1 H1 T256, g = -softplus(N(0,1)), zero h0.
2 ``gdn_bsnd_bf16``     bf16 BSND [4, 4096, 16, 128], g = -0.1 softplus(N).
3 ``gdn_packed_bf16``   bf16 TND, 32768 tokens, H32; document lengths drawn
                        uniformly in [37, 8192] until they reach 32768, the
                        last one clipped to the remainder.
4 ``kda_long_bf16``     bf16 [1, 65536, 8, 128], per-key base-2 log-gate
                        g = -0.05 softplus(N), 16 segments of 4096.
5 ``gdn_train_bf16``    bf16 [8, 8192, 16, 128], h0 ~ N(0, 0.1^2) fp32,
                        dO ~ N(0, 1).
Shared: q, k ~ N(0,1) normalised per token; v ~ N(0,1); beta = sigmoid(N(0,1)).
Sizes (and the gate scale) can be overridden for smaller or harder parity cases.

``frame_scan_f32`` (``make_frame``): the dense per-token transition scan of SANA's
distributed_scan page, fp32, BH = 16 sequences of T = 4096 positions, D = 64. The page fixes
no sizes and no value law; the recipe is contracting transitions W = 0.9 I + 0.05 N(0,1)/sqrt(D)
(spectral norm about 1, so the states stay bounded over thousands of positions) for both
states, inputs U_kv, u_z ~ N(0, 1/D), initial states ~ N(0, 1); seed 5, draws in the order
W_kv, U_kv, W_z, u_z, S0_kv, s0_z.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

NAMES = {1: "gdn_tiny_f32", 2: "gdn_bsnd_bf16", 3: "gdn_packed_bf16", 4: "kda_long_bf16",
         5: "gdn_train_bf16"}

DEFAULTS = {
    1: dict(B=1, T=256, H=1, dtype="f32", per_key=False, use_exp2=False, gscale=1.0, layout="BSND"),
    2: dict(B=4, T=4096, H=16, dtype="bf16", per_key=False, use_exp2=False, gscale=0.1, layout="BSND"),
    3: dict(B=1, T=32768, H=32, dtype="bf16", per_key=False, use_exp2=False, gscale=0.1, layout="TND"),
    4: dict(B=1, T=65536, H=8, dtype="bf16", per_key=True, use_exp2=True, gscale=0.05, layout="BSND",
            seg_len=4096),
    5: dict(B=8, T=8192, H=16, dtype="bf16", per_key=False, use_exp2=False, gscale=0.1, layout="BSND",
            h0_std=0.1, with_dO=True),
}


@dataclass
class Inputs:
    """The exact values the kernels see (bf16-rounded where dtype is bf16), as float32."""
    name: str
    layout: str
    dtype: str
    per_key: bool
    use_exp2: bool
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    h0: Optional[np.ndarray] = None
    dO: Optional[np.ndarray] = None
    cu: Optional[np.ndarray] = None
    seg_len: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def K(self):
        return self.q.shape[-1]

    @property
    def H(self):
        return self.q.shape[-2]


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x.astype(np.float32)
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def doc_lengths(rng, total: int, lo: int = 37, hi: int = 8192) -> np.ndarray:
    """Uniform integer lengths in [lo, hi] until their sum reaches ``total``; last clipped."""
    lens = []
    acc = 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return np.array(lens, dtype=np.int64)


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _softplus(x):
    return np.logaddexp(0.0, x).astype(np.float32)


def _sigmoid(x):
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def make(config: int, *, B=None, T=None, H=None, seed=None, K=128, V=128, dtype=None,
         with_h0=None, with_dO=None, gscale=None) -> Inputs:
    d = dict(DEFAULTS[config])
    if gscale is not None:
        d["gscale"] = gscale
    B = d["B"] if B is None else B
    T = d["T"] if T is None else T
    H = d["H"] if H is None else H
    dtype = d["dtype"] if dtype is None else dtype
    seed = config - 1 if seed is None else seed
    rng = np.random.default_rng(seed)
    cu = None
    if d["layout"] == "TND":
        lens = doc_lengths(rng, T)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        shape = (T, H)
    else:
        shape = (B, T, H)
    q = _round(_unit_rows(_normal(rng, shape + (K,))), dtype)
    k = _round(_unit_rows(_normal(rng, shape + (K,))), dtype)
    v = _round(_normal(rng, shape + (V,)), dtype)
    beta = _round(_sigmoid(_normal(rng, shape)), dtype)
    gshape = shape + (K,) if d["per_key"] else shape
    g = (-d["gscale"] * _softplus(_normal(rng, gshape))).astype(np.float32)
    want_h0 = ("h0_std" in d) if with_h0 is None else with_h0
    h0 = None
    if want_h0:
        nstate = (len(cu) - 1) if cu is not None else B
        h0 = (d.get("h0_std", 0.1) * _normal(rng, (nstate, H, K, V))).astype(np.float32)
    want_dO = d.get("with_dO", False) if with_dO is None else with_dO
    dO = _round(_normal(rng, shape + (V,)), dtype) if want_dO else None
    return Inputs(name=NAMES[config], layout=d["layout"], dtype=dtype, per_key=d["per_key"],
                  use_exp2=d["use_exp2"], q=q, k=k, v=v, g=g, beta=beta, h0=h0, dO=dO, cu=cu,
                  seg_len=d.get("seg_len", 0), meta=dict(config=config, seed=seed))


FRAME_DEFAULTS = dict(BH=16, T=4096, D=64, seed=5)


@dataclass
class FrameInputs:
    """Inputs of the dense per-token transition scan, float32."""
    W_kv: np.ndarray  # [BH, T, D, D]
    U_kv: np.ndarray  # [BH, T, D, D]
    W_z: np.ndarray   # [BH, T, D, D]
    u_z: np.ndarray   # [BH, T, D]
    S0_kv: np.ndarray  # [BH, D, D]
    s0_z: np.ndarray   # [BH, D]


def make_frame(*, BH=None, T=None, D=None, seed=None) -> FrameInputs:
    d = dict(FRAME_DEFAULTS)
    for k, v in (("BH", BH), ("T", T), ("D", D), ("seed", seed)):
        if v is not None:
            d[k] = v
    BH, T, D = d["BH"], d["T"], d["D"]
    rng = np.random.default_rng(d["seed"])
    eye = np.eye(D, dtype=np.float32)

    def trans():
        w = rng.standard_normal((BH, T, D, D), dtype=np.float32)
        w *= np.float32(0.05 / np.sqrt(D))
        w += np.float32(0.9) * eye
        return w

    W_kv = trans()
    U_kv = rng.standard_normal((BH, T, D, D), dtype=np.float32) * np.float32(1.0 / np.sqrt(D))
    W_z = trans()
    u_z = rng.standard_normal((BH, T, D), dtype=np.float32) * np.float32(1.0 / np.sqrt(D))
    S0 = rng.standard_normal((BH, D, D), dtype=np.float32)
    s0 = rng.standard_normal((BH, D), dtype=np.float32)
    return FrameInputs(W_kv, U_kv, W_z, u_z, S0, s0)

"""GPU parity at the edges of the gate range, on every forward and backward path.

The bf16 scalar-gate tensor-core kernels build the in-chunk decay from products of
per-block gate factors, and the per-key kernels from per-channel factors, so each
path is driven here with:

* the strong gates of the tiny workload (g = -softplus(N), scale 1) in bf16;
* a vanishing decay (g = -1e4: a_t = 0 to fp32 and fp64 alike), where every state
  forgets its past and the output has the closed form o_t = scale beta_t (k_t . q_t) v_t;
* beta = 0 (pure decay), where S_t = (prod_{s<=t} a_s) h0, a closed form too;
* positive log-gates (a_t > 1, a growing state), which the recurrence defines as well.

Closed forms are checked against the GPU directly (not only through the oracle);
everything is also compared with the fp64 oracle at the relative Frobenius bounds of
the other parity tests.
"""
import numpy as np
import pytest

from oracle import recurrence as R
from tests.conftest import cuda_available
from tests.helpers import TOL, host, rel_frob, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not cuda_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_28_gb300 import build
    build.build()


def _inputs(kind, dtype, per_key, T=200, B=2, H=2):
    from gated_delta_rule_28_gb300 import workloads
    cfg = 4 if per_key else 5
    gscale = {"strong": 1.0, "growing": -0.05}.get(kind)
    inp = workloads.make(cfg, B=B, T=T, H=H, dtype=dtype, with_h0=True, with_dO=True, gscale=gscale,
                         seed=21)
    if kind == "vanishing":
        inp.g = np.full_like(inp.g, -1e4)
    if kind == "no_write":
        inp.beta = np.zeros_like(inp.beta)
    return inp


def _fwd(inp):
    from gated_delta_rule_28_gb300 import api, binding
    d = to_dev(inp)
    out = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                         use_exp2=inp.use_exp2, return_g_cumsum=True, return_A=True)
    binding.gdn_device_status()
    return d, out


def _closed_form(inp, kind):
    """o and ht in closed form for the two degenerate gates (fp64)."""
    q, k, v, beta = (x.astype(np.float64) for x in (inp.q, inp.k, inp.v, inp.beta))
    scale = inp.K ** -0.5
    if kind == "vanishing":
        o = scale * beta[..., None] * (k * q).sum(-1, keepdims=True) * v
        ht = beta[:, -1, :, None, None] * k[:, -1, :, :, None] * v[:, -1, :, None, :]
        return o, ht
    # beta = 0: S_t = Diag(prod_{s<=t} a_s) h0
    base = 2.0 if inp.use_exp2 else np.e
    G = np.cumsum(inp.g.astype(np.float64), axis=1)  # [B, T, H] or [B, T, H, K]
    decay = base ** G
    h0 = inp.h0.astype(np.float64)  # [B, H, K, V]
    if inp.per_key:
        o = scale * np.einsum("bthk,bhkv->bthv", q * decay, h0)
        ht = decay[:, -1][..., None] * h0
    else:
        o = scale * decay[..., None] * np.einsum("bthk,bhkv->bthv", q, h0)
        ht = decay[:, -1][..., None, None] * h0
    return o, ht


KINDS = ["strong", "vanishing", "no_write", "growing"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("per_key", [False, True])
def test_forward_at_gate_extremes(kind, dtype, per_key):
    inp = _inputs(kind, dtype, per_key)
    _, out = _fwd(inp)
    o_gpu, ht_gpu = host(out["o"]), host(out["ht"])
    assert np.isfinite(o_gpu).all() and np.isfinite(ht_gpu).all()
    o, ht = R.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, per_key=inp.per_key,
                      use_exp2=inp.use_exp2)
    assert rel_frob(o_gpu, o) <= TOL[dtype], "o"
    assert rel_frob(ht_gpu, ht) <= TOL[dtype], "ht"
    if kind in ("vanishing", "no_write"):
        o_cf, ht_cf = _closed_form(inp, kind)
        assert rel_frob(o_gpu, o_cf) <= TOL[dtype], "o closed form"
        assert rel_frob(ht_gpu, ht_cf) <= TOL[dtype], "ht closed form"
        # the oracle meets the closed form to fp64 rounding
        assert rel_frob(o, o_cf) <= 1e-12 and rel_frob(ht, ht_cf) <= 1e-12


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("per_key", [False, True])
def test_backward_at_gate_extremes(kind, dtype, per_key):
    from gated_delta_rule_28_gb300 import api, binding
    inp = _inputs(kind, dtype, per_key, T=130)
    d, f = _fwd(inp)
    gr = api.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], f["g_cumsum"], d["beta"], f["A"],
                                        d["dO"], h0=d["h0"], use_exp2=inp.use_exp2)
    binding.gdn_device_status()
    want = R.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.dO, None,
                      per_key=inp.per_key, use_exp2=inp.use_exp2)
    rms = lambda x: float(np.sqrt(np.mean(np.square(np.asarray(x, np.float64)))))  # noqa: E731
    typical = rms(want["dq"])  # never zero here: dO != 0 and every state is nonzero
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        got = host(gr[name])
        assert np.isfinite(got).all(), name
        ref = want[name]
        if rms(ref) == 0.0:
            # identically zero in exact arithmetic (beta = 0 gives dk = dv = 0; a = 0 gives
            # dg = 0): the kernels' rounding residue must stay below the bound measured
            # against the size of a typical gradient element
            assert rms(got) <= TOL[dtype] * typical, (name, rms(got), typical)
        else:
            assert rel_frob(got, ref) <= TOL[dtype], (name, rel_frob(got, ref))

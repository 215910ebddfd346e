"""GPU parity of the chunked backward against the CPU fp64 reverse-mode oracle."""
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


def _run(inp, dht=None, cu=None):
    import torch
    from gated_delta_rule_28_gb300 import api, binding
    d = to_dev(inp)
    kw = dict(use_exp2=inp.use_exp2)
    if cu is not None:
        kw["cu_seqlens"] = cu
    f = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                       return_g_cumsum=True, return_A=True, **kw)
    dht_d = None if dht is None else torch.from_numpy(dht).cuda()
    g = api.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], f["g_cumsum"], d["beta"], f["A"],
                                       d["dO"], h0=d["h0"], dht=dht_d, **kw)
    binding.gdn_device_status()
    return {k: host(v) for k, v in g.items()}


def _oracle(inp, dht=None, cu=None):
    kw = dict(per_key=inp.per_key, use_exp2=inp.use_exp2)
    if cu is not None:
        kw["cu"] = cu
    return R.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.dO, dht, **kw)


def _compare(got, want, tol):
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        err = rel_frob(got[name], want[name])
        assert err <= tol, (name, err)


@pytest.mark.parametrize("T", [64, 100, 129])
def test_backward_fp32_small(T):
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(5, B=2, T=T, H=2, dtype="f32")
    dht = np.random.default_rng(3).standard_normal((2, 2, 128, 128)).astype(np.float32)
    _compare(_run(inp, dht), _oracle(inp, dht), TOL["f32"])


@pytest.mark.parametrize("per_key", [False, True])
def test_backward_gate_kinds_bf16(per_key):
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(5, B=1, T=200, H=2, with_h0=True, with_dO=True)
    if per_key:
        rng = np.random.default_rng(4)
        inp.g = (-0.05 * np.logaddexp(0, rng.standard_normal(inp.q.shape))).astype(np.float32)
        inp.per_key, inp.use_exp2 = True, True
    _compare(_run(inp), _oracle(inp), TOL["bf16"])


def test_backward_packed_documents():
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(3, T=700, H=2, with_h0=True, with_dO=True)
    inp.cu = np.array([0, 37, 100, 164, 420, 700], np.int32)
    inp.h0 = (0.1 * np.random.default_rng(6).standard_normal((5, 2, 128, 128))).astype(np.float32)
    _compare(_run(inp, cu=inp.cu), _oracle(inp, cu=inp.cu), TOL["bf16"])


def test_backward_training_workload_slice():
    """Workload 5 recipe (B8 H16, h0 ~ N(0, 0.1^2), dO ~ N(0,1)) on T = 512."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(5, T=512)
    _compare(_run(inp), _oracle(inp), TOL["bf16"])


@pytest.mark.parametrize("use_exp2", [False, True])
def test_backward_bf16_final_state_gradient(use_exp2):
    """Tensor-core path with an upstream final-state gradient, a ragged last chunk and both bases."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(5, B=2, T=130, H=2, with_h0=True, with_dO=True)
    inp.use_exp2 = use_exp2
    dht = np.random.default_rng(7).standard_normal((2, 2, 128, 128)).astype(np.float32)
    _compare(_run(inp, dht), _oracle(inp, dht), TOL["bf16"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("per_key", [False, True])
def test_forward_and_backward_with_input_maps(dtype, per_key):
    """Raw q, k (normalised by the prologue) and raw beta (sigmoid in the prologue):
    o, ht and every gradient w.r.t. the raw inputs against the oracle's chain rule."""
    import torch
    from gated_delta_rule_28_gb300 import api, binding, workloads
    inp = workloads.make(4 if per_key else 5, B=2, T=150, H=2, dtype=dtype, with_h0=True, with_dO=True)
    rng = np.random.default_rng(31)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to("cuda", dt)  # noqa: E731
    q, k = dev(2.0 * rng.standard_normal(inp.q.shape)), dev(0.3 * rng.standard_normal(inp.k.shape))
    braw = dev(rng.standard_normal(inp.beta.shape))
    d = to_dev(inp)
    kw = dict(use_exp2=inp.use_exp2, use_qk_l2norm=True, use_beta_sigmoid=True)
    f = api.chunk_gated_delta_rule_fwd(q, k, d["v"], d["g"], braw, h0=d["h0"], return_g_cumsum=True,
                                       return_A=True, **kw)
    gr = api.chunk_gated_delta_rule_bwd(q, k, d["v"], f["g_cumsum"], braw, f["A"], d["dO"], h0=d["h0"],
                                        **kw)
    binding.gdn_device_status()
    okw = dict(per_key=inp.per_key, use_exp2=inp.use_exp2, use_qk_l2norm=True, beta_sigmoid=True)
    o, ht = R.forward(host(q), host(k), inp.v, inp.g, host(braw), inp.h0, **okw)
    assert rel_frob(host(f["o"]), o) <= TOL[dtype]
    assert rel_frob(host(f["ht"]), ht) <= TOL[dtype]
    want = R.backward(host(q), host(k), inp.v, inp.g, host(braw), inp.h0, inp.dO, None, **okw)
    _compare({n: host(x) for n, x in gr.items()}, want, TOL[dtype])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("per_key", [False, True])
def test_backward_is_bit_reproducible(dtype, per_key):
    """No reduction of the backward depends on thread arrival order: two runs on the same
    inputs give identical bits in every gradient."""
    import torch
    from gated_delta_rule_28_gb300 import api, binding, workloads
    inp = workloads.make(4 if per_key else 5, B=2, T=200, H=2, dtype=dtype, with_h0=True, with_dO=True)
    d = to_dev(inp)
    kw = dict(use_exp2=inp.use_exp2)
    f = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                       return_g_cumsum=True, return_A=True, **kw)
    runs = [api.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], f["g_cumsum"], d["beta"], f["A"],
                                           d["dO"], h0=d["h0"], **kw) for _ in range(2)]
    binding.gdn_device_status()
    for name in runs[0]:
        assert torch.equal(runs[0][name], runs[1][name]), name

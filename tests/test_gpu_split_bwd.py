"""GPU parity of the split backward: backward segment summaries, their adjoint merge
through the transposed transfer maps, and every segment's backward seeded with its
exit gradient, against the fp64 oracle's unsplit reverse mode (through the C ABI)."""
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


def _split(inp, seg_len, dht=None):
    import torch
    from gated_delta_rule_28_gb300 import api, binding
    d = to_dev(inp)
    kw = dict(use_exp2=inp.use_exp2)
    f = api.split_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], seg_len, h0=d["h0"],
                          return_g_cumsum=True, return_A=True, **kw)
    dht_d = None if dht is None else torch.from_numpy(dht).cuda()
    g = api.split_backward(d["q"], d["k"], d["v"], f["g_cumsum"], d["beta"], f["A"], d["dO"], seg_len,
                           f["S_init"], f["M"], dht=dht_d, **kw)
    binding.gdn_device_status()
    return f, g


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("per_key", [False, True])
def test_split_backward_matches_unsplit_oracle(dtype, per_key):
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4 if per_key else 5, B=2, T=700, H=2, dtype=dtype, with_h0=True, with_dO=True)
    if not per_key:
        inp.use_exp2 = False
    seg = 256  # segments of 256, 256 and 188 tokens
    dht = np.random.default_rng(17).standard_normal((2, 2, 128, 128)).astype(np.float32)
    f, g = _split(inp, seg, dht)
    kw = dict(per_key=inp.per_key, use_exp2=inp.use_exp2)
    want = R.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.dO, dht, **kw)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert rel_frob(host(g[name]), want[name]) <= TOL[dtype], (name, rel_frob(host(g[name]), want[name]))
    # the stages on their own: backward summaries against the oracle's, and the adjoint merge
    # against the oracle's merge of the same (GPU) operands
    dS_ext = R.segment_summary_bwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.dO, seg, **kw)
    assert rel_frob(host(g["dS_ext"]), dS_ext) <= TOL[dtype]
    dS_exit, dh0 = R.segment_merge_bwd(host(g["dS_ext"]), host(f["M"]), dht)
    assert rel_frob(host(g["dS_exit"]), dS_exit) <= 1e-5
    assert rel_frob(host(g["dh0"]), dh0) <= 1e-5


def test_split_backward_without_final_state_gradient():
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4, B=1, T=512, H=2, with_h0=True, with_dO=True)
    f, g = _split(inp, 128)
    want = R.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.dO, None, per_key=True,
                      use_exp2=True)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert rel_frob(host(g[name]), want[name]) <= TOL["bf16"], name


def test_full_size_kda_split_backward_whole_tensors():
    """The long-context workload (T 65,536, H8, per-key base-2 gates, 16 segments of 4,096)
    with dO ~ N(0,1): every gradient of the split backward against the unsplit oracle."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4, with_dO=True)
    f, g = _split(inp, inp.seg_len)
    got = {n: host(x) for n, x in g.items() if n in ("dq", "dk", "dv", "dg", "dbeta", "dh0")}
    del f, g
    want = R.backward(inp.q, inp.k, inp.v, inp.g, inp.beta, None, inp.dO, None, per_key=True,
                      use_exp2=True)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert rel_frob(got[name], want[name]) <= TOL["bf16"], name
    for h in range(8):
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            assert rel_frob(got[name][:, :, h], want[name][:, :, h]) <= TOL["bf16"], (h, name)

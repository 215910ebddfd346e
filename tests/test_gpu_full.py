"""Full-size parity of the secondary workloads, in the launch configurations the
benchmark times: the whole problem runs on the GPU and whole output tensors are
compared with the fp64 oracle (run on every host core), and every (document or
batch row, head) slice must meet the bound on its own as well.

* workload 3: 32,768 packed tokens, H32, documents of U[37, 8192] tokens;
* workload 4: per-key base-2 gates, T 65,536, H8, split into 16 segments of 4,096
  (segment summaries, their ordered merge and the corrected scan);
* workload 5: the training step, B8 T8192 H16 with an initial state: forward with
  the saved slots, then the backward.
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


def _status():
    from gated_delta_rule_28_gb300 import binding
    binding.gdn_device_status()


def test_full_size_packed_workload_whole_tensors():
    from gated_delta_rule_28_gb300 import api, workloads
    inp = workloads.make(3)
    d = to_dev(inp)
    vl = api.Varlen(inp.cu, inp.q.shape[0], "cuda")
    out = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], varlen=vl)
    _status()
    ndoc = len(inp.cu) - 1
    assert tuple(out["ht"].shape) == (ndoc, 32, 128, 128)
    o, ht = R.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, cu=inp.cu)
    o_gpu, ht_gpu = host(out["o"]), host(out["ht"])
    assert rel_frob(o_gpu, o) <= TOL["bf16"]
    assert rel_frob(ht_gpu, ht) <= TOL["bf16"]
    for i in range(ndoc):
        a, b = int(inp.cu[i]), int(inp.cu[i + 1])
        for h in range(32):
            assert rel_frob(o_gpu[a:b, h], o[a:b, h]) <= TOL["bf16"], (i, h)
            assert rel_frob(ht_gpu[i, h], ht[i, h]) <= TOL["bf16"], (i, h)


def test_full_size_kda_long_context_split_whole_tensors():
    from gated_delta_rule_28_gb300 import api, workloads
    inp = workloads.make(4)
    assert inp.per_key and inp.use_exp2 and inp.seg_len == 4096
    d = to_dev(inp)
    out = api.split_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], inp.seg_len, use_exp2=True)
    _status()
    o_gpu, ht_gpu = host(out["o"]), host(out["ht"])
    del out, d
    o, ht = R.forward(inp.q, inp.k, inp.v, inp.g, inp.beta, per_key=True, use_exp2=True)
    assert rel_frob(o_gpu, o) <= TOL["bf16"]
    assert rel_frob(ht_gpu, ht) <= TOL["bf16"]
    for h in range(8):
        assert rel_frob(o_gpu[:, :, h], o[:, :, h]) <= TOL["bf16"], h
        assert rel_frob(ht_gpu[0, h], ht[0, h]) <= TOL["bf16"], h


def test_full_size_training_step_backward_whole_batch_rows():
    """Every gradient of the first and the last batch row (all 16 heads, 8,192 tokens)."""
    from gated_delta_rule_28_gb300 import api, workloads
    inp = workloads.make(5)
    d = to_dev(inp)
    f = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                       return_g_cumsum=True, return_A=True)
    gr = api.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], f["g_cumsum"], d["beta"], f["A"],
                                        d["dO"], h0=d["h0"])
    _status()
    for b in (0, 7):
        sl = lambda x: x[b:b + 1]  # noqa: E731
        want = R.backward(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.g), sl(inp.beta),
                          inp.h0[b:b + 1], sl(inp.dO), None)
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            got = host(gr[name][b:b + 1])
            assert rel_frob(got, want[name]) <= TOL["bf16"], (b, name)
            for h in range(16):
                assert rel_frob(got[:, :, h], want[name][:, :, h]) <= TOL["bf16"], (b, h, name)
        got = host(gr["dh0"][b:b + 1])
        assert rel_frob(got, want["dh0"]) <= TOL["bf16"], b
        for h in range(16):
            assert rel_frob(got[0, h], want["dh0"][0, h]) <= TOL["bf16"], (b, h)

"""The forward on inputs in pinned host memory (api.HostPipeline, the end-to-end path the
benchmark times): several calls in flight over rotating device buffer sets, the copies on their
own streams, must give exactly the outputs of the same forward on device tensors, and those
agree with the fp64 oracle."""
import numpy as np
import pytest

from oracle import recurrence as R
from tests.conftest import cuda_available
from tests.helpers import TOL, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not cuda_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_28_gb300 import build
    build.build()


@pytest.mark.parametrize("depth,streams", [(2, 1), (2, 2), (3, 4)])
def test_host_pipeline_matches_device_calls(depth, streams):
    import torch
    from gated_delta_rule_28_gb300 import api, binding, workloads
    Bsz, T, H = 2, 320, 2
    calls = 5  # more calls than buffer sets: every set is refilled while others are in flight
    sets = []
    for i in range(calls):
        inp = workloads.make(2, B=Bsz, T=T, H=H, seed=100 + i)
        pin = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(dt).pin_memory()  # noqa: E731
        sets.append(dict(inp=inp, q=pin(inp.q, torch.bfloat16), k=pin(inp.k, torch.bfloat16),
                         v=pin(inp.v, torch.bfloat16), g=pin(inp.g, torch.float32),
                         beta=pin(inp.beta, torch.bfloat16),
                         o=torch.empty((Bsz, T, H, 128), dtype=torch.bfloat16).pin_memory(),
                         ht=torch.empty((Bsz, H, 128, 128), dtype=torch.float32).pin_memory()))
    pipe = api.HostPipeline(Bsz, T, H, 128, 128, torch.device("cuda", 0), depth=depth, h2d_streams=streams)
    for s in sets:
        pipe.submit(s["q"], s["k"], s["v"], s["g"], s["beta"], s["o"], s["ht"])
    pipe.synchronize()
    binding.gdn_device_status()
    for i, s in enumerate(sets):
        dev = {n: s[n].cuda() for n in ("q", "k", "v", "g", "beta")}
        ref = api.chunk_gated_delta_rule_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"])
        torch.cuda.synchronize()
        assert torch.equal(s["o"], ref["o"].cpu()), i
        assert torch.equal(s["ht"], ref["ht"].cpu()), i
    # and the first call against the oracle
    inp = sets[0]["inp"]
    o_ref, ht_ref = R.forward(inp.q, inp.k, inp.v, inp.g, inp.beta)
    assert rel_frob(sets[0]["o"].float().numpy(), o_ref) <= TOL["bf16"]
    assert rel_frob(sets[0]["ht"].numpy(), ht_ref) <= TOL["bf16"]

"""The backward entry point that allocates nothing (gdn_chunk_bwd_noalloc).

It serves callers that cannot allocate device memory (runtimes that plan all
device buffers at start-up, plugin hosts that hand over only input and
output buffers): its scratch is an array built into the library. Here it is
called through the C ABI twice in a row, on two different inputs, and each
result is compared with gdn_chunk_bwd (caller workspace) on the same input.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

from tests.conftest import cuda_available

pytestmark = pytest.mark.gpu


def _problem_and_inputs(seed, T=200, H=2):
    import torch
    from gated_delta_rule_28_gb300 import api, workloads
    inp = workloads.make(5, B=1, T=T, H=H, seed=seed)
    dev = "cuda"
    t = lambda x, dt=torch.bfloat16: torch.from_numpy(np.ascontiguousarray(x)).to(dev, dt)  # noqa: E731
    d = dict(q=t(inp.q), k=t(inp.k), v=t(inp.v), beta=t(inp.beta), dO=t(inp.dO),
             g=t(inp.g, torch.float32), h0=t(inp.h0, torch.float32))
    d["dht"] = t(np.random.default_rng(seed + 7).standard_normal(inp.h0.shape).astype(np.float32),
                 torch.float32)
    f = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                       return_g_cumsum=True, return_A=True)
    d["g_cumsum"], d["A"] = f["g_cumsum"], f["A"]
    p = api.problem_for(d["q"], d["v"], d["g"])
    return p, d


def _outputs(d):
    import torch
    return dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]), dv=torch.empty_like(d["v"]),
                dg=torch.empty_like(d["g"]), dbeta=torch.empty_like(d["beta"]),
                dh0=torch.empty_like(d["h0"]))


def _args(d, o):
    return (d["q"], d["k"], d["v"], d["g_cumsum"], d["beta"], d["A"], d["dO"], d["h0"], d["dht"],
            o["dq"], o["dk"], o["dv"], o["dg"], o["dbeta"], o["dh0"])


def test_backward_without_allocation_matches_workspace_backward():
    """Same kernels, same inputs, and no step of the backward depends on the order in
    which threads arrive (no atomics): every output must be bit-identical. A stale or
    aliased word of the built-in scratch would show up as a difference."""
    if not cuda_available():
        pytest.skip("no CUDA device")
    import torch
    from gated_delta_rule_28_gb300 import binding as B, build
    build.build()
    for seed in (11, 12):  # two calls in a row, different inputs
        p, d = _problem_and_inputs(seed)
        ref = _outputs(d)
        nws = B.gdn_chunk_bwd_workspace(p)
        assert 0 < nws <= B.GDN_NOALLOC_SCRATCH_BYTES
        ws = torch.empty(nws, device="cuda", dtype=torch.uint8)
        B.gdn_chunk_bwd(p, *_args(d, ref), ws, nws)
        got = _outputs(d)
        B.gdn_chunk_bwd_noalloc(p, *_args(d, got))
        B.gdn_device_status()
        for name in ref:
            assert torch.equal(got[name], ref[name]), (seed, name)


def test_backward_without_allocation_rejects_oversized_problems():
    if not cuda_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_28_gb300 import binding as B, build
    build.build()
    # B8 T8192 H16 needs far more than the built-in scratch; rejected before any device work
    p = B.make_problem(8, 8192, 16)
    assert B.gdn_chunk_bwd_workspace(p) > B.GDN_NOALLOC_SCRATCH_BYTES
    a = 1 << 20
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_bwd_noalloc(p, *([a] * 15))
    assert e.value.status == B.GDN_ERR_WORKSPACE
    assert "built-in array" in str(e.value)

"""GPU parity of the dense per-token transition scan (``frame_scan_fwd``, SANA's
distributed_scan page) against the fp64 oracle (``oracle/frame_scan.py``), through the C ABI.

fp32 throughout, so the bar is the fp32 tolerance: relative Frobenius error <= 1e-4 over each
whole output (every position's KV and Z states, and the terminal states).
"""
import numpy as np
import pytest

from oracle import frame_scan as F
from tests.conftest import cuda_available
from tests.helpers import rel_frob

pytestmark = pytest.mark.gpu
TOL32 = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not cuda_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_28_gb300 import build
    build.build()


def _run(f, *, with_init=True, active=0, segment_len=0):
    import torch
    from gated_delta_rule_28_gb300 import api, binding
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = api.frame_scan(dev(f.W_kv), dev(f.U_kv), dev(f.W_z), dev(f.u_z),
                         S0_kv=dev(f.S0_kv) if with_init else None, s0_z=dev(f.s0_z) if with_init else None,
                         active=active, segment_len=segment_len)
    torch.cuda.synchronize()
    assert binding.gdn_device_status() == 0
    return [o.cpu().numpy().astype(np.float64) for o in out]


def _ref(f, *, with_init=True, active=0):
    return F.scan(f.W_kv, f.U_kv, f.W_z, f.u_z, f.S0_kv if with_init else None,
                  f.s0_z if with_init else None, active=active or None)


def _check(got, ref):
    for name, x, y in zip(("S_kv_all", "s_z_all", "S_kv_last", "s_z_last"), got, ref):
        err = rel_frob(x, y)
        assert err <= TOL32, f"{name}: relative Frobenius error {err:.3e}"


@pytest.mark.parametrize("D", [32, 64])
@pytest.mark.parametrize("with_init", [True, False])
def test_one_pass(D, with_init):
    from gated_delta_rule_28_gb300 import workloads
    f = workloads.make_frame(BH=3, T=37, D=D, seed=11)
    _check(_run(f, with_init=with_init), _ref(f, with_init=with_init))


@pytest.mark.parametrize("D", [32, 64])
@pytest.mark.parametrize("seg", [1, 5, 16, 36, 37, 100])
def test_split_over_segments(D, seg):
    # ragged last segments, one position per segment, and segments longer than the sequence
    from gated_delta_rule_28_gb300 import workloads
    f = workloads.make_frame(BH=2, T=37, D=D, seed=12)
    _check(_run(f, segment_len=seg), _ref(f))


@pytest.mark.parametrize("seg", [0, 8])
@pytest.mark.parametrize("active", [1, 20, 24, 37])
def test_truncate_to_active(seg, active):
    from gated_delta_rule_28_gb300 import workloads
    f = workloads.make_frame(BH=2, T=37, D=64, seed=13)
    got = _run(f, active=active, segment_len=seg)
    _check(got, _ref(f, active=active))
    # the held positions repeat the state of position active-1: exactly inside its segment;
    # later segments start from the merged entry state (S_init M + h with M = I, h = 0 for a
    # segment past active, but the segment holding active-1 composes its own map), equal up to
    # fp32 rounding
    end = 37 if seg == 0 else min(37, -(-active // seg) * seg)
    for t in range(active, 37):
        for x in got[:2]:
            if t < end:
                np.testing.assert_array_equal(x[:, t], x[:, active - 1])
            else:
                np.testing.assert_allclose(x[:, t], x[:, active - 1], rtol=1e-5, atol=1e-6)


def test_single_position_and_sequence():
    from gated_delta_rule_28_gb300 import workloads
    f = workloads.make_frame(BH=1, T=1, D=64, seed=14)
    _check(_run(f), _ref(f))
    _check(_run(f, segment_len=4), _ref(f))


def test_full_size_split_on_sampled_sequences():
    # the bench's workload (16 sequences x 4096 positions, D = 64) in the bench's launch
    # configuration (segments of 256 positions); two whole sequences against the oracle
    from gated_delta_rule_28_gb300 import workloads
    f = workloads.make_frame()
    got = _run(f, segment_len=256)
    for bh in (0, 15):
        sub = workloads.FrameInputs(*(x[bh:bh + 1] for x in (f.W_kv, f.U_kv, f.W_z, f.u_z, f.S0_kv, f.s0_z)))
        ref = _ref(sub)
        _check([g[bh:bh + 1] for g in got], ref)


def test_invalid_arguments_are_rejected():
    import torch
    from gated_delta_rule_28_gb300 import binding as B
    x = torch.zeros(64 * 64 * 4, device="cuda")
    with pytest.raises(B.GdnError) as e:
        B.frame_scan_fwd(B.make_frame_problem(1, 4, 48), x, x, x, x, None, None, x, x)
    assert e.value.status == B.GDN_ERR_UNSUPPORTED
    with pytest.raises(B.GdnError) as e:
        B.frame_scan_fwd(B.make_frame_problem(1, 4, 64, active=5), x, x, x, x, None, None, x, x)
    assert e.value.status == B.GDN_ERR_INVALID_ARGUMENT
    with pytest.raises(B.GdnError) as e:
        B.frame_scan_fwd(B.make_frame_problem(1, 4, 64), x, None, x, x, None, None, x, x)
    assert e.value.status == B.GDN_ERR_INVALID_ARGUMENT
    p = B.make_frame_problem(2, 64, 64, segment_len=8)
    need = B.frame_scan_workspace(p)
    assert need == 2 * 8 * (4 * 64 * 64 + 2 * 64) * 4
    with pytest.raises(B.GdnError) as e:
        B.frame_scan_fwd(p, x, x, x, x, None, None, x, x, ws=x, ws_bytes=need - 16)
    assert e.value.status == B.GDN_ERR_WORKSPACE

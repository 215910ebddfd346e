"""GPU parity of the chunked forward, segment summary, merge and correction
against the CPU oracle, through the C ABI (relative Frobenius error: 1e-2 for
bf16 inputs with fp32 accumulation, 1e-4 for fp32 inputs)."""
import numpy as np
import pytest

from oracle import chunk_form as CF, recurrence as R
from tests.conftest import cuda_available
from tests.helpers import TOL, chunk_ref, host, oracle_fwd, rel_frob, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not cuda_available():
        pytest.skip("no CUDA device")
    from gated_delta_rule_28_gb300 import build
    build.build()


def _api():
    from gated_delta_rule_28_gb300 import api
    return api


def _status():
    from gated_delta_rule_28_gb300 import binding
    binding.gdn_device_status()


def test_tiny_fp32_workload_all_slots():
    """Workload 1: fp32 B1 H1 T256, zero initial state; every output slot."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(1)
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                            return_g_cumsum=True, return_A=True,
                                            return_h_chunks=True)
    _status()
    o, ht = oracle_fwd(inp)
    c = chunk_ref(inp)
    assert rel_frob(host(out["o"]), o) <= TOL["f32"]
    assert rel_frob(host(out["ht"]), ht) <= TOL["f32"]
    assert rel_frob(host(out["g_cumsum"]), c["g_cumsum"]) <= 1e-6
    assert rel_frob(host(out["A"]), c["A"]) <= TOL["f32"]
    assert rel_frob(host(out["h_chunks"]), c["h_chunks"]) <= TOL["f32"]


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129, 200])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_lengths_with_initial_state(T, dtype):
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(2, B=2, T=T, H=3, dtype=dtype, with_h0=True)
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                            return_A=True, return_g_cumsum=True)
    _status()
    o, ht = oracle_fwd(inp)
    c = chunk_ref(inp)
    assert rel_frob(host(out["o"]), o) <= TOL[dtype]
    assert rel_frob(host(out["ht"]), ht) <= TOL[dtype]
    assert rel_frob(host(out["A"]), c["A"]) <= TOL[dtype]
    assert rel_frob(host(out["g_cumsum"]), c["g_cumsum"]) <= 1e-6


def test_empty_sequence_passes_state_through():
    import torch
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(2, B=2, T=0, H=2, with_h0=True)
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"])
    torch.cuda.synchronize()
    assert out["o"].numel() == 0
    np.testing.assert_array_equal(host(out["ht"]), inp.h0)


@pytest.mark.parametrize("per_key,use_exp2", [(True, True), (False, True), (True, False)])
def test_gate_kinds_and_bases(per_key, use_exp2):
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4 if per_key else 2, B=2, T=150, H=2, with_h0=True)
    inp.use_exp2 = use_exp2
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                            use_exp2=use_exp2, return_A=True)
    _status()
    o, ht = oracle_fwd(inp)
    assert rel_frob(host(out["o"]), o) <= TOL["bf16"]
    assert rel_frob(host(out["ht"]), ht) <= TOL["bf16"]
    assert rel_frob(host(out["A"]), chunk_ref(inp)["A"]) <= TOL["bf16"]


def test_packed_documents_small():
    """Workload 3 recipe at 3000 tokens: lengths below, at and above 64, per-document state."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(3, T=3000, H=4, with_h0=True)
    inp.cu = np.array([0, 1, 38, 101, 165, 229, 1000, 2049, 2113, 3000], np.int32)
    inp.h0 = np.random.default_rng(5).standard_normal((9, 4, 128, 128)).astype(np.float32) * 0.1
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                            cu_seqlens=inp.cu, return_h_chunks=True,
                                            return_g_cumsum=True, return_A=True)
    _status()
    o, ht = oracle_fwd(inp)
    c = chunk_ref(inp)
    assert rel_frob(host(out["o"]), o) <= TOL["bf16"]
    assert rel_frob(host(out["ht"]), ht) <= TOL["bf16"]
    assert rel_frob(host(out["h_chunks"]), c["h_chunks"]) <= TOL["bf16"]
    assert rel_frob(host(out["g_cumsum"]), c["g_cumsum"]) <= 1e-6
    assert rel_frob(host(out["A"]), c["A"]) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_packed_documents_per_key_gate(dtype):
    """Per-key base-2 gates on packed documents of 1 to 887 tokens with per-document states:
    every slot of the forward (the per-key tensor-core path for bf16)."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4, B=1, T=1500, H=2, dtype=dtype)
    q, k, v, beta, g = (x[0] for x in (inp.q, inp.k, inp.v, inp.beta, inp.g))
    inp.q, inp.k, inp.v, inp.beta, inp.g = q, k, v, beta, g
    inp.layout = "TND"
    inp.cu = np.array([0, 1, 64, 129, 613, 1500], np.int32)
    inp.h0 = np.random.default_rng(8).standard_normal((5, 2, 128, 128)).astype(np.float32) * 0.1
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                            cu_seqlens=inp.cu, use_exp2=True, return_h_chunks=True,
                                            return_g_cumsum=True, return_A=True)
    _status()
    o, ht = oracle_fwd(inp)
    c = chunk_ref(inp)
    assert rel_frob(host(out["o"]), o) <= TOL[dtype]
    assert rel_frob(host(out["ht"]), ht) <= TOL[dtype]
    assert rel_frob(host(out["h_chunks"]), c["h_chunks"]) <= TOL[dtype]
    assert rel_frob(host(out["g_cumsum"]), c["g_cumsum"]) <= 1e-6
    assert rel_frob(host(out["A"]), c["A"]) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("per_key", [False, True])
def test_in_kernel_l2_norm(dtype, per_key):
    """use_qk_l2norm: q, k normalised in-kernel as x / sqrt(sum x^2 + 1e-6); raw q and k
    of very different sizes, a ragged last chunk and an initial state."""
    import torch
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4 if per_key else 2, B=2, T=130, H=2, dtype=dtype, with_h0=True)
    rng = np.random.default_rng(9)
    qr = (rng.standard_normal(inp.q.shape) * 3).astype(np.float32)
    kr = (rng.standard_normal(inp.k.shape) * 0.5).astype(np.float32)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    qd, kd = torch.from_numpy(qr).to("cuda", dt), torch.from_numpy(kr).to("cuda", dt)
    qr, kr = host(qd), host(kd)  # the values the kernel reads
    nrm = lambda x: x / np.sqrt((x.astype(np.float64) ** 2).sum(-1, keepdims=True) + 1e-6)  # noqa: E731
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(qd, kd, d["v"], d["g"], d["beta"], h0=d["h0"],
                                            use_exp2=inp.use_exp2, use_qk_l2norm=True)
    _status()
    o, ht = R.forward(nrm(qr), nrm(kr), inp.v, inp.g, inp.beta, inp.h0, per_key=per_key,
                      use_exp2=inp.use_exp2)
    assert rel_frob(host(out["o"]), o) <= TOL[dtype]
    assert rel_frob(host(out["ht"]), ht) <= TOL[dtype]


@pytest.mark.parametrize("per_key", [True, False])
def test_segment_summary_merge_and_correction(per_key):
    """Split a sequence into segments: (S_ext, M) per segment against the oracle,
    their merge against the unsplit state, the corrected run against the
    unsplit scan (workload 4 recipe at 1024 tokens, 4 segments of 256)."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4 if per_key else 2, B=2, T=1000, H=2, with_h0=True)
    inp.use_exp2 = per_key
    d = to_dev(inp)
    api = _api()
    S, M = api.segment_summary(d["k"], d["v"], d["g"], d["beta"], 256, use_exp2=inp.use_exp2)
    _status()
    So, Mo = R.segment_summary(inp.k, inp.v, inp.g, inp.beta, 256, per_key=per_key,
                               use_exp2=inp.use_exp2)
    assert rel_frob(host(S), So) <= TOL["bf16"]
    assert rel_frob(host(M), Mo) <= TOL["bf16"]
    S_init, ht = api.segment_merge(S, M, d["h0"])
    Si_o, ht_o = R.segment_merge(host(S), host(M), inp.h0)  # merge alone, same operands
    assert rel_frob(host(S_init), Si_o) <= 1e-5
    assert rel_frob(host(ht), ht_o) <= 1e-5
    out = api.split_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], 256, h0=d["h0"],
                            use_exp2=inp.use_exp2, return_h_chunks=True)
    _status()
    o, ht_ref = oracle_fwd(inp)
    c = chunk_ref(inp)
    assert rel_frob(host(out["o"]), o) <= TOL["bf16"]
    assert rel_frob(host(out["ht"]), ht_ref) <= TOL["bf16"]
    assert rel_frob(host(out["h_chunks"]), c["h_chunks"]) <= TOL["bf16"]
    whole = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                           use_exp2=inp.use_exp2, return_h_chunks=True)
    # both runs round their contraction operands to bf16: they agree to the bf16 bound
    assert rel_frob(host(out["h_chunks"]), host(whole["h_chunks"])) <= TOL["bf16"]
    assert rel_frob(host(out["o"]), host(whole["o"])) <= TOL["bf16"]


def test_one_call_split_forward_equals_the_three_calls():
    """gdn_chunk_fwd_split (bf16, per-key gate) runs the chunk preparation once for both passes;
    kda_segment_summary, kda_segment_merge and gdn_chunk_fwd with segment_len run the same
    kernels on the same operands, so every output agrees bit for bit (ragged last segment,
    initial state, every optional slot)."""
    import torch
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4, B=2, T=1000, H=2, with_h0=True)
    d = to_dev(inp)
    api = _api()
    kw = dict(use_exp2=True, return_h_chunks=True, return_g_cumsum=True, return_A=True)
    one = api.split_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], 256, h0=d["h0"], **kw)
    S, M = api.segment_summary(d["k"], d["v"], d["g"], d["beta"], 256, use_exp2=True)
    S_init, _ = api.segment_merge(S, M, d["h0"])
    three = api.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=S_init,
                                           segment_len=256, **kw)
    _status()
    three.update(S_ext=S, M=M, S_init=S_init)
    for name in ("o", "ht", "g_cumsum", "A", "h_chunks", "S_ext", "M", "S_init"):
        assert torch.equal(one[name], three[name]), name


def test_split_forward_with_input_maps():
    """Segment summaries, merge and corrected run on raw k (normalised) and raw beta
    (sigmoid), per-key base-2 gates, against the unsplit oracle on the mapped inputs."""
    import torch
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(4, B=1, T=700, H=2, with_h0=True)
    rng = np.random.default_rng(33)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to("cuda", torch.bfloat16)  # noqa: E731
    q, k, braw = dev(rng.standard_normal(inp.q.shape)), dev(rng.standard_normal(inp.k.shape)), \
        dev(rng.standard_normal(inp.beta.shape))
    d = to_dev(inp)
    out = _api().split_forward(q, k, d["v"], d["g"], braw, 256, h0=d["h0"], use_exp2=True,
                               use_qk_l2norm=True, use_beta_sigmoid=True)
    _status()
    o, ht = R.forward(host(q), host(k), inp.v, inp.g, host(braw), inp.h0, per_key=True, use_exp2=True,
                      use_qk_l2norm=True, beta_sigmoid=True)
    assert rel_frob(host(out["o"]), o) <= TOL["bf16"]
    assert rel_frob(host(out["ht"]), ht) <= TOL["bf16"]


def test_device_metadata_check_flags_bad_offsets():
    """Non-increasing device offsets are skipped and reported, not faulted on."""
    import torch
    from gated_delta_rule_28_gb300 import binding as B, workloads
    inp = workloads.make(3, T=300, H=2)
    d = to_dev(inp)
    cu_bad = torch.tensor([0, 100, 90, 300], dtype=torch.int32, device="cuda")  # 90 < 100
    idx = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    p = B.make_problem(1, 300, 2, layout=B.GDN_LAYOUT_TND, cu_seqlens=cu_bad, num_seqs=3,
                       chunk_indices=idx, num_chunks=5)
    o = torch.zeros_like(d["v"])
    nws = B.gdn_chunk_fwd_workspace(p)
    ws = torch.empty(max(nws, 1), device="cuda", dtype=torch.uint8)
    B.gdn_chunk_fwd(p, d["q"], d["k"], d["v"], d["g"], d["beta"], None, o, ws=ws, ws_bytes=nws)
    with pytest.raises(B.GdnError) as e:
        B.gdn_device_status()
    assert e.value.status == B.GDN_ERR_DEVICE_CHECK
    B.gdn_device_status()  # cleared


def test_bounded_wait_runs_out_and_reports_timeout():
    """The kernels' bounded mbarrier wait, on a barrier nothing arrives on, gives up,
    raises the timeout flag and returns; the context stays usable afterwards."""
    import torch
    from gated_delta_rule_28_gb300 import binding as B, workloads
    B.gdn_device_status()  # start clean
    B.gdn_selftest_wait_timeout(64)
    with pytest.raises(B.GdnError) as e:
        B.gdn_device_status()
    assert e.value.status == B.GDN_ERR_TIMEOUT
    B.gdn_device_status()  # read and cleared
    inp = workloads.make(2, B=1, T=100, H=1)
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"])
    torch.cuda.synchronize()
    _status()
    o, _ = oracle_fwd(inp)
    assert rel_frob(host(out["o"]), o) <= TOL["bf16"]


def test_full_size_bsnd_workload_whole_tensors():
    """Workload 2 at full size (B4 T4096 H16) in the benchmark's launch: the whole o and
    ht against the oracle (all 64 (batch, head) pairs, the oracle on every host core)."""
    from gated_delta_rule_28_gb300 import workloads
    inp = workloads.make(2)
    d = to_dev(inp)
    out = _api().chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"])
    _status()
    o, ht = R.forward(inp.q, inp.k, inp.v, inp.g, inp.beta)
    assert rel_frob(host(out["o"]), o) <= TOL["bf16"]
    assert rel_frob(host(out["ht"]), ht) <= TOL["bf16"]
    # and no (batch, head) pair hides behind the others: each one meets the bound alone
    o_gpu, ht_gpu = host(out["o"]), host(out["ht"])
    for b in range(4):
        for h in range(16):
            assert rel_frob(o_gpu[b, :, h], o[b, :, h]) <= TOL["bf16"], (b, h)
            assert rel_frob(ht_gpu[b, h], ht[b, h]) <= TOL["bf16"], (b, h)

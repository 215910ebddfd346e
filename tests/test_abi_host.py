"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol the header declares, derives packed metadata bit-exactly and
rejects contract violations before any launch."""
import os
import re

import numpy as np
import pytest

from gated_delta_rule_28_gb300 import binding as B
from gated_delta_rule_28_gb300 import build as gbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(B.EXPORTS) <= set(names) | {"gdn_last_error"}
    for name in names:
        assert hasattr(lib, name), name


def _restated_chunk_indices(offsets):
    # the pages' rule: for every document in order, one (document, chunk) pair
    # per 64-token chunk, ceil(len / 64) chunks
    pairs = []
    for n in range(len(offsets) - 1):
        length = offsets[n + 1] - offsets[n]
        for c in range(-(-length // 64)):
            pairs.append((n, c))
    return np.array(pairs, dtype=np.int32).reshape(-1, 2)


@pytest.mark.parametrize("lens", [[1], [64], [65], [37, 63, 64, 65, 128, 129, 8192], list(range(1, 200, 7))])
def test_prepare_varlen_bit_exact(lib, lens):
    cu = np.concatenate([[0], np.cumsum(lens)])
    idx, n = B.gdn_prepare_varlen(cu, int(cu[-1]))
    want = _restated_chunk_indices(cu.tolist())
    assert n == len(want)
    assert np.array_equal(idx, want)


def test_prepare_varlen_for_the_packed_workload(lib):
    from gated_delta_rule_28_gb300 import workloads
    rng = np.random.default_rng(2)
    lens = workloads.doc_lengths(rng, 32768)
    assert lens.sum() == 32768 and lens[:-1].min() >= 37 and lens.max() <= 8192
    cu = np.concatenate([[0], np.cumsum(lens)])
    idx, n = B.gdn_prepare_varlen(cu, 32768)
    assert np.array_equal(idx, _restated_chunk_indices(cu.tolist()))


@pytest.mark.parametrize("cu,total", [([0], 0), ([1, 5], 5), ([0, 5, 5, 9], 9), ([0, 6, 4, 9], 9),
                                      ([0, 5, 9], 10)])
def test_prepare_varlen_rejects_bad_offsets(lib, cu, total):
    with pytest.raises(B.GdnError) as e:
        B.gdn_prepare_varlen(cu, total)
    assert e.value.status == B.GDN_ERR_INVALID_ARGUMENT


def _fake(n=16):
    return 1 << 20  # a 16-byte-aligned non-null address; never dereferenced


@pytest.mark.parametrize("field,value,status", [
    ("K", 64, B.GDN_ERR_UNSUPPORTED), ("V", 96, B.GDN_ERR_UNSUPPORTED),
    ("chunk_size", 32, B.GDN_ERR_UNSUPPORTED), ("layout", 7, B.GDN_ERR_INVALID_ARGUMENT),
    ("gate_kind", 3, B.GDN_ERR_INVALID_ARGUMENT), ("dtype", 5, B.GDN_ERR_INVALID_ARGUMENT),
    ("B", 0, B.GDN_ERR_INVALID_ARGUMENT), ("T", -1, B.GDN_ERR_INVALID_ARGUMENT),
    ("segment_len", 100, B.GDN_ERR_INVALID_ARGUMENT), ("use_exp2", 2, B.GDN_ERR_INVALID_ARGUMENT),
])
def test_problem_validation(lib, field, value, status):
    p = B.make_problem(2, 256, 4)
    setattr(p, field, value)
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_fwd_workspace(p)
    assert e.value.status == status
    assert B.gdn_last_error()


def test_packed_layout_contract(lib):
    p = B.make_problem(2, 256, 4, layout=B.GDN_LAYOUT_TND)
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_fwd_workspace(p)
    assert "batch size one" in str(e.value)
    p = B.make_problem(1, 256, 4, layout=B.GDN_LAYOUT_TND)  # no offsets
    with pytest.raises(B.GdnError):
        B.gdn_chunk_fwd_workspace(p)


def test_null_and_misaligned_pointers_are_rejected_before_launch(lib):
    p = B.make_problem(1, 128, 2)
    a = _fake()
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_fwd(p, a, a, a, a, a, None, None, stream=0)  # o missing
    assert e.value.status == B.GDN_ERR_INVALID_ARGUMENT and "o must not be NULL" in str(e.value)
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_fwd(p, a + 2, a, a, a, a, None, a, stream=0)
    assert "aligned" in str(e.value)
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_bwd(p, a, a, a, a, a, a, a, None, None, a, a, a, a, a, None, None, 0, stream=0)
    assert e.value.status == B.GDN_ERR_WORKSPACE


def test_backward_workspace_size(lib):
    slots = 2 * 3 * 3  # B * H * ceil(130/64)
    # fp32: entry states and exit-state gradients (fp32 [K, V] per chunk and head), dv_new per token
    p = B.make_problem(2, 130, 3, dtype=B.GDN_DTYPE_F32)
    assert B.gdn_chunk_bwd_workspace(p) >= 2 * slots * 128 * 128 * 4 + 2 * 130 * 3 * 128 * 4
    # bf16 scalar gate: the same as bf16 tiles (K x V per chunk and head, 64 x V for dv_new), then
    # the forward's X pair (128 x 64 bf16) and gate table (9 x 64 fp32) per chunk and head
    p = B.make_problem(2, 130, 3)
    assert B.gdn_chunk_bwd_workspace(p) >= (2 * slots * 128 * 128 * 2 + slots * 64 * 128 * 2
                                            + slots * 128 * 64 * 2 + slots * 9 * 64 * 4)


@pytest.mark.parametrize("polls", [0, (1 << 20) + 1])
def test_wait_selftest_rejects_a_budget_out_of_range(lib, polls):
    with pytest.raises(B.GdnError) as e:
        B.gdn_selftest_wait_timeout(polls, 0)
    assert e.value.status == B.GDN_ERR_INVALID_ARGUMENT


def test_frame_scan_contract_checks(lib):
    # validation runs before any device work: fake aligned addresses are never touched
    fake = 4096
    p = B.make_frame_problem(2, 64, 64, segment_len=8)
    need = B.frame_scan_workspace(p)
    assert need == 2 * 8 * (4 * 64 * 64 + 2 * 64) * 4
    assert B.frame_scan_workspace(B.make_frame_problem(2, 64, 64)) == 0
    assert B.frame_scan_workspace(B.make_frame_problem(2, 64, 32, segment_len=64)) == 0
    cases = [
        (B.make_frame_problem(1, 4, 48), [fake] * 4, B.GDN_ERR_UNSUPPORTED),
        (B.make_frame_problem(1, 4, 64, active=5), [fake] * 4, B.GDN_ERR_INVALID_ARGUMENT),
        (B.make_frame_problem(1, 4, 64, active=-1), [fake] * 4, B.GDN_ERR_INVALID_ARGUMENT),
        (B.make_frame_problem(0, 4, 64), [fake] * 4, B.GDN_ERR_INVALID_ARGUMENT),
        (B.make_frame_problem(1, 4, 64, segment_len=-2), [fake] * 4, B.GDN_ERR_INVALID_ARGUMENT),
        (B.make_frame_problem(1, 4, 64), [fake, None, fake, fake], B.GDN_ERR_INVALID_ARGUMENT),
        (B.make_frame_problem(1, 4, 64), [fake, fake + 4, fake, fake], B.GDN_ERR_INVALID_ARGUMENT),
    ]
    for prob, (w, u, wz, uz), status in cases:
        with pytest.raises(B.GdnError) as e:
            B.frame_scan_fwd(prob, w, u, wz, uz, None, None, fake, fake, stream=0)
        assert e.value.status == status
    with pytest.raises(B.GdnError) as e:
        B.frame_scan_fwd(p, fake, fake, fake, fake, None, None, fake, fake, ws=fake, ws_bytes=need - 16,
                         stream=0)
    assert e.value.status == B.GDN_ERR_WORKSPACE


def test_one_call_split_forward_contract_checks(lib):
    # bf16 inputs with a per-key gate, BSND: the workspace is the preparation's blobs
    fake = 4096
    pk = dict(gate_kind=B.GDN_GATE_PER_KEY, use_exp2=True)
    p = B.make_problem(2, 1000, 3, **pk)
    need = B.gdn_chunk_fwd_split_workspace(p, 256)
    assert need >= 2 * 16 * 3 * 64 * 128 * 2 * 4  # per chunk and head: w, u and the scaled operands
    assert need == B.gdn_chunk_fwd_split_workspace(p, 512)  # one blob per chunk, whatever the split
    for prob, seg, status in [
        (B.make_problem(2, 1000, 3), 256, B.GDN_ERR_UNSUPPORTED),  # scalar gate
        (B.make_problem(2, 1000, 3, dtype=B.GDN_DTYPE_F32, **pk), 256, B.GDN_ERR_UNSUPPORTED),
        (p, 100, B.GDN_ERR_INVALID_ARGUMENT),
        (p, 0, B.GDN_ERR_INVALID_ARGUMENT),
    ]:
        with pytest.raises(B.GdnError) as e:
            B.gdn_chunk_fwd_split_workspace(prob, seg)
        assert e.value.status == status
    # pointers and the workspace are checked before any device work
    a = [fake] * 5
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_fwd_split(p, *a, None, 256, fake, None, fake, None, fake, ws=fake, ws_bytes=need, stream=0)
    assert e.value.status == B.GDN_ERR_INVALID_ARGUMENT and "M must not be NULL" in str(e.value)
    with pytest.raises(B.GdnError) as e:
        B.gdn_chunk_fwd_split(p, *a, None, 256, fake, None, fake, fake, fake, ws=fake, ws_bytes=need - 16,
                              stream=0)
    assert e.value.status == B.GDN_ERR_WORKSPACE

"""The C-ABI library builds, loads, exports every declared symbol, and rejects bad
arguments on the host before any launch (no GPU needed)."""

import os
import re

import pytest

import quantized_routed_expert_03_gb300 as qre
from quantized_routed_expert_03_gb300 import build as qbuild

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qre.load_library()


def _declared():
    with open(os.path.join(ROOT, "include", "qre.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"QRE_API\s+[\w\s\*]+?\b(qre_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(qre.EXPORTS) == names


def test_version_and_status_strings(lib):
    assert qre.qre_version() >= 100
    assert qre.qre_status_string(qre.QRE_ERR_WORKSPACE) == "QRE_ERR_WORKSPACE"


SHAPE = dict(hidden=4096, inter=2048, n_experts=288, top_k=8, group=128)


def _shape(**kw):
    d = dict(SHAPE)
    d.update(kw)
    return qre.make_shape(d["hidden"], d["inter"], d["n_experts"], d["top_k"], d["group"])


def _status(fn):
    with pytest.raises(qre.QreError) as ei:
        fn()
    return ei.value.status, str(ei.value)


@pytest.mark.parametrize("kw,code", [
    (dict(group=96), qre.QRE_ERR_UNSUPPORTED),
    (dict(hidden=4160), qre.QRE_ERR_UNSUPPORTED),
    (dict(hidden=8192), qre.QRE_ERR_UNSUPPORTED),
    (dict(inter=100), qre.QRE_ERR_UNSUPPORTED),
    (dict(n_experts=2048), qre.QRE_ERR_UNSUPPORTED),
    (dict(top_k=17, n_experts=32), qre.QRE_ERR_UNSUPPORTED),
    (dict(top_k=9, n_experts=8), qre.QRE_ERR_INVALID_ARG),
    (dict(top_k=0), qre.QRE_ERR_INVALID_ARG),
])
def test_bad_shapes_rejected(lib, kw, code):
    st, msg = _status(lambda: qre.qre_workspace_size(_shape(**kw), 4))
    assert st == code, msg


def test_workspace_size_grows_with_tokens(lib):
    s = _shape()
    sizes = [qre.qre_workspace_size(s, T) for T in (1, 8, 8192)]
    assert all(b % 256 == 0 and b > 0 for b in sizes)
    assert sizes[0] < sizes[1]
    st, _ = _status(lambda: qre.qre_workspace_size(s, 8193))   # T*k > 65536
    assert st == qre.QRE_ERR_UNSUPPORTED
    st, _ = _status(lambda: qre.qre_workspace_size(s, -1))
    assert st == qre.QRE_ERR_INVALID_ARG


A = 0x10000            # an aligned fake address: never dereferenced, the checks fail first
MIS = 0x10008          # 8-byte aligned only


def test_route_argument_errors(lib):
    s = _shape()
    ws = qre.qre_workspace_size(s, 4)
    st, msg = _status(lambda: qre.qre_route(s, 4, None, A, None, A, A, A, ws, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "x_bf16" in msg
    st, msg = _status(lambda: qre.qre_route(s, 4, MIS, A, None, A, A, A, ws, stream=0))
    assert st == qre.QRE_ERR_MISALIGNED and "x_bf16" in msg
    st, msg = _status(lambda: qre.qre_route(s, 4, A, A, MIS, A, A, A, ws, stream=0))
    assert st == qre.QRE_ERR_MISALIGNED and "bias" in msg
    st, msg = _status(lambda: qre.qre_route(s, 4, A, A, None, A, A, A, 16, stream=0))
    assert st == qre.QRE_ERR_WORKSPACE
    assert "needs" in qre.qre_last_error()


def test_other_argument_errors(lib):
    s = _shape()
    st, msg = _status(lambda: qre.qre_dispatch(s, 4, A, A, A, None, A, A, A, A, 1 << 20, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "perm" in msg
    st, msg = _status(lambda: qre.qre_expert_ffn(s, 4, A, A, A, A, A, MIS, A, A, 1 << 20, stream=0))
    assert st == qre.QRE_ERR_MISALIGNED and "n_active" in msg
    st, msg = _status(lambda: qre.qre_combine(s, 4, A, A, A, None, None, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "y_f32" in msg
    st, msg = _status(lambda: qre.qre_quantize(4, 100, 32, A, A, A, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG
    st, msg = _status(lambda: qre.qre_quantize(4, 128, 48, A, A, A, stream=0))
    assert st == qre.QRE_ERR_UNSUPPORTED
    st, msg = _status(lambda: qre.qre_quantize_gate_up(24, 128, 32, A, A, A, A, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG
    # the tiled storage needs whole 128-row blocks and 64-column stages
    st, msg = _status(lambda: qre.qre_quantize(100, 128, 32, A, A, A, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "128" in msg
    st, msg = _status(lambda: qre.qre_quantize(128, 96, 32, A, A, A, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG
    st, msg = _status(lambda: qre.qre_quantize_gate_up(96, 128, 32, A, A, A, A, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG


def test_empty_calls_launch_nothing(lib):
    s = _shape()
    qre.qre_route(s, 0, None, None, None, None, None, None, 0, stream=0)
    qre.qre_dispatch(s, 0, None, None, None, None, None, None, None, None, 0, stream=0)
    qre.qre_expert_ffn(s, 0, None, None, None, None, None, None, None, None, 0, stream=0)
    qre.qre_combine(s, 0, None, None, None, None, None, stream=0)
    qre.qre_quantize(0, 128, 32, None, None, None, stream=0)


def test_validate_slots_host_checks(lib):
    s = _shape(n_experts=2, top_k=1)
    good = (A, A + 4096, A + 8192, A + 12288, 0)
    st, msg = _status(lambda: qre.qre_validate_slots(s, qre.slot_array([good, good, (A, None, A, A, 0)])))
    assert st == qre.QRE_ERR_INVALID_ARG and "slot 2" in msg and "s_gate_up" in msg
    st, msg = _status(lambda: qre.qre_validate_slots(s, qre.slot_array([good, (A, A, MIS, A, 0), good])))
    assert st == qre.QRE_ERR_MISALIGNED and "slot 1" in msg
    st, msg = _status(lambda: qre.qre_validate_slots(s, qre.slot_array([(A, A, A, A, 3), good, good])))
    assert st == qre.QRE_ERR_INVALID_ARG and "tier" in msg
    arr = qre.slot_array([good, good, good])
    arr[1].reserved = 5
    st, msg = _status(lambda: qre.qre_validate_slots(s, arr))
    assert st == qre.QRE_ERR_INVALID_ARG and "reserved" in msg


def test_cache_argument_errors(lib):
    s = _shape()
    st, msg = _status(lambda: qre.qre_cache_update(s, 0, 0.995, A, A, A, A, A, A, A, A, A, A, 8, stream=0))
    assert st == qre.QRE_ERR_UNSUPPORTED and "n_slots" in msg
    st, msg = _status(lambda: qre.qre_cache_update(s, 8, 1.5, A, A, A, A, A, A, A, A, A, A, 8, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "decay" in msg
    st, msg = _status(lambda: qre.qre_cache_update(s, 8, 0.995, A, A, A, A, MIS, A, A, A, A, A, 8, stream=0))
    assert st == qre.QRE_ERR_MISALIGNED and "slot_expert" in msg
    st, msg = _status(lambda: qre.qre_cache_copy(s, A, None, A, A, 8, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "slot_mem" in msg


def test_wait_test_hook_checks_its_arguments(lib):
    st, msg = _status(lambda: qre.qre_debug_wait_test(2_000_000_000, 0))
    assert st == qre.QRE_ERR_INVALID_ARG and "wait_limit_ns" in msg
    st, msg = _status(lambda: qre.qre_debug_wait_test(0, 500_000_000))
    assert st == qre.QRE_ERR_INVALID_ARG and "stall_ns" in msg
    qre.qre_debug_wait_test(0, 0)      # the defaults


def test_split_expert_ffn_checks_its_arguments(lib):
    shape = _shape()
    n = qre.qre_shared_workspace_size(shape, 1)
    assert n >= 2 * 8 * 2048 * 2
    assert qre.qre_shared_workspace_size(shape, 4096) >= 4096 * (4096 + 2048) * 2
    st, msg = _status(lambda: qre.qre_expert_ffn_shared(shape, 1, None, 16, 16, 16, n, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "x_bf16" in msg
    st, msg = _status(lambda: qre.qre_expert_ffn_routed(shape, 1, 16, 16, None, 16, 16, 16, 16, 16, 1 << 30,
                                                        stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "offsets" in msg


def test_stage_experts_checks_its_arguments(lib):
    shape = _shape(n_experts=4, top_k=2)
    table = qre.slot_array([(16, 16, 16, 16, 0)] * 5)
    bad_staging = qre.slot_array([(16, 16, 16, 16, 1)])
    st, msg = _status(lambda: qre.qre_stage_experts(shape, table, bad_staging, 16, 16, stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "staging slot 0" in msg
    bad_table = qre.slot_array([(16, 16, 16, 16, 0)] * 4 + [(0, 16, 16, 16, 1)])
    st, msg = _status(lambda: qre.qre_stage_experts(shape, bad_table, qre.slot_array([(16, 16, 16, 16, 0)]), 16, 16,
                                                    stream=0))
    assert st == qre.QRE_ERR_INVALID_ARG and "slot 4" in msg

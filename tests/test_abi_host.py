"""The C-ABI library on the host: loading, exports and argument checks.

No case here reaches a kernel: every call either fails host validation
before any CUDA call, or (only where no GPU is present) stops at the
device check with MOE_ERR_NO_DEVICE.
"""
import ctypes
import os
import re

import pytest
import torch

from tests.conftest import ROOT

lib_mod = pytest.importorskip("sparse_expert_gb300._lib")
lib = lib_mod.lib

OK, INVALID, UNSUPPORTED, CUDA, TIMEOUT, BAD_INDEX, WORKSPACE, NO_DEVICE = range(8)
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")
FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: every use below fails validation first
NULL = None


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
        assert n in lib_mod.SIGNATURES, f"{n} has no binding"


def test_only_the_abi_is_exported():
    out = os.popen(f"nm -D --defined-only {lib_mod.LIB_PATH}").read()
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == declared_functions()


def test_abi_version_matches_header():
    m = re.search(r"#define MOE_GB300_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.moe_abi_version() == int(m.group(1))


def test_status_strings():
    for s in range(8):
        assert lib.moe_status_string(s)
    assert lib.moe_status_string(99) == b"unknown status"


def _last():
    return lib.moe_last_error().decode()


def test_route_argument_errors():
    assert lib.moe_route_topk(FAKE, -1, 8, 2, 1, FAKE, FAKE, NULL) == INVALID
    assert lib.moe_route_topk(FAKE, 10, 0, 1, 1, FAKE, FAKE, NULL) == UNSUPPORTED
    assert lib.moe_route_topk(FAKE, 10, 1025, 2, 1, FAKE, FAKE, NULL) == UNSUPPORTED
    assert lib.moe_route_topk(FAKE, 10, 8, 9, 1, FAKE, FAKE, NULL) == UNSUPPORTED
    assert lib.moe_route_topk(FAKE, 10, 64, 33, 1, FAKE, FAKE, NULL) == UNSUPPORTED
    assert lib.moe_route_topk(FAKE, 10, 8, 0, 1, FAKE, FAKE, NULL) == UNSUPPORTED
    assert lib.moe_route_topk(FAKE, 1 << 29, 8, 4, 1, FAKE, FAKE, NULL) == UNSUPPORTED  # T*k = 2^31
    assert "2^31" in _last()
    assert lib.moe_route_topk(NULL, 10, 8, 2, 1, FAKE, FAKE, NULL) == INVALID
    assert lib.moe_route_topk(FAKE, 10, 8, 2, 1, NULL, FAKE, NULL) == INVALID
    # T == 0 needs no pointers and no device
    assert lib.moe_route_topk(NULL, 0, 8, 2, 1, NULL, NULL, NULL) == OK


def test_dispatch_argument_errors():
    need = lib.moe_dispatch_workspace_bytes(100, 8, 2)
    assert need > 256
    args = dict(T=100, E=8, k=2)
    base = [FAKE, FAKE, args["T"], args["E"], args["k"], FAKE, FAKE, FAKE, FAKE, FAKE]
    assert lib.moe_dispatch_scan(*base, NULL, need, NULL) == WORKSPACE
    assert lib.moe_dispatch_scan(*base, FAKE, need - 1, NULL) == WORKSPACE
    assert lib.moe_dispatch_scan(*base, ctypes.c_void_p((1 << 20) + 8), need, NULL) == WORKSPACE  # misaligned
    assert lib.moe_dispatch_scan(FAKE, NULL, 100, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, NULL) == INVALID
    assert lib.moe_dispatch_scan(NULL, FAKE, 100, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, NULL) == INVALID
    assert lib.moe_dispatch_scan(FAKE, FAKE, 100, 8, 2, NULL, FAKE, FAKE, FAKE, FAKE, FAKE, need, NULL) == INVALID
    assert lib.moe_dispatch_scan(FAKE, FAKE, 100, 8, 9, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need, NULL) == UNSUPPORTED


def test_workspace_sizes_grow_with_the_problem():
    a = lib.moe_dispatch_workspace_bytes(1000, 64, 8)
    b = lib.moe_dispatch_workspace_bytes(2000, 64, 8)
    c = lib.moe_dispatch_workspace_bytes(2000, 128, 8)
    assert 0 < a < b < c
    assert lib.moe_dispatch_workspace_bytes(-1, 8, 2) == 0
    assert lib.moe_grouped_swiglu_workspace_bytes() == 256
    assert lib.moe_packed_weight_bytes(384, 6144, 1792) == 3 * 384 * 6144 * 1792 * 2
    assert lib.moe_packed_weight_bytes(0, 64, 64) == 0


def test_forward_layout_is_aligned_and_disjoint():
    T, E, k, d, f = 16384, 384, 8, 6144, 1792
    lay = lib_mod.ForwardLayout()
    assert lib.moe_forward_layout(T, E, k, d, f, ctypes.byref(lay)) == OK
    P = T * k
    spans = {
        "counts": (lay.counts, E * 4), "offsets": (lay.offsets, (E + 1) * 4),
        "topk_idx": (lay.topk_idx, P * 4), "topk_w": (lay.topk_w, P * 4),
        "src_token": (lay.src_token, P * 4), "dest_row": (lay.dest_row, P * 4), "row_w": (lay.row_w, P * 4),
        "x_perm": (lay.x_perm, P * d * 2), "h": (lay.h, P * f * 2), "y": (lay.y, P * d * 2),
    }
    ivals = sorted(spans.values())
    for (o1, n1), (o2, _) in zip(ivals, ivals[1:]):
        assert o1 + n1 <= o2
    for name, (o, n) in spans.items():
        assert o % 256 == 0, name
        assert o + n <= lay.total
    assert lay.counts >= 256          # after the status header
    assert lay.total == lib.moe_forward_workspace_bytes(T, E, k, d, f)
    assert lib.moe_forward_layout(T, E, k, 100, f, ctypes.byref(lay)) == UNSUPPORTED


def test_gemm_and_forward_argument_errors():
    ws = lib.moe_grouped_swiglu_workspace_bytes()
    # d, f not multiples of 64
    assert lib.moe_grouped_swiglu(FAKE, FAKE, 512, 8, 96, 64, FAKE, NULL, FAKE, FAKE, FAKE, ws, NULL) == UNSUPPORTED
    assert lib.moe_grouped_swiglu(FAKE, FAKE, 512, 8, 128, 100, FAKE, NULL, FAKE, FAKE, FAKE, ws, NULL) == UNSUPPORTED
    assert lib.moe_grouped_swiglu(FAKE, FAKE, -1, 8, 128, 64, FAKE, NULL, FAKE, FAKE, FAKE, ws, NULL) == UNSUPPORTED
    assert lib.moe_grouped_swiglu(FAKE, NULL, 512, 8, 128, 64, FAKE, NULL, FAKE, FAKE, FAKE, ws, NULL) == INVALID
    assert lib.moe_grouped_swiglu(FAKE, FAKE, 512, 8, 128, 64, FAKE, NULL, FAKE, FAKE, FAKE, 255, NULL) == WORKSPACE
    assert lib.moe_grouped_swiglu(ctypes.c_void_p((1 << 20) + 2), FAKE, 512, 8, 128, 64, FAKE, NULL, FAKE, FAKE,
                                  FAKE, ws, NULL) == INVALID  # x_perm not 16-byte aligned
    need = lib.moe_forward_workspace_bytes(256, 8, 2, 128, 64)
    fwd = [FAKE, FAKE, FAKE, 256, 128, 8, 2, 64, 1, FAKE, NULL, NULL]
    assert lib.moe_forward(*fwd, FAKE, need - 256, NULL) == WORKSPACE
    assert lib.moe_forward(*fwd, NULL, need, NULL) == WORKSPACE
    bad = list(fwd)
    bad[2] = NULL
    assert lib.moe_forward(*bad, FAKE, need, NULL) == INVALID
    bad = list(fwd)
    bad[4] = 130
    assert lib.moe_forward(*bad, FAKE, need, NULL) == UNSUPPORTED
    assert lib.moe_combine(FAKE, FAKE, NULL, 10, 2, 12, FAKE, NULL) == UNSUPPORTED  # d % 8
    assert lib.moe_permute(FAKE, 10, 16, FAKE, 0, FAKE, NULL) == INVALID
    assert lib.moe_pack_weights(FAKE, FAKE, NULL, 8, 128, 64, FAKE, NULL) == INVALID
    assert lib.moe_read_device_status(NULL, NULL, NULL) == INVALID


def test_timed_entry_points_reject_a_null_event_array():
    need = lib.moe_forward_workspace_bytes(256, 8, 2, 128, 64)
    fwd = [FAKE, FAKE, FAKE, 256, 128, 8, 2, 64, 1, FAKE, FAKE, need, NULL]
    for name in ("moe_forward_timed", "moe_forward_gathered_timed", "moe_forward_fp8_timed"):
        assert getattr(lib, name)(*fwd, NULL) == INVALID, name
        assert "events" in _last(), name
    bwd = [FAKE, FAKE, FAKE, FAKE, 256, 128, 8, 2, 64, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
           lib.moe_backward_workspace_bytes(256, 8, 2, 128, 64), NULL]
    assert lib.moe_backward_timed(*bwd, NULL) == INVALID
    assert "events" in _last()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_a_device_reports_no_device():
    assert lib.moe_route_topk(FAKE, 10, 8, 2, 1, FAKE, FAKE, NULL) == NO_DEVICE
    assert "device" in _last()


def test_wait_check_argument_errors():
    assert lib.moe_selftest_wait_timeout(FAKE, 256, 0, NULL) == INVALID
    assert lib.moe_selftest_wait_timeout(FAKE, 256, 3_000_000_000, NULL) == INVALID
    assert lib.moe_selftest_wait_timeout(NULL, 256, 1000, NULL) == WORKSPACE
    assert lib.moe_selftest_wait_timeout(FAKE, 255, 1000, NULL) == WORKSPACE


def test_activation_check_argument_errors():
    assert lib.moe_selftest_activation(FAKE, -1, FAKE, FAKE, NULL) == INVALID
    assert lib.moe_selftest_activation(NULL, 4, FAKE, FAKE, NULL) == INVALID
    assert lib.moe_selftest_activation(FAKE, 4, FAKE, NULL, NULL) == INVALID


def test_tile_schedule_argument_errors():
    assert lib.moe_set_tile_schedule(2) == INVALID
    assert lib.moe_set_tile_schedule(-1) == INVALID
    assert lib.moe_set_tile_schedule(1) == 0
    assert lib.moe_set_tile_schedule(0) == 0  # back to the default


# The boundary the hot path was specified against: each call with its
# parameter names (bf16 buffers are void*, cudaStream_t is moe_stream_t).
CONTRACT = {
    "moe_status_string": ["status"],
    "moe_route_topk": ["logits", "T", "E", "k", "renormalize", "topk_idx", "topk_w", "stream"],
    "moe_dispatch_workspace_bytes": ["T", "E", "k"],
    "moe_dispatch_scan": ["topk_idx", "T", "E", "k", "counts", "offsets", "src_token", "dest_row", "topk_w", "row_w",
                          "workspace", "workspace_bytes", "stream"],
    "moe_permute": ["x", "T", "d", "src_token", "P", "x_perm", "stream"],
    "moe_packed_weight_bytes": ["E", "d", "f"],
    "moe_pack_weights": ["w_gate", "w_up", "w_down", "E", "d", "f", "packed", "stream"],
    "moe_grouped_swiglu": ["x_perm", "offsets", "E", "d", "f", "packed", "row_scale", "h", "y", "workspace",
                           "workspace_bytes", "stream"],
    "moe_combine": ["y", "dest_row", "topk_w", "T", "k", "d", "out", "stream"],
    "moe_forward_workspace_bytes": ["T", "E", "k", "d", "f"],
    "moe_forward": ["x", "logits", "packed", "T", "d", "E", "k", "f", "renormalize", "out", "topk_idx_out",
                    "topk_w_out", "workspace", "workspace_bytes", "stream"],
    "moe_get_device_status": ["workspace", "stream"],
}

# Where the exported call departs from that form, and why (the same three
# lines stand in the design notes of the boundary).
DEVIATIONS = {
    "moe_dispatch_scan": (["topk_idx", "topk_w", "T", "E", "k", "counts", "offsets", "src_token", "dest_row", "row_w",
                           "workspace", "workspace_bytes", "stream"],
                          "the optional gates sit beside the indices they belong to"),
    "moe_permute": (["x", "T", "d", "dest_row", "k", "x_perm", "stream"],
                    "scatter from the token side: each x row is read once and written to its k rows"),
    "moe_grouped_swiglu": (["x_perm", "offsets", "P", "E", "d", "f", "packed", "row_scale", "h", "y", "workspace",
                            "workspace_bytes", "stream"],
                           "P sizes x_perm, h and y on the host without reading offsets[E] back from the device"),
}


def declared_params(name):
    text = open(HEADER).read()
    m = re.search(r"MOE_API\s+[\w\s\*]+?\b" + name + r"\s*\((.*?)\);", text, re.S)
    assert m, name
    params = [p.strip() for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
    return [re.findall(r"\w+", p)[-1] for p in params]


@pytest.mark.parametrize("name", sorted(CONTRACT))
def test_contract_call_is_exported_as_specified_or_recorded(name):
    assert hasattr(lib, name), f"{name} is not exported"
    assert name in lib_mod.SIGNATURES, f"{name} has no binding"
    want = DEVIATIONS[name][0] if name in DEVIATIONS else CONTRACT[name]
    assert declared_params(name) == want
    assert len(lib_mod.SIGNATURES[name][1]) == len(want)


def test_get_device_status_argument_check():
    assert lib.moe_get_device_status(NULL, NULL) == INVALID

"""Failure detection on the GPU without a fault: every spin in the kernels is
a bounded wait that gives up, records MOE_ERR_TIMEOUT in the workspace status
word and returns.  Here a wait on an mbarrier phase that nothing completes
runs out (a short limit), the host reads the status, and the context is
still usable for a full layer forward afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import assert_values_close, to_np

pytestmark = pytest.mark.gpu
TIMEOUT = 4


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    return m


def test_bounded_wait_runs_out_and_reports(moe):
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    moe.moe_selftest_wait_timeout(ws, 20_000_000)          # 20 ms
    status = moe.moe_read_device_status(ws)
    elapsed = time.perf_counter() - t0
    assert status == TIMEOUT
    assert 0.015 < elapsed < 1.5, elapsed


def test_context_usable_after_a_timeout(moe):
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    moe.moe_selftest_wait_timeout(ws, 5_000_000)
    assert moe.moe_read_device_status(ws) == TIMEOUT
    cfg = workloads.get("tiny")
    inp = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in workloads.generate(cfg, seed=4).items()}
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    fws = torch.empty(moe.moe_forward_workspace_bytes(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f), dtype=torch.uint8,
                      device="cuda")
    out = moe.moe_forward(inp["x"], inp["logits"], packed, cfg.E, cfg.k, cfg.f, cfg.renormalize, workspace=fws)
    assert moe.moe_read_device_status(fws) == 0
    ref = oracle.moe_forward(to_np(inp["x"]), to_np(inp["logits"]), to_np(inp["w_gate"]), to_np(inp["w_up"]),
                             to_np(inp["w_down"]), cfg.k, cfg.renormalize)
    assert_values_close(to_np(out), ref["out"], "out after a timeout")

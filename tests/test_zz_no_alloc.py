"""moe_dispatch_scan_noalloc: the dispatch pass for callers that cannot
allocate device memory (plugins handed only their input and output
buffers, loops that must not call cudaMalloc).  It uses the library's
fixed device scratch instead of a caller workspace, so it must give exactly
what moe_dispatch_scan gives, call after call, whatever the previous call
left in that shared scratch.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads


def _routing(name_or_cfg, seed):
    cfg = workloads.get(name_or_cfg)
    l = workloads.generate_logits(cfg, seed).numpy()
    idx, w = oracle.route_topk(l, cfg.k)
    return cfg, torch.from_numpy(idx.astype(np.int32)), torch.from_numpy(w.astype(np.float32))


@pytest.mark.gpu
def test_noalloc_dispatch_matches_workspace_dispatch_on_consecutive_calls():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import sparse_expert_gb300 as moe

    cases = [
        _routing("t1", 0),                                                  # 131,072 pairs: 64 chunks
        _routing(workloads.custom("few", T=300, d=64, E=8, k=2, f=64), 1),  # smaller call right after
        _routing(workloads.custom("wide", T=20000, d=64, E=384, k=8, f=64), 5),  # 79 chunks: a wider count table
        _routing("skew", 2),                                                # many empty experts
        _routing(workloads.custom("few2", T=77, d=64, E=16, k=3, f=64), 6),  # a small call after the wide ones
    ]
    for cfg, idx, w in cases:
        idx_d, w_d = idx.cuda(), w.cuda()
        want = moe.moe_dispatch_scan(idx_d, cfg.E, topk_w=w_d)
        got = moe.moe_dispatch_scan_noalloc(idx_d, cfg.E, topk_w=w_d)
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "src_token", "dest_row", "row_w"):
            assert torch.equal(got[key], want[key]), f"{cfg.name}: {key} differs"
        assert int(got["offsets"][-1]) == cfg.T * cfg.k
        assert moe.moe_dispatch_noalloc_status() == 0


@pytest.mark.gpu
def test_noalloc_dispatch_out_of_range_expert_index():
    """A pair whose expert index is outside [0, E) gets dest_row = -1 and the
    status reads MOE_ERR_BAD_INDEX; every other pair is placed exactly as the
    workspace path places it, and the next clean call clears the status."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import sparse_expert_gb300 as moe

    cfg, idx, w = _routing(workloads.custom("bad", T=3000, d=64, E=64, k=4, f=64), 7)
    bad_pair = 1234
    idx.view(-1)[bad_pair] = cfg.E + 3
    idx_d, w_d = idx.cuda(), w.cuda()
    want = moe.moe_dispatch_scan(idx_d, cfg.E, topk_w=w_d)
    got = moe.moe_dispatch_scan_noalloc(idx_d, cfg.E, topk_w=w_d)
    torch.cuda.synchronize()
    assert moe.moe_dispatch_noalloc_status() == 5  # MOE_ERR_BAD_INDEX
    assert moe.moe_read_device_status(want["workspace"]) == 5
    assert int(got["dest_row"][bad_pair]) == -1
    placed = cfg.T * cfg.k - 1
    assert int(got["offsets"][-1]) == placed
    for key in ("counts", "offsets", "dest_row"):
        assert torch.equal(got[key], want[key]), key
    for key in ("src_token", "row_w"):  # the last row has no pair
        assert torch.equal(got[key][:placed], want[key][:placed]), key
    cfg, idx, w = _routing(workloads.custom("clean", T=100, d=64, E=8, k=2, f=64), 8)
    moe.moe_dispatch_scan_noalloc(idx.cuda(), cfg.E, topk_w=w.cuda())
    assert moe.moe_dispatch_noalloc_status() == 0


def test_noalloc_status_reader_argument_check():
    from sparse_expert_gb300._lib import lib

    assert lib.moe_dispatch_noalloc_status(None, None) == 1  # MOE_ERR_INVALID_ARG


def test_noalloc_rejects_problems_beyond_its_scratch():
    from sparse_expert_gb300._lib import lib

    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    status = lib.moe_dispatch_scan_noalloc(fake, fake, 800000, 384, 8, fake, fake, fake, fake, fake, None)
    assert status == 2  # MOE_ERR_UNSUPPORTED
    msg = lib.moe_last_error().decode()
    assert "static scratch" in msg and str(4 << 20) in msg

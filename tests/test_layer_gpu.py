"""Parity of the whole layer forward (moe_forward) with the fp64 oracle.

tiny and small: every intermediate and every output element.
t1, skew, long (the 1T-model layer shape, 25 GB of weights): routing,
counts, offsets and both index maps for all tokens bit for bit, and the
values of H, Y and the output on a seeded sample of 256 random tokens plus
the tokens of the rows at the edges of the paired GEMM's token tiles (first
and last row of every tile, both sides of the 256-token MMA split) in the
largest, the smallest and four random non-empty expert groups -- for the
skewed workload every tile of its ~16,000-row group.  This is the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import (ExpertSlices, assert_gates_close, assert_values_close, pick_sample_tokens, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    return m


def _run_forward(moe, inp):
    cfg = inp["cfg"]
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    ws = torch.empty(moe.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
    out = moe.moe_forward(inp["x"], inp["logits"], packed, E, k, f, cfg.renormalize, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return out, ws, packed


def _check_routing_and_index(inter, ridx, rw, E, k):
    counts, offsets, src, dst = oracle.dispatch(ridx, E)
    assert np.array_equal(to_np(inter["topk_idx"]), ridx)
    assert_gates_close(to_np(inter["topk_w"]), rw, k)
    assert np.array_equal(to_np(inter["counts"]), counts)
    assert np.array_equal(to_np(inter["offsets"]), offsets)
    assert np.array_equal(to_np(inter["src_token"]), src)
    assert np.array_equal(to_np(inter["dest_row"]), dst)
    return counts, offsets, src, dst


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_forward_full_parity(moe, name):
    cfg = workloads.get(name)
    inp = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in workloads.generate(cfg, seed=1).items()}
    out, ws, _ = _run_forward(moe, inp)
    inter = moe.forward_intermediates(ws, cfg.T, cfg.E, cfg.k, cfg.d, cfg.f)
    ref = oracle.moe_forward(to_np(inp["x"]), to_np(inp["logits"]), to_np(inp["w_gate"]), to_np(inp["w_up"]),
                             to_np(inp["w_down"]), cfg.k, cfg.renormalize)
    _check_routing_and_index(inter, ref["idx"], ref["w"], cfg.E, cfg.k)
    assert np.array_equal(to_np(inter["x_perm"]), ref["x_perm"])
    assert_values_close(to_np(inter["h"]), ref["h"], "h")
    # y holds the ungated expert rows (the gates enter in the output reduction)
    assert_values_close(to_np(inter["y"]), ref["y"], "y")
    assert_values_close(to_np(out), ref["out"], "out")


# Paired-GEMM token tiles of every kind, checked in full: groups of at most
# 256 rows (one MMA per K step), groups of 257..512 rows in one tile (two
# MMAs per K step) and groups split into near-equal tiles.  The skewed case
# has groups of 9..2,330 rows (tiles of 310, 384, 464, 466 and 469 rows among
# them); forced-uniform routing gives every expert 350 rows.
@pytest.mark.parametrize("T,E,k,routing,seed", [(3000, 16, 2, "zipf", 12), (1400, 8, 2, "fur", 14)])
def test_forward_full_parity_token_tile_kinds(moe, T, E, k, routing, seed):
    cfg = workloads.custom(f"tiles_{routing}", T=T, d=512, E=E, k=k, f=256, routing=routing)
    inp = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in workloads.generate(cfg, seed=seed).items()}
    out, ws, _ = _run_forward(moe, inp)
    inter = moe.forward_intermediates(ws, cfg.T, cfg.E, cfg.k, cfg.d, cfg.f)
    ref = oracle.moe_forward(to_np(inp["x"]), to_np(inp["logits"]), to_np(inp["w_gate"]), to_np(inp["w_up"]),
                             to_np(inp["w_down"]), cfg.k, cfg.renormalize)
    _check_routing_and_index(inter, ref["idx"], ref["w"], cfg.E, cfg.k)
    assert_values_close(to_np(inter["h"]), ref["h"], "h")
    assert_values_close(to_np(inter["y"]), ref["y"], "y")
    assert_values_close(to_np(out), ref["out"], "out")


@pytest.mark.parametrize("name", ["t1", "skew", "long"])
def test_forward_full_size_sampled(moe, name):
    cfg = workloads.get(name)
    inp = workloads.generate(cfg, seed=0, device="cuda")
    out, ws, packed = _run_forward(moe, inp)
    del packed
    inter = moe.forward_intermediates(ws, cfg.T, cfg.E, cfg.k, cfg.d, cfg.f)
    logits = to_np(inp["logits"])
    ridx, rw = oracle.route_topk(logits, cfg.k, cfg.renormalize)
    counts, offsets, src, dst = _check_routing_and_index(inter, ridx, rw, cfg.E, cfg.k)
    if name == "long":
        assert set(counts.tolist()) == {1365, 1366}
    if name == "skew":
        assert (counts == 0).sum() > 100 and counts.max() > 10000
    toks = pick_sample_tokens(ridx, counts, n_random=256, seed=7, offsets=offsets, src_token=src)
    x_rows = to_np(inp["x"][torch.from_numpy(toks).cuda()])
    ref = oracle.moe_forward_tokens(x_rows, logits[toks], ExpertSlices(inp["w_gate"]), ExpertSlices(inp["w_up"]),
                                    ExpertSlices(inp["w_down"]), cfg.k, cfg.renormalize)
    rows = dst.reshape(cfg.T, cfg.k)[toks]                        # [n, k]
    rows_t = torch.from_numpy(rows.reshape(-1)).cuda()
    xp = to_np(inter["x_perm"][rows_t]).reshape(len(toks), cfg.k, cfg.d)
    assert np.array_equal(xp, np.repeat(x_rows[:, None, :], cfg.k, axis=1))
    h = to_np(inter["h"][rows_t]).reshape(len(toks), cfg.k, cfg.f)
    y = to_np(inter["y"][rows_t]).reshape(len(toks), cfg.k, cfg.d)
    assert_values_close(h, ref["h"], "h (sampled)")
    assert_values_close(y, ref["y"], "y (sampled, ungated)")
    assert_values_close(to_np(out[torch.from_numpy(toks).cuda()]), ref["out"], "out (sampled)")
    # every output row is finite and rows of untouched tokens were written
    assert torch.isfinite(out.float()).all()


def test_forward_is_deterministic(moe):
    cfg = workloads.get("small")
    inp = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in workloads.generate(cfg, seed=2).items()}
    out1, ws, packed = _run_forward(moe, inp)
    out2 = moe.moe_forward(inp["x"], inp["logits"], packed, cfg.E, cfg.k, cfg.f, True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_forward_from_host_buffers_matches(moe):
    cfg = workloads.get("tiny")
    inp = workloads.generate(cfg, seed=3)
    dev = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in inp.items()}
    out_dev, ws, packed = _run_forward(moe, dev)
    x_h = inp["x"].pin_memory()
    l_h = inp["logits"].pin_memory()
    out_h = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(dev["x"])
    l_d = torch.empty_like(dev["logits"])
    o_d = torch.empty_like(dev["x"])
    moe.moe_forward_host(x_h, l_h, out_h, x_d, l_d, o_d, packed, cfg.E, cfg.k, cfg.f, ws)
    assert torch.equal(out_h, out_dev.cpu())


def test_forward_without_renormalisation(moe):
    cfg = workloads.custom("norenorm", T=300, d=128, E=16, k=4, f=128, renormalize=False)
    inp = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in workloads.generate(cfg, seed=4).items()}
    out, ws, _ = _run_forward(moe, inp)
    ref = oracle.moe_forward(to_np(inp["x"]), to_np(inp["logits"]), to_np(inp["w_gate"]), to_np(inp["w_up"]),
                             to_np(inp["w_down"]), cfg.k, False)
    inter = moe.forward_intermediates(ws, cfg.T, cfg.E, cfg.k, cfg.d, cfg.f)
    assert_gates_close(to_np(inter["topk_w"]), ref["w"], cfg.E)
    assert_values_close(to_np(out), ref["out"], "out")


def test_forward_zero_tokens(moe):
    cfg = workloads.custom("empty", T=0, d=128, E=8, k=2, f=64)
    packed = torch.zeros(moe.moe_packed_weight_bytes(8, 128, 64), dtype=torch.uint8, device="cuda")
    ws = torch.empty(max(256, moe.moe_forward_workspace_bytes(0, 8, 2, 128, 64)), dtype=torch.uint8, device="cuda")
    out = moe.moe_forward(torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"),
                          torch.empty(0, 8, device="cuda"), packed, 8, 2, 64, workspace=ws)
    assert out.shape == (0, 128)
    assert moe.moe_read_device_status(ws) == 0


# ------------------------------------------------- gathered A (no x_perm)
@pytest.mark.parametrize("name", ["tiny", "small", "t1", "skew"])
def test_gathered_forward_equals_permuted_forward(moe, name):
    """The gate/up GEMM fed by TMA gathers of x[src_token[r]] sees the same A
    rows in the same order as the one reading x_perm, so every intermediate
    and the output are bit-identical; at oracle sizes it is also held to the
    oracle directly."""
    cfg = workloads.get(name)
    inp = workloads.generate(cfg, seed=3, device="cuda")
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    nbytes = moe.moe_forward_workspace_bytes(T, E, k, d, f)
    ws1 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out1 = moe.moe_forward(inp["x"], inp["logits"], packed, E, k, f, cfg.renormalize, workspace=ws1)
    out2 = moe.moe_forward_gathered(inp["x"], inp["logits"], packed, E, k, f, cfg.renormalize, workspace=ws2)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws2) == 0
    i1 = moe.forward_intermediates(ws1, T, E, k, d, f)
    i2 = moe.forward_intermediates(ws2, T, E, k, d, f)
    for key in ("topk_idx", "offsets", "src_token", "dest_row", "h", "y"):
        assert torch.equal(i1[key], i2[key]), key
    assert torch.equal(out1, out2)
    if name == "tiny":
        ref = oracle.moe_forward(to_np(inp["x"]), to_np(inp["logits"]), to_np(inp["w_gate"]), to_np(inp["w_up"]),
                                 to_np(inp["w_down"]), k, cfg.renormalize)
        assert_values_close(to_np(out2), ref["out"], "out (gathered)")


def test_gathered_forward_zero_tokens(moe):
    E, d, f, k = 4, 128, 64, 2
    g = torch.Generator().manual_seed(2)
    w = [(torch.randn(E, d, f, generator=g) / 11).to(torch.bfloat16).cuda() for _ in range(2)]
    wd = (torch.randn(E, f, d, generator=g) / 8).to(torch.bfloat16).cuda()
    packed = moe.moe_pack_weights(w[0], w[1], wd)
    out = moe.moe_forward_gathered(torch.empty(0, d, dtype=torch.bfloat16, device="cuda"),
                                   torch.empty(0, E, device="cuda"), packed, E, k, f)
    assert out.shape == (0, d)


def test_forward_host_stream_matches_device_forward(moe):
    """Five batches from pinned host memory through the pipelined entry point
    (copies on their own streams, two device slots) give, batch by batch,
    the bit-identical outputs of moe_forward on device copies."""
    cfg = workloads.get("small")
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    w = workloads.generate(cfg, seed=11, device="cuda")
    packed = moe.moe_pack_weights(w["w_gate"], w["w_up"], w["w_down"])
    batches = [workloads.generate(cfg, seed=20 + b, weights=False) for b in range(5)]
    xh = [b["x"].pin_memory() for b in batches]
    lh = [b["logits"].pin_memory() for b in batches]
    oh = [torch.empty(T, d, dtype=torch.bfloat16).pin_memory() for _ in batches]
    xd = [torch.empty(T, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ld = [torch.empty(T, E, dtype=torch.float32, device="cuda") for _ in range(2)]
    od = [torch.empty(T, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ws = torch.empty(moe.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
    moe.moe_forward_host_stream(xh, lh, oh, xd, ld, od, packed, E, k, f, ws, cfg.renormalize)
    for b in range(5):
        ref = moe.moe_forward(batches[b]["x"].cuda(), batches[b]["logits"].cuda(), packed, E, k, f, cfg.renormalize)
        assert torch.equal(oh[b], ref.cpu()), b

"""Parity of the backward expert GEMMs and of the whole layer backward with
the fp64 oracle, through the C ABI.

The expert GEMMs of the backward ("Scalable Pretraining of Large MoE LMs on
Aurora Super Computer", §3.1, Algorithm 1, stage 4, differentiated) take
bf16 operands with fp32 accumulation; their outputs, and the intermediates
they read (G, U, H, dG, dU), are rounded to bf16.  They are held to the
rule of tests/parity.py for bf16 GEMM outputs against exact fp64:
max|err| <= 2e-2 max|ref| and mean|err| <= 5e-3 mean|ref|, per output
tensor.  The router-logit gradient of the layer backward, a difference of
nearly equal terms for most entries, is held to the same relative-L1 rule.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import ExpertSlices, assert_values_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    return m


def _weights(g, E, d, f):
    wg = (torch.randn(E, d, f, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    wu = (torch.randn(E, d, f, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    wd = (torch.randn(E, f, d, generator=g) / math.sqrt(f)).to(torch.bfloat16)
    return wg, wu, wd


def _expert_case(moe, T, d, E, k, f, seed=0, skew=0.0):
    """Route and index on the host (oracle), then the GPU gate/up GEMM that
    keeps G and U, and the GPU backward GEMMs, against the oracle."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    l = torch.randn(T, E, generator=g)
    if skew:
        l = l - skew * torch.log(torch.arange(1, E + 1, dtype=torch.float32))[None, :]
    wg, wu, wd = _weights(g, E, d, f)
    idx, _ = oracle.route_topk(l.numpy(), k)
    counts, offsets, src, _ = oracle.dispatch(idx, E)
    xp = oracle.permute(x.float().numpy(), src)
    dy = (torch.randn(T * k, d, generator=g) * 0.5).to(torch.bfloat16)
    wg_np, wu_np, wd_np = wg.float().numpy(), wu.float().numpy(), wd.float().numpy()

    packed = moe.moe_pack_weights(wg.cuda(), wu.cuda(), wd.cuda())
    xp_t = torch.from_numpy(xp).to(torch.bfloat16).cuda()
    off_t = torch.from_numpy(offsets.astype(np.int32)).cuda()
    h, gu = moe.moe_grouped_gate_up_save(xp_t, off_t, E, f, packed)
    G, U = moe.gu_split(gu, f)
    rG, rU = oracle.expert_gate_up(xp, offsets, wg_np, wu_np)
    rh, _ = oracle.expert_mlp(xp, offsets, wg_np, wu_np, wd_np)
    assert_values_close(to_np(G), rG, "G")
    assert_values_close(to_np(U), rU, "U")
    assert_values_close(to_np(h), rh, "h")

    r = moe.moe_grouped_swiglu_backward(xp_t, h, gu, dy.cuda(), off_t, E, f, packed)
    rdx, rdwg, rdwu, rdwd, rdG, rdU = oracle.expert_mlp_backward(xp, offsets, wg_np, wu_np, wd_np,
                                                                 dy.double().numpy(), return_preact_grads=True)
    dG, dU = moe.gu_split(r["dgu"], f)
    assert_values_close(to_np(dG), rdG, "dG")
    assert_values_close(to_np(dU), rdU, "dU")
    assert_values_close(to_np(r["dx_perm"]), rdx, "dx_perm")
    assert_values_close(to_np(r["dw_gate"]), rdwg, "dw_gate")
    assert_values_close(to_np(r["dw_up"]), rdwu, "dw_up")
    assert_values_close(to_np(r["dw_down"]), rdwd, "dw_down")
    empty = np.nonzero(counts == 0)[0]
    for name in ("dw_gate", "dw_up", "dw_down"):
        assert not r[name][torch.from_numpy(empty).cuda()].any(), f"{name} of an expert without rows"
    return counts


@pytest.mark.parametrize("T,d,E,k,f", [
    (256, 128, 8, 2, 64),      # gate/up half tile 64, down tile 128; every group ragged
    (300, 256, 4, 2, 128),     # N tiles of 256
    (129, 192, 3, 1, 192),     # d = 192: down tile 64, a 64-row partial M tile in the gate/up wgrad
    (1, 128, 2, 1, 64),        # one row
    (1000, 512, 16, 4, 256),   # many partial tiles
    (640, 384, 5, 1, 320),     # f = 320: gate/up half 64, dgrad N tile 64
])
def test_swiglu_backward_matches_oracle(moe, T, d, E, k, f):
    _expert_case(moe, T, d, E, k, f, seed=T + d + f)


def test_swiglu_backward_empty_and_huge_groups(moe):
    counts = _expert_case(moe, 2048, 256, 32, 4, 128, seed=5, skew=3.0)
    assert (counts == 0).sum() > 0 and counts.max() > 1000


def test_swiglu_backward_paired_empty_and_huge_groups(moe):
    # d and f multiples of 256: both dgrad GEMMs run on SM pairs, here with
    # experts without rows and experts spanning several 512-token tiles
    counts = _expert_case(moe, 2048, 512, 32, 4, 256, seed=6, skew=3.0)
    assert (counts == 0).sum() > 0 and counts.max() > 1000


def test_swiglu_backward_max_experts(moe):
    # E = MOE_MAX_EXPERTS with d and f multiples of 256: paired dgrad and the
    # weight gradients over ~16 rows per expert (one partial K block each)
    counts = _expert_case(moe, 2048, 256, 1024, 8, 256, seed=12)
    assert len(counts) == 1024


def test_swiglu_backward_single_expert_long_k(moe):
    # E = 1: every row in one group; the weight gradients contract over 700 rows
    _expert_case(moe, 700, 1024, 1, 1, 256, seed=9)


def test_swiglu_backward_rows_multiple_of_64(moe):
    # group sizes that end exactly on a 64-row K block: no tail zeroing
    T, d, E, k, f = 256, 128, 4, 1, 128
    g = torch.Generator().manual_seed(13)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wg, wu, wd = _weights(g, E, d, f)
    offsets = np.arange(0, T + 1, T // E, dtype=np.int64)
    packed = moe.moe_pack_weights(wg.cuda(), wu.cuda(), wd.cuda())
    off_t = torch.from_numpy(offsets.astype(np.int32)).cuda()
    h, gu = moe.moe_grouped_gate_up_save(x.cuda(), off_t, E, f, packed)
    dy = torch.randn(T, d, generator=g).to(torch.bfloat16)
    r = moe.moe_grouped_swiglu_backward(x.cuda(), h, gu, dy.cuda(), off_t, E, f, packed)
    ref = oracle.expert_mlp_backward(x.double().numpy(), offsets, wg.float().numpy(), wu.float().numpy(),
                                     wd.float().numpy(), dy.double().numpy())
    for name, want in zip(("dx_perm", "dw_gate", "dw_up", "dw_down"), ref):
        assert_values_close(to_np(r[name]), want, name)


# --------------------------------------------------------- layer backward
def _layer_inputs(name, seed=0, device="cpu"):
    cfg = workloads.get(name)
    inp = workloads.generate(name, seed, device=device)
    dout = (torch.randn(cfg.T, cfg.d, generator=torch.Generator().manual_seed(seed + 77)) * 0.1).to(torch.bfloat16)
    return cfg, inp, dout.to(device)


def _gpu_backward(moe, cfg, inp, dout, renorm=True):
    packed = moe.moe_pack_weights(inp["w_gate"].cuda(), inp["w_up"].cuda(), inp["w_down"].cuda())
    g = moe.moe_backward(inp["x"].cuda(), inp["logits"].cuda(), packed, dout.cuda(), cfg.E, cfg.k, cfg.f,
                         renormalize=renorm)
    del packed
    return g


@pytest.mark.parametrize("name,renorm", [("tiny", True), ("tiny", False), ("small", True)])
def test_layer_backward_matches_oracle(moe, name, renorm):
    cfg, inp, dout = _layer_inputs(name)
    g = _gpu_backward(moe, cfg, inp, dout, renorm)
    ref = oracle.moe_backward(inp["x"].float().numpy(), inp["logits"].numpy(), inp["w_gate"].float().numpy(),
                              inp["w_up"].float().numpy(), inp["w_down"].float().numpy(), dout.double().numpy(),
                              cfg.k, renorm)
    for key in ("dx", "d_logits", "dw_gate", "dw_up", "dw_down"):
        assert_values_close(to_np(g[key]), ref[key], key)


def test_layer_backward_token_tile_kinds(moe):
    """The recompute's paired gate/up GEMM (which also keeps G and U) on token
    tiles of every kind: groups of 9..2,330 rows, so tiles of up to 256 rows
    (one MMA per K step), of 257..512 (two) and groups split over several."""
    cfg = workloads.custom("tiles_zipf", T=3000, d=512, E=16, k=2, f=256, routing="zipf")
    cfg, inp, dout = _layer_inputs(cfg, seed=12)
    g = _gpu_backward(moe, cfg, inp, dout)
    ref = oracle.moe_backward(inp["x"].float().numpy(), inp["logits"].numpy(), inp["w_gate"].float().numpy(),
                              inp["w_up"].float().numpy(), inp["w_down"].float().numpy(), dout.double().numpy(),
                              cfg.k, True)
    for key in ("dx", "d_logits", "dw_gate", "dw_up", "dw_down"):
        assert_values_close(to_np(g[key]), ref[key], key)


def test_layer_backward_is_deterministic(moe):
    cfg, inp, dout = _layer_inputs("tiny", seed=3)
    a = _gpu_backward(moe, cfg, inp, dout)
    b = _gpu_backward(moe, cfg, inp, dout)
    for key in a:
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("name", ["t1", "skew", "long"])
def test_layer_backward_full_size_sampled(moe, name):
    """16384 tokens, d = 6144, 384 experts, k = 8, f = 1792 (normal routing,
    the Zipf-skewed routing whose largest group holds ~16,000 rows and ~200
    experts none, and 65,536 tokens with forced-uniform routing: three
    455-row tiles per expert): the whole backward runs on the GPU; the oracle
    recomputes, one by one, the rows of a seeded token sample (all k slots
    of each) and of two whole experts (the largest group and a random one,
    which may be empty: its weight gradients must then be exactly zero),
    and the gradients that depend only on those rows are compared: dx and
    d_logits of the sampled tokens, the three weight gradients of the
    sampled experts."""
    cfg, inp, dout = _layer_inputs(name, device="cuda")
    g = _gpu_backward(moe, cfg, inp, dout)
    torch.cuda.synchronize()
    logits = to_np(inp["logits"])
    idx, w = oracle.route_topk(logits, cfg.k)
    counts, offsets, src, dst = oracle.dispatch(idx, cfg.E)
    rng = np.random.default_rng(17)
    toks = np.sort(rng.choice(cfg.T, 24, replace=False))
    experts = np.array(sorted({int(np.argmax(counts)), int(rng.integers(cfg.E))}))
    rows = set(dst.reshape(cfg.T, cfg.k)[toks].reshape(-1).tolist())
    for e in experts:
        rows.update(range(int(offsets[e]), int(offsets[e + 1])))
    rows = np.array(sorted(rows))                      # expert-sorted: rows of one expert stay together
    row_expert = np.searchsorted(offsets, rows, side="right") - 1
    sub_off = np.searchsorted(row_expert, np.arange(cfg.E + 1), side="left")
    xs = to_np(inp["x"][torch.from_numpy(src[rows]).cuda()]).astype(np.float64)
    wg, wu, wd = (ExpertSlices(inp[n]) for n in ("w_gate", "w_up", "w_down"))
    dout_np = to_np(dout).astype(np.float64)
    # the gradient of each row's expert output: gate * dout of its token
    row_of = {int(r): i for i, r in enumerate(rows)}
    flat_w = w.reshape(-1)
    pos = np.empty(cfg.T * cfg.k, dtype=np.int64)
    pos[dst] = np.arange(cfg.T * cfg.k)                # row -> flat (token, slot)
    dys = flat_w[pos[rows]][:, None] * dout_np[src[rows]]
    _, ys = oracle.expert_mlp(xs, sub_off, wg, wu, wd)
    dxs, dwg, dwu, dwd = oracle.expert_mlp_backward(xs, sub_off, wg, wu, wd, dys)
    # tokens: dx sums the token's k rows; d_logits from <y_r, dout_t>
    ref_dx = np.zeros((len(toks), cfg.d))
    dw_tok = np.zeros((len(toks), cfg.k))
    for i, t in enumerate(toks):
        for j in range(cfg.k):
            r = row_of[int(dst[t * cfg.k + j])]
            ref_dx[i] += dxs[r]
            dw_tok[i, j] = ys[r] @ dout_np[t]
    ref_dl = oracle.route_backward(logits[toks].astype(np.float64), idx[toks], dw_tok)
    t_idx = torch.from_numpy(toks).cuda()
    assert_values_close(to_np(g["dx"][t_idx]), ref_dx, "dx (sampled tokens)")
    assert_values_close(to_np(g["d_logits"][t_idx]), ref_dl, "d_logits (sampled tokens)")
    for e in experts:
        assert_values_close(to_np(g["dw_gate"][int(e)]), dwg[e], f"dw_gate[{e}]")
        assert_values_close(to_np(g["dw_up"][int(e)]), dwu[e], f"dw_up[{e}]")
        assert_values_close(to_np(g["dw_down"][int(e)]), dwd[e], f"dw_down[{e}]")


def test_layer_backward_zero_tokens(moe):
    E, d, f, k = 4, 128, 64, 2
    g = torch.Generator().manual_seed(1)
    wg, wu, wd = _weights(g, E, d, f)
    packed = moe.moe_pack_weights(wg.cuda(), wu.cuda(), wd.cuda())
    out = moe.moe_backward(torch.empty(0, d, dtype=torch.bfloat16, device="cuda"),
                           torch.empty(0, E, device="cuda"), packed,
                           torch.empty(0, d, dtype=torch.bfloat16, device="cuda"), E, k, f)
    assert out["dx"].shape == (0, d)
    for name in ("dw_gate", "dw_up", "dw_down"):
        assert not out[name].any()

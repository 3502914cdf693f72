"""Parity of each CUDA stage with the fp64 oracle, through the C ABI.

Inputs are seeded synthetic tensors (workloads/); each test feeds the same
inputs to the kernel and to the oracle.  Integer outputs must match bit for
bit; values follow tests/parity.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import assert_gates_close, assert_values_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m  # must load: no fallback exists
    return m


def _logits_for(name, seed=0):
    return workloads.generate_logits(name, seed).contiguous()


# ------------------------------------------------------------------ route
ROUTE_CASES = [("tiny", True), ("tiny", False), ("small", True), ("t1", True), ("t1", False), ("skew", True),
               ("long", True)]


@pytest.mark.parametrize("name,renorm", ROUTE_CASES)
def test_route_matches_oracle(moe, name, renorm):
    cfg = workloads.get(name)
    l = _logits_for(name)
    idx, w = moe.moe_route_topk(l.cuda(), cfg.k, renorm)
    ridx, rw = oracle.route_topk(l.numpy(), cfg.k, renorm)
    assert np.array_equal(to_np(idx), ridx)
    assert_gates_close(to_np(w), rw, cfg.k if renorm else cfg.E)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (33, 7, 7), (100, 32, 32), (64, 1024, 32), (257, 1024, 8),
                                   (50, 33, 3), (40, 64, 64 // 2)])
@pytest.mark.parametrize("ties", [False, True])
def test_route_shapes_and_ties(moe, T, E, k, ties):
    g = torch.Generator().manual_seed(T * 131 + E)
    l = torch.randn(T, E, generator=g)
    if ties:
        l = torch.round(l * 2) / 2
        l[torch.rand(T, E, generator=g) < 0.1] = -0.0
        l[torch.rand(T, E, generator=g) < 0.1] = 0.0
    idx, w = moe.moe_route_topk(l.cuda(), k, True)
    ridx, rw = oracle.route_topk(l.numpy(), k, True)
    assert np.array_equal(to_np(idx), ridx)
    assert_gates_close(to_np(w), rw, k)


def test_route_empty(moe):
    idx, w = moe.moe_route_topk(torch.empty(0, 8, device="cuda"), 2)
    assert idx.shape == (0, 2)


# --------------------------------------------------------------- dispatch
def _check_dispatch(moe, ridx, E, w=None):
    T, k = ridx.shape
    idx_t = torch.from_numpy(ridx.astype(np.int32)).cuda()
    w_t = None if w is None else torch.from_numpy(np.asarray(w, dtype=np.float32)).cuda()
    res = moe.moe_dispatch_scan(idx_t, E, topk_w=w_t)
    counts, offsets, src, dst = oracle.dispatch(ridx, E)
    assert np.array_equal(to_np(res["counts"]), counts)
    assert np.array_equal(to_np(res["offsets"]), offsets)
    assert np.array_equal(to_np(res["src_token"]), src)
    assert np.array_equal(to_np(res["dest_row"]), dst)
    if w is not None:
        row_w = np.empty(T * k, dtype=np.float32)
        row_w[dst] = np.asarray(w, dtype=np.float32).reshape(-1)
        assert np.array_equal(to_np(res["row_w"]), row_w)   # a copy: bit exact
    assert moe.moe_read_device_status(res["workspace"]) == 0


@pytest.mark.parametrize("name", ["tiny", "small", "t1", "skew", "long"])
def test_dispatch_matches_oracle(moe, name):
    cfg = workloads.get(name)
    ridx, rw = oracle.route_topk(_logits_for(name).numpy(), cfg.k)
    _check_dispatch(moe, ridx, cfg.E, rw)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (1, 8, 8), (3, 1024, 5), (1023, 4, 1), (1025, 4, 1),
                                   (4096, 64, 8), (777, 300, 6), (2000, 1024, 32)])
def test_dispatch_shapes(moe, T, E, k):
    rng = np.random.default_rng(T + E + k)
    # concentrate routing on a few experts so that many groups are empty
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[:, : max(1, E // 10)] += 3.0
    ridx, rw = oracle.route_topk(l, k)
    _check_dispatch(moe, ridx, E, rw)


def test_dispatch_hand_example(moe, golden):
    g = golden("alg1_index_example.json")
    idx = np.array(g["indices"], dtype=np.int32)
    res = moe.moe_dispatch_scan(torch.from_numpy(idx).cuda(), g["N"])
    assert to_np(res["offsets"]).tolist() == g["no_ep"]["cum_token_counts"]
    assert to_np(res["src_token"]).tolist() == g["no_ep"]["input_indices"]
    assert to_np(res["dest_row"]).tolist() == g["no_ep"]["output_indices"]


def test_dispatch_empty(moe):
    res = moe.moe_dispatch_scan(torch.empty(0, 4, dtype=torch.int32, device="cuda"), 16)
    assert to_np(res["offsets"]).tolist() == [0] * 17
    assert to_np(res["counts"]).tolist() == [0] * 16


def test_dispatch_reports_out_of_range_expert(moe):
    idx = torch.tensor([[0, 1], [2, 9], [1, 3]], dtype=torch.int32, device="cuda")
    res = moe.moe_dispatch_scan(idx, 4)
    assert moe.moe_read_device_status(res["workspace"]) == 5  # MOE_ERR_BAD_INDEX
    assert to_np(res["dest_row"])[3] == -1
    assert to_np(res["counts"]).tolist() == [1, 2, 1, 1]


# ---------------------------------------------------------------- permute
@pytest.mark.parametrize("T,d,k", [(256, 128, 2), (1000, 2048, 8), (37, 8, 3), (5, 6144, 8), (300, 136, 1)])
def test_permute_is_exact(moe, T, d, k):
    g = torch.Generator().manual_seed(T + d)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    dest = torch.randperm(T * k, generator=g).to(torch.int32)
    xp = moe.moe_permute(x.cuda(), dest.cuda(), k)
    src = np.empty(T * k, dtype=np.int64)
    src[dest.numpy()] = np.arange(T * k) // k
    ref = oracle.permute(x.float().numpy(), src)
    assert np.array_equal(to_np(xp), ref)


# ---------------------------------------------------------------- combine
@pytest.mark.parametrize("T,d,k", [(256, 128, 2), (999, 2048, 8), (16, 6144, 8), (77, 24, 5)])
@pytest.mark.parametrize("gated", [True, False])
def test_combine_matches_oracle(moe, T, d, k, gated):
    g = torch.Generator().manual_seed(T * d + k)
    y = torch.randn(T * k, d, generator=g).to(torch.bfloat16)
    dest = torch.randperm(T * k, generator=g).to(torch.int32)
    w = torch.rand(T, k, generator=g) if gated else None
    out = moe.moe_combine(y.cuda(), dest.cuda(), T, k, None if w is None else w.cuda())
    ref = oracle.combine(y.float().numpy(), dest.numpy(), w.numpy() if gated else np.ones((T, k)))
    assert_values_close(to_np(out), ref, "combine")


def test_combine_single_slot_is_exact(moe):
    T, d = 300, 512
    g = torch.Generator().manual_seed(1)
    y = torch.randn(T, d, generator=g).to(torch.bfloat16)
    dest = torch.randperm(T, generator=g).to(torch.int32)
    out = moe.moe_combine(y.cuda(), dest.cuda(), T, 1)
    assert torch.equal(out.cpu(), y[dest.long()])


# ------------------------------------------------------------------- pack
def _tile_major(w_nk, bn):
    """[E, N, K] (K contiguous) -> blocks of bn rows x 64 K values, block order (e, N tile, K block)."""
    E, N, K = w_nk.shape
    return w_nk.reshape(E, N // bn, bn, K // 64, 64).permute(0, 1, 3, 2, 4).reshape(-1)


@pytest.mark.parametrize("E,d,f", [(8, 128, 64), (3, 256, 384), (2, 192, 192), (2, 640, 128)])
def test_pack_layout(moe, E, d, f):
    g = torch.Generator().manual_seed(E * d + f)
    wg = torch.randn(E, d, f, generator=g).to(torch.bfloat16)
    wu = torch.randn(E, d, f, generator=g).to(torch.bfloat16)
    wd = torch.randn(E, f, d, generator=g).to(torch.bfloat16)
    packed = moe.moe_pack_weights(wg.cuda(), wu.cuda(), wd.cuda()).cpu()
    h = 64
    # gate/up: N tiles of [h gate columns | the same h up columns], each a row of K = d weights
    gt = wg.transpose(1, 2).reshape(E, f // h, h, d)
    ut = wu.transpose(1, 2).reshape(E, f // h, h, d)
    gu_nk = torch.stack([gt, ut], dim=2).reshape(E, 2 * f, d)
    bn_down = 256 if d % 256 == 0 else 128 if d % 128 == 0 else 64
    dn_nk = wd.transpose(1, 2).contiguous()
    got = packed.view(torch.bfloat16)
    assert torch.equal(got[: E * 2 * f * d], _tile_major(gu_nk, 2 * h))
    assert torch.equal(got[E * 2 * f * d:], _tile_major(dn_nk, bn_down))


# ------------------------------------------------------ grouped SwiGLU GEMM
def _gemm_case(moe, T, d, E, k, f, seed=0, skew=0.0, scale_rows=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    l = torch.randn(T, E, generator=g)
    if skew:
        l = l + skew * torch.log(torch.arange(1, E + 1, dtype=torch.float32))[None, :].neg()
    wg = (torch.randn(E, d, f, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    wu = (torch.randn(E, d, f, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    wd = (torch.randn(E, f, d, generator=g) / math.sqrt(f)).to(torch.bfloat16)
    idx, w = oracle.route_topk(l.numpy(), k)
    counts, offsets, src, dst = oracle.dispatch(idx, E)
    xp = oracle.permute(x.float().numpy(), src)
    row_w = np.empty(T * k)
    row_w[dst] = w.reshape(-1)
    packed = moe.moe_pack_weights(wg.cuda(), wu.cuda(), wd.cuda())
    xp_t = torch.from_numpy(xp).to(torch.bfloat16).cuda()
    off_t = torch.from_numpy(offsets.astype(np.int32)).cuda()
    rs = torch.from_numpy(row_w.astype(np.float32)).cuda() if scale_rows else None
    h, y = moe.moe_grouped_swiglu(xp_t, off_t, E, f, packed, row_scale=rs)
    rh, ry = oracle.expert_mlp(xp, offsets, wg.float().numpy(), wu.float().numpy(), wd.float().numpy())
    assert_values_close(to_np(h), rh, "h")
    ref_y = ry * (row_w.astype(np.float32).astype(np.float64)[:, None] if scale_rows else 1.0)
    assert_values_close(to_np(y), ref_y, "y")
    return counts


@pytest.mark.parametrize("T,d,E,k,f", [
    (256, 128, 8, 2, 64),      # tiny layer: N tile 128 (64 gate + 64 up), down N tile 128
    (300, 256, 4, 2, 128),     # N tile 256 gate/up, down 256
    (129, 192, 3, 1, 192),     # gate/up halves of 64, down N tile 64, ragged M
    (1, 128, 2, 1, 64),        # one row
    (1000, 512, 16, 4, 256),   # many partial M tiles
])
def test_grouped_swiglu_matches_oracle(moe, T, d, E, k, f):
    _gemm_case(moe, T, d, E, k, f, seed=T + d)


def test_grouped_swiglu_unscaled(moe):
    _gemm_case(moe, 200, 128, 4, 2, 128, seed=3, scale_rows=False)


def test_grouped_swiglu_empty_and_huge_groups(moe):
    counts = _gemm_case(moe, 2048, 256, 32, 4, 128, seed=5, skew=3.0)
    assert (counts == 0).sum() > 0 and counts.max() > 1000


def test_grouped_swiglu_max_experts(moe):
    # E = MOE_MAX_EXPERTS: the largest expert tables in the paired GEMM's shared
    # memory, ~16 rows per expert (one 16-token MMA per tile)
    counts = _gemm_case(moe, 2048, 256, 1024, 8, 128, seed=11)
    assert len(counts) == 1024


def test_grouped_swiglu_single_expert_long_k(moe):
    # E=1: one group covering every row; d = 2048 gives 32 K blocks
    _gemm_case(moe, 700, 2048, 1, 1, 256, seed=9)


# ---------------------------------------------------- group-limited routing
@pytest.mark.parametrize("T,E,k,G,ties", [(16384, 384, 8, 4, False), (16384, 384, 8, 8, False), (500, 8, 4, 2, True),
                                          (300, 64, 8, 2, True), (200, 48, 6, 3, False), (100, 64, 32, 4, False),
                                          (257, 1024, 8, 4, True)])
def test_grouped_route_matches_oracle(moe, T, E, k, G, ties):
    g = torch.Generator().manual_seed(T + E + k + G)
    l = torch.randn(T, E, generator=g)
    if ties:
        l = torch.round(l * 2) / 2
        l[torch.rand(T, E, generator=g) < 0.1] = -0.0
    for renorm in (True, False):
        idx, w = moe.moe_route_topk(l.cuda(), k, renorm, n_groups=G)
        ridx, rw = oracle.route_topk_grouped(l.numpy(), k, G, renorm)
        assert np.array_equal(to_np(idx), ridx)
        assert_gates_close(to_np(w), rw, k if renorm else E)


def test_grouped_route_balances_expert_groups_on_gpu(moe):
    cfg = workloads.get("skew")  # a router that strongly prefers a few experts
    l = _logits_for("skew").cuda()
    G = 4
    idx, w = moe.moe_route_topk(l, cfg.k, True, n_groups=G)
    res = moe.moe_dispatch_scan(idx, cfg.E, topk_w=w)
    per_group = to_np(res["counts"]).reshape(G, -1).sum(axis=1)
    assert per_group.tolist() == [cfg.T * cfg.k // G] * G

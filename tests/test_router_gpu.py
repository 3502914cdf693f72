"""The fused router (router GEMM + Softmax + TopK in one kernel) against the
fp64 oracle.

The kernel ranks fp32 logits accumulated on the tensor cores, the oracle
exact fp64 logits, so experts whose logits are closer than the fp32
accumulation error can legitimately swap.  For every token and selected
expert e the check is: logit64[e] >= (the oracle's k-th best logit) - eps,
with eps = (d + 2) * 2^-24 * sum_i |x_i w_ie| + 2^-20 (a rigorous bound on
fp32 accumulation of d products in any order), and the same bound on the
order of the slots.  Tokens whose oracle margins all exceed 2*eps must
match exactly, and at least 95 % of all tokens must (typical errors are
far below the worst-case bound); gates are checked against the oracle's
softmax over the experts the kernel chose.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import assert_values_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    return m


def _check_router(idx_gpu, w_gpu, x, wr, k, renorm):
    x64 = x.astype(np.float64)
    w64 = wr.astype(np.float64)
    ridx, rw, logits = oracle.router_topk(x64, w64, k, renorm)
    absdot = np.abs(x64) @ np.abs(w64)
    d = x.shape[1]
    eps = (d + 2) * 2.0 ** -24 * absdot + 2.0 ** -20
    T, E = logits.shape
    srt = -np.sort(-logits, axis=1)
    kth = srt[:, k - 1]
    exact_tokens = 0
    same = 0
    for t in range(T):
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == k and sel.min() >= 0 and sel.max() < E
        # every chosen expert is a valid top-k choice within the error bound
        assert np.all(logits[t, sel] >= kth[t] - eps[t, sel] - eps[t].max()), t
        # slots in descending order up to the bound
        assert np.all(logits[t, sel[:-1]] >= logits[t, sel[1:]] - eps[t, sel[:-1]] - eps[t, sel[1:]]), t
        same += list(sel) == list(ridx[t])
        margins = np.abs(np.diff(srt[t, : min(E, k + 1)]))
        if margins.size == 0 or margins.min() > 2 * eps[t].max():
            assert list(sel) == list(ridx[t]), t
            exact_tokens += 1
        # gates: softmax over the chosen experts (renormalised) or over all E
        z = np.exp(logits[t] - logits[t].max())
        ref = z[sel] / (z[sel].sum() if renorm else z.sum())
        # a logit error of eps moves a softmax probability by at most ~2*eps relative
        assert np.all(np.abs(w_gpu[t] - ref) <= 4 * eps[t].max() * ref.max() + 1e-6), t
    return exact_tokens, same / T


@pytest.mark.parametrize("T,d,E,k", [(256, 128, 8, 2), (1000, 2048, 64, 8), (300, 6144, 384, 8), (129, 256, 512, 32),
                                     (77, 64, 130, 3)])
@pytest.mark.parametrize("renorm", [True, False])
def test_router_topk_matches_oracle(moe, T, d, E, k, renorm):
    g = torch.Generator().manual_seed(T + d + E)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    wr = (torch.randn(d, E, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    packed = moe.moe_pack_router_weights(wr.cuda())
    idx, w = moe.moe_router_topk(x.cuda(), packed, E, k, renorm)
    _, same = _check_router(to_np(idx), to_np(w), to_np(x), to_np(wr), k, renorm)
    # the bound is worst case; actual fp32 errors are far smaller, so nearly
    # every token picks exactly the oracle's experts in the oracle's order
    assert same >= 0.95


def test_router_at_the_1t_layer_shape_matches_oracle_on_a_sample(moe):
    cfg = workloads.get("t1")
    x = workloads.generate(cfg, seed=0, device="cuda", weights=False)["x"]
    wr = workloads.generate_router(cfg, seed=0, device="cuda")
    packed = moe.moe_pack_router_weights(wr)
    idx, w = moe.moe_router_topk(x, packed, cfg.E, cfg.k)
    rows = torch.arange(0, cfg.T, 97, device="cuda")
    _, same = _check_router(to_np(idx[rows]), to_np(w[rows]), to_np(x[rows]), to_np(wr), cfg.k, True)
    assert same >= 0.95


def test_forward_from_router_weights_matches_oracle(moe):
    cfg = workloads.custom("routed", T=512, d=256, E=16, k=4, f=128)
    inp = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in workloads.generate(cfg, seed=6).items()}
    wr = workloads.generate_router(cfg, seed=6, device="cuda")
    rp = moe.moe_pack_router_weights(wr)
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    ws = torch.empty(moe.moe_forward_workspace_bytes(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f), dtype=torch.uint8,
                     device="cuda")
    out = moe.moe_forward_routed(inp["x"], rp, packed, cfg.E, cfg.k, cfg.f, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    inter = moe.forward_intermediates(ws, cfg.T, cfg.E, cfg.k, cfg.d, cfg.f)
    x = to_np(inp["x"])
    ridx, rw, logits = oracle.router_topk(x, to_np(wr), cfg.k)
    gidx = to_np(inter["topk_idx"])
    # the layer output is compared on tokens where the kernel chose the oracle's experts
    same = np.all(gidx == ridx, axis=1)
    assert same.mean() > 0.9
    ref_layer = oracle.moe_forward_tokens(x, None, to_np(inp["w_gate"]), to_np(inp["w_up"]), to_np(inp["w_down"]),
                                          cfg.k, True, routing=(ridx, rw))
    assert_values_close(to_np(out)[same], ref_layer["out"][same], "out (routed)")

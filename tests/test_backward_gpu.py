"""Parity of the backward kernels with the fp64 oracle, through the C ABI.

Output reduction, backward ("Scalable Pretraining of Large MoE LMs on Aurora
Super Computer", §3.1, Algorithm 1, stage 5): the gated row gradient is one
fp32 product rounded to bf16, so each element is held to one bf16 unit in
the last place, |err| <= 2^-7 |ref|; the gate gradient is an fp32 sum of d
exact bf16 x bf16 products, |err| <= d 2^-24 sum|y g| (the recursive-summation
bound).  Router-logit backward: fp32 softmax and sums against fp64,
|err_e| <= (2R + 2n + k + 16) 2^-24 (|w_e dw_e| + q_e sum_j |w_j dw_j|), n
the number of softmax terms and R the token's largest |l - max l| over them
(the rounding of l - max l moves exp by a relative R 2^-24); entries outside
the normalisation set are exactly 0 when the gates are renormalised.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import to_np

pytestmark = pytest.mark.gpu
U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    return m


def _bf16(gen, *shape, scale=1.0):
    return (torch.randn(*shape, generator=gen) * scale).to(torch.bfloat16)


def _check_combine_backward(dy, dw, dout, y, dst, w):
    """dout, y: bf16 host tensors; dst, w: host numpy; compare with the oracle."""
    g64 = dout.double().numpy()
    y64 = y.double().numpy()
    rdy, rdw = oracle.combine_backward(g64, y64, dst, w.astype(np.float64))
    got = to_np(dy).astype(np.float64)
    assert np.all(np.abs(got - rdy) <= 2.0 ** -7 * np.abs(rdy)), "d_mlp_out beyond one bf16 ulp"
    T, k = w.shape
    d = g64.shape[1]
    rows = np.asarray(dst, dtype=np.int64).reshape(T, k)
    bound = np.stack([np.abs(y64[rows[:, j]] * g64).sum(axis=1) for j in range(k)], axis=1) * d * U32
    err = np.abs(to_np(dw).astype(np.float64) - rdw)
    assert np.all(err <= bound + 1e-30), f"d_topk_w: worst excess {np.max(err - bound):.3e}"


@pytest.mark.parametrize("T,d,E,k", [(1, 8, 1, 1), (37, 136, 7, 3), (256, 128, 8, 2), (999, 2048, 64, 8),
                                     (300, 6144, 384, 8), (64, 24, 4, 4)])
def test_combine_backward_matches_oracle(moe, T, d, E, k):
    gen = torch.Generator().manual_seed(T * 7 + d)
    l = torch.randn(T, E, generator=gen)
    idx, w = oracle.route_topk(l.numpy(), k)
    _, _, _, dst = oracle.dispatch(idx, E)
    dout = _bf16(gen, T, d)
    y = _bf16(gen, T * k, d, scale=3.0)
    w32 = w.astype(np.float32)
    dy, dw = moe.moe_combine_backward(dout.cuda(), y.cuda(), torch.from_numpy(dst.astype(np.int32)).cuda(),
                                      torch.from_numpy(w32).cuda())
    _check_combine_backward(dy, dw, dout, y, dst, w32)


def test_combine_backward_full_layer_sampled(moe):
    """16384 tokens, d = 6144, k = 8, 384 experts: every output is computed,
    a seeded sample of 256 tokens (and their 2048 rows) checked."""
    cfg = workloads.get("t1")
    l = workloads.generate_logits("t1", 0)
    idx, w = moe.moe_route_topk(l.cuda(), cfg.k)
    res = moe.moe_dispatch_scan(idx, cfg.E)
    gen = torch.Generator().manual_seed(5)
    dout = _bf16(gen, cfg.T, cfg.d).cuda()
    y = _bf16(gen, cfg.T * cfg.k, cfg.d, scale=3.0).cuda()
    dy, dw = moe.moe_combine_backward(dout, y, res["dest_row"], w)
    torch.cuda.synchronize()
    sample = np.sort(np.random.default_rng(6).choice(cfg.T, 256, replace=False))
    rows = to_np(res["dest_row"]).astype(np.int64).reshape(cfg.T, cfg.k)[sample]
    compact = np.arange(rows.size)            # token i, slot j -> row i*k + j of the gathered rows
    flat = rows.reshape(-1)
    _check_combine_backward(dy[torch.from_numpy(flat).cuda()], dw[torch.from_numpy(sample).cuda()],
                            dout[torch.from_numpy(sample).cuda()].cpu(), y[torch.from_numpy(flat).cuda()].cpu(),
                            compact, to_np(w)[sample])


def test_combine_backward_empty(moe):
    dy, dw = moe.moe_combine_backward(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"),
                                      torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"),
                                      torch.empty(0, dtype=torch.int32, device="cuda"),
                                      torch.empty(0, 2, dtype=torch.float32, device="cuda"))
    assert dy.shape == (0, 64) and dw.shape == (0, 2)


def _check_route_backward(got, l, idx, dw, renorm):
    l64 = np.asarray(l, dtype=np.float64)
    ref = oracle.route_backward(l64, idx, dw.astype(np.float64), renorm)
    T, E = l64.shape
    k = idx.shape[1]
    ii = idx.astype(np.int64)
    if renorm:
        z = np.exp(np.take_along_axis(l64, ii, axis=1) - l64.max(axis=1, keepdims=True))
        wts = z / z.sum(axis=1, keepdims=True)
        q = np.zeros((T, E))
        np.put_along_axis(q, ii, wts, axis=1)
        sel = np.take_along_axis(l64, ii, axis=1)
        R = sel.max(axis=1, keepdims=True) - sel.min(axis=1, keepdims=True)
        n = k
    else:
        q = oracle.softmax_rows(l64)
        wts = np.take_along_axis(q, ii, axis=1)
        R = l64.max(axis=1, keepdims=True) - l64.min(axis=1, keepdims=True)
        n = E
    own = np.zeros((T, E))
    np.put_along_axis(own, ii, np.abs(wts * dw), axis=1)
    bound = (2 * R + 2 * n + k + 16) * U32 * (own + q * np.abs(wts * dw).sum(axis=1, keepdims=True))
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-38), f"d_logits: worst excess {np.max(err - bound):.3e}"
    if renorm:
        outside = np.ones((T, E), dtype=bool)
        np.put_along_axis(outside, ii, False, axis=1)
        assert np.all(got[outside] == 0.0)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (33, 7, 7), (100, 32, 32), (64, 1024, 32), (257, 1024, 8),
                                   (50, 33, 3), (513, 384, 8), (40, 400, 6)])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_backward_matches_oracle(moe, T, E, k, renorm):
    gen = torch.Generator().manual_seed(T * 131 + E)
    l = torch.randn(T, E, generator=gen) * 2
    idx, _ = moe.moe_route_topk(l.cuda(), k, renorm)
    dw = torch.randn(T, k, generator=gen)
    got = moe.moe_route_backward(l.cuda(), idx, dw.cuda(), renorm)
    _check_route_backward(to_np(got), l.numpy(), to_np(idx), dw.numpy(), renorm)


@pytest.mark.parametrize("renorm", [True, False])
def test_route_backward_full_layer(moe, renorm):
    cfg = workloads.get("t1")
    l = workloads.generate_logits("t1", 0)
    idx, _ = moe.moe_route_topk(l.cuda(), cfg.k, renorm)
    dw = torch.randn(cfg.T, cfg.k, generator=torch.Generator().manual_seed(9))
    got = moe.moe_route_backward(l.cuda(), idx, dw.cuda(), renorm)
    _check_route_backward(to_np(got), l.numpy(), to_np(idx), dw.numpy(), renorm)


def test_route_backward_empty(moe):
    out = moe.moe_route_backward(torch.empty(0, 8, device="cuda"), torch.empty(0, 2, dtype=torch.int32,
                                                                               device="cuda"),
                                 torch.empty(0, 2, device="cuda"))
    assert out.shape == (0, 8)

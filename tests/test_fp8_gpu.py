"""Blockwise FP8 weight encoding on the GPU against the reference.

Codes, scales and dequantised weights are integer/bit-level decisions taken
in the precision the page fixes (fp32 scale and division, E4M3 round to
nearest even, bf16 result), so they must match the reference bit for bit.
The layer run from FP8-stored weights is compared with the oracle on the
same dequantised weights, to the usual value tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import fp8_oracle as f8
from tests.parity import assert_values_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    return m


def _awkward_weights(n_blocks, seed):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal(n_blocks * 128).astype(np.float32)
    w *= np.repeat(10.0 ** rng.uniform(-6, 2, n_blocks), 128).astype(np.float32)   # per-block magnitudes
    w[:128] = 0.0                                  # an all-zero block
    w[128:256:3] = -0.0                            # signed zeros
    w[256:384] *= 1e-4                             # values that land in E4M3's subnormal range
    w[384] = 1e4                                   # one large outlier in its block
    return torch.from_numpy(w).to(torch.bfloat16)


@pytest.mark.parametrize("n_blocks,seed", [(1, 0), (40, 1), (4096, 2)])
def test_quantize_and_dequantize_match_reference_bit_for_bit(moe, n_blocks, seed):
    w = _awkward_weights(max(n_blocks, 4), seed)
    codes, scales = moe.moe_quantize_fp8_blockwise(w.cuda())
    rc, rs = f8.quantize_blockwise(w)
    assert np.array_equal(to_np(codes), rc)
    assert np.array_equal(to_np(scales), rs)
    back = moe.moe_dequantize_fp8_blockwise(codes, scales)
    assert torch.equal(back.cpu().view(torch.int16), f8.dequantize_blockwise(rc, rs).view(torch.int16))


def test_expert_weights_of_the_1t_layer_sampled(moe):
    cfg = workloads.get("t1")
    g = torch.Generator(device="cuda").manual_seed(0)
    w = (torch.randn(16, cfg.d, cfg.f, generator=g, device="cuda") / math.sqrt(cfg.d)).to(torch.bfloat16)
    codes, scales = moe.moe_quantize_fp8_blockwise(w)
    for e in (0, 7, 15):
        n = cfg.d * cfg.f
        rc, rs = f8.quantize_blockwise(w[e].cpu())
        assert np.array_equal(to_np(codes[e * n:(e + 1) * n]), rc)
        assert np.array_equal(to_np(scales[e * n // 128:(e + 1) * n // 128]), rs)


def test_layer_from_fp8_weights_matches_oracle(moe):
    cfg = workloads.get("small")
    inp = workloads.generate(cfg, seed=4)
    deq = {}
    packed_in = {}
    for name in ("w_gate", "w_up", "w_down"):
        w = inp[name]
        codes, scales = moe.moe_quantize_fp8_blockwise(w.cuda())
        packed_in[name] = moe.moe_dequantize_fp8_blockwise(codes, scales, shape=w.shape)
        rc, rs = f8.quantize_blockwise(w)
        deq[name] = f8.dequantize_blockwise(rc, rs).view(w.shape)
        assert torch.equal(packed_in[name].cpu(), deq[name])
    packed = moe.moe_pack_weights(packed_in["w_gate"], packed_in["w_up"], packed_in["w_down"])
    x, logits = inp["x"].cuda(), inp["logits"].cuda()
    out = moe.moe_forward(x, logits, packed, cfg.E, cfg.k, cfg.f)
    torch.cuda.synchronize()
    toks = np.arange(0, cfg.T, 37)
    ref = oracle.moe_forward_tokens(inp["x"][toks].float().numpy(), inp["logits"][toks].numpy(),
                                    deq["w_gate"].float().numpy(), deq["w_up"].float().numpy(),
                                    deq["w_down"].float().numpy(), cfg.k)
    assert_values_close(to_np(out)[toks], ref["out"], "out (fp8 weights)")
    # and the FP8 weights change the layer by about the page's weight error
    ref_bf16 = oracle.moe_forward_tokens(inp["x"][toks].float().numpy(), inp["logits"][toks].numpy(),
                                         inp["w_gate"].float().numpy(), inp["w_up"].float().numpy(),
                                         inp["w_down"].float().numpy(), cfg.k)
    rel = np.abs(ref["out"] - ref_bf16["out"]).mean() / np.abs(ref_bf16["out"]).mean()
    assert 1e-3 < rel < 0.1

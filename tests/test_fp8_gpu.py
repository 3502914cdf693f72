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


# ------------------------------------------- FP8 weights read by the GEMMs
def _fp8_layer(moe, cfg, inp):
    """(packed FP8 weights, packed bf16 copies of the dequantised weights)."""
    q = {}
    deq = {}
    for name in ("w_gate", "w_up", "w_down"):
        w = inp[name]
        q[name] = moe.moe_quantize_fp8_blockwise(w.reshape(-1))
        deq[name] = moe.moe_dequantize_fp8_blockwise(*q[name], shape=w.shape)
    packed_fp8 = moe.moe_pack_weights_fp8(q["w_gate"], q["w_up"], q["w_down"], cfg.E, cfg.d, cfg.f)
    packed_deq = moe.moe_pack_weights(deq["w_gate"], deq["w_up"], deq["w_down"])
    return packed_fp8, packed_deq, deq


FP8_CASES = [
    workloads.custom("fp8_pairs", T=1536, d=256, E=8, k=2, f=128),    # tiles of > 256 tokens, ragged groups
    workloads.custom("fp8_wide", T=700, d=512, E=16, k=4, f=384),     # three gate/up scale blocks per row
    "small", "t1", "skew",
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: c if isinstance(c, str) else c.name)
def test_fp8_weight_forward_is_bit_identical_to_dequantised_weights(moe, case):
    """moe_forward_fp8 dequantises each stage's codes in shared memory to
    exactly moe_dequantize_fp8_blockwise's bf16 values, so H, Y and the
    output equal moe_forward's on the dequantised weights bit for bit."""
    cfg = workloads.get(case)
    inp = workloads.generate(cfg, seed=5, device="cuda")
    packed_fp8, packed_deq, _ = _fp8_layer(moe, cfg, inp)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    nbytes = moe.moe_forward_workspace_bytes(T, E, k, d, f)
    ws1 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ref = moe.moe_forward(inp["x"], inp["logits"], packed_deq, E, k, f, cfg.renormalize, workspace=ws1)
    got = moe.moe_forward_fp8(inp["x"], inp["logits"], packed_fp8, E, k, f, cfg.renormalize, workspace=ws2)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws2) == 0
    i1 = moe.forward_intermediates(ws1, T, E, k, d, f)
    i2 = moe.forward_intermediates(ws2, T, E, k, d, f)
    assert torch.equal(i1["h"], i2["h"]), "h"
    assert torch.equal(i1["y"], i2["y"]), "y"
    assert torch.equal(ref, got)


def test_fp8_weight_forward_against_oracle(moe):
    """The same layer held to the fp64 oracle on the dequantised weights."""
    cfg = workloads.custom("fp8_oracle", T=1536, d=256, E=8, k=2, f=128)
    inp = workloads.generate(cfg, seed=6)
    dev = {kk: (v.cuda() if torch.is_tensor(v) else v) for kk, v in inp.items()}
    packed_fp8, _, deq = _fp8_layer(moe, cfg, dev)
    out = moe.moe_forward_fp8(dev["x"], dev["logits"], packed_fp8, cfg.E, cfg.k, cfg.f)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(inp["x"].float().numpy(), inp["logits"].numpy(), to_np(deq["w_gate"]),
                             to_np(deq["w_up"]), to_np(deq["w_down"]), cfg.k, True)
    assert_values_close(to_np(out), ref["out"], "out (FP8 weights in the GEMMs)")


def test_fp8_pack_layout_of_codes_and_scales(moe):
    """Bytes of the packed layout against their definition: code (e, n, k) of
    gate/up tile t and K block b at row 32g + 16h + r, down tile t at row n %
    128; scale records of 136 (gate/up) and 64 (down) floats."""
    E, d, f = 2, 256, 256
    g = torch.Generator().manual_seed(7)
    ws = [(torch.randn(E, d, f, generator=g) / 16).to(torch.bfloat16) for _ in range(2)]
    wd = (torch.randn(E, f, d, generator=g) / 16).to(torch.bfloat16)
    q = [moe.moe_quantize_fp8_blockwise(w.reshape(-1).cuda()) for w in (ws[0], ws[1], wd)]
    packed = moe.moe_pack_weights_fp8(q[0], q[1], q[2], E, d, f).cpu().numpy()
    gc, uc, dc = (to_np(c).reshape(E, -1) for c, _ in q)
    gs, us, ds = (to_np(s) for _, s in q)
    gate_c = gc.reshape(E, d, f)
    up_c = uc.reshape(E, d, f)
    down_c = dc.reshape(E, f, d)
    codes_gu = packed[:E * 2 * f * d].reshape(E, 2 * f // 128, d // 64, 128, 64)
    for e, t, b, s_ in ((0, 0, 0, 0), (1, 3, 2, 77), (1, 2, 3, 127), (0, 1, 1, 40)):
        gq, h, r = s_ // 32, (s_ // 16) % 2, s_ % 16
        feat = 64 * t + 16 * gq + r
        src = (up_c if h else gate_c)[e, 64 * b:64 * b + 64, feat]
        assert np.array_equal(codes_gu[e, t, b, s_], src), (e, t, b, s_)
    codes_dn = packed[E * 2 * f * d:E * 3 * f * d].reshape(E, d // 128, f // 64, 128, 64)
    for e, t, b, s_ in ((0, 0, 0, 0), (1, 1, 3, 99)):
        assert np.array_equal(codes_dn[e, t, b, s_], down_c[e, 64 * b:64 * b + 64, 128 * t + s_])
    off = 3 * E * d * f
    rec_gu = packed[off:off + E * (f // 128) * (d // 64) * 136 * 4].view(np.float32).reshape(E, f // 128, d // 64, 136)
    gsr = gs.reshape(E, d, f // 128)
    usr = us.reshape(E, d, f // 128)
    for e, fb, b in ((0, 0, 0), (1, 1, 3)):
        assert np.array_equal(rec_gu[e, fb, b, :64], gsr[e, 64 * b:64 * b + 64, fb])
        assert np.array_equal(rec_gu[e, fb, b, 68:132], usr[e, 64 * b:64 * b + 64, fb])
        assert not rec_gu[e, fb, b, 64:68].any() and not rec_gu[e, fb, b, 132:].any()
    off2 = off + ((E * (f // 128) * (d // 64) * 136 * 4 + 255) // 256) * 256
    rec_dn = packed[off2:off2 + E * (d // 128) * (f // 64) * 64 * 4].view(np.float32).reshape(E, d // 128, f // 64, 64)
    dsr = ds.reshape(E, f, d // 128)
    for e, db, b in ((0, 0, 0), (1, 1, 2)):
        assert np.array_equal(rec_dn[e, db, b], dsr[e, 64 * b:64 * b + 64, db])

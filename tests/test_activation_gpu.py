"""Error of the activation functions the expert-GEMM epilogues apply.

Silu(z) = z * sigmoid(z) ("Scalable Pretraining of Large MoE LMs on Aurora
Super Computer", §3.1, Algorithm 1, stage 4: Silu(gate) * up; the backward
uses sigmoid for Silu').  The device computes both through the hardware tanh,
sigmoid(z) = (1 + tanh(z / 2)) / 2; the bounds below are checked against the
fp64 definitions on a dense grid and at the saturating ends.
"""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m  # must load: no fallback exists
    return m

BF16_ULP = 2.0 ** -8  # relative spacing of bf16 values


def _ref(z):
    zd = z.double()
    sig = torch.sigmoid(zd)
    return zd * sig, sig


def test_activation_matches_fp64_definition(moe):
    z = torch.linspace(-20.0, 20.0, 2_000_001, dtype=torch.float32)
    silu, sig = moe.moe_selftest_activation(z.cuda())
    silu_ref, sig_ref = _ref(z)
    silu, sig = silu.cpu().double(), sig.cpu().double()
    assert (sig - sig_ref).abs().max().item() <= 1e-5
    err = (silu - silu_ref).abs()
    assert err.max().item() <= 2e-5
    zd = z.double()
    rel = err / silu_ref.abs().clamp_min(1e-30)
    assert rel[zd >= -4].max().item() <= 2e-4
    assert rel[(zd >= -8) & (zd < -4)].max().item() <= BF16_ULP


def test_activation_special_values(moe):
    z = torch.tensor([0.0, -0.0, 1e-30, -1e-30, 88.0, -88.0, 1e4, -1e4, math.inf, -math.inf, math.nan])
    silu, sig = moe.moe_selftest_activation(z.cuda())
    silu, sig = silu.cpu(), sig.cpu()
    assert silu[0].item() == 0.0 and silu[1].item() == 0.0
    assert sig[0].item() == 0.5
    assert silu[6].item() == 1e4 and silu[7].item() == 0.0
    assert sig[6].item() == 1.0 and sig[7].item() == 0.0
    assert silu[4].item() == pytest.approx(88.0, rel=1e-6) and abs(silu[5].item()) < 1e-5
    assert sig[8].item() == 1.0 and sig[9].item() == 0.0
    assert math.isnan(silu[10].item()) and math.isnan(sig[10].item())


def test_activation_empty(moe):
    silu, sig = moe.moe_selftest_activation(torch.empty(0, device="cuda"))
    assert silu.numel() == 0 and sig.numel() == 0

"""The expert GEMMs under the static tile schedule and beside a kernel
that holds part of the GPU.

The static schedule (pair i takes tiles i, i + pairs, ...) changes only
which SM pair runs a tile and when, so every output equals the dynamically
scheduled one bit for bit.  With moe_occupy_sms holding 40 SMs on another
stream, the layer runs on the remaining SMs (and on all of them once the
occupier returns) with the same outputs.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    yield m
    m.moe_set_tile_schedule(m.TILE_SCHEDULE_DYNAMIC)


def _case(name):
    if name == "pairs":
        return workloads.custom("pairs", T=1536, d=256, E=8, k=2, f=128)
    return workloads.get(name)


@pytest.mark.parametrize("name", ["small", "pairs"])
def test_static_schedule_gives_the_same_layer(moe, name):
    cfg = _case(name)
    inp = workloads.generate(cfg, seed=0, device="cuda")
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    args = (inp["x"], inp["logits"], packed, cfg.E, cfg.k, cfg.f, cfg.renormalize)
    moe.moe_set_tile_schedule(moe.TILE_SCHEDULE_DYNAMIC)
    ref = moe.moe_forward(*args)
    moe.moe_set_tile_schedule(moe.TILE_SCHEDULE_STATIC)
    got = moe.moe_forward(*args)
    moe.moe_set_tile_schedule(moe.TILE_SCHEDULE_DYNAMIC)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("mode", ["dynamic", "static"])
def test_layer_beside_an_occupier_gives_the_same_layer(moe, mode):
    cfg = _case("small")
    inp = workloads.generate(cfg, seed=1, device="cuda")
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    args = (inp["x"], inp["logits"], packed, cfg.E, cfg.k, cfg.f, cfg.renormalize)
    ref = moe.moe_forward(*args)
    torch.cuda.synchronize()
    moe.moe_set_tile_schedule(moe.TILE_SCHEDULE_STATIC if mode == "static" else moe.TILE_SCHEDULE_DYNAMIC)
    side = torch.cuda.Stream()
    moe.moe_occupy_sms(40, 2_000_000, stream=side)  # 2 ms on 40 SMs
    got = moe.moe_forward(*args)
    torch.cuda.synchronize()
    moe.moe_set_tile_schedule(moe.TILE_SCHEDULE_DYNAMIC)
    assert torch.equal(got, ref)


def test_occupier_argument_errors(moe):
    n = torch.cuda.get_device_properties(0).multi_processor_count
    for bad in ((-1, 1000), (n + 1, 1000), (1, -1), (1, 10_000_000_001)):
        with pytest.raises(RuntimeError):
            moe.moe_occupy_sms(*bad)
    moe.moe_occupy_sms(0, 0)
    torch.cuda.synchronize()

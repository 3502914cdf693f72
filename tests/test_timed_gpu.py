"""The timed entry points: stage events recorded on the launching stream.

moe_forward_timed (and its FP8, gathered and backward siblings) must compute
exactly what the untimed call computes; an event array may hold NULL entries,
which record nothing, so that a caller can bracket one kernel alone.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import sparse_expert_gb300 as m
    return m


def _setup(moe):
    cfg = workloads.custom("timed", T=1536, d=256, E=8, k=2, f=128)
    inp = workloads.generate(cfg, seed=0, device="cuda")
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    ws = torch.empty(moe.moe_forward_workspace_bytes(cfg.T, cfg.E, cfg.k, cfg.d, cfg.f), dtype=torch.uint8,
                     device="cuda")
    return cfg, inp, packed, ws


@pytest.mark.parametrize("keep", [(0, 1, 2, 3, 4, 5, 6), (3, 4, 5), (), (0, 6)])
def test_forward_timed_with_partial_events_matches_forward(moe, keep):
    cfg, inp, packed, ws = _setup(moe)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    x, logits = inp["x"], inp["logits"]
    ref = moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    n = len(moe.FORWARD_STAGES) + 1
    ev = [torch.cuda.Event(enable_timing=True) if i in keep else None for i in range(n)]
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward_timed(x, logits, packed, E, k, f, ws, out, ev, cfg.renormalize, stream)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    assert torch.equal(out, ref)
    kept = [e for e in ev if e is not None]
    for a, b in zip(kept, kept[1:]):
        assert a.query() and b.query()
        assert a.elapsed_time(b) >= 0.0


def test_backward_timed_with_partial_events_matches_backward(moe):
    cfg, inp, packed, _ = _setup(moe)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    x, logits = inp["x"], inp["logits"]
    dout = torch.randn(T, d, generator=torch.Generator(device="cuda").manual_seed(5), device="cuda",
                       dtype=torch.float32).to(torch.bfloat16)
    wsb = torch.empty(moe.moe_backward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
    ref = {n: t.clone() for n, t in moe.moe_backward(x, logits, packed, dout, E, k, f, cfg.renormalize,
                                                    workspace=wsb).items()}
    torch.cuda.synchronize()
    n = len(moe.BACKWARD_STAGES) + 1
    keep = (1, 2, 5, 7, 9)  # includes boundaries inside the backward GEMM launcher
    ev = [torch.cuda.Event(enable_timing=True) if i in keep else None for i in range(n)]
    grads = {nm: torch.empty_like(t) for nm, t in ref.items()}
    moe.moe_backward_timed(x, logits, packed, dout, E, k, f, wsb, grads, ev, cfg.renormalize)
    torch.cuda.synchronize()
    for nm, t in ref.items():
        assert torch.equal(grads[nm], t), nm
    kept = [e for e in ev if e is not None]
    for a, b in zip(kept, kept[1:]):
        assert a.elapsed_time(b) >= 0.0

"""The layer forward captured into a CUDA graph and replayed.

moe_forward and moe_forward_routed put every step on the caller's stream
with no host synchronisation (the workspace header, the count table and the
GEMMs' tile counter are cleared by stream operations), so a whole layer can
be captured once and replayed.  A replay must give exactly what a direct
call gives on the same inputs, also after the inputs change in place between
replays (the graph reads the buffers, not a snapshot).
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


def _inputs(moe, name, seed):
    cfg = workloads.get(name) if name in ("tiny", "small") else workloads.custom(name, T=1536, d=256, E=8, k=2, f=128)
    inp = workloads.generate(cfg, seed=seed, device="cuda")
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    return cfg, inp, packed


@pytest.mark.parametrize("name", ["tiny", "small", "pairs"])
def test_forward_graph_replay_matches_direct_calls(moe, name):
    cfg, inp, packed = _inputs(moe, name, seed=0)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    x, logits = inp["x"], inp["logits"]
    ws = torch.empty(moe.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")

    # warm up outside the capture (first launches set kernel attributes)
    moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, topk_idx=idx,
                            topk_w=w, stream=stream)

    for seed in (1, 2):
        # new inputs written in place, then one replay and one direct call
        _, new, _ = _inputs(moe, name, seed=seed)
        x.copy_(new["x"])
        logits.copy_(new["logits"])
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(ws) == 0
        got = (out.clone(), idx.clone(), w.clone())
        ref_out = moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize)
        ref_idx = torch.empty_like(idx)
        ref_w = torch.empty_like(w)
        moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, topk_idx=ref_idx, topk_w=ref_w)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref_out), seed
        assert torch.equal(got[1], ref_idx), seed
        assert torch.equal(got[2], ref_w), seed


def test_routed_forward_graph_replay_matches_direct_call(moe):
    cfg = workloads.custom("routed_graph", T=512, d=256, E=16, k=4, f=128)
    inp = workloads.generate(cfg, seed=0, device="cuda")
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    wr = workloads.generate_router(cfg, seed=0, device="cuda")
    rp = moe.moe_pack_router_weights(wr)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    x = inp["x"]
    ws = torch.empty(moe.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward_routed(x, rp, packed, E, k, f, cfg.renormalize, workspace=ws, out=out)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            moe.moe_forward_routed(x, rp, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
    x.copy_(workloads.generate(cfg, seed=3, device="cuda")["x"])
    graph.replay()
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    ref = moe.moe_forward_routed(x, rp, packed, E, k, f, cfg.renormalize)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)

"""Dynamic tile schedule and per-expert readiness counts of the weights-on-M
bf16 expert GEMMs (the down GEMM runs as a programmatic dependent of gate/up
and waits per expert for its h rows): the counters live in the workspace
header and every call must leave them at zero.  Repeated calls (and a CUDA
graph replayed several times) give bit-identical results, and the counters
read back as zero after each."""
import numpy as np
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCHED_WORDS = slice(32, 36)  # header words of the two schedule counter pairs
DONE_WORDS = slice(64, 64 + 256)  # per-expert published gate/up tiles


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


def header_words(ws):
    torch.cuda.synchronize()
    return ws[:2048].view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("name,T", [("tiny", 64), ("decode", 64)])
def test_repeated_forwards_identical_and_counters_zero(lib, name, T):
    cfg = mi.CONFIGS[name].with_T(T)
    x, wr, b = (t.to(DEV) for t in mi.make_router_inputs(cfg, seed=4))
    ex = lib.Experts(*mi.make_expert_weights(cfg, device=DEV, seed=4))
    d = lib.dims_of(cfg)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD)
    ys = []
    for _ in range(5):
        y = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=DEV)
        lib.moe_forward(d, x, wr, b, ex, y, ws)
        h = header_words(ws)
        assert h[0] == 0 and not h[SCHED_WORDS].any() and not h[DONE_WORDS].any(), h[:80]
        ys.append(y)
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_graph_replays_identical_and_counters_zero(lib):
    cfg = mi.CONFIGS["decode"]
    x, wr, b = (t.to(DEV) for t in mi.make_router_inputs(cfg, seed=5))
    ex = lib.Experts(*mi.make_expert_weights(cfg, device=DEV, seed=5))
    d = lib.dims_of(cfg)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD)
    y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    lib.moe_forward(d, x, wr, b, ex, y, ws)
    ref = y.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lib.moe_forward(d, x, wr, b, ex, y, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lib.moe_forward(d, x, wr, b, ex, y, ws)
    for _ in range(4):
        y.zero_()
        g.replay()
        h = header_words(ws)
        assert h[0] == 0 and not h[SCHED_WORDS].any() and not h[DONE_WORDS].any(), h[:80]
        assert torch.equal(y, ref)

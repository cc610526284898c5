"""moe_forward under CUDA graph capture: the C ABI allocates nothing and never
synchronises, so a captured forward replays the same kernels.  Replays must
equal eager calls bit for bit (the path is deterministic), including after the
input buffer's contents change between replays."""
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


@pytest.mark.parametrize("T,weights", [(64, "bf16"), (2048, "bf16"), (200, "nvfp4-a4"),
                                       (64, "nvfp4"), (2048, "nvfp4"), (64, "fp8"), (2048, "fp8")])
def test_graph_replay_matches_eager(lib, T, weights):
    """The packed W4A16 / W8A16 cases cover both packed GEMM paths (T=64: the
    tensor-memory GEMMs and their chain of four dependent launches; T=2048:
    the token-major ones with the scaled gather and the h rescaling)."""
    cfg = mi.CONFIGS["tiny"].with_T(T)
    if weights != "bf16":
        cfg = mi.MoeConfig("tiny-packed", T=T, H=256, E=32, n_group=8, topk_group=2, top_k=4, I=256,
                           weights="nvfp4")
    x, wr, b = (t.to(DEV) for t in mi.make_router_inputs(cfg, seed=3))
    w = mi.make_expert_weights(cfg, device=DEV, seed=3)
    if weights == "bf16":
        ex = lib.Experts(*w)
    elif weights == "fp8":
        packed = [mi.quantize_experts_fp8(t) for t in w]
        ex = lib.Experts(*[p[0] for p in packed], None, None, None, *[p[1] for p in packed])
    else:
        packed = [mi.quantize_experts_nvfp4(t) for t in w]
        a4 = (mi.A4_X_GLOBAL, mi.A4_H_GLOBAL) if weights == "nvfp4-a4" else None
        ex = lib.Experts(*[p[i] for i in range(3) for p in packed], a4=a4)
    d = lib.dims_of(cfg)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, ex.dtype)
    y = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(T, cfg.top_k, dtype=torch.int32, device=DEV)
    tw = torch.empty(T, cfg.top_k, dtype=torch.float32, device=DEV)

    def fwd():
        lib.moe_forward(d, x, wr, b, ex, y, ws, idx, tw)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fwd()  # first call outside capture: kernel attributes, tensor-map entry point
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    y_eager = y.clone()
    idx_eager = idx.clone()

    g = torch.cuda.CUDAGraph()
    y.zero_()
    with torch.cuda.graph(g):
        fwd()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)
    assert torch.equal(idx, idx_eager)

    # new input contents, same buffers: a replay equals a fresh eager call
    x.copy_(torch.roll(x, shifts=1, dims=0))
    g.replay()
    torch.cuda.synchronize()
    y_replay = y.clone()
    fwd()
    torch.cuda.synchronize()
    assert torch.equal(y_replay, y)
    assert lib.workspace_status(ws) == 0

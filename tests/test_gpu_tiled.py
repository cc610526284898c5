"""MMA-tiled bf16 expert weights (moe_pack_bf16, layout MOE_LAYOUT_TILED): the
packed bytes follow the documented tile order and swizzle, and a forward with
packed weights equals the row-major forward bit for bit on both GEMM paths
(weights on M for small batches, token-major for large ones)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


def test_pack_layout(lib):
    E, N, K = 2, 256, 192
    w = torch.arange(E * N * K, dtype=torch.int32).remainder(30011).to(torch.float32)
    w = (w / 64).to(torch.bfloat16).reshape(E, N, K).to(DEV)
    p = lib.moe_pack_bf16(w)
    torch.cuda.synchronize()
    src = w.cpu().view(torch.int16).numpy().reshape(E * N, K // 8, 8)  # 16-byte chunks
    got = p.cpu().view(torch.int16).numpy().reshape(-1, 8)
    ktiles = K // 64
    for row in range(E * N):
        rblk, r = divmod(row, 128)
        for kc in range(K // 8):
            kt, c = divmod(kc, 8)
            tile = rblk * ktiles + kt
            pos = tile * 1024 + (r // 8) * 64 + (r % 8) * 8 + (c ^ (r % 8))
            assert np.array_equal(got[pos], src[row, kc])


def test_pack_rejects_bad_shapes(lib):
    with pytest.raises(lib.MoeError):
        lib.moe_pack_bf16(torch.zeros(1, 100, 64, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(lib.MoeError):
        lib.moe_pack_bf16(torch.zeros(1, 128, 96, dtype=torch.bfloat16, device=DEV))


@pytest.mark.parametrize("name,T", [("tiny", 64), ("tiny", 2048), ("decode", 64)])
def test_tiled_forward_equals_row_major(lib, name, T):
    cfg = mi.CONFIGS[name].with_T(T)
    x, wr, b = (t.to(DEV) for t in mi.make_router_inputs(cfg, seed=2))
    wg, wu, wd = mi.make_expert_weights(cfg, device=DEV, seed=2)
    d = lib.dims_of(cfg)

    def fwd(ex):
        ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD)
        y = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=DEV)
        lib.moe_forward(d, x, wr, b, ex, y, ws)
        assert lib.workspace_status(ws) == 0
        return y

    y_rm = fwd(lib.Experts(wg, wu, wd))
    packed = [lib.moe_pack_bf16(t) for t in (wg, wu, wd)]
    del wg, wu, wd
    torch.cuda.empty_cache()
    y_t = fwd(lib.Experts(*packed, tiled=True))
    assert torch.equal(y_t, y_rm)


def test_tiled_rejected_for_packed_formats(lib):
    cfg = mi.CONFIGS["tiny"]
    d = lib.dims_of(cfg)
    q = torch.zeros(cfg.E, cfg.I, cfg.H, dtype=torch.uint8, device=DEV)
    qd = torch.zeros(cfg.E, cfg.H, cfg.I, dtype=torch.uint8, device=DEV)
    g = torch.ones(cfg.E, cfg.I, dtype=torch.float32, device=DEV)
    gd = torch.ones(cfg.E, cfg.H, dtype=torch.float32, device=DEV)
    ex = lib.Experts(q, q, qd, None, None, None, g, g, gd)
    st = ex.struct(d)
    st.layout = lib.MOE_LAYOUT_TILED
    x = torch.zeros(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros(cfg.E, cfg.H, dtype=torch.float32, device=DEV)
    b = torch.zeros(cfg.E, dtype=torch.float32, device=DEV)
    y = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=DEV)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, lib.MOE_W_FP8)
    import ctypes
    rc = lib.native().moe_forward(ctypes.byref(d), x.data_ptr(), wr.data_ptr(), b.data_ptr(),
                                  ctypes.byref(st), y.data_ptr(), None, None, ws.data_ptr(),
                                  ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 2  # MOE_ERR_UNSUPPORTED

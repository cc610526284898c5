"""Tiled expert weights (layout MOE_LAYOUT_TILED): the bytes written by
moe_pack_bf16, moe_pack_nvfp4 and moe_pack_fp8 follow the documented tile
order (and, for bf16, the swizzle), and a forward with tiled bf16 weights
equals the row-major forward bit for bit on both GEMM paths (weights on M for
small batches, token-major for large ones).  The NVFP4 and FP8 forwards with
tiled weights are checked in their own parity files."""
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


def _tiles(a, ktiles, row_bytes):
    """[E*N, K-bytes] -> [row block, k block, 128, row_bytes]: the tile grid of
    the documented layouts."""
    rows = a.shape[0]
    return a.reshape(rows // 128, 128, ktiles, row_bytes).transpose(0, 2, 1, 3)


def test_pack_nvfp4_layout(lib):
    E, N, K = 2, 256, 512
    g = torch.Generator().manual_seed(11)
    q = torch.randint(0, 256, (E, N, K // 2), generator=g, dtype=torch.uint8)
    s = torch.randint(0, 256, (E, N, K // 16), generator=g, dtype=torch.uint8)
    p = lib.moe_pack_nvfp4(q.to(DEV), s.to(DEV))
    assert p.shape == (E, N, K * 9 // 16)
    got = p.cpu().numpy().reshape(-1, 4608)
    kt = K // 64
    codes = _tiles(q.numpy().reshape(E * N, K // 2), kt, 32).reshape(-1, 128 * 32)
    scales = _tiles(s.numpy().reshape(E * N, K // 16), kt, 4).reshape(-1, 128 * 4)
    assert np.array_equal(got, np.concatenate([codes, scales], axis=1))


def test_pack_fp8_layout(lib):
    E, N, K = 3, 128, 192
    g = torch.Generator().manual_seed(12)
    q = torch.randint(0, 256, (E, N, K), generator=g, dtype=torch.uint8)
    p = lib.moe_pack_fp8(q.to(DEV))
    got = p.cpu().numpy().reshape(-1, 8192)
    want = _tiles(q.numpy().reshape(E * N, K), K // 64, 64).reshape(-1, 8192)
    assert np.array_equal(got, want)


def test_pack_packed_rejects_bad_shapes(lib):
    u8 = torch.uint8
    with pytest.raises(lib.MoeError):
        lib.moe_pack_nvfp4(torch.zeros(1, 100, 64, dtype=u8, device=DEV),
                           torch.zeros(1, 100, 8, dtype=u8, device=DEV))
    with pytest.raises(lib.MoeError):
        lib.moe_pack_nvfp4(torch.zeros(1, 128, 48, dtype=u8, device=DEV),
                           torch.zeros(1, 128, 6, dtype=u8, device=DEV))
    with pytest.raises(lib.MoeError):
        lib.moe_pack_fp8(torch.zeros(1, 128, 96, dtype=u8, device=DEV))


def test_tiled_rejected_for_w4a4(lib):
    """W4A4 takes row-major NVFP4 weights only."""
    c = mi.MoeConfig("tiny-a4", T=64, H=256, E=32, n_group=8, topk_group=2, top_k=4, I=256)
    d = lib.dims_of(c)
    u8 = torch.uint8
    qg = torch.zeros(c.E, c.I, c.H // 2, dtype=u8, device=DEV)
    sg = torch.zeros(c.E, c.I, c.H // 16, dtype=u8, device=DEV)
    qd = torch.zeros(c.E, c.H, c.I // 2, dtype=u8, device=DEV)
    sd = torch.zeros(c.E, c.H, c.I // 16, dtype=u8, device=DEV)
    g = torch.ones(c.E, dtype=torch.float32, device=DEV)
    ex = lib.Experts(qg, qg, qd, sg, sg, sd, g, g, g, a4=(mi.A4_X_GLOBAL, mi.A4_H_GLOBAL))
    st = ex.struct(d)
    st.layout = lib.MOE_LAYOUT_TILED
    x = torch.zeros(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros(c.E, c.H, dtype=torch.float32, device=DEV)
    b = torch.zeros(c.E, dtype=torch.float32, device=DEV)
    y = torch.empty(c.T, c.H, dtype=torch.bfloat16, device=DEV)
    ws = lib.alloc_workspace(d, lib.MOE_OP_FORWARD, lib.MOE_W_NVFP4_A4)
    import ctypes
    rc = lib.native().moe_forward(ctypes.byref(d), x.data_ptr(), wr.data_ptr(), b.data_ptr(),
                                  ctypes.byref(st), y.data_ptr(), None, None, ws.data_ptr(),
                                  ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 2  # MOE_ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        ex.to_tiled()

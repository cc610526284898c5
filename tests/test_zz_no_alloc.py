"""moe_permute_noalloc, the dispatch entry point for callers that cannot
allocate device memory (a plug-in handed only its tensors, or a loop that
forbids allocation after start-up): it must give exactly what moe_permute
gives, on two calls in a row that share its built-in scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process (its
first call performs the per-device set-up)."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    import group_limited_routing_bias_b300 as m
    return m


def _routing(T, E, k, seed, skew):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -skew
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _outputs(T, E, k, H):
    Tk = T * k
    return (torch.full((Tk, H), 7, dtype=torch.bfloat16, device=DEV),
            torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
            torch.full((Tk,), -7, dtype=torch.int32, device=DEV),
            torch.full((Tk,), -7, dtype=torch.int32, device=DEV))


def test_noalloc_matches_workspace_permute_twice(lib):
    H = 512
    # two calls in a row with different sizes and routings: the second must not
    # see anything the first left in the shared scratch
    for T, E, k, seed, skew in [(3000, 256, 8, 0, 1.5), (777, 32, 4, 1, 0.0)]:
        d = lib.make_dims(T, H, E, 8, 4 if E == 256 else 2, k, 128, 2.5)
        idx = torch.from_numpy(_routing(T, E, k, seed, skew)).to(DEV)
        x = torch.randn(T, H, device=DEV).to(torch.bfloat16)
        ref = _outputs(T, E, k, H)
        ws = lib.alloc_workspace(d, lib.MOE_OP_PERMUTE)
        lib.moe_permute(d, idx, x, *ref, ws)
        got = _outputs(T, E, k, H)
        lib.moe_permute_noalloc(d, idx, x, *got)
        torch.cuda.synchronize()
        assert lib.workspace_status(ws) == 0
        for a, b in zip(ref, got):
            assert torch.equal(a, b)


def _scratch_bytes(Tk, E):
    """The scratch a call needs: a 256-byte header, then the counts and the
    bases tables, each 4 * E * ceil(Tk / 4096) bytes rounded up to 256."""
    nchunks = max(1, -(-Tk // 4096))
    table = -(-(4 * E * nchunks) // 256) * 256
    return 256 + 2 * table


def test_noalloc_rejects_oversize_before_launch(lib):
    # T*k beyond the scratch limit: refused with MOE_ERR_UNSUPPORTED, no pointer is read
    fake = ctypes.c_void_p(1 << 20)
    d = lib.make_dims(300000, 512, 256, 8, 4, 8, 128, 2.5)
    assert lib.native().moe_permute_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake, fake,
                                            None) == 2
    # E = 32 with 4095 chunks: 4 * 32 * 4095 bytes is not a multiple of 256, and
    # with the rounding the two tables need 256 bytes more than 1 MiB holds
    T = 4095 * 4096 // 16
    assert _scratch_bytes(T * 16, 32) > 1 << 20
    d = lib.make_dims(T, 128, 32, 8, 4, 16, 128, 2.5)
    assert lib.native().moe_permute_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake, fake,
                                            None) == 2


def test_noalloc_accepts_the_largest_call_that_fits(lib):
    """E = 32 with 4094 chunks of 4096 entries (16.8 M entries, top_k 16) is the
    largest E = 32 call the 1 MiB scratch holds; it runs and sorts stably."""
    E, k, H = 32, 16, 128
    T = 4094 * 4096 // k
    assert _scratch_bytes(T * k, E) <= 1 << 20 < _scratch_bytes(T * k + 1, E)
    gen = torch.Generator(device=DEV).manual_seed(11)
    idx = torch.randint(0, E, (T, k), dtype=torch.int32, device=DEV, generator=gen)
    x = torch.randn(T, H, device=DEV, generator=gen).to(torch.bfloat16)
    d = lib.make_dims(T, H, E, 8, 4, k, 128, 2.5)
    got = _outputs(T, E, k, H)
    lib.moe_permute_noalloc(d, idx, x, *got)
    torch.cuda.synchronize()
    flat = idx.view(-1).cpu().numpy()
    order = np.argsort(flat, kind="stable")
    offs = np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))])
    np.testing.assert_array_equal(got[1].cpu().numpy(), offs)
    np.testing.assert_array_equal(got[3].cpu().numpy(), order)
    rows = torch.from_numpy(np.arange(0, T * k, 9973)).to(DEV)
    src = torch.from_numpy(order[::9973] // k).long().to(DEV)
    assert torch.equal(got[0][rows], x[src])
    del got, x, idx
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,E,k", [(100, 32, 4), (3000, 256, 8)])
def test_noalloc_drops_bad_indices_like_permute(lib, T, E, k):
    """Indices outside [0, E) (here -1 and E) are dropped: expert_offsets[E]
    counts only the valid entries, slot_of is -1 for the dropped ones, and
    every output equals moe_permute's.  T*k = 400 runs the one-CTA dispatch,
    24000 the multi-CTA one."""
    H = 256
    idx = _routing(T, E, k, 3, 0.0)
    bad = [(7, 2, E), (T // 2, 0, -1), (T - 1, k - 1, E), (T - 1, 0, -1)]
    for t, j, v in bad:
        idx[t, j] = v
    idx_d = torch.from_numpy(idx).to(DEV)
    x = torch.randn(T, H, device=DEV).to(torch.bfloat16)
    d = lib.make_dims(T, H, E, 8, 4 if E == 256 else 2, k, 128, 2.5)
    ref = _outputs(T, E, k, H)
    ws = lib.alloc_workspace(d, lib.MOE_OP_PERMUTE)
    lib.moe_permute(d, idx_d, x, *ref, ws)
    assert lib.workspace_status(ws) == lib.MOE_DEV_BAD_INDEX
    got = _outputs(T, E, k, H)
    lib.moe_permute_noalloc(d, idx_d, x, *got)
    torch.cuda.synchronize()
    assert int(got[1][E]) == T * k - len(bad)
    so = got[2].cpu().numpy()
    for t, j, _ in bad:
        assert so[t * k + j] == -1
    for a, b in zip(ref, got):
        assert torch.equal(a, b)

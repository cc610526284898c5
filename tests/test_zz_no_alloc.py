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


def test_noalloc_rejects_oversize_before_launch(lib):
    # T*k beyond the scratch limit: refused with MOE_ERR_UNSUPPORTED, no pointer is read
    d = lib.make_dims(300000, 512, 256, 8, 4, 8, 128, 2.5)
    fake = ctypes.c_void_p(1 << 20)
    assert lib.native().moe_permute_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake, fake,
                                        None) == 2

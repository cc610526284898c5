"""The C ABI without a GPU: the library loads, exports every function that
include/beam_moe.h declares, sizes workspaces, and rejects bad arguments
before launching anything (none of these calls reaches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam_moe.h")


@pytest.fixture(scope="module")
def lib():
    from group_limited_routing_bias_b300 import build
    build.build()
    import group_limited_routing_bias_b300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("moe_route", "moe_permute", "moe_experts_swiglu", "moe_combine",
                     "moe_forward", "moe_workspace_size"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), name
    assert set(declared_functions()) == set(lib.EXPORTED)


def beam_dims(lib, T=64):
    return lib.make_dims(T, 5120, 256, 8, 4, 8, 2560, 2.5)


def test_check_dims(lib):
    assert lib.check_dims(beam_dims(lib)) == 0
    assert lib.check_dims(lib.make_dims(64, 256, 32, 8, 2, 4, 128, 2.5)) == 0
    assert lib.check_dims(beam_dims(lib, T=0)) == 0
    bad_arg = [lib.make_dims(64, 5120, 256, 7, 4, 8, 2560, 2.5),    # E % n_group
               lib.make_dims(64, 5120, 256, 8, 9, 8, 2560, 2.5),    # topk_group > n_group
               lib.make_dims(64, 5120, 256, 8, 1, 33, 2560, 2.5),   # top_k > kept experts
               lib.make_dims(-1, 5120, 256, 8, 4, 8, 2560, 2.5)]
    for d in bad_arg:
        assert lib.check_dims(d) == 1
    unsupported = [lib.make_dims(64, 5000, 256, 8, 4, 8, 2560, 2.5),  # H % 128
                   lib.make_dims(64, 5120, 512, 8, 4, 8, 2560, 2.5),  # E > 256
                   lib.make_dims(64, 5120, 96, 8, 4, 8, 2560, 2.5),   # group size 12
                   lib.make_dims(64, 5120, 256, 8, 4, 17, 2560, 2.5)]  # top_k > 16
    for d in unsupported:
        assert lib.check_dims(d) == 2


def test_workspace_sizes(lib):
    d = beam_dims(lib, T=16384)
    sizes = {op: lib.workspace_size(d, op) for op in range(4)}
    Tk = 16384 * 8
    # the forward workspace holds x_perm, h and y_partial in bf16
    assert sizes[lib.MOE_OP_FORWARD] >= Tk * (5120 + 2560 + 5120) * 2
    assert sizes[lib.MOE_OP_EXPERTS] >= Tk * 2560 * 2
    assert sizes[lib.MOE_OP_FORWARD] > max(sizes[o] for o in range(3))
    assert lib.workspace_size(lib.make_dims(64, 5000, 256, 8, 4, 8, 2560, 2.5), 3) == 0
    # packed weights add the per-row factors of x and h and the row maxima of
    # h ([Tk] fp32 each); the staged experts call also an f16 copy of x_perm
    for wd in (lib.MOE_W_NVFP4, lib.MOE_W_FP8):
        fwd = lib.workspace_size(d, lib.MOE_OP_FORWARD, wd)
        exp = lib.workspace_size(d, lib.MOE_OP_EXPERTS, wd)
        assert fwd >= sizes[lib.MOE_OP_FORWARD] + 3 * Tk * 4
        assert exp >= sizes[lib.MOE_OP_EXPERTS] + Tk * 5120 * 2 + 3 * Tk * 4


def test_argument_errors_return_before_launch(lib):
    d = beam_dims(lib)
    P = ctypes.c_void_p
    fake = P(1 << 20)        # never dereferenced: the checks fail first
    mis = P((1 << 20) + 4)   # misaligned
    so = lib.native()
    ws_n = lib.workspace_size(d, lib.MOE_OP_ROUTE)
    # null pointer
    assert so.moe_route(ctypes.byref(d), None, fake, fake, fake, fake, fake, ws_n, None) == 1
    # misaligned pointer
    assert so.moe_route(ctypes.byref(d), mis, fake, fake, fake, fake, fake, ws_n, None) == 1
    # workspace too small / missing
    assert so.moe_route(ctypes.byref(d), fake, fake, fake, fake, fake, fake, ws_n - 1, None) == 3
    assert so.moe_route(ctypes.byref(d), fake, fake, fake, fake, fake, None, ws_n, None) == 3
    # unsupported shape
    d2 = lib.make_dims(64, 5000, 256, 8, 4, 8, 2560, 2.5)
    assert so.moe_route(ctypes.byref(d2), fake, fake, fake, fake, fake, fake, ws_n, None) == 2
    ex = lib.MoeExperts(lib.MOE_W_BF16, None, fake, fake, None, None, None, None, None, None)
    n = lib.workspace_size(d, lib.MOE_OP_FORWARD)
    assert so.moe_forward(ctypes.byref(d), fake, fake, fake, ctypes.byref(ex), fake, None, None,
                          fake, n, None) == 1
    assert so.moe_combine(ctypes.byref(d), fake, None, fake, None) == 1
    assert so.moe_permute(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, 0, None) == 3


def test_status_strings(lib):
    for s in range(7):
        assert lib.status_string(s)
    assert lib.version() >= 100

"""Plain CPU oracle for the Beam MoE block forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  It shares no code
with the CUDA library and imports nothing from it.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, OpenMP over tokens
or rows); this module only builds it with gcc, marshals numpy arrays, and
strings the three steps together (route -> per-expert SwiGLU -> weighted
combine) in the order the pages state the layer:

* "Hugging Face releases Beam ..." (deliver-ai.xyz), third paragraph: 256
  experts, SwiGLU with intermediate 2,560, top 8 experts from the top 4 of 8
  groups of 32.
* "Reflection Releases Beam ..." (telohudelo.online), section "Where Beam
  Saves and Where the Memory Bill Comes In": sigmoid scores, group limits,
  no shared expert, normalised and scaled by 2.5.
* "Beam 1.0" (interestana.com): per-expert bias from auxiliary-loss-free
  balancing.

Readings of open points are stated at the top of ``moe_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Callable, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` with gcc into ``libmoe_oracle.so`` (in-tree)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", _SO, "-lm"]
        subprocess.run(cmd, check=True)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i, f, d = ctypes.c_int, ctypes.c_float, ctypes.c_double
    lib.oracle_route.argtypes = [i, i, i, i, i, i, f, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_route.restype = i
    lib.oracle_expert_swiglu.argtypes = [i, i, i, P, i, P, P, d, P, P, d, P, P, d, P]
    lib.oracle_expert_swiglu.restype = i
    lib.oracle_combine.argtypes = [i, i, i, P, P, P]
    lib.oracle_combine.restype = i
    lib.oracle_decode_matrix.argtypes = [i, i, i, P, P, d, P]
    lib.oracle_decode_matrix.restype = i
    lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_value.restype = d
    lib.oracle_bias_update.argtypes = [i, i, i, P, P, d, i, i]
    lib.oracle_bias_update.restype = f
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = d
    lib.oracle_e2m1_rne.argtypes = [f]
    lib.oracle_e2m1_rne.restype = ctypes.c_uint8
    lib.oracle_e4m3_rne.argtypes = [f]
    lib.oracle_e4m3_rne.restype = ctypes.c_uint8
    lib.oracle_quantize_nvfp4.argtypes = [i, i, P, f, P, P]
    lib.oracle_quantize_nvfp4.restype = i
    lib.oracle_expert_swiglu_w4a4.argtypes = [i, i, i, P, P, P, d, P, P, d, P, P, d, f, f, P]
    lib.oracle_expert_swiglu_w4a4.restype = i
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


# ---------------------------------------------------------------- routing


@dataclass
class Routing:
    idx: np.ndarray            # int32 [T, k], descending biased score
    w: np.ndarray              # fp32 [T, k], sums to routed_scale
    logits: Optional[np.ndarray] = None       # fp32 [T, E]
    scores: Optional[np.ndarray] = None       # fp32 [T, E]  sigmoid(logit)
    biased: Optional[np.ndarray] = None       # fp32 [T, E]  scores + bias
    group_score: Optional[np.ndarray] = None  # fp32 [T, G]
    group_kept: Optional[np.ndarray] = None   # uint8 [T, G]


def route(x_bf16: np.ndarray, w_router: np.ndarray, bias: np.ndarray, n_group: int,
          topk_group: int, top_k: int, routed_scale: float, details: bool = False) -> Routing:
    """Sigmoid router with selection bias and group-limited top-k.

    ``x_bf16`` holds bf16 bit patterns as uint16 [T, H].
    """
    lib = _load()
    x = _c(x_bf16, np.uint16)
    wr = _c(w_router, np.float32)
    b = _c(bias, np.float32)
    T, H = x.shape
    E = wr.shape[0]
    idx = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    extra = {}
    if details:
        extra = dict(logits=np.empty((T, E), np.float32), scores=np.empty((T, E), np.float32),
                     biased=np.empty((T, E), np.float32),
                     group_score=np.empty((T, n_group), np.float32),
                     group_kept=np.empty((T, n_group), np.uint8))
    rc = lib.oracle_route(T, H, E, n_group, topk_group, top_k, routed_scale, _ptr(x), _ptr(wr),
                          _ptr(b), _ptr(idx), _ptr(w), _ptr(extra.get("logits")),
                          _ptr(extra.get("scores")), _ptr(extra.get("biased")),
                          _ptr(extra.get("group_score")), _ptr(extra.get("group_kept")))
    if rc != 0:
        raise ValueError("oracle_route: bad arguments")
    return Routing(idx=idx, w=w, **extra)


def routed_weights(scores_row: np.ndarray, idx_row: Sequence[int], routed_scale: float) -> np.ndarray:
    """Weights for a given selection: routed_scale * s_e / sum(s), fp64 sum, fp32 result."""
    s = np.asarray(scores_row, np.float64)[np.asarray(idx_row)]
    return (routed_scale * s / s.sum()).astype(np.float32)


# ---------------------------------------------------------------- experts


@dataclass
class Nvfp4Matrix:
    """NVFP4 weight [N, K]: packed e2m1 uint8 [N, K/2] (low nibble = even k),
    e4m3 block scales uint8 [N, K/16], and one fp32 global scale."""
    q: np.ndarray
    s: np.ndarray
    g: float


@dataclass
class Fp8Matrix:
    """FP8 weight [N, K]: e4m3 codes uint8 [N, K] and one fp32 scale per row [N]."""
    q: np.ndarray
    row_scale: np.ndarray


def _mat_args(m):
    if isinstance(m, Nvfp4Matrix):
        return 1, _c(m.q, np.uint8), _c(m.s, np.uint8), float(m.g)
    if isinstance(m, Fp8Matrix):
        return 2, _c(m.q, np.uint8), _c(m.row_scale, np.float32), 1.0
    return 0, _c(m, np.uint16), None, 1.0


def expert_swiglu(x_rows: np.ndarray, wg, wu, wd) -> np.ndarray:
    """One SwiGLU expert on n rows; returns fp64 [n, H].

    Weights are bf16 bit patterns (uint16 [I,H], [I,H], [H,I]), ``Nvfp4Matrix`` or
    ``Fp8Matrix``.
    """
    lib = _load()
    x = _c(x_rows, np.uint16)
    n, H = x.shape
    dg, qg, sg, gg = _mat_args(wg)
    du, qu, su, gu = _mat_args(wu)
    dd, qd, sd, gd = _mat_args(wd)
    assert dg == du == dd
    I = qg.shape[0]
    o = np.empty((n, H), np.float64)
    rc = lib.oracle_expert_swiglu(n, H, I, _ptr(x), dg, _ptr(qg), _ptr(sg), gg, _ptr(qu), _ptr(su),
                                  gu, _ptr(qd), _ptr(sd), gd, _ptr(o))
    if rc != 0:
        raise ValueError("oracle_expert_swiglu: bad arguments")
    return o


def combine(topk_w: np.ndarray, o: np.ndarray) -> np.ndarray:
    """y[t] = sum_k topk_w[t,k] * o[t,k,:] in k order, fp64."""
    lib = _load()
    w = _c(topk_w, np.float32)
    oo = _c(o, np.float64)
    T, k, H = oo.shape
    y = np.empty((T, H), np.float64)
    if lib.oracle_combine(T, k, H, _ptr(w), _ptr(oo), _ptr(y)) != 0:
        raise ValueError("oracle_combine: bad arguments")
    return y


def decode_matrix(m) -> np.ndarray:
    """Widen a bf16 or NVFP4 weight matrix to fp64 [N, K]."""
    lib = _load()
    dt, q, s, g = _mat_args(m)
    N = q.shape[0]
    K = q.shape[1] * (2 if dt == 1 else 1)
    out = np.empty((N, K), np.float64)
    if lib.oracle_decode_matrix(dt, N, K, _ptr(q), _ptr(s), g, _ptr(out)) != 0:
        raise ValueError("oracle_decode_matrix: bad arguments")
    return out


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code)


def e2m1_rne(v: float) -> int:
    """fp32 -> E2M1 code (round to nearest, ties to even mantissa, saturate at 6)."""
    return _load().oracle_e2m1_rne(v)


def e4m3_rne(v: float) -> int:
    """fp32 -> E4M3 code (round to nearest, ties to even, saturate at 448)."""
    return _load().oracle_e4m3_rne(v)


def quantize_nvfp4(v: np.ndarray, g: float):
    """NVFP4 activation quantiser (readings in moe_oracle.c): fp32 [rows, cols]
    and a global scale -> (codes uint8 [rows, cols/2], scales uint8 [rows, cols/16])."""
    lib = _load()
    a = _c(v, np.float32)
    rows, cols = a.shape
    q = np.empty((rows, cols // 2), np.uint8)
    sc = np.empty((rows, cols // 16), np.uint8)
    if lib.oracle_quantize_nvfp4(rows, cols, _ptr(a), g, _ptr(q), _ptr(sc)) != 0:
        raise ValueError("oracle_quantize_nvfp4: bad arguments")
    return q, sc


def expert_swiglu_w4a4(x_rows: np.ndarray, wg: Nvfp4Matrix, wu: Nvfp4Matrix, wd: Nvfp4Matrix,
                       gx: float, gh: float) -> np.ndarray:
    """One SwiGLU expert with NVFP4 weights and NVFP4 activations (x quantised
    with global gx, h with gh); returns fp64 [n, H]."""
    lib = _load()
    x = _c(x_rows, np.uint16)
    n, H = x.shape
    I = wg.q.shape[0]
    o = np.empty((n, H), np.float64)
    args = []
    for m in (wg, wu, wd):
        args += [_ptr(_c(m.q, np.uint8)), _ptr(_c(m.s, np.uint8)), float(m.g)]
    if lib.oracle_expert_swiglu_w4a4(n, H, I, _ptr(x), *args, gx, gh, _ptr(o)) != 0:
        raise ValueError("oracle_expert_swiglu_w4a4: bad arguments")
    return o


ExpertFn = Callable[[int], tuple]


def experts_forward(x_bf16: np.ndarray, idx: np.ndarray, w: np.ndarray, get_expert: ExpertFn,
                    tokens: Optional[Sequence[int]] = None,
                    a4: Optional[tuple] = None) -> np.ndarray:
    """Expert path for a given routing: per-expert SwiGLU, then the combine.

    ``get_expert(e)`` returns the three weight matrices of expert e (so large
    weight sets can be fetched one expert at a time).  ``tokens`` restricts
    the outputs to a subset of token indices (rows of the result follow it).
    ``a4 = (gx, gh)`` selects NVFP4 activations (W4A4) with those global
    scales; the weights must then be ``Nvfp4Matrix``.
    Returns fp64 [len(tokens), H].
    """
    x = _c(x_bf16, np.uint16)
    sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, np.int64)
    k = idx.shape[1]
    H = x.shape[1]
    sub_idx = idx[sel]
    o = np.zeros((len(sel), k, H), np.float64)
    for e in np.unique(sub_idx):
        rr, kk = np.nonzero(sub_idx == e)
        wg, wu, wd = get_expert(int(e))
        if a4 is None:
            o[rr, kk] = expert_swiglu(x[sel[rr]], wg, wu, wd)
        else:
            o[rr, kk] = expert_swiglu_w4a4(x[sel[rr]], wg, wu, wd, a4[0], a4[1])
    return combine(np.ascontiguousarray(w[sel]), o)


def moe_forward(x_bf16, w_router, bias, get_expert: ExpertFn, n_group: int, topk_group: int,
                top_k: int, routed_scale: float, tokens=None, details: bool = False):
    """The whole block: route all tokens, then the expert path for ``tokens``
    (all by default).  Returns (y fp64, Routing)."""
    r = route(x_bf16, w_router, bias, n_group, topk_group, top_k, routed_scale, details)
    y = experts_forward(x_bf16, r.idx, r.w, get_expert, tokens)
    return y, r


def bias_update(topk_idx: np.ndarray, bias: np.ndarray, E: int, gamma_max: float, step: int,
                total_steps: int):
    """Auxiliary-loss-free bias update (readings in moe_oracle.c).  Returns
    (new bias fp32 [E], gamma_t used)."""
    lib = _load()
    idx = _c(topk_idx, np.int32)
    b = np.array(bias, dtype=np.float32, copy=True)
    T, k = idx.shape
    g = lib.oracle_bias_update(T, k, E, _ptr(idx), _ptr(b), gamma_max, step, total_steps)
    return b, g

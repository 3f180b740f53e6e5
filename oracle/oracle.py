"""ctypes wrapper around ``libspear_oracle.so`` (plain C++17, see spear_oracle.cpp).

TEST INFRASTRUCTURE ONLY -- the parity oracle.  Each function restates one
step of the method in the SPEAR explainer (gist.science, Technical Summary
2.1 A for the layer, 2.1 B for module selection) and is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.

Arrays are numpy; bf16 and fp16 values travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spear_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_build", "libspear_oracle.so")
_lock = threading.Lock()
_lib = None

__all__ = [
    "build_oracle", "f32_to_f16_ru", "f16_to_f32", "f32_to_bf16_rn", "bf16_to_f32",
    "quantize_pack", "unpack_codes", "unpack_zeros", "dequant", "linear",
    "linear_vector_gate", "layer_select_mask", "chunk_select", "linear_cka", "packed_sizes",
]


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with g++ (no CUDA) into oracle/_build/."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(os.path.join(_HERE, "spear_oracle.h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-o", tmp, _SRC, "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build_oracle())
        P = ctypes.c_void_p
        i, f, d = ctypes.c_int, ctypes.c_float, ctypes.c_double
        lib.oracle_f32_to_f16_ru.argtypes = [f]; lib.oracle_f32_to_f16_ru.restype = ctypes.c_uint16
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]; lib.oracle_f16_to_f32.restype = f
        lib.oracle_f32_to_bf16_rn.argtypes = [f]; lib.oracle_f32_to_bf16_rn.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]; lib.oracle_bf16_to_f32.restype = f
        lib.oracle_quantize_pack.argtypes = [P, i, i, i, i, P, P, P]
        lib.oracle_unpack_codes.argtypes = [P, i, i, P]
        lib.oracle_unpack_zeros.argtypes = [P, i, i, i, i, P]
        lib.oracle_dequant.argtypes = [P, P, P, i, i, i, i, P]
        lib.oracle_linear.argtypes = [i, i, i, i, P, P, P, i, P, P, P, f, f, i, P, i, P, i, i, i,
                                      P, P, P]
        lib.oracle_linear_vector_gate.argtypes = [i, i, i, i, P, P, P, i, P, P, i, P, P, P, P, f,
                                                  P, i, i, P, P]
        lib.oracle_layer_select_mask.argtypes = [P, P, i, d, i, i, P, P]
        for name in ("oracle_quantize_pack", "oracle_unpack_codes", "oracle_unpack_zeros",
                     "oracle_dequant", "oracle_linear", "oracle_linear_vector_gate",
                     "oracle_layer_select_mask"):
            getattr(lib, name).restype = i
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle: {what} rejected its arguments (status {rc})")


# ------------------------------------------------------------------ numbers

def f32_to_f16_ru(v: float) -> int:
    return int(_load().oracle_f32_to_f16_ru(float(v)))


def f16_to_f32(h: int) -> float:
    return float(_load().oracle_f16_to_f32(int(h)))


def f32_to_bf16_rn(v: float) -> int:
    return int(_load().oracle_f32_to_bf16_rn(float(v)))


def bf16_to_f32(b: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(b)))


# ---------------------------------------------------------------- quantiser

def packed_sizes(N: int, K: int, G: int, sym: bool):
    """Bytes of (qweight, scales, zeros) in the canonical packed format."""
    ng = K // G
    return N * (K // 2), N * ng * 2, 0 if sym else N * ((ng + 1) // 2)


def quantize_pack(W: np.ndarray, G: int, sym: bool):
    """Round-to-nearest int4 quantisation + nibble packing of W [N][K] fp32.

    Returns (qweight uint8 [N][K/2], scales uint16 (fp16 bits) [N][K/G],
    zeros uint8 [N][ceil(K/G/2)] or None)."""
    W = _c(W, np.float32)
    N, K = W.shape
    ng = K // G
    q = np.zeros((N, K // 2), np.uint8)
    s = np.zeros((N, ng), np.uint16)
    z = None if sym else np.zeros((N, (ng + 1) // 2), np.uint8)
    _check(_load().oracle_quantize_pack(_ptr(W), N, K, G, int(bool(sym)), _ptr(q), _ptr(s), _ptr(z)),
           "quantize_pack")
    return q, s, z


def unpack_codes(qweight: np.ndarray, K: int) -> np.ndarray:
    qweight = _c(qweight, np.uint8)
    N = qweight.shape[0]
    u = np.zeros((N, K), np.uint8)
    _check(_load().oracle_unpack_codes(_ptr(qweight), N, K, _ptr(u)), "unpack_codes")
    return u


def unpack_zeros(zeros, N: int, K: int, G: int, sym: bool) -> np.ndarray:
    zeros = _c(zeros, np.uint8)
    z = np.zeros((N, K // G), np.uint8)
    _check(_load().oracle_unpack_zeros(_ptr(zeros), N, K, G, int(bool(sym)), _ptr(z)), "unpack_zeros")
    return z


def dequant(qweight, scales, zeros, K: int, G: int, sym: bool) -> np.ndarray:
    qweight, scales, zeros = _c(qweight, np.uint8), _c(scales, np.uint16), _c(zeros, np.uint8)
    N = qweight.shape[0]
    dq = np.zeros((N, K), np.float64)
    _check(_load().oracle_dequant(_ptr(qweight), _ptr(scales), _ptr(zeros), N, K, G, int(bool(sym)),
                                  _ptr(dq)), "dequant")
    return dq


# -------------------------------------------------------------------- layer

def linear(layer: dict, x_bf16: np.ndarray, *, n_idx=None, accum_double: bool = True,
           nthreads: int = 1, want_corr: bool = False, want_gate: bool = False):
    """y[m][c] for output rows n_idx (all rows if None), fp64 (see spear_oracle.h).

    ``layer`` holds N, K, G, sym, qweight, scales, zeros, r, A, B, w_g (bf16
    bits), b_g, alpha, comp_enabled.  Returns y, or (y, corr, gate)."""
    L = layer
    x = _c(x_bf16, np.uint16)
    M = x.shape[0] if x.ndim == 2 else 0
    N, K, G = L["N"], L["K"], L["G"]
    idx = None if n_idx is None else np.ascontiguousarray(n_idx, dtype=np.int32)
    cols = N if idx is None else idx.shape[0]
    y = np.zeros((M, cols), np.float64)
    corr = np.zeros((M, cols), np.float64) if want_corr else None
    gate = np.zeros((M,), np.float64) if want_gate else None
    r = int(L.get("r", 0))
    rc = _load().oracle_linear(
        N, K, G, int(bool(L["sym"])),
        _ptr(_c(L["qweight"], np.uint8)), _ptr(_c(L["scales"], np.uint16)),
        _ptr(_c(L.get("zeros"), np.uint8)),
        r, _ptr(_c(L.get("A"), np.uint16)), _ptr(_c(L.get("B"), np.uint16)),
        _ptr(_c(L.get("w_g"), np.uint16)),
        float(L.get("b_g", 0.0)), float(L.get("alpha", 1.0)), int(L.get("comp_enabled", 1)),
        _ptr(x), M, _ptr(idx), cols, int(bool(accum_double)), int(nthreads),
        _ptr(y), _ptr(corr), _ptr(gate))
    _check(rc, "linear")
    if want_corr or want_gate:
        return y, corr, gate
    return y


def linear_vector_gate(layer: dict, x_bf16, W1, c1, W2, c2, *, nthreads: int = 1):
    """The paper's bottleneck-MLP gate gamma(Ax) on the rank-r code; returns (y, gamma)."""
    L = layer
    x = _c(x_bf16, np.uint16)
    M = x.shape[0]
    N, K, G, r = L["N"], L["K"], L["G"], int(L["r"])
    W1, c1, W2, c2 = (_c(a, np.float32) for a in (W1, c1, W2, c2))
    h = W1.shape[0]
    y = np.zeros((M, N), np.float64)
    gam = np.zeros((M, r), np.float64)
    rc = _load().oracle_linear_vector_gate(
        N, K, G, int(bool(L["sym"])), _ptr(_c(L["qweight"], np.uint8)),
        _ptr(_c(L["scales"], np.uint16)), _ptr(_c(L.get("zeros"), np.uint8)),
        r, _ptr(_c(L["A"], np.uint16)), _ptr(_c(L["B"], np.uint16)),
        h, _ptr(W1), _ptr(c1), _ptr(W2), _ptr(c2), float(L.get("alpha", 1.0)),
        _ptr(x), M, int(nthreads), _ptr(y), _ptr(gam))
    _check(rc, "linear_vector_gate")
    return y, gam


# --------------------------------------------------------- linear CKA

def linear_cka(X, Y) -> float:
    """Linear CKA from its definition (Technical Summary 2.1 B names CKA as
    the damage proxy): K = X X^T, L = Y Y^T on the raw activations, the
    centring matrix H = I - 1 1^T / n, HSIC(K, L) = tr(K H L H), and
    CKA = HSIC(K, L) / sqrt(HSIC(K, K) HSIC(L, L)); fp64 numpy."""
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    n = X.shape[0]
    H = np.eye(n) - np.ones((n, n)) / n
    K, L = X @ X.T, Y @ Y.T
    hsic = lambda a, b: float(np.trace(a @ H @ b @ H))
    return hsic(K, L) / np.sqrt(hsic(K, K) * hsic(L, L))


# --------------------------------------------------------- chunk selection

def chunk_select(prefill_curves, decode_curves, decode_tokens: int, choices, itl_target_us: float):
    """SLO-constrained chunk choice (Technical Summary 2.2 C), written out
    plainly: a curve is (M list, microseconds list); its latency at M is the
    line through the two points bracketing M (the nearest two outside the
    range; one point: constant).  A chunk C > 0 costs the sum of the prefill
    curves at C + D; C = 0 the sum of the decode curves at D (0 without
    decode tokens).  Returns (largest C within the target, else the smallest C;
    that C's latency)."""
    def at(curve, M):
        Ms, us = [float(v) for v in curve[0]], [float(v) for v in curve[1]]
        if len(Ms) == 1:
            return us[0]
        i = 0
        while i + 2 < len(Ms) and M > Ms[i + 1]:
            i += 1
        return us[i] + (us[i + 1] - us[i]) * (M - Ms[i]) / (Ms[i + 1] - Ms[i])

    def step(C):
        if C > 0:
            return sum(at(c, C + decode_tokens) for c in prefill_curves)
        return sum(at(c, decode_tokens) for c in decode_curves) if decode_tokens > 0 else 0.0

    ok = [C for C in choices if step(C) <= itl_target_us]
    C = max(ok) if ok else min(choices)
    return C, step(C)


# --------------------------------------------------------- module selection

def layer_select_mask(damage, cost, budget_bytes: float, rank_min: int, rank_max: int):
    d = _c(damage, np.float32)
    c = _c(cost, np.float32)
    L = d.shape[0]
    mask = np.zeros(L, np.uint8)
    rank = np.zeros(L, np.int32)
    _check(_load().oracle_layer_select_mask(_ptr(d), _ptr(c), L, float(budget_bytes), int(rank_min),
                                            int(rank_max), _ptr(mask), _ptr(rank)),
           "layer_select_mask")
    return mask, rank

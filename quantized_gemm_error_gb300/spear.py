"""Thin Python binding of ``libspear.so`` (C ABI in ``include/spear.h``).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Torch provides device memory and streams.  There is no CPU
fallback -- if the library cannot be loaded every call raises.

Function names follow the C ABI:
  spear_pack_w4, spear_linear_decode, spear_linear_prefill,
  spear_layer_select_mask, plus the workspace / status helpers.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libspear.so")

SPEAR_OK = 0
STATUS_NAMES = {0: "SPEAR_OK", 1: "SPEAR_ERR_INVALID_ARG", 2: "SPEAR_ERR_UNSUPPORTED",
                3: "SPEAR_ERR_WORKSPACE", 4: "SPEAR_ERR_CUDA", 5: "SPEAR_ERR_TIMEOUT", 6: "SPEAR_ERR_BOUNDS"}
PREFILL_AUTO, PREFILL_FUSED, PREFILL_STREAM = 0, 1, 2
OUT_BF16, OUT_F32 = 0, 1

# every symbol include/spear.h declares
EXPORTS = ["spear_pack_w4_sizes", "spear_pack_w4", "spear_decode_workspace_bytes",
           "spear_linear_decode", "spear_linear_decode_noalloc", "spear_prefill_workspace_bytes", "spear_linear_prefill",
           "spear_workspace_init", "spear_set_launch_overlap", "spear_set_wait_limit_ns", "spear_layer_select_mask",
           "spear_chunk_select",
           "spear_linear_cka", "spear_cka_damage",
           "spear_get_device_status", "spear_status_string", "spear_last_error", "spear_version"]


class SpearError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


class _Layer(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("K", ctypes.c_int), ("group_size", ctypes.c_int),
                ("symmetric", ctypes.c_int), ("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p), ("rank", ctypes.c_int), ("A", ctypes.c_void_p),
                ("B", ctypes.c_void_p), ("w_g", ctypes.c_void_p), ("b_g", ctypes.c_float),
                ("alpha", ctypes.c_float), ("comp_enabled", ctypes.c_int), ("gate_hidden", ctypes.c_int),
                ("gate_w1", ctypes.c_void_p), ("gate_c1", ctypes.c_void_p), ("gate_w2", ctypes.c_void_p),
                ("gate_c2", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Loads the CUDA library (once).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libspear.so not found at {path}: build it first "
                               "(python -m quantized_gemm_error_gb300.build)")
        lib = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        LP = ctypes.POINTER(_Layer)
        sig = {
            "spear_pack_w4_sizes": [I, I, I, I, ctypes.POINTER(S), ctypes.POINTER(S), ctypes.POINTER(S)],
            "spear_pack_w4": [P, I, I, I, I, P, P, P, P],
            "spear_decode_workspace_bytes": [LP, I, ctypes.POINTER(S)],
            "spear_linear_decode": [LP, P, I, P, I, P, S, P],
            "spear_linear_decode_noalloc": [LP, P, I, P, I, P],
            "spear_prefill_workspace_bytes": [LP, I, I, ctypes.POINTER(S)],
            "spear_linear_prefill": [LP, P, I, P, I, I, P, S, P, P],
            "spear_workspace_init": [P, S, P],
            "spear_layer_select_mask": [P, P, I, ctypes.c_double, I, I, P, P],
            "spear_chunk_select": [P, P, I, I, P, I, ctypes.c_double, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double)],
            "spear_linear_cka": [P, P, I, I, I, ctypes.POINTER(ctypes.c_double)],
            "spear_cka_damage": [P, P, I, I, I, ctypes.POINTER(ctypes.c_double)],
            "spear_get_device_status": [ctypes.POINTER(I), P],
            "spear_set_launch_overlap": [I],
            "spear_set_wait_limit_ns": [ctypes.c_uint64],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I
        lib.spear_status_string.argtypes = [I]
        lib.spear_status_string.restype = ctypes.c_char_p
        lib.spear_last_error.argtypes = []
        lib.spear_last_error.restype = ctypes.c_char_p
        lib.spear_version.argtypes = []
        lib.spear_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(rc: int, where: str):
    if rc != SPEAR_OK:
        detail = load().spear_last_error().decode(errors="replace")
        raise SpearError(rc, where, detail)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


@dataclass
class W4Layer:
    """A packed layer plus its compensator (all tensors on the same CUDA device)."""
    N: int
    K: int
    group_size: int
    symmetric: bool
    qweight: torch.Tensor                 # uint8 [N][K/2]
    scales: torch.Tensor                  # fp16  [N][K/G]
    zeros: Optional[torch.Tensor] = None  # uint8 [N][ceil(K/G/2)]
    rank: int = 0
    A: Optional[torch.Tensor] = None      # bf16 [rank][K]
    B: Optional[torch.Tensor] = None      # bf16 [N][rank]
    w_g: Optional[torch.Tensor] = None    # bf16 [K]
    b_g: float = 0.0
    alpha: float = 1.0
    comp_enabled: bool = True
    # the vector gate gamma(A x) = sigmoid(W2 relu(W1 (A x) + c1) + c2), fp32 device
    # tensors W1 [h][rank], c1 [h], W2 [rank][h], c2 [rank]; None: the scalar gate
    gate_w1: Optional[torch.Tensor] = None
    gate_c1: Optional[torch.Tensor] = None
    gate_w2: Optional[torch.Tensor] = None
    gate_c2: Optional[torch.Tensor] = None

    def check(self):
        """Shapes and dtypes of the layer's tensors, which the C ABI (plain
        pointers) cannot see; the library checks the rest (shape rules, rank,
        hidden width, alignment)."""
        N, K, G, r = self.N, self.K, self.group_size, self.rank
        if G <= 0 or K % G:
            raise ValueError(f"group_size={G} must divide K={K}")

        def need(t, name, dtype, shape):
            if t is None:
                raise ValueError(f"{name} is missing")
            if t.dtype != dtype or tuple(t.shape) != tuple(shape):
                raise ValueError(f"{name} must be {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")

        need(self.qweight, "qweight", torch.uint8, (N, K // 2))
        need(self.scales, "scales", torch.float16, (N, K // G))
        if not self.symmetric:
            need(self.zeros, "zeros", torch.uint8, (N, (K // G + 1) // 2))
        if self.comp_enabled and r > 0:
            need(self.A, "A", torch.bfloat16, (r, K))
            need(self.B, "B", torch.bfloat16, (N, r))
            if self.gate_w1 is None:
                need(self.w_g, "w_g", torch.bfloat16, (K,))
            else:
                h = int(self.gate_w1.shape[0]) if self.gate_w1.dim() == 2 else -1
                need(self.gate_w1, "gate_w1", torch.float32, (h, r))
                need(self.gate_c1, "gate_c1", torch.float32, (h,))
                need(self.gate_w2, "gate_w2", torch.float32, (r, h))
                need(self.gate_c2, "gate_c2", torch.float32, (r,))

    def c_struct(self) -> _Layer:
        self.check()
        h = int(self.gate_w1.shape[0]) if self.gate_w1 is not None else 0
        return _Layer(self.N, self.K, self.group_size, int(self.symmetric), _ptr(self.qweight),
                      _ptr(self.scales), _ptr(self.zeros), int(self.rank), _ptr(self.A), _ptr(self.B),
                      _ptr(self.w_g), float(self.b_g), float(self.alpha), int(self.comp_enabled), h,
                      _ptr(self.gate_w1), _ptr(self.gate_c1), _ptr(self.gate_w2), _ptr(self.gate_c2))

    def with_comp(self, enabled: bool) -> "W4Layer":
        d = dict(self.__dict__)
        d["comp_enabled"] = enabled
        return W4Layer(**d)


# ------------------------------------------------------------------ pack

def spear_pack_w4_sizes(N: int, K: int, group_size: int, symmetric: bool):
    q, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().spear_pack_w4_sizes(N, K, group_size, int(symmetric), ctypes.byref(q), ctypes.byref(s),
                                      ctypes.byref(z)), "spear_pack_w4_sizes")
    return q.value, s.value, z.value


def spear_pack_w4(W: torch.Tensor, group_size: int, symmetric: bool, *, out=None, stream=None):
    """Quantise + pack W (CUDA fp32 [N][K]); returns (qweight, scales, zeros)."""
    if W.dtype != torch.float32 or W.dim() != 2:
        raise ValueError("W must be a 2-D float32 CUDA tensor")
    N, K = W.shape
    qb, sb, zb = spear_pack_w4_sizes(N, K, group_size, symmetric)
    if out is None:
        q = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
        s = torch.empty((N, K // group_size), dtype=torch.float16, device=W.device)
        z = None if symmetric else torch.empty((N, zb // N), dtype=torch.uint8, device=W.device)
    else:
        q, s, z = out
    _check(load().spear_pack_w4(_ptr(W), N, K, group_size, int(symmetric), _ptr(q), _ptr(s), _ptr(z),
                                _stream(stream)), "spear_pack_w4")
    return q, s, z


# ---------------------------------------------------------------- layer

def spear_decode_workspace_bytes(layer: W4Layer, M: int) -> int:
    n = ctypes.c_size_t()
    L = layer.c_struct()
    _check(load().spear_decode_workspace_bytes(ctypes.byref(L), M, ctypes.byref(n)),
           "spear_decode_workspace_bytes")
    return n.value


def spear_prefill_workspace_bytes(layer: W4Layer, M: int, mode: int = PREFILL_AUTO) -> int:
    n = ctypes.c_size_t()
    L = layer.c_struct()
    _check(load().spear_prefill_workspace_bytes(ctypes.byref(L), M, mode, ctypes.byref(n)),
           "spear_prefill_workspace_bytes")
    return n.value


def new_workspace(nbytes: int, device, zero: bool = True) -> torch.Tensor:
    """A 256-byte aligned device buffer (torch allocations are) of at least nbytes."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    if zero:
        spear_workspace_init(ws)
    return ws


# Workspaces of the calls made without one: one per (kind, device, stream),
# grown when a call needs more and otherwise reused.  Calls on one stream run
# in order, so they never use it at the same time; a decode workspace is left
# ready for the next call by the kernel itself.
_default_ws = {}


def _default_workspace(kind: str, nbytes: int, device, stream, zero: bool) -> torch.Tensor:
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    key = (kind, idx, _stream(stream).value or 0)
    ws = _default_ws.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=torch.device("cuda", idx))
        if isinstance(stream, torch.cuda.Stream):
            ws.record_stream(stream)                  # freed (when replaced) only after that stream's work
        if zero:
            spear_workspace_init(ws, stream)          # on the stream the calls use
        _default_ws[key] = ws
    return ws


def reset_default_workspaces() -> None:
    """Drops the workspaces kept for calls made without one (the next call
    makes a zeroed one): after spear_get_device_status reports
    SPEAR_ERR_TIMEOUT, or to release the memory."""
    _default_ws.clear()


def spear_workspace_init(ws: torch.Tensor, stream=None):
    _check(load().spear_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "spear_workspace_init")


def _check_io(layer: W4Layer, x: torch.Tensor, y: Optional[torch.Tensor], out_dtype: int):
    """Shapes and dtypes the C ABI cannot see: x bf16 [M][K]; y, when given,
    [M][N] in the requested output type (a wrong type would be written past
    its end)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != layer.K:
        raise ValueError(f"x must be a bfloat16 [M][{layer.K}] tensor, got {x.dtype} {tuple(x.shape)}")
    if out_dtype not in (OUT_BF16, OUT_F32):
        raise ValueError(f"out_dtype must be OUT_BF16 or OUT_F32, got {out_dtype}")
    if y is not None:
        want = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
        if y.dtype != want or tuple(y.shape) != (x.shape[0], layer.N):
            raise ValueError(f"y must be a {want} [{x.shape[0]}][{layer.N}] tensor, got {y.dtype} "
                             f"{tuple(y.shape)}")


def _out(y, M, N, out_dtype, device):
    if y is not None:
        return y
    return torch.empty((M, N), dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16, device=device)


def spear_linear_decode(layer: W4Layer, x: torch.Tensor, *, y=None, out_dtype: int = OUT_BF16,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = dequant(Wq) x + alpha g(x) B (A x) for M <= 64 tokens, one kernel launch.
    Without `workspace` the call uses the binding's workspace for this device
    and stream (made once, zeroed, then reused; see reset_default_workspaces)."""
    _check_io(layer, x, y, out_dtype)
    M = x.shape[0]
    y = _out(y, M, layer.N, out_dtype, x.device)
    if workspace is None:
        workspace = _default_workspace("decode", spear_decode_workspace_bytes(layer, M), x.device, stream, True)
    L = layer.c_struct()
    _check(load().spear_linear_decode(ctypes.byref(L), _ptr(x), M, _ptr(y), out_dtype, _ptr(workspace),
                                      workspace.numel(), _stream(stream)), "spear_linear_decode")
    return y


def spear_linear_decode_noalloc(layer: W4Layer, x: torch.Tensor, *, y: torch.Tensor,
                                out_dtype: int = OUT_BF16, stream=None) -> torch.Tensor:
    """Decode for callers that cannot allocate device memory: the library keeps
    the scratch in a fixed 8 MiB array of its own, so the caller passes only
    inputs and the output buffer.  Calls that overlap on the GPU race."""
    _check_io(layer, x, y, out_dtype)
    L = layer.c_struct()
    _check(load().spear_linear_decode_noalloc(ctypes.byref(L), _ptr(x), x.shape[0], _ptr(y), out_dtype,
                                              _stream(stream)), "spear_linear_decode_noalloc")
    return y


def spear_linear_prefill(layer: W4Layer, x: torch.Tensor, *, y=None, out_dtype: int = OUT_BF16,
                         mode: int = PREFILL_AUTO, workspace: Optional[torch.Tensor] = None,
                         stream=None, stream_aux=None) -> torch.Tensor:
    """Same layer for large M on the tcgen05 tensor-core path."""
    _check_io(layer, x, y, out_dtype)
    M = x.shape[0]
    y = _out(y, M, layer.N, out_dtype, x.device)
    if workspace is None:
        workspace = _default_workspace("prefill", spear_prefill_workspace_bytes(layer, M, mode), x.device, stream,
                                       False)
    L = layer.c_struct()
    aux = None if stream_aux is None else _stream(stream_aux)
    _check(load().spear_linear_prefill(ctypes.byref(L), _ptr(x), M, _ptr(y), out_dtype, mode,
                                       _ptr(workspace), workspace.numel(), _stream(stream), aux),
           "spear_linear_prefill")
    return y


# ------------------------------------------------------- module selection

def spear_layer_select_mask(damage, cost, budget_bytes: float, rank_min: int, rank_max: int):
    d = np.ascontiguousarray(damage, dtype=np.float32)
    c = np.ascontiguousarray(cost, dtype=np.float32)
    mask = np.zeros(d.shape[0], np.uint8)
    rank = np.zeros(d.shape[0], np.int32)
    _check(load().spear_layer_select_mask(d.ctypes.data_as(ctypes.c_void_p), c.ctypes.data_as(ctypes.c_void_p),
                                          d.shape[0], float(budget_bytes), int(rank_min), int(rank_max),
                                          mask.ctypes.data_as(ctypes.c_void_p),
                                          rank.ctypes.data_as(ctypes.c_void_p)), "spear_layer_select_mask")
    return mask, rank


def spear_linear_cka(X, Y) -> float:
    """Linear CKA of two host activation matrices [n][dx], [n][dy] (fp32)."""
    x = np.ascontiguousarray(X, dtype=np.float32)
    y = np.ascontiguousarray(Y, dtype=np.float32)
    if x.ndim != 2 or y.ndim != 2 or x.shape[0] != y.shape[0]:
        raise ValueError("X and Y must be [n][d] with the same n")
    out = ctypes.c_double()
    _check(load().spear_linear_cka(x.ctypes.data_as(ctypes.c_void_p), y.ctypes.data_as(ctypes.c_void_p),
                                   x.shape[0], x.shape[1], y.shape[1], ctypes.byref(out)), "spear_linear_cka")
    return out.value


def spear_cka_damage(X_ref, Y_quant) -> float:
    """1 - CKA(X_ref, Y_quant) of two host matrices [n][dx], [n][dy] (fp32),
    computed by the library: one module's damage score."""
    x = np.ascontiguousarray(X_ref, dtype=np.float32)
    y = np.ascontiguousarray(Y_quant, dtype=np.float32)
    if x.ndim != 2 or y.ndim != 2 or x.shape[0] != y.shape[0]:
        raise ValueError("X_ref and Y_quant must be [n][d] with the same n")
    out = ctypes.c_double()
    _check(load().spear_cka_damage(x.ctypes.data_as(ctypes.c_void_p), y.ctypes.data_as(ctypes.c_void_p),
                                   x.shape[0], x.shape[1], y.shape[1], ctypes.byref(out)), "spear_cka_damage")
    return out.value


def cka_damage(reference_outputs, quantised_outputs):
    """Per-module damage scores for the module-selection rule (one
    spear_cka_damage call per module); each argument a list of host [n][d]
    matrices."""
    return np.array([spear_cka_damage(a, b) for a, b in zip(reference_outputs, quantised_outputs)],
                    dtype=np.float32)


class _Curve(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("M", ctypes.c_void_p), ("us", ctypes.c_void_p)]


def spear_chunk_select(prefill_curves, decode_curves, decode_tokens: int, choices, itl_target_us: float):
    """prefill_curves / decode_curves: per layer, a pair (M list, microseconds list).
    Returns (chunk, predicted step microseconds)."""
    keep = []

    def curves(cs):
        arr = (_Curve * len(cs))()
        for i, (Ms, us) in enumerate(cs):
            m = np.ascontiguousarray(Ms, dtype=np.int32)
            u = np.ascontiguousarray(us, dtype=np.float32)
            keep.extend([m, u])
            arr[i] = _Curve(m.shape[0], m.ctypes.data, u.ctypes.data)
        return arr
    pre, dec = curves(prefill_curves), curves(decode_curves)
    ch = np.ascontiguousarray(choices, dtype=np.int32)
    out = ctypes.c_int()
    step = ctypes.c_double()
    _check(load().spear_chunk_select(ctypes.cast(pre, ctypes.c_void_p), ctypes.cast(dec, ctypes.c_void_p),
                                     len(prefill_curves), int(decode_tokens), ch.ctypes.data_as(ctypes.c_void_p),
                                     ch.shape[0], float(itl_target_us), ctypes.byref(out), ctypes.byref(step)),
           "spear_chunk_select")
    return out.value, step.value


# ------------------------------------------------------------ status

def spear_get_device_status(stream=None) -> int:
    out = ctypes.c_int()
    _check(load().spear_get_device_status(ctypes.byref(out), _stream(stream)), "spear_get_device_status")
    return out.value


def spear_set_launch_overlap(enable: bool) -> None:
    """Process-wide: decode launches may start while the previous kernel on
    their stream finishes (programmatic dependent launch).  The caller
    guarantees that the kernel right before a decode call does not write that
    layer's weights; see include/spear.h."""
    _check(load().spear_set_launch_overlap(1 if enable else 0), "spear_set_launch_overlap")


def spear_set_wait_limit_ns(ns: int) -> None:
    """Process-wide limit of the device-side waits on other thread blocks (0:
    the defaults); a wait that runs out records SPEAR_ERR_TIMEOUT.  For tests
    and diagnostics; see include/spear.h."""
    _check(load().spear_set_wait_limit_ns(int(ns)), "spear_set_wait_limit_ns")


def version() -> str:
    return load().spear_version().decode()

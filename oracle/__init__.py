"""The oracle: TEST INFRASTRUCTURE ONLY.

A plain, slow CPU restatement of the routed expert layer in fp64 (``oracle.c``),
wrapped here for numpy. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the library (``routed_expert_layer_gb300``)
never does, and the two share no code.

Parity status of each function (what pins it) is listed in the tests under
``tests/test_oracle_pins.py``; "parity unpinned" items are named there and in the
design notes: the gate-weight values beyond their invariants (no worked example
on the pages) and fidelity to the real checkpoint (no checkpoint available).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c (-O2, OpenMP, no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11",
               _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class _Layer(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int64), ("I", ctypes.c_int64), ("E", ctypes.c_int64),
                ("gu_codes", ctypes.c_void_p), ("gu_scales", ctypes.c_void_p), ("gu_global", ctypes.c_void_p),
                ("dn_codes", ctypes.c_void_p), ("dn_scales", ctypes.c_void_p), ("dn_global", ctypes.c_void_p),
                ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p)]


class _Block(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("d", ctypes.c_int64), ("Is", ctypes.c_int64),
                ("proj_down", ctypes.c_void_p), ("proj_up", ctypes.c_void_p), ("shared_gu", ctypes.c_void_p),
                ("shared_dn", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i64, p, d = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        _lib.oracle_e2m1.restype = d
        _lib.oracle_e2m1.argtypes = [ctypes.c_uint]
        _lib.oracle_e4m3.restype = d
        _lib.oracle_e4m3.argtypes = [ctypes.c_uint]
        _lib.oracle_bf16.restype = d
        _lib.oracle_bf16.argtypes = [ctypes.c_uint16]
        _lib.oracle_dequant.argtypes = [i64, i64, p, p, d, p]
        _lib.oracle_router_logits.argtypes = [i64, i64, i64, p, p, p, p]
        _lib.oracle_router_abs.argtypes = [i64, i64, i64, p, p, p]
        _lib.oracle_select.argtypes = [i64, i64, i64, p, p, p]
        _lib.oracle_permute.argtypes = [i64, i64, i64, p, p, p, p, p, p]
        _lib.oracle_expert_gateup.argtypes = [ctypes.POINTER(_Layer), i64, i64, p, p]
        _lib.oracle_expert_down.argtypes = [ctypes.POINTER(_Layer), i64, i64, p, p]
        _lib.oracle_moe_forward.argtypes = [ctypes.POINTER(_Layer), i64, i64, p, p, p, p, p]
        _lib.oracle_moe_tokens.argtypes = [ctypes.POINTER(_Layer), i64, i64, p, p, p, p, p]
        _lib.oracle_moe_routed.argtypes = [ctypes.POINTER(_Layer), i64, i64, p, p, p, i64, p, p]
        _lib.oracle_moe_block.argtypes = [ctypes.POINTER(_Layer), ctypes.POINTER(_Block), i64, i64, p, p, p, p, p]
        _lib.oracle_num_threads.restype = ctypes.c_int
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e4m3(byte: int) -> float:
    return lib().oracle_e4m3(byte)


def bf16(bits: int) -> float:
    return lib().oracle_bf16(bits)


def dequant(codes: np.ndarray, scales: np.ndarray, global_scale: float) -> np.ndarray:
    rows, half = codes.shape
    K = 2 * half
    out = np.empty((rows, K), dtype=np.float64)
    lib().oracle_dequant(rows, K, _ptr(codes), _ptr(scales), float(global_scale), _ptr(out))
    return out


def router_logits(x_bits: np.ndarray, W_r: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    T, H = x_bits.shape
    E = W_r.shape[1]
    out = np.empty((T, E), dtype=np.float64)
    if T:
        lib().oracle_router_logits(T, H, E, _ptr(x_bits), _ptr(W_r), _ptr(bias), _ptr(out))
    return out


def router_abs(x_bits: np.ndarray, W_r: np.ndarray) -> np.ndarray:
    """sum_h |x_h * W_r[h, e]| per (token, expert)."""
    T, H = x_bits.shape
    E = W_r.shape[1]
    out = np.empty((T, E), dtype=np.float64)
    if T:
        lib().oracle_router_abs(T, H, E, _ptr(x_bits), _ptr(W_r), _ptr(out))
    return out


def select(logits: np.ndarray, k: int):
    """(idx int32 [T][k], w float64 [T][k]) from logits [T][E] (any float dtype, widened exactly)."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    if T:
        lib().oracle_select(T, E, k, _ptr(logits), _ptr(idx), _ptr(w))
    return idx, w


def permute(idx: np.ndarray, E: int):
    """(counts [E], offsets [E+1], perm [T*k], slot [T*k], inv [T*k]) -- all int32."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    slot = np.empty(T * k, dtype=np.int32)
    inv = np.empty(T * k, dtype=np.int32)
    lib().oracle_permute(T, E, k, _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(slot), _ptr(inv))
    return counts, offsets, perm, slot, inv


class Layer:
    """Holds references to a synthetic layer's arrays (see ``synth.Layer``) for the C oracle."""

    def __init__(self, layer):
        self.src = layer
        self.arrays = [np.ascontiguousarray(a) for a in (
            layer.gu_codes, layer.gu_scales, layer.gu_global, layer.dn_codes, layer.dn_scales,
            layer.dn_global, layer.router_w)]
        self.bias = None if layer.router_bias is None else np.ascontiguousarray(layer.router_bias, np.float32)
        gc, gs, gg, dc, ds, dg, rw = self.arrays
        self.c = _Layer(layer.H, layer.I, layer.E, gc.ctypes.data, gs.ctypes.data, gg.ctypes.data,
                        dc.ctypes.data, ds.ctypes.data, dg.ctypes.data, rw.ctypes.data,
                        None if self.bias is None else self.bias.ctypes.data)
        self.H, self.I, self.E = layer.H, layer.I, layer.E


def expert_gateup(L: Layer, e: int, xs: np.ndarray) -> np.ndarray:
    xs = np.ascontiguousarray(xs, dtype=np.float64)
    n = xs.shape[0]
    hs = np.empty((n, L.I), dtype=np.float64)
    lib().oracle_expert_gateup(ctypes.byref(L.c), e, n, _ptr(xs), _ptr(hs))
    return hs


def expert_down(L: Layer, e: int, hs: np.ndarray) -> np.ndarray:
    hs = np.ascontiguousarray(hs, dtype=np.float64)
    n = hs.shape[0]
    ys = np.empty((n, L.H), dtype=np.float64)
    lib().oracle_expert_down(ctypes.byref(L.c), e, n, _ptr(hs), _ptr(ys))
    return ys


def moe_forward(L: Layer, x_bits: np.ndarray, k: int):
    """Whole layer: returns (out fp64 [T][H], idx [T][k], w [T][k], logits [T][E])."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T = x_bits.shape[0]
    out = np.empty((T, L.H), dtype=np.float64)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    logits = np.empty((T, L.E), dtype=np.float64)
    if T:
        lib().oracle_moe_forward(ctypes.byref(L.c), T, k, _ptr(x_bits), _ptr(out), _ptr(idx), _ptr(w), _ptr(logits))
    return out, idx, w, logits


def moe_tokens(L: Layer, x_rows: np.ndarray, k: int):
    """The layer one token at a time (for sampled rows): (out, idx, w, logits)."""
    x_rows = np.ascontiguousarray(x_rows, dtype=np.uint16)
    n = x_rows.shape[0]
    out = np.empty((n, L.H), dtype=np.float64)
    idx = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float64)
    logits = np.empty((n, L.E), dtype=np.float64)
    if n:
        lib().oracle_moe_tokens(ctypes.byref(L.c), n, k, _ptr(x_rows), _ptr(out), _ptr(idx), _ptr(w), _ptr(logits))
    return out, idx, w, logits


def moe_routed(L: Layer, x_bits: np.ndarray, idx: np.ndarray, w: np.ndarray, e0: int = 0):
    """The expert stage on given routing for a worker holding experts [e0, e0 + L.E) (L
    holds those experts only): (out fp64 [T][H], served int32 [T][k])."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    T, k = idx.shape
    out = np.empty((T, L.H), dtype=np.float64)
    served = np.empty((T, k), dtype=np.int32)
    if T:
        lib().oracle_moe_routed(ctypes.byref(L.c), T, k, _ptr(x_bits), _ptr(idx), _ptr(w), e0, _ptr(out),
                                _ptr(served))
    return out, served


def moe_block(L: Layer, x_rows: np.ndarray, k: int):
    """A LatentMoE block one token at a time (L from a synth.block_layer: experts at the
    latent width, the hidden width and the bf16 dense weights): (out [n][hidden], idx,
    w, logits)."""
    src = L.src
    x_rows = np.ascontiguousarray(x_rows, dtype=np.uint16)
    n = x_rows.shape[0]
    Is = 0 if src.shared_gu is None else src.shared_gu.shape[0] // 2
    keep = [np.ascontiguousarray(a, dtype=np.uint16) if a is not None else None
            for a in (src.proj_down, src.proj_up, src.shared_gu, src.shared_dn)]
    B = _Block(src.hidden, src.H, Is, *[None if a is None else a.ctypes.data for a in keep])
    out = np.empty((n, src.hidden), dtype=np.float64)
    idx = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float64)
    logits = np.empty((n, L.E), dtype=np.float64)
    if n:
        lib().oracle_moe_block(ctypes.byref(L.c), ctypes.byref(B), n, k, _ptr(x_rows), _ptr(out), _ptr(idx), _ptr(w),
                               _ptr(logits))
    return out, idx, w, logits


def num_threads() -> int:
    return lib().oracle_num_threads()

"""Seeded synthetic inputs for the routed expert layer (numpy in, numpy out).

Holds no arithmetic of the layer itself: a counter-based Gaussian generator, the
NVFP4 encoder that turns Gaussian weights into E2M1 codes with E4M3 block scales
and an fp32 tensor scale, and a Zipf router bias. Used by the oracle-side tests
and by the CUDA-side tests and benchmark alike; neither of those imports the
other. The C source is ``synth.c`` beside this file.

Recipe (seeds are arguments; the tests and the benchmark use weights=1,
router=2, x=3+batch, Zipf permutation=4):
  x        bf16 ~ N(0, 1)                         [T][H]
  W_r      fp32 ~ N(0, 1/H)                       [H][E]
  experts  N(0, 1/fan_in), fan_in = H (gate, up) or I (down), then NVFP4
  Zipf     bias_e = -s * ln(rank_e), ranks over a seeded permutation
  LatentMoE block (bf16 dense weights, seed = weights seed):
           routed-down [d][H] ~ N(0, 1/H), routed-up [H][d] ~ N(0, 1/d),
           shared gate/up [2Is][H] ~ N(0, 1/H), shared down [H][Is] ~ N(0, 1/Is)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library next to this file."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11",
               _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        p = ctypes.c_void_p
        _lib.synth_hash.restype = u64
        _lib.synth_hash.argtypes = [u64, u64, u64]
        _lib.synth_normal.restype = ctypes.c_double
        _lib.synth_normal.argtypes = [u64, u64, u64]
        _lib.synth_normal_f32.argtypes = [u64, u64, i64, ctypes.c_float, p]
        _lib.synth_x_bf16.argtypes = [u64, i64, i64, p]
        _lib.synth_router.argtypes = [u64, i64, i64, p]
        _lib.synth_logits.argtypes = [u64, i64, i64, p]
        _lib.synth_e4m3_encode.restype = ctypes.c_uint8
        _lib.synth_e4m3_encode.argtypes = [ctypes.c_double]
        _lib.synth_e2m1_encode.restype = ctypes.c_uint8
        _lib.synth_e2m1_encode.argtypes = [ctypes.c_double]
        _lib.synth_quantize_nvfp4.argtypes = [p, i64, i64, p, p, p]
        _lib.synth_experts.argtypes = [u64, i64, i64, i64, p, p, p, p, p, p]
        _lib.synth_zipf_bias.argtypes = [u64, i64, ctypes.c_double, p]
        _lib.synth_bf16_normal.argtypes = [u64, u64, i64, ctypes.c_float, p]
        _lib.synth_num_threads.restype = ctypes.c_int
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def x_bf16(seed: int, T: int, H: int) -> np.ndarray:
    """Activations as bf16 bit patterns, uint16 [T][H]."""
    out = np.empty((T, H), dtype=np.uint16)
    if T * H:
        lib().synth_x_bf16(seed, T, H, _ptr(out))
    return out


def router(seed: int, H: int, E: int) -> np.ndarray:
    out = np.empty((H, E), dtype=np.float32)
    lib().synth_router(seed, H, E, _ptr(out))
    return out


def logits(seed: int, T: int, E: int) -> np.ndarray:
    out = np.empty((T, E), dtype=np.float32)
    if T * E:
        lib().synth_logits(seed, T, E, _ptr(out))
    return out


def normal_f32(seed: int, stream: int, n: int, scale: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_normal_f32(seed, stream, n, scale, _ptr(out))
    return out


def quantize_nvfp4(w: np.ndarray):
    """w float32 [rows][K] -> (codes uint8 [rows][K/2], scales uint8 [rows][K/16], global fp32)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, K = w.shape
    assert K % 16 == 0
    codes = np.empty((rows, K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // 16), dtype=np.uint8)
    g = np.empty(1, dtype=np.float32)
    lib().synth_quantize_nvfp4(_ptr(w), rows, K, _ptr(codes), _ptr(scales), _ptr(g))
    return codes, scales, float(g[0])


def bf16_normal(seed: int, which: int, rows: int, cols: int, scale: float) -> np.ndarray:
    """A bf16 dense weight [rows][cols] ~ N(0, scale^2) as bit patterns (uint16)."""
    out = np.empty((rows, cols), dtype=np.uint16)
    lib().synth_bf16_normal(seed, which, rows * cols, scale, _ptr(out))
    return out


def zipf_bias(seed: int, E: int, s: float = 1.1) -> np.ndarray:
    out = np.empty(E, dtype=np.float32)
    lib().synth_zipf_bias(seed, E, s, _ptr(out))
    return out


@dataclass
class Layer:
    """One routed-expert layer in the host layout the C-ABI loads.

    gu_codes  uint8 [E][2I][H/2]   rows 0..I-1 gate, I..2I-1 up; element k of a row
                                   is in byte k/2, low nibble = even k
    gu_scales uint8 [E][2I][H/16]  E4M3 block scales along K
    gu_global fp32  [E][2]         (gate, up) tensor scales
    dn_codes  uint8 [E][H][I/2]
    dn_scales uint8 [E][H][I/16]
    dn_global fp32  [E]
    router_w  fp32  [H][E]
    router_bias fp32 [E] or None
    """
    H: int
    I: int
    E: int
    gu_codes: np.ndarray
    gu_scales: np.ndarray
    gu_global: np.ndarray
    dn_codes: np.ndarray
    dn_scales: np.ndarray
    dn_global: np.ndarray
    router_w: np.ndarray
    router_bias: np.ndarray | None = None
    # LatentMoE block (None for a plain layer): the experts above work in width H = d (the
    # routed latent); the layer's rows are `hidden` wide and the router reads them
    # (router_w is [hidden][E]).
    hidden: int | None = None
    proj_down: np.ndarray | None = None  # bf16 bits [d][hidden]
    proj_up: np.ndarray | None = None    # bf16 bits [hidden][d]
    shared_gu: np.ndarray | None = None  # bf16 bits [2 Is][hidden]: gate rows, then up rows
    shared_dn: np.ndarray | None = None  # bf16 bits [hidden][Is]

    @property
    def expert_bytes(self) -> int:
        """Bytes of one expert: codes + block scales + the three fp32 tensor scales
        + three fp32 input scales (kept in the census, unused with bf16 activations)."""
        H, I = self.H, self.I
        return 3 * H * I // 2 + 3 * H * I // 16 + 6 * 4


def layer(H: int, I: int, E: int, seed_weights: int = 1, seed_router: int = 2,
          zipf_seed: int | None = None, zipf_s: float = 1.1) -> Layer:
    assert H % 16 == 0 and I % 16 == 0
    gu_codes = np.empty((E, 2 * I, H // 2), dtype=np.uint8)
    gu_scales = np.empty((E, 2 * I, H // 16), dtype=np.uint8)
    gu_global = np.empty((E, 2), dtype=np.float32)
    dn_codes = np.empty((E, H, I // 2), dtype=np.uint8)
    dn_scales = np.empty((E, H, I // 16), dtype=np.uint8)
    dn_global = np.empty((E,), dtype=np.float32)
    lib().synth_experts(seed_weights, H, I, E, _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_global),
                        _ptr(dn_codes), _ptr(dn_scales), _ptr(dn_global))
    bias = zipf_bias(zipf_seed, E, zipf_s) if zipf_seed is not None else None
    return Layer(H, I, E, gu_codes, gu_scales, gu_global, dn_codes, dn_scales, dn_global,
                 router(seed_router, H, E), bias)


def block_layer(hidden: int, d: int, I: int, E: int, shared_inter: int = 0, seed_weights: int = 1,
                seed_router: int = 2, zipf_seed: int | None = None, zipf_s: float = 1.1) -> Layer:
    """A LatentMoE block: experts at width d (NVFP4, as layer()), a router over the hidden
    rows, the bf16 routed-down / routed-up projections and, when shared_inter > 0, the
    shared experts (all of them as one gate/up and one down tensor)."""
    L = layer(d, I, E, seed_weights, seed_router, zipf_seed, zipf_s)
    L.router_w = router(seed_router, hidden, E)
    L.hidden = hidden
    L.proj_down = bf16_normal(seed_weights, 1, d, hidden, 1.0 / np.sqrt(hidden))
    L.proj_up = bf16_normal(seed_weights, 2, hidden, d, 1.0 / np.sqrt(d))
    if shared_inter:
        L.shared_gu = bf16_normal(seed_weights, 3, 2 * shared_inter, hidden, 1.0 / np.sqrt(hidden))
        L.shared_dn = bf16_normal(seed_weights, 4, hidden, shared_inter, 1.0 / np.sqrt(shared_inter))
    return L


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact): a storage conversion, not layer arithmetic."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# Workloads (sizes from the configurations the layer is measured on).
TINY = dict(H=256, I=128, E=32, k=4)
K3 = dict(H=7168, I=1536, E=896, k=16)

"""routed_expert_layer_gb300 -- a routed Mixture-of-Experts layer for GB300 (sm_103a).

Thin Python binding over the C ABI declared in ``include/moe_gb300.h``: argument
marshalling only. Every step of the layer runs in the library's CUDA kernels;
PyTorch is used by callers for device memory and streams. There is no CPU path:
if the CUDA library is missing, importing ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_BUILD = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD, "libmoe_gb300.so")
_SOURCES = ["api.cu", "route.cu", "router_tc.cu", "expert_tc.cu", "noalloc.cu", "block.cu"]
_HEADERS = ["moe_internal.cuh", "tc_ptx.cuh"]
NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr"]

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_NOT_LOADED = 0, -1, -2, -3
MOE_ERR_OOM, MOE_ERR_CUDA, MOE_ERR_DEVICE_FLAG = -4, -5, -6

EXPORTED = ["moe_create", "moe_load_layer", "moe_forward", "moe_forward_host", "moe_destroy", "moe_status_str",
            "moe_get_error", "moe_debug_route", "moe_debug_select", "moe_debug_experts", "moe_profile_stages",
            "moe_profile_stage_name", "moe_profile_begin", "moe_profile_end", "moe_device_bytes", "moe_launch_count",
            "moe_route_noalloc", "moe_plan", "moe_forward_routed", "moe_debug_pdl_copy"]

# Revision of each kernel's code; a stored ncu traffic figure is only reported while
# the revision it was measured on is current. "gateup" and "down" are the decode grouped
# GEMM (the bench's dominant kernel), "prefill" the prefill / midfill grouped GEMM.
KERNEL_REV = {"router": "tc3-1", "select": "warp-6", "permute": "mask-6", "gather": "f16-6",
              "gateup": "tc-14", "down": "tc-14", "prefill": "tc-18", "combine": "f32-6"}


def _nvcc() -> str:
    for p in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(p):
            return p
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library in-tree for sm_103a (one -gencode, parallel TUs)."""
    os.makedirs(_BUILD, exist_ok=True)
    deps = [os.path.join(_CSRC, f) for f in _SOURCES + _HEADERS] + [os.path.join(_ROOT, "include", "moe_gb300.h")]
    newest = max(os.path.getmtime(d) for d in deps)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(_BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *NVCC_ARCH, *NVCC_FLAGS, "-c", os.path.join(_CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(_SOURCES)) as ex:
        objs = list(ex.map(compile_one, _SOURCES))
    tmp = LIB_PATH + ".tmp"
    r = subprocess.run([nvcc, *NVCC_ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("expert_begin", ctypes.c_int32), ("expert_count", ctypes.c_int32), ("latent", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32)]


class LayerHost(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("gu_codes", ctypes.POINTER(ctypes.c_void_p)), ("gu_scales", ctypes.POINTER(ctypes.c_void_p)),
                ("gu_global", ctypes.c_void_p),
                ("dn_codes", ctypes.POINTER(ctypes.c_void_p)), ("dn_scales", ctypes.POINTER(ctypes.c_void_p)),
                ("dn_global", ctypes.c_void_p), ("proj_down", ctypes.c_void_p), ("proj_up", ctypes.c_void_p),
                ("shared_gu", ctypes.c_void_p), ("shared_dn", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded C library. Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} (run __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, vp = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
        L.moe_create.argtypes = [ctypes.POINTER(Config), ctypes.c_int, ctypes.POINTER(vp)]
        L.moe_load_layer.argtypes = [vp, ctypes.POINTER(LayerHost)]
        L.moe_forward.argtypes = [vp, vp, p, p, i32]
        L.moe_forward_host.argtypes = [vp, vp, p, p, i32]
        L.moe_forward_routed.argtypes = [vp, vp, p, p, p, p, i32, p]
        L.moe_destroy.argtypes = [vp]
        L.moe_status_str.restype = ctypes.c_char_p
        L.moe_status_str.argtypes = [ctypes.c_int]
        L.moe_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.moe_debug_route.argtypes = [vp, vp, p, i32, p, p, p, p, p, p, p]
        L.moe_debug_select.argtypes = [vp, vp, p, i32, p, p, p, p, p, p]
        L.moe_debug_experts.argtypes = [vp, vp, p, i32, p, p, p]
        L.moe_debug_pdl_copy.argtypes = [vp, p, p, ctypes.c_int64]
        L.moe_profile_stage_name.restype = ctypes.c_char_p
        L.moe_profile_stage_name.argtypes = [ctypes.c_int]
        L.moe_profile_begin.argtypes = [vp, i32]
        L.moe_profile_end.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(i32), i32]
        L.moe_device_bytes.restype = ctypes.c_int64
        L.moe_device_bytes.argtypes = [vp]
        L.moe_plan.argtypes = [ctypes.POINTER(Config), ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64)]
        L.moe_launch_count.restype = ctypes.c_int64
        L.moe_launch_count.argtypes = [vp]
        L.moe_route_noalloc.argtypes = [vp, p, p, p, i32, i32, i32, i32, p, p, p, p, p, p, p]
        _lib = L
    return _lib


def route_noalloc(x, router_w, router_bias, k, idx, w, offsets, perm, slot, inv, err=None, stream=None) -> None:
    """Routing without any device allocation (see moe_route_noalloc in the header).
    Every argument is a contiguous CUDA tensor on the current device; the outputs are
    caller-allocated: idx int32 [T][k], w float32 [T][k], offsets int32 [E+1], perm, slot,
    inv int32 [T*k]; err (optional) a uint32/int32 word the kernels OR their error bits
    into. The C entry point only sees plain pointers, so every size is checked here."""
    import torch
    if x.dim() != 2 or x.element_size() != 2:
        raise ValueError("x: expected [T][H] with 2-byte (bf16) elements")
    T, H = x.shape
    if router_w.dim() != 2 or router_w.shape[0] != H or router_w.dtype != torch.float32:
        raise ValueError(f"router_w: expected float32 [{H}][E], got {router_w.dtype} {list(router_w.shape)}")
    E = router_w.shape[1]
    expect = {"idx": (idx, (T, k), torch.int32), "w": (w, (T, k), torch.float32),
              "offsets": (offsets, (E + 1,), torch.int32), "perm": (perm, (T * k,), torch.int32),
              "slot": (slot, (T * k,), torch.int32), "inv": (inv, (T * k,), torch.int32)}
    if router_bias is not None:
        expect["router_bias"] = (router_bias, (E,), torch.float32)
    if err is not None:
        if err.numel() != 1 or err.element_size() != 4:
            raise ValueError("err: expected one 4-byte word")
        expect["err"] = (err, tuple(err.shape), err.dtype)
    tensors = {"x": (x, (T, H), x.dtype), "router_w": (router_w, (H, E), torch.float32), **expect}
    for name, (t, shape, dtype) in tensors.items():
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name}: expected {dtype} {list(shape)}, got {t.dtype} {list(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")
        if not t.is_cuda:
            raise ValueError(f"{name}: expected a CUDA tensor")
    dev = torch.cuda.current_device()
    for name, (t, _, _) in tensors.items():
        if t.device.index != dev:
            raise ValueError(f"{name}: expected a tensor on the current device cuda:{dev}, got {t.device}")
    _check(lib().moe_route_noalloc(_stream(stream), _dptr(x), _dptr(router_w), _dptr(router_bias), H, E, k, T,
                                   _dptr(idx), _dptr(w), _dptr(offsets), _dptr(perm), _dptr(slot), _dptr(inv),
                                   _dptr(err)),
           "moe_route_noalloc")


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {lib().moe_status_str(status).decode()} ({status})")
        self.status = status


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _dptr(t):
    """Device pointer of a torch tensor (or None)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _rows(t, H: int, what: str, cuda: bool) -> int:
    """Check that t is a contiguous [T][H] array of 2-byte elements (a CUDA tensor when
    cuda, else a numpy array or a host torch tensor) and return T. The C entry points
    take plain pointers, so this is where a wrong shape is caught."""
    shape = tuple(t.shape)
    if len(shape) != 2 or shape[1] != H:
        raise ValueError(f"{what}: expected shape [T][{H}], got {list(shape)}")
    if isinstance(t, np.ndarray):
        if cuda:
            raise ValueError(f"{what}: expected a CUDA tensor, got a numpy array")
        if t.itemsize != 2 or not t.flags["C_CONTIGUOUS"]:
            raise ValueError(f"{what}: expected contiguous 2-byte elements")
        return shape[0]
    if t.element_size() != 2 or not t.is_contiguous():
        raise ValueError(f"{what}: expected contiguous 2-byte elements")
    if t.is_cuda != cuda:
        raise ValueError(f"{what}: expected a {'CUDA' if cuda else 'host'} tensor")
    return shape[0]


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def debug_pdl_copy(src, dst, stream=None) -> None:
    """moe_debug_pdl_copy: dst = src (same-size contiguous device tensors, bytes a multiple
    of 16) by a kernel launched as a programmatic dependent of the stream's previous one."""
    if src.nbytes != dst.nbytes or not src.is_contiguous() or not dst.is_contiguous():
        raise ValueError("debug_pdl_copy: src and dst must be contiguous and of the same size")
    if not src.is_cuda or not dst.is_cuda:
        raise ValueError("debug_pdl_copy: device tensors expected")
    _check(lib().moe_debug_pdl_copy(_stream(stream), _dptr(src), _dptr(dst), src.nbytes), "moe_debug_pdl_copy")


PLAN_FIELDS = ("prefill", "rows_per_item", "gateup_splits", "down_splits", "gemm_ctas", "router_splits",
               "router_ctas", "fused_routing", "chunk_capacity", "workspace_bytes", "cold_rows")


def plan(hidden: int, inter: int, n_experts: int, top_k: int, max_tokens: int, sm_count: int, T: int) -> dict:
    """The launch plan moe_forward uses for T tokens (host only, no GPU needed)."""
    cfg = Config(hidden, inter, n_experts, top_k, max_tokens, 0)
    out = (ctypes.c_int64 * len(PLAN_FIELDS))()
    _check(lib().moe_plan(ctypes.byref(cfg), sm_count, T, out), "moe_plan")
    return {k: int(v) for k, v in zip(PLAN_FIELDS, out)}


class MoeLayer:
    """One routed expert layer on one GPU (wraps a moe_ctx). expert_begin / expert_count
    select the experts this context holds (0 / 0: all of them); latent > 0 makes it a
    LatentMoE block whose experts work in `latent` dimensions between bf16 routed-down and
    routed-up projections, with shared experts of total intermediate size shared_inter."""

    def __init__(self, hidden: int, inter: int, n_experts: int, top_k: int, max_tokens: int, device: int = 0,
                 expert_begin: int = 0, expert_count: int = 0, latent: int = 0, shared_inter: int = 0):
        self.cfg = Config(hidden, inter, n_experts, top_k, max_tokens, 0, expert_begin, expert_count, latent,
                          shared_inter)
        self.device = device
        self.ctx = ctypes.c_void_p()
        _check(lib().moe_create(ctypes.byref(self.cfg), device, ctypes.byref(self.ctx)), "moe_create")

    @property
    def H(self):
        return self.cfg.hidden

    @property
    def k(self):
        return self.cfg.top_k

    @property
    def D(self):
        """Width the routed experts work in."""
        return self.cfg.latent or self.cfg.hidden

    @property
    def n_local(self):
        """Experts this context holds."""
        return self.cfg.expert_count or self.cfg.n_experts

    def load(self, layer) -> None:
        """layer: object with numpy arrays gu_codes [n][2I][D/2], gu_scales, gu_global [n][2],
        dn_codes [n][D][I/2], dn_scales, dn_global [n], router_w [H][E], router_bias [E] or None,
        where n is either the context's expert count (its experts only) or E (the whole
        layer, of which the context's range is taken) and D the experts' width; for a
        LatentMoE block also proj_down [d][H], proj_up [H][d], shared_gu [2Is][H] and
        shared_dn [H][Is] (bf16 bit patterns)."""
        E, H, I, D = self.cfg.n_experts, self.cfg.hidden, self.cfg.inter, self.D
        n, e0 = self.n_local, self.cfg.expert_begin
        expert_arrays = ("gu_codes", "gu_scales", "gu_global", "dn_codes", "dn_scales", "dn_global")
        if n != E and len(np.shape(layer.gu_codes)) and np.shape(layer.gu_codes)[0] == E:
            import dataclasses
            layer = dataclasses.replace(layer, **{a: getattr(layer, a)[e0:e0 + n] for a in expert_arrays})
        expect = {"gu_codes": (n, 2 * I, D // 2), "gu_scales": (n, 2 * I, D // 16), "gu_global": (n, 2),
                  "dn_codes": (n, D, I // 2), "dn_scales": (n, D, I // 16), "dn_global": (n,), "router_w": (H, E)}
        d, Is = self.cfg.latent, self.cfg.shared_inter
        if d:
            expect.update(proj_down=(d, H), proj_up=(H, d))
        if Is:
            expect.update(shared_gu=(2 * Is, H), shared_dn=(H, Is))
        for name, shape in expect.items():  # the library reads these sizes through plain pointers
            if tuple(np.shape(getattr(layer, name))) != shape:
                raise ValueError(f"{name}: expected shape {list(shape)}, got {list(np.shape(getattr(layer, name)))}")
        if layer.router_bias is not None and tuple(np.shape(layer.router_bias)) != (E,):
            raise ValueError(f"router_bias: expected shape [{E}]")
        keep = []

        def arr(a, dtype):
            a = np.ascontiguousarray(a, dtype=dtype)
            keep.append(a)
            return a

        def per_expert(a):
            a = arr(a, np.uint8)
            assert a.shape[0] == n
            ptrs = (ctypes.c_void_p * n)(*[a.ctypes.data + e * a.strides[0] for e in range(n)])
            keep.append(ptrs)
            return ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p))

        rw = arr(layer.router_w, np.float32)
        rb = None if layer.router_bias is None else arr(layer.router_bias, np.float32)

        def dense(name):
            a = getattr(layer, name, None)
            return None if a is None or name not in expect else arr(a, np.uint16).ctypes.data

        lh = LayerHost(rw.ctypes.data, None if rb is None else rb.ctypes.data,
                       per_expert(layer.gu_codes), per_expert(layer.gu_scales),
                       arr(layer.gu_global, np.float32).ctypes.data,
                       per_expert(layer.dn_codes), per_expert(layer.dn_scales),
                       arr(layer.dn_global, np.float32).ctypes.data,
                       dense("proj_down"), dense("proj_up"), dense("shared_gu"), dense("shared_dn"))
        _check(lib().moe_load_layer(self.ctx, ctypes.byref(lh)), "moe_load_layer")

    def forward(self, x, out, stream=None) -> None:
        """x, out: CUDA tensors of bf16 [T][H] (any dtype with 2-byte elements)."""
        T = _rows(x, self.H, "x", True)
        if _rows(out, self.H, "out", True) != T:
            raise ValueError("out: expected as many rows as x")
        _check(lib().moe_forward(self.ctx, _stream(stream), _dptr(x), _dptr(out), T), "moe_forward")

    def forward_routed(self, x, idx, w, out, served=None, stream=None) -> None:
        """The expert stage on caller-given routing (moe_forward_routed): x and out [T][D]
        (the experts' width), idx int32 [T][k] global expert ids (-1 masked), w float32
        [T][k], served int32 [T][k] or None."""
        import torch
        T = _rows(x, self.D, "x", True)
        if _rows(out, self.D, "out", True) != T:
            raise ValueError("out: expected as many rows as x")
        for name, t, dt in (("idx", idx, torch.int32), ("w", w, torch.float32), ("served", served, torch.int32)):
            if t is None and name == "served":
                continue
            if tuple(t.shape) != (T, self.k) or t.dtype != dt or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name}: expected a contiguous CUDA {dt} tensor of shape [{T}][{self.k}]")
        _check(lib().moe_forward_routed(self.ctx, _stream(stream), _dptr(x), _dptr(idx), _dptr(w), _dptr(out), T,
                                        _dptr(served)), "moe_forward_routed")

    def forward_host(self, x_host, out_host, stream=None) -> None:
        """x_host, out_host: host buffers (numpy uint16 or pinned torch tensors) of [T][H] bf16."""
        T = _rows(x_host, self.H, "x_host", False)
        if _rows(out_host, self.H, "out_host", False) != T:
            raise ValueError("out_host: expected as many rows as x_host")
        xp = x_host.ctypes.data if isinstance(x_host, np.ndarray) else x_host.data_ptr()
        op = out_host.ctypes.data if isinstance(out_host, np.ndarray) else out_host.data_ptr()
        _check(lib().moe_forward_host(self.ctx, _stream(stream), ctypes.c_void_p(xp), ctypes.c_void_p(op), T),
               "moe_forward_host")

    def debug_route(self, x, logits=None, idx=None, w=None, offsets=None, perm=None, slot=None, inv=None,
                    stream=None):
        _rows(x, self.H, "x", True)
        _check(lib().moe_debug_route(self.ctx, _stream(stream), _dptr(x), x.shape[0], _dptr(logits), _dptr(idx),
                                     _dptr(w), _dptr(offsets), _dptr(perm), _dptr(slot), _dptr(inv)),
               "moe_debug_route")

    def debug_select(self, logits, idx=None, w=None, offsets=None, perm=None, slot=None, inv=None, stream=None):
        _check(lib().moe_debug_select(self.ctx, _stream(stream), _dptr(logits), logits.shape[0], _dptr(idx),
                                      _dptr(w), _dptr(offsets), _dptr(perm), _dptr(slot), _dptr(inv)),
               "moe_debug_select")

    def debug_experts(self, x, h=None, y=None, lat=None, stream=None):
        _rows(x, self.H, "x", True)
        _check(lib().moe_debug_experts(self.ctx, _stream(stream), _dptr(x), x.shape[0], _dptr(h), _dptr(y),
                                       _dptr(lat)), "moe_debug_experts")

    def get_error(self) -> int:
        bits = ctypes.c_uint32(0)
        st = lib().moe_get_error(self.ctx, ctypes.byref(bits))
        if st not in (MOE_OK, MOE_ERR_DEVICE_FLAG):
            _check(st, "moe_get_error")
        return bits.value

    def profile_begin(self, max_calls: int) -> None:
        _check(lib().moe_profile_begin(self.ctx, max_calls), "moe_profile_begin")

    def profile_end(self) -> dict:
        n = lib().moe_profile_stages()
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int32 * n)()
        _check(lib().moe_profile_end(self.ctx, ms, cnt, n), "moe_profile_end")
        return {lib().moe_profile_stage_name(i).decode(): (ms[i], cnt[i]) for i in range(n)}

    def launch_count(self) -> int:
        """Kernels this layer has enqueued so far."""
        return lib().moe_launch_count(self.ctx)

    def device_bytes(self) -> int:
        return lib().moe_device_bytes(self.ctx)

    def close(self) -> None:
        if self.ctx:
            lib().moe_destroy(self.ctx)
            self.ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

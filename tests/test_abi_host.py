"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before touching a GPU (no CUDA call is reached here)."""
import ctypes
import os
import re

import pytest

import routed_expert_layer_gb300 as rel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    rel.build()
    return rel.lib()


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            with open(os.path.join(inc, f)) as fh:
                names |= set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", fh.read(), flags=re.M))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 15
    for n in sorted(names):
        assert hasattr(L, n), n
    assert set(rel.EXPORTED) <= names


def test_status_strings(L):
    assert L.moe_status_str(0) == b"ok"
    assert L.moe_status_str(-2).startswith(b"unsupported")
    assert L.moe_status_str(123) == b"unknown status"


def _cfg(**kw):
    base = dict(hidden=256, inter=128, n_experts=32, top_k=4, max_tokens=8, flags=0)
    base.update(kw)
    return rel.Config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(hidden=0), rel.MOE_ERR_INVALID_ARG),
    (dict(max_tokens=0), rel.MOE_ERR_INVALID_ARG),
    (dict(flags=1), rel.MOE_ERR_INVALID_ARG),
    (dict(hidden=300), rel.MOE_ERR_UNSUPPORTED),
    (dict(inter=96), rel.MOE_ERR_UNSUPPORTED),
    (dict(top_k=33, n_experts=64), rel.MOE_ERR_UNSUPPORTED),
    (dict(top_k=8, n_experts=4), rel.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=2048), rel.MOE_ERR_UNSUPPORTED),
    (dict(hidden=16384), rel.MOE_ERR_UNSUPPORTED),
    (dict(max_tokens=2**28, top_k=16), rel.MOE_ERR_UNSUPPORTED),
    (dict(expert_begin=-1, expert_count=4), rel.MOE_ERR_INVALID_ARG),
    (dict(expert_count=-1), rel.MOE_ERR_INVALID_ARG),
    (dict(expert_begin=5, expert_count=0), rel.MOE_ERR_INVALID_ARG),
    (dict(expert_begin=30, expert_count=3), rel.MOE_ERR_INVALID_ARG),
    (dict(latent=-256), rel.MOE_ERR_INVALID_ARG),
    (dict(latent=100), rel.MOE_ERR_UNSUPPORTED),
    (dict(shared_inter=64), rel.MOE_ERR_UNSUPPORTED),              # shared experts need the block
    (dict(latent=256, shared_inter=32), rel.MOE_ERR_UNSUPPORTED),
    (dict(latent=256, expert_begin=0, expert_count=16), rel.MOE_ERR_UNSUPPORTED),  # a block is one context
    (dict(latent=256, shared_inter=64, expert_begin=16, expert_count=16), rel.MOE_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_config_on_host(L, kw, status):
    out = ctypes.c_void_p(1234)
    cfg = _cfg(**kw)
    assert L.moe_create(ctypes.byref(cfg), 0, ctypes.byref(out)) == status
    assert out.value is None


def test_null_arguments(L):
    cfg = _cfg()
    assert L.moe_create(ctypes.byref(cfg), 0, None) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_create(None, 0, ctypes.byref(ctypes.c_void_p())) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_destroy(None) == rel.MOE_OK
    assert L.moe_forward(None, None, None, None, 1) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_forward_host(None, None, None, None, 1) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_load_layer(None, None) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_get_error(None, None) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_debug_route(None, None, None, 1, None, None, None, None, None, None, None) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_debug_select(None, None, None, 1, None, None, None, None, None, None) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_profile_begin(None, 1) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_device_bytes(None) == 0


def test_binding_pdl_copy_checks_tensors():
    import torch
    with pytest.raises(ValueError):
        rel.debug_pdl_copy(torch.zeros(8, dtype=torch.int16), torch.zeros(8, dtype=torch.int16))  # host tensors
    with pytest.raises(ValueError):
        rel.debug_pdl_copy(torch.zeros(8, dtype=torch.int16), torch.zeros(16, dtype=torch.int16))  # sizes differ


def test_pdl_copy_checks_its_arguments_before_launching(L):
    """moe_debug_pdl_copy rejects NULL, misaligned, overlapping and odd-sized arguments on the
    host (the pointers below are never dereferenced), and a zero-byte copy enqueues nothing."""
    a, b = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    bad = rel.MOE_ERR_INVALID_ARG
    assert L.moe_debug_pdl_copy(None, None, b, 16) == bad
    assert L.moe_debug_pdl_copy(None, a, None, 16) == bad
    assert L.moe_debug_pdl_copy(None, ctypes.c_void_p(0x10008), b, 16) == bad  # src not 16-byte aligned
    assert L.moe_debug_pdl_copy(None, a, ctypes.c_void_p(0x20004), 16) == bad  # dst not 16-byte aligned
    assert L.moe_debug_pdl_copy(None, a, b, 24) == bad                         # not a multiple of 16
    assert L.moe_debug_pdl_copy(None, a, b, -16) == bad
    assert L.moe_debug_pdl_copy(None, a, ctypes.c_void_p(0x10010), 64) == bad  # ranges overlap
    assert L.moe_debug_pdl_copy(None, a, b, 0) == rel.MOE_OK


def test_profile_stage_names(L):
    n = L.moe_profile_stages()
    names = [L.moe_profile_stage_name(i).decode() for i in range(n)]
    assert names[:3] == ["router", "select", "permute"] and "combine" in names
    assert L.moe_profile_stage_name(n) == b""


def test_binding_checks_token_arrays():
    """The binding checks shapes before it hands plain pointers to the library."""
    import numpy as np
    import torch
    import routed_expert_layer_gb300 as rel
    assert rel._rows(torch.zeros(3, 256, dtype=torch.int16), 256, "x", False) == 3
    assert rel._rows(np.zeros((0, 256), dtype=np.uint16), 256, "x", False) == 0
    bad = [(torch.zeros(3, 128, dtype=torch.int16), False),          # wrong H
           (torch.zeros(3, 256, dtype=torch.float32), False),        # 4-byte elements
           (torch.zeros(256, 3, dtype=torch.int16).t(), False),      # not contiguous
           (torch.zeros(3, 256, dtype=torch.int16), True),           # host tensor where CUDA is needed
           (np.zeros((3, 256), dtype=np.uint16), True),              # numpy where CUDA is needed
           (np.zeros((3, 256), dtype=np.float32), False),
           (torch.zeros(768, dtype=torch.int16), False)]             # not 2-D
    for t, cuda in bad:
        with pytest.raises(ValueError):
            rel._rows(t, 256, "x", cuda)


def test_binding_checks_layer_shapes():
    """load() rejects weight arrays whose shapes do not match the context's config before
    the library reads them (checked on a stand-in object, no device needed)."""
    import dataclasses
    import numpy as np
    import synth
    import routed_expert_layer_gb300 as rel
    L = synth.layer(256, 128, 32, seed_weights=1, seed_router=2)

    class Stub(rel.MoeLayer):  # skips moe_create: only the host-side checks run
        def __init__(self):
            self.cfg = rel.Config(256, 128, 32, 4, 8, 0)
            self.ctx = None

    for name in ("gu_codes", "dn_scales", "router_w"):
        bad = dataclasses.replace(L, **{name: np.zeros((1, 2), dtype=getattr(L, name).dtype)})
        with pytest.raises(ValueError):
            Stub().load(bad)
    with pytest.raises(ValueError):
        Stub().load(dataclasses.replace(L, router_bias=np.zeros(31, dtype=np.float32)))


def test_header_is_plain_c(tmp_path):
    """include/moe_gb300.h is a C header: a C99 translation unit that takes the address
    of every declared entry point compiles without warnings (and so does C++)."""
    import re
    import shutil
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    inc = os.path.join(root, "include")
    text = open(os.path.join(inc, "moe_gb300.h")).read()
    names = re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)
    assert len(names) >= 18
    src = tmp_path / "abi.c"
    src.write_text('#include "moe_gb300.h"\n'
                   "typedef void (*fn)(void);\n"
                   "fn entry_points[] = {" + ", ".join(f"(fn){n}" for n in names) + "};\n")
    for cc, std in (("gcc", "-std=c99"), ("g++", "-std=c++17")):
        exe = shutil.which(cc)
        if exe is None:
            pytest.skip(f"{cc} not found")
        lang = ["-x", "c++"] if cc == "g++" else []
        r = subprocess.run([exe, *lang, std, "-Wall", "-Wextra", "-Werror", "-I", inc, "-c", str(src), "-o",
                            str(tmp_path / f"abi_{cc}.o")], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_binding_checks_noalloc_arguments():
    """route_noalloc checks every tensor's dtype, shape and contiguity (and that it is a
    CUDA tensor) before it hands plain pointers to moe_route_noalloc; each check raises on
    host tensors here, before any CUDA call."""
    import torch
    import routed_expert_layer_gb300 as rel
    T, H, E, k = 4, 128, 16, 2

    def args(**kw):
        a = dict(x=torch.zeros(T, H, dtype=torch.int16), router_w=torch.zeros(H, E, dtype=torch.float32),
                 router_bias=None, k=k, idx=torch.zeros(T, k, dtype=torch.int32),
                 w=torch.zeros(T, k, dtype=torch.float32), offsets=torch.zeros(E + 1, dtype=torch.int32),
                 perm=torch.zeros(T * k, dtype=torch.int32), slot=torch.zeros(T * k, dtype=torch.int32),
                 inv=torch.zeros(T * k, dtype=torch.int32))
        a.update(kw)
        return a

    bad = [dict(x=torch.zeros(T, H, dtype=torch.float32)),                  # 4-byte x
           dict(router_w=torch.zeros(H + 64, E, dtype=torch.float32)),      # H mismatch
           dict(router_w=torch.zeros(H, E, dtype=torch.float64)),           # router dtype
           dict(router_bias=torch.zeros(E - 1, dtype=torch.float32)),       # bias size
           dict(idx=torch.zeros(T, k + 1, dtype=torch.int32)),              # idx shape
           dict(w=torch.zeros(T, k, dtype=torch.float16)),                  # w dtype
           dict(offsets=torch.zeros(E, dtype=torch.int32)),                 # offsets size
           dict(perm=torch.zeros(T * k - 1, dtype=torch.int32)),            # perm size
           dict(slot=torch.zeros(T * k, dtype=torch.int64)),                # slot dtype
           dict(inv=torch.zeros(2 * T * k, dtype=torch.int32)[::2]),        # not contiguous
           dict(err=torch.zeros(2, dtype=torch.int32)),                     # err not one word
           {}]                                                              # host tensors
    for kw in bad:
        with pytest.raises(ValueError):
            rel.route_noalloc(**args(**kw))


def test_plan_of_an_expert_range():
    """A context holding a quarter of the experts plans for its own experts: fewer row
    chunks, as many K splits or more (fewer touched experts must still fill the GPU), the
    same variant choice (rows per expert follow the layer's routing rate, not the range's
    size)."""
    full = rel.plan(7168, 1536, 896, 16, 512, 152, 53)
    cfg = rel.Config(7168, 1536, 896, 16, 512, 0, 224, 224)
    out = (ctypes.c_int64 * len(rel.PLAN_FIELDS))()
    assert rel.lib().moe_plan(ctypes.byref(cfg), 152, 53, out) == rel.MOE_OK
    part = {k: int(v) for k, v in zip(rel.PLAN_FIELDS, out)}
    assert part["prefill"] == full["prefill"] and part["rows_per_item"] == full["rows_per_item"]
    assert part["chunk_capacity"] < full["chunk_capacity"]
    assert part["gateup_splits"] >= full["gateup_splits"] and part["down_splits"] >= full["down_splits"]

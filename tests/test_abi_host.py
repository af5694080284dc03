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


def test_profile_stage_names(L):
    n = L.moe_profile_stages()
    names = [L.moe_profile_stage_name(i).decode() for i in range(n)]
    assert names[:3] == ["router", "select", "permute"] and "combine" in names
    assert L.moe_profile_stage_name(n) == b""

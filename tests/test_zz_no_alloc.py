"""The allocation-free routing entry point against the regular one.

moe_route_noalloc serves callers that may not allocate device memory (engines that
reserve their HBM budget at start-up, plugin hosts, decode loops that cannot take
the synchronisation an allocation may cause): its scratch is a fixed array inside
the library. Here it is called through the C ABI twice in a row on different
batches (the second call finds the first call's leftovers in the shared scratch),
and each result must match moe_debug_route on the same inputs: indices and the
permutation bit-exact, gate weights within the tests' weight tolerance. This file
is collected last so a failure here comes after every other test has run.
"""
import numpy as np
import pytest

import synth
from helpers import SHAPES, layer

pytestmark = pytest.mark.gpu


def outputs(T, E, k):
    import torch
    return dict(idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
                w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
                offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
                perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
                slot=torch.empty(T * k, dtype=torch.int32, device="cuda"),
                inv=torch.empty(T * k, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("name,zipf", [("mid", False), ("mid", True)])
def test_noalloc_route_matches_regular_route(name, zipf):
    import torch
    import routed_expert_layer_gb300 as rel
    s = SHAPES[name]
    H, E, k = s["H"], s["E"], s["k"]
    L = layer(name, zipf)
    moe = rel.MoeLayer(H, s["I"], E, k, 256)
    try:
        moe.load(L)
        rw = torch.from_numpy(L.router_w).cuda()
        rb = None if L.router_bias is None else torch.from_numpy(L.router_bias).cuda()
        for call, T in enumerate((256, 37)):  # two calls in a row, the second smaller
            x = torch.from_numpy(synth.x_bf16(4000 + T + call, T, H).view(np.int16)).cuda()
            ref = outputs(T, E, k)
            moe.debug_route(x, **ref)
            got = outputs(T, E, k)
            rel.route_noalloc(x, rw, rb, k, **got)
            torch.cuda.synchronize()
            for key in ("idx", "offsets", "perm", "slot", "inv"):
                assert torch.equal(got[key], ref[key]), (call, key)
            assert torch.allclose(got["w"], ref["w"], rtol=2e-6, atol=1e-7), call
    finally:
        moe.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import routed_expert_layer_gb300 as rel
    H, E, k = 512, 64, 8
    rw = torch.zeros(H, E, dtype=torch.float32, device="cuda")
    x = torch.zeros(257, H, dtype=torch.int16, device="cuda")
    out = outputs(257, E, k)
    with pytest.raises(rel.MoeError) as ei:
        rel.route_noalloc(x, rw, None, k, **out)
    assert ei.value.status == rel.MOE_ERR_UNSUPPORTED
    rw_big = torch.zeros(H, 1025, dtype=torch.float32, device="cuda")
    out = outputs(4, 1025, k)
    with pytest.raises(rel.MoeError) as ei:
        rel.route_noalloc(x[:4], rw_big, None, k, **out)
    assert ei.value.status == rel.MOE_ERR_UNSUPPORTED

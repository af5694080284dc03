"""The allocation-free routing entry point, through the C ABI.

moe_route_noalloc serves callers that may not allocate device memory (engines that
reserve their HBM budget at start-up, plugin hosts that only hand out planned buffers,
decode loops that cannot take the synchronisation an allocation may cause): its
scratch is a fixed array inside the library. It is called twice in a row on different
batches (the second call finds the first call's leftovers in the shared scratch), and
each result is checked

  - against the oracle: the expert sets equal except on tokens whose fp64 logits have
    a gap at the k / k+1 boundary within twice the logit bound (rounding of fp32 logits
    may swap those), the order equal elsewhere, gate weights within the fp32 logit
    error, and offsets / perm / slot / inv bit-exact against the oracle's permutation of
    the returned expert ids;
  - against the regular routing entry point (moe_debug_route, whose tensor-core router
    rounds differently in the last bits) under the same near-tie rule;
  - with its device error word read back as zero.

This file is collected last so that a failure here comes after every other test.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import LOGIT_REL, SHAPES, layer, near_tie_tokens

pytestmark = pytest.mark.gpu


def outputs(T, E, k):
    import torch
    return dict(idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
                w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
                offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
                perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
                slot=torch.empty(T * k, dtype=torch.int32, device="cuda"),
                inv=torch.empty(T * k, dtype=torch.int32, device="cuda"))


def check_against(got, ref_idx, ref_w, ties, E, what):
    """Expert ids and weights of `got` against a reference routing; the permutation
    bit-exact against the oracle's permutation of got's own ids."""
    idx = got["idx"]
    same = np.all(np.sort(idx, axis=1) == np.sort(ref_idx, axis=1), axis=1)
    assert not (~same & ~ties).any(), f"{what}: routing differs on tokens {np.nonzero(~same & ~ties)[0][:10]}"
    ok = same & ~ties
    assert np.array_equal(idx[ok], ref_idx[ok]), what
    if ref_w is not None:
        assert np.allclose(got["w"][ok], ref_w[ok], rtol=0, atol=1e-3), what
    counts, offs, perm, slot, inv = oracle.permute(idx, E)
    for key, ref in (("offsets", offs), ("perm", perm), ("slot", slot), ("inv", inv)):
        assert np.array_equal(got[key], ref), (what, key)


@pytest.mark.parametrize("name,zipf", [("mid", False), ("mid", True)])
def test_noalloc_route_matches_oracle_and_regular_route(name, zipf):
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
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for call, T in enumerate((256, 37)):  # two calls in a row, the second smaller
            xb = synth.x_bf16(4000 + T + call, T, H)
            x = torch.from_numpy(xb.view(np.int16)).cuda()
            got = outputs(T, E, k)
            rel.route_noalloc(x, rw, rb, k, **got, err=err)
            reg = outputs(T, E, k)
            moe.debug_route(x, **reg)
            torch.cuda.synchronize()
            got = {key: v.cpu().numpy() for key, v in got.items()}
            reg = {key: v.cpu().numpy() for key, v in reg.items()}
            ref_logits = oracle.router_logits(xb, L.router_w, L.router_bias)
            ref_idx, ref_w = oracle.select(ref_logits, k)
            bound = LOGIT_REL * oracle.router_abs(xb, L.router_w)
            ties = near_tie_tokens(ref_logits, k, 2.0 * float(bound.max()))
            check_against(got, ref_idx, ref_w, ties, E, f"call {call} vs oracle")
            check_against(got, reg["idx"], reg["w"], ties, E, f"call {call} vs regular route")
            assert int(err.item()) == 0
            print(f"noalloc call {call} T={T}: near-tie tokens {int(ties.sum())}")
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

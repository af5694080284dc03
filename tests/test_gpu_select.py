"""S2 + S3 on the GPU, bit-exact against the oracle given the same logits.

The logits come from the seeded generator (not from the GPU router), with planted
ties, -0/+0 pairs and runs of equal values longer than k, so both sides decide on
identical fp32 values.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

CASES = [  # (E, k, T)
    (32, 4, 1), (32, 4, 4), (32, 4, 37),
    (64, 8, 300),
    (896, 16, 1), (896, 16, 53), (896, 16, 64), (896, 16, 257), (896, 16, 4099), (896, 16, 8192),
    (1024, 32, 33),
]


def planted(T, E, seed):
    l = synth.logits(seed, T, E)
    l[0, :] = 0.0
    l[0, 3] = -0.0
    if T > 1:
        l[1, 5] = l[1, 9] = l[1, E - 1] = 7.0
        l[1, 10] = -0.0
        l[1, 11] = 0.0
    if T > 2:
        l[2, ::2] = 1.25
    if T > 3:
        l[3, :] = -3.0
        l[3, E // 2:] = -3.0000002  # a second plateau one ulp-ish lower
    if T > 5:
        l[5:T:7, 1] = l[5:T:7, 2]  # equal pairs in many rows
    return np.ascontiguousarray(l, dtype=np.float32)


@pytest.fixture(scope="module")
def ctxs():
    import routed_expert_layer_gb300 as rel
    out = {}
    for E, k, T in CASES:
        key = (E, k)
        Tm = max(t for e_, k_, t in CASES if (e_, k_) == key)
        if key not in out:
            out[key] = rel.MoeLayer(256, 128, E, k, Tm)
    yield out
    for m in out.values():
        m.close()


@pytest.mark.parametrize("E,k,T", CASES)
def test_select_and_permute_bit_exact(ctxs, E, k, T):
    import torch
    moe = ctxs[(E, k)]
    l = planted(T, E, 1000 + T + E)
    ref_idx, ref_w = oracle.select(l, k)
    counts, offsets, perm, slot, inv = oracle.permute(ref_idx, E)
    dev = dict(idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               slot=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               inv=torch.empty(T * k, dtype=torch.int32, device="cuda"))
    moe.debug_select(torch.from_numpy(l).cuda(), **dev)
    torch.cuda.synchronize()
    got = {n: v.cpu().numpy() for n, v in dev.items()}
    assert np.array_equal(got["idx"], ref_idx)
    assert np.array_equal(got["offsets"], offsets)
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["slot"], slot)
    assert np.array_equal(got["inv"], inv)
    assert np.allclose(got["w"], ref_w, rtol=2e-6, atol=1e-7)
    assert moe.get_error() == 0


def test_select_is_deterministic(ctxs):
    import torch
    moe = ctxs[(896, 16)]
    l = torch.from_numpy(planted(4099, 896, 7)).cuda()
    a = torch.empty(4099 * 16, dtype=torch.int32, device="cuda")
    b = torch.empty_like(a)
    moe.debug_select(l, perm=a)
    moe.debug_select(l, perm=b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("H,I,E,k,T", [(256, 128, 32, 4, 1), (256, 128, 32, 4, 32), (512, 256, 64, 8, 7),
                                       (256, 128, 896, 16, 1), (256, 128, 896, 16, 8), (256, 128, 896, 16, 32),
                                       (256, 128, 1024, 32, 17), (256, 128, 896, 16, 33)])
def test_small_batch_route_matches_general_path(H, I, E, k, T):
    """Batches of at most 32 tokens are routed by one fused kernel (reduce, select and
    permute in one CTA). Given the logits it produced, the general select and permute
    kernels must give bit-identical results; T = 33 takes the general path on both sides."""
    import torch
    import routed_expert_layer_gb300 as rel
    moe = rel.MoeLayer(H, I, E, k, 64)
    try:
        moe.load(synth.layer(H, I, E, seed_weights=11, seed_router=12))
        x = torch.from_numpy(synth.x_bf16(900 + T, T, H).view(np.int16)).cuda()
        names = ("idx", "w", "offsets", "perm", "slot", "inv")
        shapes = dict(idx=((T, k), torch.int32), w=((T, k), torch.float32), offsets=((E + 1,), torch.int32),
                      perm=((T * k,), torch.int32), slot=((T * k,), torch.int32), inv=((T * k,), torch.int32))
        a = {n: torch.empty(*shapes[n][0], dtype=shapes[n][1], device="cuda") for n in names}
        b = {n: torch.empty(*shapes[n][0], dtype=shapes[n][1], device="cuda") for n in names}
        logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
        moe.debug_route(x, logits=logits, **a)
        moe.debug_select(logits, **b)
        torch.cuda.synchronize()
        for n in names:
            assert torch.equal(a[n], b[n]), n
        ref_idx, _ = oracle.select(logits.cpu().numpy(), k)
        assert np.array_equal(a["idx"].cpu().numpy(), ref_idx)
        assert moe.get_error() == 0
    finally:
        moe.close()

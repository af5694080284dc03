"""Expert ranges and caller-given routing on the GPU, through the C ABI, against the
oracle ("Kimi-K3 NVFP4 station eight sparks", section "What has to be built": the split
of one model's experts across workers is a mask on the router's chosen ids, a worker
takes each token's 16 global expert ids with -1 for a masked one and returns rows plus
the ids it served).

  - A context holding experts [e0, e0 + n) routes over all experts and returns the part
    of the layer's output its experts contribute: compared with the oracle's routed step
    on that range, and the partial outputs of contexts partitioning the experts add up
    to the layer.
  - moe_forward_routed takes the routing from the caller: masked (-1) and other workers'
    ids are skipped, `served` reports the routes computed; an id outside [-1, E) and a
    token listing one expert twice raise their error bits.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from helpers import (SHAPES, bf16_bits_to_f64, bf16_half_ulp, check_output, check_routing, gpu_forward, gpu_route,
                     layer)

pytestmark = pytest.mark.gpu

MID = SHAPES["mid"]  # H=512, I=256, E=64, k=8
EXPERT_ARRAYS = ("gu_codes", "gu_scales", "gu_global", "dn_codes", "dn_scales", "dn_global")


def expert_slice(L, e0, n):
    return dataclasses.replace(L, E=n, **{a: getattr(L, a)[e0:e0 + n] for a in EXPERT_ARRAYS})


def make(s, L, max_tokens, e0=0, n=0):
    import routed_expert_layer_gb300 as rel
    m = rel.MoeLayer(s["H"], s["I"], s["E"], s["k"], max_tokens, expert_begin=e0, expert_count=n)
    m.load(L)
    return m


RANGES = ((0, 24), (24, 1), (25, 39))  # a partition of the 64 experts, one of them a single expert


@pytest.fixture(scope="module")
def mid_ranges():
    L = layer("mid")
    ms = [make(MID, L, 512, e0, n) for e0, n in RANGES]
    yield ms
    for m in ms:
        m.close()


@pytest.mark.parametrize("T", [9, 20, 300])
def test_expert_ranges_partition_the_layer(mid_ranges, T):
    """Decode (T=9), the fused small-batch routing (T=20) and prefill (T=300): each
    context's partial output against the oracle's routed step on its range, and the sum
    of the partials against the whole layer."""
    L = layer("mid")
    k, E = MID["k"], MID["E"]
    x = synth.x_bf16(1300 + T, T, MID["H"])
    ref, ref_idx, ref_w, ref_logits = oracle.moe_forward(oracle.Layer(L), x, k)
    ref_abs = oracle.router_abs(x, L.router_w)
    total = np.zeros_like(ref)
    slack = np.zeros_like(ref)
    ties = np.zeros(T, dtype=bool)
    for (e0, n), m in zip(RANGES, mid_ranges):
        r = gpu_route(m, x, E, k)
        ties |= check_routing(r["logits"], r["idx"], ref_logits, ref_abs, ref_idx, k)
        # rows served here (a range context fills offsets[0..n] only)
        assert r["offsets"][n] == int(((r["idx"] >= e0) & (r["idx"] < e0 + n)).sum())
        out = gpu_forward(m, x)
        part, _ = oracle.moe_routed(oracle.Layer(expert_slice(L, e0, n)), x, ref_idx, ref_w, e0)
        rms_full = float(np.sqrt(np.mean(ref[~ties] ** 2)))
        err = np.max(np.maximum(np.abs(out - part) - bf16_half_ulp(out), 0.0)[~ties]) if (~ties).any() else 0.0
        assert err <= 2e-2 * rms_full, (e0, n, err / rms_full)
        assert m.get_error() == 0
        total += out
        slack += bf16_half_ulp(out)
    err = np.max(np.maximum(np.abs(total - ref) - slack, 0.0)[~ties])
    assert err <= 2e-2 * float(np.sqrt(np.mean(ref[~ties] ** 2)))


def random_routing(T, k, E, seed, masked=0.25):
    """Distinct expert ids per token, a fraction of them masked with -1, positive weights."""
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[rng.random((T, k)) < masked] = -1
    w = rng.random((T, k)).astype(np.float32) + 0.05
    return idx, w


def run_routed(m, L_local, e0, x_bits, idx, w):
    import torch
    xd = torch.from_numpy(x_bits.view(np.int16)).cuda()
    out = torch.empty_like(xd)
    served = torch.empty(idx.shape, dtype=torch.int32, device="cuda")
    m.forward_routed(xd, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), out, served)
    torch.cuda.synchronize()
    got = bf16_bits_to_f64(out.cpu().numpy().view(np.uint16))
    ref, ref_served = oracle.moe_routed(oracle.Layer(L_local), x_bits, idx, w.astype(np.float64), e0)
    return got, ref, served.cpu().numpy(), ref_served


@pytest.mark.parametrize("T", [5, 37, 300])
@pytest.mark.parametrize("e0,n", [(0, 0), (10, 30)])
def test_forward_routed_vs_oracle(T, e0, n):
    """Caller-given routing (a quarter of the ids masked, the rest random distinct experts,
    random positive weights) on the whole layer and on the range [10, 40)."""
    L = layer("mid")
    m = make(MID, L, 512, e0, n)
    try:
        idx, w = random_routing(T, MID["k"], MID["E"], 1400 + T)
        x = synth.x_bf16(1500 + T, T, MID["H"])
        Ll = expert_slice(L, e0, n) if n else L
        got, ref, served, ref_served = run_routed(m, Ll, e0, x, idx, w)
        assert np.array_equal(served, ref_served)
        check_output(got, ref)
        assert m.get_error() == 0
    finally:
        m.close()


def test_forward_routed_all_masked_gives_zeros():
    L = layer("mid")
    m = make(MID, L, 64)
    try:
        T, k = 16, MID["k"]
        idx = np.full((T, k), -1, dtype=np.int32)
        w = np.ones((T, k), dtype=np.float32)
        got, ref, served, _ = run_routed(m, L, 0, synth.x_bf16(1600, T, MID["H"]), idx, w)
        assert np.all(got == 0.0) and np.all(served == -1)
        assert m.get_error() == 0
    finally:
        m.close()


def test_forward_routed_bad_id_and_duplicate_raise_error_bits():
    """An id outside [-1, E) is skipped and raises bit 1; the other tokens stay exact. A
    token listing one expert twice raises bit 16."""
    L = layer("mid")
    m = make(MID, L, 64)
    try:
        T, k, E = 12, MID["k"], MID["E"]
        idx, w = random_routing(T, k, E, 1700)
        idx[3, 2] = E + 5
        x = synth.x_bf16(1701, T, MID["H"])
        got, ref, served, ref_served = run_routed(m, L, 0, x, idx, w)
        assert served[3, 2] == -1 and np.array_equal(served, ref_served)
        check_output(got, ref)
        assert m.get_error() & 1
        idx2, w2 = random_routing(T, k, E, 1702, masked=0.0)
        idx2[5, 1] = idx2[5, 0]
        run_routed(m, L, 0, x, idx2, w2)
        assert m.get_error() & 16
        assert m.get_error() == 0
    finally:
        m.close()


K3 = SHAPES["k3"]


@pytest.fixture(scope="module")
def k3_half():
    m = make(K3, layer("k3"), 4096, 448, 448)
    yield m
    m.close()


@pytest.mark.parametrize("T", [53, 4096])
def test_k3_expert_range(k3_half, T):
    """The K3 layer's upper half of the experts (448..895) on one context: sampled rows of
    its partial output against the oracle's routed step on that range."""
    L = layer("k3")
    x = synth.x_bf16(1800 + T, T, K3["H"])
    out = gpu_forward(k3_half, x)
    r = gpu_route(k3_half, x, K3["E"], K3["k"])
    rows = np.unique(np.concatenate([np.arange(0, T, max(1, T // 24)), [T - 1]]))[:32]
    _, ref_idx, ref_w, ref_logits = oracle.moe_tokens(oracle.Layer(L), x[rows], K3["k"])
    ties = check_routing(r["logits"][rows], r["idx"][rows], ref_logits, oracle.router_abs(x[rows], L.router_w),
                         ref_idx, K3["k"])
    part, _ = oracle.moe_routed(oracle.Layer(expert_slice(L, 448, 448)), x[rows], ref_idx, ref_w, 448)
    check_output(out[rows], part, ~ties)
    assert k3_half.get_error() == 0
    assert r["offsets"][448] == int((r["idx"] >= 448).sum())  # offsets[0..448] of the range

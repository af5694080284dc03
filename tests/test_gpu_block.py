"""A LatentMoE block on the GPU, through the C ABI, against the oracle's block step.

"Kimi K3 optimization on GB300, Part I", sections "Routed-down projection" and
"Routed-up projection": the block projects the hidden state (7,168) into the routed
latent (3,584) with a bf16 weight and back after the routed experts; "Serving Kimi K3
End to End", section 3.3: 2 shared experts that every token uses, unquantized. The GPU
computes the routed-down projection together with the shared experts' gate/up (one
tensor-core GEMM), the routed experts in the latent, and the routed-up projection
together with the shared experts' down projection (one GEMM whose fp32 accumulator sums
the two); the oracle follows the block token by token in fp64.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import bf16_bits_to_f64, bf16_half_ulp, check_output, check_routing, gpu_forward, gpu_route

pytestmark = pytest.mark.gpu

MIDB = dict(H=512, d=256, I=256, E=64, k=8)


def make(s, Is, max_tokens):
    import routed_expert_layer_gb300 as rel
    L = synth.block_layer(s["H"], s["d"], s["I"], s["E"], Is, seed_weights=11, seed_router=12)
    m = rel.MoeLayer(s["H"], s["I"], s["E"], s["k"], max_tokens, latent=s["d"], shared_inter=Is)
    m.load(L)
    return m, L


@pytest.fixture(scope="module", params=[0, 256], ids=["latent", "latent+shared"])
def midb(request):
    m, L = make(MIDB, request.param, 512)
    yield m, L
    m.close()


def run_block(m, L, s, rows_x, rows=None):
    x = rows_x
    out = gpu_forward(m, x)
    r = gpu_route(m, x, s["E"], s["k"])
    sel = np.arange(x.shape[0]) if rows is None else rows
    ref, ref_idx, ref_w, ref_logits = oracle.moe_block(oracle.Layer(L), x[sel], s["k"])
    ties = check_routing(r["logits"][sel], r["idx"][sel], ref_logits, oracle.router_abs(x[sel], L.router_w), ref_idx,
                         s["k"])
    ratio = check_output(out[sel], ref, ~ties)
    assert m.get_error() == 0
    return ratio


@pytest.mark.parametrize("T", [1, 9, 37, 300, 512])
def test_mid_block(midb, T):
    """Decode, the fused small-batch routing and prefill sizes, with and without shared
    experts."""
    m, L = midb
    run_block(m, L, MIDB, synth.x_bf16(2100 + T, T, MIDB["H"]))


def test_block_latent_is_the_routed_down_projection(midb):
    """The latent the experts read is bf16(x W_down^T): within the rounding of bf16 plus
    the fp32 accumulation over K = hidden."""
    import torch
    m, L = midb
    T = 40
    x = synth.x_bf16(2200, T, MIDB["H"])
    lat = torch.empty(T, MIDB["d"], dtype=torch.int16, device="cuda")
    m.debug_experts(torch.from_numpy(x.view(np.int16)).cuda(), lat=lat)
    torch.cuda.synchronize()
    got = bf16_bits_to_f64(lat.cpu().numpy().view(np.uint16))
    ref = bf16_bits_to_f64(x) @ bf16_bits_to_f64(L.proj_down).T
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= bf16_half_ulp(got) + 1e-5 * rms)


KB = dict(H=7168, d=3584, I=3072, E=896, k=16)
K3_SHARED = 6144  # two shared experts of the routed experts' intermediate width 3072


@pytest.fixture(scope="module")
def k3_block():
    m, L = make(KB, K3_SHARED, 4096)
    yield m, L
    m.close()


@pytest.mark.parametrize("T", [1, 53, 4096])
def test_k3_block(k3_block, T):
    """The K3 block (hidden 7168, latent 3584, 896 experts of 3584 x 3072, top-16, shared
    experts 6144 wide) on sampled rows."""
    m, L = k3_block
    x = synth.x_bf16(2300 + T, T, KB["H"])
    rows = np.unique(np.concatenate([np.arange(0, T, max(1, T // 24)), [T - 1]]))[:32]
    ratio = run_block(m, L, KB, x, rows)
    print(f"K3 block T={T}: rows={len(rows)} err/rms={ratio:.3e}")

"""The layer at the K3 shape (H=7168, I=1536, E=896, k=16, NVFP4 experts of
18,579,480 bytes, 16.6 GB per layer) on the GPU, in the launch configuration the
benchmark times: decode T=1, 8, 53; verify/batched decode T=64, 128, 256;
prefill T=2048, 4096, 8192; Zipf(1.1)-skewed routing at T=64 and 4096.

Sampled output rows (at least 64 per batch, among them every row of the largest
bucket's first and last row chunk and the last row of a partial chunk) are checked
against the oracle token by token (each row depends only on its own token); the
permutation of the whole batch is compared bit for bit with the oracle's permutation
of the GPU's expert ids; the selection at full size is checked bit-exactly in
test_gpu_select.py."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from helpers import SHAPES, check_output, check_routing, forward_vs_caller_routed, gpu_forward, gpu_route, layer

pytestmark = pytest.mark.gpu

K3 = SHAPES["k3"]
T_MAX = 8192


@pytest.fixture(scope="module")
def k3():
    import routed_expert_layer_gb300 as rel
    m = rel.MoeLayer(K3["H"], K3["I"], K3["E"], K3["k"], T_MAX)
    m.load(layer("k3"))
    yield m
    m.close()


@pytest.fixture(scope="module")
def k3_zipf():
    import routed_expert_layer_gb300 as rel
    m = rel.MoeLayer(K3["H"], K3["I"], K3["E"], K3["k"], 4096)
    m.load(layer("k3", zipf=True))
    yield m
    m.close()


def rows_per_item(s, T):
    import torch
    import routed_expert_layer_gb300 as rel
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    return rel.plan(s["H"], s["I"], s["E"], s["k"], T, sm, T)["rows_per_item"]


def sample_rows(r, T, nmax, n=64, per_chunk=24, seed=0):
    """Every token if T <= n; else the first, middle and last tokens, the tokens of the
    largest bucket's first and last row chunk (all of them for chunks of at most
    per_chunk rows, else per_chunk spread over the chunk), the last row of the last
    expert whose bucket ends in a partial chunk, and random tokens up to n."""
    if T <= n:
        return np.arange(T)
    offs, perm = r["offsets"], r["perm"]
    counts = np.diff(offs)
    e = int(np.argmax(counts))
    c = int(counts[e])
    first = perm[offs[e]:offs[e] + min(nmax, c)]
    last = perm[offs[e] + ((c - 1) // nmax) * nmax:offs[e + 1]]
    rows = {0, T // 2, T - 1}
    for ch in (first, last):
        pick = ch if len(ch) <= per_chunk else ch[np.linspace(0, len(ch) - 1, per_chunk).astype(int)]
        rows |= set(int(v) for v in pick)
    partial = np.nonzero(counts % nmax != 0)[0]
    if len(partial):
        rows.add(int(perm[offs[partial[-1] + 1] - 1]))
    rng = np.random.default_rng(seed + T)
    while len(rows) < n:
        rows.add(int(rng.integers(0, T)))
    return np.array(sorted(rows))


def check_permutation_exact(r, E):
    """The GPU's offsets, perm, slot and inv equal the oracle's permutation of the GPU's
    own expert ids, bit for bit, over the whole batch."""
    counts, offs, perm, slot, inv = oracle.permute(r["idx"], E)
    for key, ref in (("offsets", offs), ("perm", perm), ("slot", slot), ("inv", inv)):
        assert np.array_equal(r[key], ref), key


def scaled_bits(x_bits, a):
    """bf16 bits of x * 2^a (exact for a power of two away from the format's limits)."""
    f = synth.bf16_bits_to_f32(x_bits) * np.float32(2.0 ** a)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def run_k3(moe, T, zipf=False, name="k3", L=None, x_scale=0):
    s = SHAPES[name]
    L = layer(name, zipf) if L is None else L
    x = synth.x_bf16(3 + T, T, s["H"])
    if x_scale:
        x = scaled_bits(x, x_scale)
    out = gpu_forward(moe, x)
    r = gpu_route(moe, x, s["E"], s["k"])
    check_permutation_exact(r, s["E"])
    rows = sample_rows(r, T, rows_per_item(s, T))
    ref, ref_idx, ref_w, ref_logits = oracle.moe_tokens(oracle.Layer(L), x[rows], s["k"])
    ref_abs = oracle.router_abs(x[rows], L.router_w)
    ties = check_routing(r["logits"][rows], r["idx"][rows], ref_logits, ref_abs, ref_idx, s["k"])
    ratio = check_output(out[rows], ref, ~ties)
    raw = float(np.max(np.abs(out[rows][~ties] - ref[~ties])) / np.sqrt(np.mean(ref[~ties] ** 2)))
    assert moe.get_error() == 0
    counts = np.diff(r["offsets"])
    if zipf and T >= 2048:  # both GEMMs run: experts of at most 16 rows on the decode one
        assert ((counts > 0) & (counts <= 16)).any() and (counts > 16).any()
    print(f"{name.upper()} T={T} zipf={zipf} x_scale={x_scale}: touched={int((counts > 0).sum())} "
          f"max_rows={int(counts.max())} rows_checked={len(rows)} err/rms={ratio:.3e} (with bf16 output rounding "
          f"{raw:.3e}) near_ties={int(ties.sum())}")


@pytest.mark.parametrize("T", [1, 8, 53, 64, 128, 256, 2048, 4096, 8192])
def test_k3_uniform(k3, T):
    run_k3(k3, T)


@pytest.mark.parametrize("T", [64, 4096])
def test_k3_zipf(k3_zipf, T):
    run_k3(k3_zipf, T, zipf=True)


@pytest.mark.parametrize("T", [53, 4096])
@pytest.mark.parametrize("xa", [-8, 8])
def test_k3_scaled_x(k3, T, xa):
    """x scaled by 2^-8 and 2^8 at the decode and prefill sizes."""
    run_k3(k3, T, x_scale=xa)


def k3_scaled_layer():
    base = layer("k3")
    return dataclasses.replace(base, gu_global=(base.gu_global * np.float32(64.0)).astype(np.float32),
                               dn_global=(base.dn_global * np.float32(1 / 64.0)).astype(np.float32))


@pytest.fixture(scope="module")
def k3_scaled():
    import routed_expert_layer_gb300 as rel
    m = rel.MoeLayer(K3["H"], K3["I"], K3["E"], K3["k"], 4096)
    m.load(k3_scaled_layer())
    yield m
    m.close()


@pytest.mark.parametrize("T", [53, 4096])
def test_k3_scaled_tensor_scales(k3_scaled, T):
    """Gate/up tensor scales x 2^6 and down tensor scales x 2^-6."""
    run_k3(k3_scaled, T, L=k3_scaled_layer())


@pytest.fixture(scope="module")
def latent():
    import routed_expert_layer_gb300 as rel
    s = SHAPES["latent"]
    m = rel.MoeLayer(s["H"], s["I"], s["E"], s["k"], 4096)
    m.load(layer("latent"))
    yield m
    m.close()


@pytest.mark.parametrize("T", [1, 53, 4096])
def test_latent_expert_shape(latent, T):
    """The pages' own expert geometry (d = 3584, f = 3072, 896 experts, top-16): the same
    kernels, shape-parametric, decode and prefill."""
    run_k3(latent, T, name="latent")


@pytest.mark.parametrize("T", [1, 16, 53])
def test_k3_forward_matches_caller_routed_expert_stage(k3, T):
    """K3 forwards (K-split gate/up at T = 1, fused routing at T <= 32) against the expert
    stage on the same routing through moe_forward_routed: bit for bit."""
    a, b = forward_vs_caller_routed(k3, synth.x_bf16(2200 + T, T, K3["H"]), K3["H"], K3["k"])
    assert np.array_equal(a, b)
    assert k3.get_error() == 0

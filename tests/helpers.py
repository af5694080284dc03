"""Helpers shared by the GPU parity tests (imported by test modules, not a test)."""
from __future__ import annotations

import dataclasses
import functools

import numpy as np

import synth

# Output tolerance: max |out_gpu - out_ref| <= TOL_RMS * RMS(out_ref) over the rows compared.
TOL_RMS = 2e-2
# GPU fp32 logits must be within this multiple of sum_h |x_h W_r[h,e]| of the fp64 logits.
LOGIT_REL = 2.0 ** -16

SHAPES = {
    "tiny": dict(H=256, I=128, E=32, k=4),
    "mid": dict(H=512, I=256, E=64, k=8),
    "k3": dict(H=7168, I=1536, E=896, k=16),
    # degenerate routings: one expert (the layer is one SwiGLU MLP) and k = E = 32 (every
    # token uses every expert: a dense softmax mixture); the widest supported row, H = 14336
    "single": dict(H=256, I=128, E=1, k=1),
    "dense": dict(H=256, I=128, E=32, k=32),
    "wide": dict(H=14336, I=256, E=16, k=4),
    # the pages' own expert geometry (latent experts d = 3584, f = 3072; same bytes per expert)
    "latent": dict(H=3584, I=3072, E=896, k=16),
}


@functools.lru_cache(maxsize=None)
def layer(name: str, zipf: bool = False):
    """Synthetic layer of a named shape (weights seed 1, router seed 2); the Zipf
    variant shares the experts and adds the router bias (permutation seed 4)."""
    s = SHAPES[name]
    if zipf:
        return dataclasses.replace(layer(name, False), router_bias=synth.zipf_bias(4, s["E"], 1.1))
    return synth.layer(s["H"], s["I"], s["E"], seed_weights=1, seed_router=2)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def gpu_forward(moe, x_bits: np.ndarray) -> np.ndarray:
    """Run the C-ABI forward on device copies of x; returns out as float64 [T][H]."""
    import torch
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    out = torch.empty_like(x)
    moe.forward(x, out)
    torch.cuda.synchronize()
    return bf16_bits_to_f64(out.cpu().numpy().view(np.uint16))


def gpu_route(moe, x_bits: np.ndarray, E: int, k: int):
    import torch
    T = x_bits.shape[0]
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    dev = dict(logits=torch.empty(T, E, dtype=torch.float32, device="cuda"),
               idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               slot=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               inv=torch.empty(T * k, dtype=torch.int32, device="cuda"))
    moe.debug_route(x, **dev)
    torch.cuda.synchronize()
    return {k_: v.cpu().numpy() for k_, v in dev.items()}


def near_tie_tokens(ref_logits: np.ndarray, k: int, delta: float) -> np.ndarray:
    """Tokens whose fp64 logits have a gap smaller than delta between the k-th and
    (k+1)-th largest: rounding of fp32 logits may legitimately swap them."""
    if ref_logits.shape[1] <= k:
        return np.zeros(ref_logits.shape[0], dtype=bool)
    srt = -np.sort(-ref_logits, axis=1)
    return (srt[:, k - 1] - srt[:, k]) <= delta


def check_routing(gpu_logits, gpu_idx, ref_logits, ref_abs, ref_idx, k):
    """GPU logits within LOGIT_REL * sum|xW| of fp64; idx identical except on near ties.
    Returns the boolean mask of near-tie tokens (excluded from output comparisons)."""
    err = np.abs(gpu_logits.astype(np.float64) - ref_logits)
    assert np.all(err <= LOGIT_REL * ref_abs + 1e-30), f"logit error {err.max()} vs bound"
    print(f"logit error / sum|xW|: max {float(np.max(err / (ref_abs + 1e-300))):.3e} (bound {LOGIT_REL:.3e})")
    delta = 2.0 * float(err.max()) + 1e-12
    ties = near_tie_tokens(ref_logits, k, delta)
    same = np.all(np.sort(gpu_idx, axis=1) == np.sort(ref_idx, axis=1), axis=1)
    bad = ~same & ~ties
    assert not bad.any(), f"routing differs on tokens {np.nonzero(bad)[0][:10]} beyond rounding"
    # where the sets agree and the token is not near a tie, the order must agree too
    ok = same & ~ties
    assert np.array_equal(gpu_idx[ok], ref_idx[ok])
    return ties


def bf16_half_ulp(v):
    """Half a unit in the last place of bf16 in the binade of each |v|: the largest error
    of rounding a real number in that binade to bf16 (8 significant bits)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 8), 2.0 ** -134)


# The largest relative error of storing a value in f16 (11 significant bits): half an ulp
# at the bottom of a binade. The SwiGLU and down-projection rows are stored in f16 in
# normalised units (a factor that is not a power of two away from true units), so in true
# units only this relative bound holds, not a binade-exact one.
F16_STORE_REL = 2.0 ** -11


def check_output(out_gpu, out_ref, rows_mask=None, tol=TOL_RMS, bf16_out=True, f16_store=False):
    """max |out_gpu - out_ref| <= tol * RMS(out_ref) over the compared rows. For the layer's
    bf16 output the rounding of each element to bf16 (at most half an ulp of the stored
    value) is the output format's, not the path's, and is allowed on top: the oracle's own
    exact result rounded to bf16 would otherwise fail the bound on heavy-tailed rows (on
    Zipf-routed K3 rows it is 2.8e-2 of RMS off). f16_store allows instead the rounding of
    a value stored in f16 (F16_STORE_REL of it). Returns (max error excess) / RMS."""
    if rows_mask is not None:
        out_gpu, out_ref = out_gpu[rows_mask], out_ref[rows_mask]
    rms = float(np.sqrt(np.mean(out_ref ** 2)))
    assert np.all(np.isfinite(out_gpu))
    diff = np.abs(out_gpu - out_ref)
    if f16_store:
        diff = np.maximum(diff - F16_STORE_REL * np.abs(out_gpu), 0.0)
    elif bf16_out:
        diff = np.maximum(diff - bf16_half_ulp(out_gpu), 0.0)
    err = float(np.max(diff)) if out_ref.size else 0.0
    assert err <= tol * rms, f"max|err| {err:.4g} > {tol} * RMS {rms:.4g} (ratio {err / rms:.4g})"
    return err / rms if rms > 0 else 0.0


def forward_vs_caller_routed(m, x_bits, H, k):
    """The layer's forward, and the expert stage on the routing that forward chose given
    back through moe_forward_routed (which always gathers the routed rows): two outputs
    that must agree bit for bit, returned as uint16 arrays."""
    import torch
    T = x_bits.shape[0]
    xd = torch.from_numpy(x_bits.view(np.int16)).cuda()
    out_a = torch.empty_like(xd)
    m.forward(xd, out_a)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    m.debug_route(xd, idx=idx, w=w)
    out_b = torch.empty_like(xd)
    m.forward_routed(xd, idx, w, out_b)
    torch.cuda.synchronize()
    return out_a.cpu().numpy().view(np.uint16), out_b.cpu().numpy().view(np.uint16)

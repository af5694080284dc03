"""Pins for the oracle: each check ties it to something other than itself.

Sources of truth used here: values printed on the pages (byte census), the
hand-written format tables in ``golden/formats.json``, library routines
(torch's float8_e4m3fn and bfloat16 decoders, numpy fp64 matmul and sort),
brute force on tiny inputs, closed forms and invariants. The last group plants
plausible mistakes in numpy restatements and checks the pins would catch them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---- independent decoders (library routines + hand table) -------------------------

def e4m3_lib(b):
    return torch.tensor(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_lib(bits):
    return torch.tensor(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


E2M1_HAND = np.array([float(v) for _, v in sorted(_gold("formats.json")["e2m1"].items(), key=lambda kv: int(kv[0]))])


def dequant_lib(codes, scales, g):
    """NVFP4 -> fp64 with the hand E2M1 table and torch's E4M3 decoder."""
    lo = codes & 0xF
    hi = codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    s = np.repeat(e4m3_lib(scales), 16, axis=1)
    return E2M1_HAND[c] * s * np.float64(g)


# ---- P-A decode tables ----------------------------------------------------------------

def test_e2m1_table_hand():
    for code, v in _gold("formats.json")["e2m1"].items():
        assert oracle.e2m1(int(code)) == v


def test_e4m3_hand_values():
    for b, v in _gold("formats.json")["e4m3"].items():
        assert oracle.e4m3(int(b, 16)) == v


def test_e4m3_all_bytes_vs_torch():
    ref = e4m3_lib(np.arange(256))
    got = np.array([oracle.e4m3(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F, 0xFF
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_vs_torch():
    bits = np.array([0x0000, 0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F, 0x8000, 0x3DCD, 0xC2F7], dtype=np.uint16)
    ref = bf16_lib(bits)
    got = np.array([oracle.bf16(int(b)) for b in bits])
    assert np.array_equal(ref, got)


# ---- P-B byte census (numbers printed on the pages) --------------------------------

@pytest.mark.parametrize("H,I", [(7168, 1536), (3584, 3072)])
def test_census_expert_bytes(H, I):
    g = _gold("census.json")
    L = synth.Layer(H, I, 1, *([None] * 7))
    assert L.expert_bytes == g["expert_bytes"]


def test_census_totals():
    g = _gold("census.json")
    assert g["moe_layers"] * g["experts_per_layer"] == g["experts_total"]
    assert g["experts_total"] * g["expert_bytes"] == g["routed_expert_bytes_total"]
    assert abs(g["routed_expert_bytes_total"] / 2**30 - g["routed_expert_gib_total"]) < 0.005
    d, f = g["expert_params_shape"][1:]
    total = 3 * d * f * g["experts_total"]
    assert round(total / 1e12, 2) == 2.72
    assert round(100 * g["experts_per_token"] / g["experts_per_layer"], 1) == g["fraction_read_per_token_percent"]


# ---- dequantisation and the encoder ------------------------------------------------------

def test_dequant_vs_library_decoders():
    w = synth.normal_f32(11, 99, 64 * 256, 0.05).reshape(64, 256)
    codes, scales, g = synth.quantize_nvfp4(w)
    assert np.array_equal(oracle.dequant(codes, scales, g), dequant_lib(codes, scales, g))


def test_quantizer_round_trip_bound():
    w = synth.normal_f32(12, 99, 128 * 512, 1 / math.sqrt(512)).reshape(128, 512)
    codes, scales, g = synth.quantize_nvfp4(w)
    deq = oracle.dequant(codes, scales, g)
    s = np.repeat(e4m3_lib(scales), 16, axis=1) * g
    bmax = np.repeat(np.abs(w.reshape(128, -1, 16)).max(axis=2), 16, axis=1)
    bound = np.maximum(s * 1.0, bmax / 15.0) + 1e-12
    assert np.all(np.abs(deq - w) <= bound)
    assert not np.any(np.isnan(e4m3_lib(scales)))
    rel = np.linalg.norm(deq - w) / np.linalg.norm(w)
    assert rel < 0.12  # 4-bit grid with 16-element blocks


def test_e2m1_encoder_ties_to_even():
    lib = synth.lib()
    # midpoints between grid values go to the even code
    for v, code in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6), (7.0, 7), (-0.75, 10)]:
        assert lib.synth_e2m1_encode(v) == code, v


# ---- S1 router -------------------------------------------------------------------------

def test_router_vs_numpy_matmul():
    x = synth.x_bf16(3, 5, 256)
    W = synth.router(2, 256, 32)
    bias = synth.zipf_bias(4, 32)
    ref = bf16_lib(x) @ W.astype(np.float64) + bias.astype(np.float64)
    got = oracle.router_logits(x, W, bias)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_router_abs_vs_numpy_and_triangle_inequality():
    """sum_h |x_h W[h, e]| (the scale every routing check's logit bound is measured in)
    against numpy fp64 |x| @ |W|; it bounds |logit| (triangle inequality), with equality
    when every product is non-negative; a signed sum (the plausible slip) fails the pin."""
    x = synth.x_bf16(5, 6, 256)
    W = synth.router(2, 256, 32)
    got = oracle.router_abs(x, W)
    ref = np.abs(bf16_lib(x)) @ np.abs(W.astype(np.float64))
    assert np.allclose(got, ref, rtol=1e-13, atol=0)
    logits = oracle.router_logits(x, W)
    assert np.all(np.abs(logits) <= got * (1 + 1e-12))
    xp = x & np.uint16(0x7FFF)  # clear the bf16 sign bits: every product is >= 0
    Wp = np.abs(W)
    assert np.allclose(oracle.router_abs(xp, Wp), oracle.router_logits(xp, Wp), rtol=1e-13, atol=0)
    signed = np.abs(bf16_lib(x) @ W.astype(np.float64))
    assert np.max(np.abs(signed - got) / got) > 0.5


# ---- P-C select ----------------------------------------------------------------------------

def _brute_select(logits, k):
    T, E = logits.shape
    idx = np.array([[e for _, e in sorted((-float(l) + 0.0, e) for e, l in enumerate(row))][:k] for row in logits],
                   dtype=np.int32).reshape(T, k)
    # softmax over all experts, then renormalised over the selected ones
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    p = z / z.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx, axis=1)
    return idx, sel / sel.sum(axis=1, keepdims=True)


def _planted_logits(T, E, seed):
    l = synth.logits(seed, T, E).astype(np.float64)
    l[0, :] = 0.0                      # all equal: a run longer than k
    l[0, 5] = -0.0
    if T > 1:
        l[1, 3] = l[1, 7] = l[1, 11] = 9.0  # equal maxima
        l[1, E - 2] = -0.0
        l[1, E - 1] = 0.0
    if T > 2:
        l[2, ::2] = 1.5                 # half the experts tied
    return l


@pytest.mark.parametrize("T,E,k", [(7, 32, 4), (5, 64, 16), (3, 16, 16), (9, 40, 1)])
def test_select_vs_brute_force(T, E, k):
    l = _planted_logits(T, E, 50 + T)
    idx, w = oracle.select(l, k)
    ridx, rw = _brute_select(l, k)
    assert np.array_equal(idx, ridx)
    assert np.allclose(w, rw, rtol=1e-12, atol=1e-15)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 1e-15)  # listed by descending logit


# ---- P-D permutation -------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (13, 32, 4), (40, 16, 16)])
def test_permute_invariants_and_brute(T, E, k):
    l = synth.logits(70 + T, T, E)
    idx, _ = oracle.select(l, k)
    counts, offsets, perm, slot, inv = oracle.permute(idx, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and np.all(np.diff(offsets) == counts)
    # brute force: bucket e lists (t, j) with idx[t, j] == e, ascending t
    p = 0
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    assert perm[p] == t and slot[p] == j and inv[t * k + j] == p
                    p += 1
    assert p == T * k
    # every token appears exactly k times, and each of its experts exactly once
    assert np.array_equal(np.bincount(perm, minlength=T), np.full(T, k))
    assert np.array_equal(np.sort(inv), np.arange(T * k))
    assert np.array_equal(idx.reshape(-1)[perm * k + slot].reshape(-1),
                          np.repeat(np.arange(E), counts))


# ---- P-E / P-F / P-G whole-layer special cases -----------------------------------------

def _dense_ffn(L, e, xf):
    """Dense numpy SwiGLU MLP of expert e on rows xf [n][H], weights decoded by the library decoders."""
    H, I = L.H, L.I
    Wgu = dequant_lib(L.gu_codes[e], L.gu_scales[e], 1.0)
    Wg = Wgu[:I] * np.float64(L.gu_global[e, 0])
    Wu = Wgu[I:] * np.float64(L.gu_global[e, 1])
    Wd = dequant_lib(L.dn_codes[e], L.dn_scales[e], L.dn_global[e])
    g = xf @ Wg.T
    u = xf @ Wu.T
    h = g * (1.0 / (1.0 + np.exp(-g))) * u
    return h @ Wd.T


def test_single_expert_is_a_swiglu_mlp():
    """E=1, k=1 reduces to one dense SwiGLU MLP."""
    L = synth.layer(H=128, I=64, E=1, seed_weights=21, seed_router=22)
    x = synth.x_bf16(23, 6, 128)
    out, idx, w, _ = oracle.moe_forward(oracle.Layer(L), x, 1)
    ref = _dense_ffn(L, 0, bf16_lib(x))
    assert np.all(idx == 0) and np.all(w == 1.0)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_all_experts_is_dense_softmax_mixture():
    """k=E: the renormalised top-k is the softmax over all experts."""
    L = synth.layer(H=64, I=32, E=6, seed_weights=31, seed_router=32)
    x = synth.x_bf16(33, 5, 64)
    out, idx, w, _ = oracle.moe_forward(oracle.Layer(L), x, 6)
    xf = bf16_lib(x)
    logits = xf @ L.router_w.astype(np.float64)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ref = sum(p[:, e:e + 1] * _dense_ffn(L, e, xf) for e in range(6))
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_all_equal_weights_closed_form():
    """All codes 1.0, all scales 1.0, tensor scales c, c_d: every output column is
    I * c_d * silu(c*S) * c*S with S = sum_h x_h (the gate weights sum to 1)."""
    H, I, E, k = 64, 32, 8, 3
    L = synth.layer(H=H, I=I, E=E, seed_weights=41, seed_router=42)
    L.gu_codes[:] = 0x22  # E2M1 code 2 = 1.0 in both nibbles
    L.dn_codes[:] = 0x22
    L.gu_scales[:] = 0x38  # E4M3 1.0
    L.dn_scales[:] = 0x38
    c, cd = 0.03125, 0.5
    L.gu_global[:] = c
    L.dn_global[:] = cd
    x = synth.x_bf16(43, 4, H)
    out, _, w, _ = oracle.moe_forward(oracle.Layer(L), x, k)
    S = bf16_lib(x).sum(axis=1)
    a = c * S
    ref = I * cd * a / (1 + np.exp(-a)) * a
    assert np.allclose(out, np.repeat(ref[:, None], H, axis=1), rtol=1e-12, atol=1e-12)


def test_forward_equals_token_by_token():
    L = synth.layer(**{k: v for k, v in synth.TINY.items() if k != "k"}, seed_weights=1, seed_router=2)
    OL = oracle.Layer(L)
    x = synth.x_bf16(3, 9, L.H)
    out, idx, w, logits = oracle.moe_forward(OL, x, 4)
    out2, idx2, w2, logits2 = oracle.moe_tokens(OL, x[[8, 0, 3]], 4)
    assert np.array_equal(idx[[8, 0, 3]], idx2)
    assert np.array_equal(out[[8, 0, 3]], out2)
    assert np.array_equal(logits[[8, 0, 3]], logits2)


def test_tiny_layer_invariants():
    L = synth.layer(H=256, I=128, E=32, seed_weights=1, seed_router=2)
    x = synth.x_bf16(3, 4, 256)
    out, idx, w, logits = oracle.moe_forward(oracle.Layer(L), x, 4)
    assert out.shape == (4, 256) and np.all(np.isfinite(out))
    assert np.allclose(w.sum(axis=1), 1.0)
    for t in range(4):
        assert len(set(idx[t])) == 4
        assert np.all(logits[t, idx[t]] >= np.sort(logits[t])[-4])


def test_zipf_bias_is_a_permuted_log_rank():
    b = synth.zipf_bias(4, 896, 1.1)
    assert np.allclose(np.sort(b)[::-1], -1.1 * np.log(np.arange(1, 897)), atol=1e-5)
    assert len(set(np.argsort(b)[-5:])) == 5


# ---- caller-given routing on an expert range (a worker of an expert-parallel split) --------

def _expert_slice(L, e0, n):
    import dataclasses
    return dataclasses.replace(L, E=n, **{a: getattr(L, a)[e0:e0 + n] for a in (
        "gu_codes", "gu_scales", "gu_global", "dn_codes", "dn_scales", "dn_global")})


def test_routed_full_range_equals_the_layer():
    """With the layer's own routing and all experts, the routed expert stage is the layer
    (same operations in the same order: byte-equal)."""
    L = synth.layer(H=128, I=64, E=12, seed_weights=61, seed_router=62)
    x = synth.x_bf16(63, 7, 128)
    out, idx, w, _ = oracle.moe_forward(oracle.Layer(L), x, 3)
    got, served = oracle.moe_routed(oracle.Layer(L), x, idx, w, 0)
    assert np.array_equal(got, out)
    assert np.array_equal(served, idx)


def test_routed_ranges_partition_the_layer():
    """Workers whose expert ranges partition the experts add up to the layer."""
    L = synth.layer(H=128, I=64, E=12, seed_weights=61, seed_router=62)
    x = synth.x_bf16(64, 9, 128)
    out, idx, w, _ = oracle.moe_forward(oracle.Layer(L), x, 4)
    parts, served_any = [], np.full(idx.shape, -1)
    for e0, n in ((0, 5), (5, 1), (6, 6)):
        got, served = oracle.moe_routed(oracle.Layer(_expert_slice(L, e0, n)), x, idx, w, e0)
        mine = (idx >= e0) & (idx < e0 + n)
        assert np.array_equal(served, np.where(mine, idx, -1))
        served_any = np.where(mine, served, served_any)
        parts.append(got)
    assert np.array_equal(served_any, idx)  # every route served exactly once
    assert np.allclose(sum(parts), out, rtol=1e-12, atol=1e-14)


def test_routed_masked_and_foreign_ids_vs_dense_numpy():
    """Ids -1 and other workers' ids are skipped; the kept routes are weighted as given
    (dense numpy SwiGLU with the library decoders); no route gives zeros."""
    L = synth.layer(H=128, I=64, E=10, seed_weights=71, seed_router=72)
    x = synth.x_bf16(73, 5, 128)
    idx = np.array([[3, -1, 7, 0], [-1, -1, -1, -1], [9, 4, 5, 2], [6, 3, -1, 8], [1, 2, 3, 4]], dtype=np.int32)
    w = synth.normal_f32(74, 1, idx.size, 1.0).reshape(idx.shape).astype(np.float64)
    e0, n = 2, 5  # this worker holds experts 2..6
    got, served = oracle.moe_routed(oracle.Layer(_expert_slice(L, e0, n)), x, idx, w, e0)
    xf = bf16_lib(x)
    ref = np.zeros((5, 128))
    for t in range(5):
        for j in range(4):
            if e0 <= idx[t, j] < e0 + n:
                ref[t] += w[t, j] * _dense_ffn(L, int(idx[t, j]), xf[t:t + 1])[0]
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-12)
    assert np.all(got[1] == 0.0)
    assert np.array_equal(served, np.where((idx >= e0) & (idx < e0 + n), idx, -1))


# ---- a LatentMoE block -------------------------------------------------------------------------

def test_block_with_identity_projections_is_the_layer():
    """Routed-down and routed-up projections equal to the identity (d = hidden) and no
    shared experts: the block is the plain layer, byte for byte."""
    L = synth.block_layer(128, 128, 64, 8, 0, seed_weights=81, seed_router=82)
    eye = np.where(np.eye(128, dtype=bool), np.uint16(0x3F80), np.uint16(0))  # bf16 1.0 on the diagonal
    L.proj_down = eye.copy()
    L.proj_up = eye.copy()
    x = synth.x_bf16(83, 5, 128)
    out, idx, w, logits = oracle.moe_block(oracle.Layer(L), x, 3)
    ref, ridx, rw, rlog = oracle.moe_tokens(oracle.Layer(L), x, 3)
    assert np.array_equal(out, ref) and np.array_equal(idx, ridx) and np.array_equal(logits, rlog)


def test_block_dense_mixture_vs_numpy():
    """k = E (the routed part is the dense softmax mixture) with random bf16 projections and
    two shared experts of width 32 given as one of width 64, against numpy fp64 with the
    library decoders and the two shared experts computed separately."""
    Hm, d, I, E, f = 128, 64, 32, 5, 32
    L = synth.block_layer(Hm, d, I, E, 2 * f, seed_weights=91, seed_router=92)
    x = synth.x_bf16(93, 4, Hm)
    out, idx, w, _ = oracle.moe_block(oracle.Layer(L), x, E)
    xf = bf16_lib(x)
    logits = xf @ L.router_w.astype(np.float64)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    lat = xf @ bf16_lib(L.proj_down).T
    routed = sum(p[:, e:e + 1] * _dense_ffn(L, e, lat) for e in range(E))
    up = routed @ bf16_lib(L.proj_up).T
    gu, dn = bf16_lib(L.shared_gu), bf16_lib(L.shared_dn)
    silu = lambda v: v / (1 + np.exp(-v))
    shared = 0.0
    for s0 in (0, f):  # expert s: gate rows s0.., up rows 2f + s0.., down columns s0..
        g = xf @ gu[s0:s0 + f].T
        u = xf @ gu[2 * f + s0:2 * f + s0 + f].T
        shared = shared + (silu(g) * u) @ dn[:, s0:s0 + f].T
    assert np.allclose(out, up + shared, rtol=1e-10, atol=1e-12)
    assert np.allclose(np.sort(w, axis=1), np.sort(p, axis=1), rtol=1e-12, atol=1e-15)


# ---- the pins catch plausible mistakes ------------------------------------------------------

def test_pins_catch_planted_mistakes():
    L = synth.layer(H=128, I=64, E=1, seed_weights=21, seed_router=22)
    x = synth.x_bf16(23, 6, 128)
    xf = bf16_lib(x)
    out, _, _, _ = oracle.moe_forward(oracle.Layer(L), x, 1)
    I = L.I
    Wgu = dequant_lib(L.gu_codes[0], L.gu_scales[0], 1.0)
    Wg, Wu = Wgu[:I] * L.gu_global[0, 0], Wgu[I:] * L.gu_global[0, 1]
    Wd = dequant_lib(L.dn_codes[0], L.dn_scales[0], L.dn_global[0])
    silu = lambda v: v / (1 + np.exp(-v))
    mistakes = {
        "gate/up swapped": silu(xf @ Wu.T) * (xf @ Wg.T) @ Wd.T,
        "block scale dropped": silu(xf @ (Wg / np.repeat(e4m3_lib(L.gu_scales[0, :I]), 16, 1)).T) * (xf @ Wu.T) @ Wd.T,
        "nibbles swapped": None,
        "sign of the silu": (-xf @ Wg.T) / (1 + np.exp(xf @ Wg.T)) * (xf @ Wu.T) @ Wd.T,
    }
    codes = L.gu_codes[0]
    swapped = ((codes & 0xF) << 4) | (codes >> 4)
    Wgs = dequant_lib(swapped, L.gu_scales[0], 1.0)
    mistakes["nibbles swapped"] = silu(xf @ (Wgs[:I] * L.gu_global[0, 0]).T) * (xf @ (Wgs[I:] * L.gu_global[0, 1]).T) @ Wd.T
    rms = np.sqrt(np.mean(out ** 2))
    for name, wrong in mistakes.items():
        assert np.max(np.abs(wrong - out)) > 0.1 * rms, name


# ---- the oracle's result does not depend on its thread count --------------------------------

_THREADS_SNIPPET = """
import sys, numpy as np
sys.path.insert(0, {root!r})
import oracle, synth
L = synth.layer(256, 128, 32, seed_weights=41, seed_router=42)
x = synth.x_bf16(43, 19, 256)
out, idx, w, logits = oracle.moe_forward(oracle.Layer(L), x, 4)
sys.stdout.buffer.write(out.tobytes() + idx.tobytes() + w.tobytes() + logits.tobytes())
"""


def test_oracle_is_independent_of_thread_count():
    """Every output's reduction order is fixed, so one OpenMP thread and several give
    the same bytes (the oracle's timing runs use all host cores)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = _THREADS_SNIPPET.format(root=root)
    outs = []
    for n in ("1", "4"):
        env = dict(os.environ, OMP_NUM_THREADS=n)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, env=env, timeout=300)
        assert r.returncode == 0, r.stderr.decode()[-2000:]
        outs.append(r.stdout)
    assert len(outs[0]) > 0 and outs[0] == outs[1]

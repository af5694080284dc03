"""The whole layer on the GPU through the C ABI against the oracle, at sizes the
oracle finishes in seconds: the tiny configuration (T=4, H=256, I=128, E=32, k=4)
and a mid shape spanning several tiles with ragged token counts; plus the ABI's
edge cases (T=0, T=max, bad pointers, forward before load), determinism, the
host-buffer entry point and the stage hooks."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from helpers import (SHAPES, bf16_bits_to_f64, check_output, check_routing, forward_vs_caller_routed, gpu_forward,
                     gpu_route, layer)

pytestmark = pytest.mark.gpu


def make(name, max_tokens, zipf=False):
    import routed_expert_layer_gb300 as rel
    s = SHAPES[name]
    m = rel.MoeLayer(s["H"], s["I"], s["E"], s["k"], max_tokens)
    m.load(layer(name, zipf))
    return m


@pytest.fixture(scope="module")
def tiny():
    m = make("tiny", 64)
    yield m
    m.close()


@pytest.fixture(scope="module")
def mid():
    m = make("mid", 512)
    yield m
    m.close()


def run_case(moe, name, T, seed, zipf=False):
    s = SHAPES[name]
    return run_layer_case(moe, layer(name, zipf), s, synth.x_bf16(seed, T, s["H"]))


def run_layer_case(moe, L, s, x):
    """The whole layer on x (bf16 bits) through the C ABI against the oracle on L."""
    ref, ref_idx, ref_w, ref_logits = oracle.moe_forward(oracle.Layer(L), x, s["k"])
    r = gpu_route(moe, x, s["E"], s["k"])
    ref_abs = oracle.router_abs(x, L.router_w)
    ties = check_routing(r["logits"], r["idx"], ref_logits, ref_abs, ref_idx, s["k"])
    out = gpu_forward(moe, x)
    ratio = check_output(out, ref, ~ties)
    assert moe.get_error() == 0
    return ratio


def test_tiny_config(tiny):
    """The tiny configuration exactly: T=4, H=256, I=128, E=32, k=4, seed 3."""
    run_case(tiny, "tiny", 4, 3)


@pytest.mark.parametrize("T", [1, 2, 5, 33, 64])
def test_tiny_sizes(tiny, T):
    run_case(tiny, "tiny", T, 100 + T)


@pytest.mark.parametrize("T", [1, 7, 37, 300, 512])
def test_mid_sizes(mid, T):
    run_case(mid, "mid", T, 200 + T)


def test_mid_zipf_routing():
    """A skewed prefill-sized batch: experts of at most 16 rows run on the decode GEMM and
    the others on the prefill GEMM in the same call."""
    m = make("mid", 300, zipf=True)
    try:
        run_case(m, "mid", 300, 77, zipf=True)
        r = gpu_route(m, synth.x_bf16(77, 300, SHAPES["mid"]["H"]), SHAPES["mid"]["E"], SHAPES["mid"]["k"])
        counts = np.diff(r["offsets"])
        assert ((counts > 0) & (counts <= 16)).any() and (counts > 16).any()
    finally:
        m.close()


@pytest.mark.parametrize("T", [1, 2, 7, 16, 33])
def test_forward_matches_caller_routed_expert_stage(mid, T):
    """The forward (routed by the fused small-batch kernel up to 32 tokens, by the general
    kernels above) and the expert stage given that forward's routing back through
    moe_forward_routed (the general permutation, and its own gather): the same output bit
    for bit."""
    s = SHAPES["mid"]
    a, b = forward_vs_caller_routed(mid, synth.x_bf16(2100 + T, T, s["H"]), s["H"], s["k"])
    assert np.array_equal(a, b)
    assert mid.get_error() == 0


# h and y are kept in f16 (11 significant bits) between the GEMMs and before the
# combine. Each stored element's own rounding (at most 2^-11 of it, helpers.F16_STORE_REL)
# is allowed per element; what remains is fp32 accumulation and exp() error (about 1e-6
# relative) for h and for y against the down projection of the GPU's own h, and for y
# against the oracle's exact h additionally h's rounding carried through W_d (a sum of
# I independent errors of at most 2^-11 each: about 2^-11 / sqrt(3) of RMS(y) per
# element, up to ~4 times that at the extremes of a bucket).
H_TOL = 1e-3
Y_TOL = 2e-3


@pytest.mark.parametrize("T", [9, 300, 512])
def test_expert_stage_h_and_y(mid, T):
    """h (SwiGLU) and y (down projection) per routed row against the oracle's expert
    functions, for the decode variant (T=9) and the midfill variants with 64-row items
    (T=300, 37.5 rows per expert on average) and 128-row items (T=512, 64 rows)."""
    import torch
    s = SHAPES["mid"]
    L = layer("mid")
    OL = oracle.Layer(L)
    k = s["k"]
    x = synth.x_bf16(55, T, s["H"])
    r = gpu_route(mid, x, s["E"], k)
    h = torch.empty(T * k, s["I"], dtype=torch.float32, device="cuda")
    y = torch.empty(T * k, s["H"], dtype=torch.float32, device="cuda")
    mid.debug_experts(torch.from_numpy(x.view(np.int16)).cuda(), h=h, y=y)
    torch.cuda.synchronize()
    h, y = h.cpu().numpy().astype(np.float64), y.cpu().numpy().astype(np.float64)
    xf = bf16_bits_to_f64(x)
    offs = r["offsets"]
    for e in np.nonzero(np.diff(offs))[0]:
        rows = np.arange(offs[e], offs[e + 1])
        toks = r["perm"][rows]
        href = oracle.expert_gateup(OL, int(e), xf[toks])
        yref = oracle.expert_down(OL, int(e), href)
        check_output(h[rows], href, tol=H_TOL, f16_store=True)
        check_output(y[rows], oracle.expert_down(OL, int(e), h[rows]), tol=H_TOL, f16_store=True)
        check_output(y[rows], yref, tol=Y_TOL, f16_store=True)


def test_dependent_kernel_after_forward_reads_the_finished_output(mid):
    """At decode sizes the forward's last kernel lets the next kernel on the stream launch
    before it has finished. A consumer launched that way which waits on its grid
    dependency before reading (moe_debug_pdl_copy, as the header asks of such kernels)
    gets the finished output: bit for bit the output, never the sentinel it was filled
    with before the forward."""
    import torch
    import routed_expert_layer_gb300 as rel
    s = SHAPES["mid"]
    T = 5  # T*k/E = 0.6: decode plan, kernels launched with programmatic dependent launch
    assert rel.plan(s["H"], s["I"], s["E"], s["k"], 512, 152, T)["prefill"] == 0
    xd = torch.from_numpy(synth.x_bf16(2300, T, s["H"]).view(np.int16)).cuda()
    sentinel = 0x7FC1  # a bf16 NaN: never a value of the layer's finite output
    for _ in range(20):
        out = torch.full((T, s["H"]), sentinel, dtype=torch.int16, device="cuda")
        copy = torch.zeros_like(out)
        mid.forward(xd, out)
        rel.debug_pdl_copy(out, copy)
        torch.cuda.synchronize()
        assert not bool((out == sentinel).any())
        assert torch.equal(copy, out)
    assert mid.get_error() == 0


def test_zero_tokens_is_a_noop(tiny):
    import torch
    import routed_expert_layer_gb300 as rel
    x = torch.zeros(0, 256, dtype=torch.int16, device="cuda")
    tiny.forward(x, torch.zeros(0, 256, dtype=torch.int16, device="cuda"))
    assert rel.lib().moe_forward(tiny.ctx, None, None, None, 0) == 0


def test_max_tokens_and_beyond(tiny):
    import torch
    import routed_expert_layer_gb300 as rel
    run_case(tiny, "tiny", 64, 9)
    x = torch.zeros(65, 256, dtype=torch.int16, device="cuda")
    with pytest.raises(rel.MoeError) as ei:
        tiny.forward(x, torch.zeros_like(x))
    assert ei.value.status == rel.MOE_ERR_INVALID_ARG


def test_bad_pointers_rejected(tiny):
    import ctypes
    import torch
    import routed_expert_layer_gb300 as rel
    L = rel.lib()
    buf = torch.zeros(3 * 256 + 8, dtype=torch.int16, device="cuda")
    base = buf.data_ptr()
    # misaligned
    assert L.moe_forward(tiny.ctx, None, ctypes.c_void_p(base + 2), ctypes.c_void_p(base + 2048), 1) == rel.MOE_ERR_INVALID_ARG
    # out overlaps x
    assert L.moe_forward(tiny.ctx, None, ctypes.c_void_p(base), ctypes.c_void_p(base + 256), 1) == rel.MOE_ERR_INVALID_ARG
    assert L.moe_forward(tiny.ctx, None, None, ctypes.c_void_p(base), 1) == rel.MOE_ERR_INVALID_ARG
    assert tiny.get_error() == 0


def test_forward_before_load():
    import torch
    import routed_expert_layer_gb300 as rel
    m = rel.MoeLayer(256, 128, 32, 4, 4)
    try:
        x = torch.zeros(2, 256, dtype=torch.int16, device="cuda")
        with pytest.raises(rel.MoeError) as ei:
            m.forward(x, torch.zeros_like(x))
        assert ei.value.status == rel.MOE_ERR_NOT_LOADED
    finally:
        m.close()


def test_deterministic_and_host_entry_point(mid):
    import torch
    x = synth.x_bf16(999, 300, 512)
    a = gpu_forward(mid, x)
    b = gpu_forward(mid, x)
    assert np.array_equal(a, b)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    mid.forward_host(xh, oh)
    assert np.array_equal(bf16_bits_to_f64(oh.numpy().view(np.uint16)), a)


def test_profile_hooks(tiny):
    import torch
    x = torch.from_numpy(synth.x_bf16(5, 16, 256).view(np.int16)).cuda()
    out = torch.empty_like(x)
    tiny.profile_begin(3)
    for _ in range(3):
        tiny.forward(x, out)
    prof = tiny.profile_end()
    assert prof["gateup"][1] == 3 and prof["gateup"][0] > 0


def test_forward_in_cuda_graph(mid):
    """moe_forward allocates nothing and never syncs the host, so it can be captured in
    a CUDA graph; replays give exactly the eager result."""
    import torch
    x = torch.from_numpy(synth.x_bf16(321, 37, 512).view(np.int16)).cuda()
    eager = torch.empty_like(x)
    mid.forward(x, eager)
    s = torch.cuda.Stream()
    out = torch.zeros_like(x)
    with torch.cuda.stream(s):
        mid.forward(x, out, s)  # first call outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mid.forward(x, out, s)
    out.zero_()
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert mid.get_error() == 0


def test_profile_hooks_under_graph_capture(mid):
    import torch
    x = torch.from_numpy(synth.x_bf16(77, 37, 512).view(np.int16)).cuda()
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mid.forward(x, out, s)
    torch.cuda.synchronize()
    mid.profile_begin(1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mid.forward(x, out, s)
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    prof = mid.profile_end()
    assert prof["gateup"][1] == 1 and prof["gateup"][0] > 0 and prof["down"][0] > 0


@pytest.mark.parametrize("name,T", [("single", 1), ("single", 9), ("dense", 3), ("dense", 40), ("wide", 5),
                                    ("wide", 33)])
def test_degenerate_and_extreme_shapes(name, T):
    """E = k = 1 (one SwiGLU MLP), k = E = 32 (every expert for every token) and the
    widest supported hidden size (H = 14336), through the whole layer."""
    m = make(name, 64)
    try:
        run_case(m, name, T, 600 + T)
    finally:
        m.close()


# ---- the size of x and of the tensor scales ------------------------------------------------

def scaled_bits(x_bits, a):
    """bf16 bits of x * 2^a (exact for a power of two away from the format's limits)."""
    f = synth.bf16_bits_to_f32(x_bits) * np.float32(2.0 ** a)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


SCALINGS = [(-8, 0, 0), (8, 0, 0), (0, 6, 0), (0, -6, 0), (0, 0, 6), (0, 0, -6), (8, -6, 6), (-8, 6, -6)]


@pytest.mark.parametrize("name,T", [("mid", 9), ("mid", 300), ("wide", 5)])
@pytest.mark.parametrize("xa,ga,da", SCALINGS)
def test_scale_of_inputs(name, T, xa, ga, da):
    """x scaled by 2^xa, the gate/up tensor scales by 2^ga and the down tensor scales by
    2^da: the layer meets the same tolerance against the oracle at every size of its
    inputs, for the decode variant (mid T=9), the prefill variant (mid T=300) and the
    K-split decode path with its separate SwiGLU pass (wide T=5)."""
    import routed_expert_layer_gb300 as rel
    s = SHAPES[name]
    base = layer(name)
    L = dataclasses.replace(base, gu_global=(base.gu_global * np.float32(2.0 ** ga)).astype(np.float32),
                            dn_global=(base.dn_global * np.float32(2.0 ** da)).astype(np.float32))
    x = scaled_bits(synth.x_bf16(900 + T, T, s["H"]), xa)
    m = rel.MoeLayer(s["H"], s["I"], s["E"], s["k"], T)
    try:
        m.load(L)
        run_layer_case(m, L, s, x)
    finally:
        m.close()


def test_out_of_range_intermediate_raises_the_error_word():
    """An input whose SwiGLU values leave the f16 range of the normalised store sets the
    device error word instead of being clamped silently: every gate/up weight at its
    largest block value (+6 x 448) and every x element 1.0, so all H = 14336 products of
    a row add up (normalised gate and up sums of about H/3 each, h about 3e5 > 65504)."""
    import torch
    import routed_expert_layer_gb300 as rel
    s = SHAPES["wide"]
    base = layer("wide")
    L = dataclasses.replace(base, gu_codes=np.full_like(base.gu_codes, 0x77),
                            gu_scales=np.full_like(base.gu_scales, 0x7E))
    m = rel.MoeLayer(s["H"], s["I"], s["E"], s["k"], 4)
    try:
        m.load(L)
        x = torch.full((4, s["H"]), 0x3F80, dtype=torch.int16, device="cuda")  # bf16 1.0
        out = torch.empty_like(x)
        m.forward(x, out)
        torch.cuda.synchronize()
        assert m.get_error() & 8
        assert m.get_error() == 0  # read and cleared
    finally:
        m.close()

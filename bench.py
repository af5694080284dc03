"""Benchmark of the routed expert layer at the K3 shape on GB300.

One step = one moe_forward over one batch of T tokens (router, select, permute,
gate/up + SwiGLU, down, combine) on the K3-shaped layer (H=7168, I=1536, E=896,
k=16, NVFP4 experts, 16.6 GB resident in HBM). The headline workload is decode at
T=53 tokens (the serving pages' concurrency cap). Inputs are synthetic and seeded
(x ~ N(0,1) bf16, router N(0,1/H), experts N(0,1/fan_in) quantised to NVFP4) and
already resident in HBM when the timed region starts; 8 x batches rotate so the
routing (and the ~10 GB of touched expert weights) changes every step, which is
larger than the 129 MB L2, so no L2 flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs an independent
replica on its own GPU (weak scaling: the layer does not exchange data between
replicas); value = tokens of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at K3 shape; % HBM roofline (decode) / % tensor peak (prefill)"
K3 = dict(H=7168, I=1536, E=896, k=16)
EXPERT_BYTES = 3 * K3["H"] * K3["I"] // 2 + 3 * K3["H"] * K3["I"] // 16 + 6 * 4  # 18,579,480
GU_BYTES = 2 * K3["I"] * K3["H"] // 2 + 2 * K3["I"] * K3["H"] // 16 + 8            # gate+up codes, scales, 2 scales
DN_BYTES = K3["H"] * K3["I"] // 2 + K3["H"] * K3["I"] // 16 + 4
N_BATCHES = 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--T", type=int, default=53)
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-configuration side measurements")
    ap.add_argument("--cpu-sample", type=int, default=0, help="tokens in the oracle sample (0 = auto)")
    ap.add_argument("--profile-run", action="store_true",
                    help="only run warmup+steps forwards of a K3-shaped layer with --experts experts "
                         "(no timing line): the command the ncu captures in profiles/ use")
    ap.add_argument("--experts", type=int, default=896, help="experts in the layer (--profile-run only)")
    ap.add_argument("--inter", type=int, default=0,
                    help="expert intermediate size (--profile-run only; 0 = K3's 1536): a small layer with "
                         "K3's router for captures of the routing kernels")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def job_throughput(ms, T, world, device):
    """Max over ranks of the per-step time (ms) and the whole-job throughput:
    tokens of all ranks per step / that time. Every rank must call it."""
    ms_all = float(ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_all], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_all = float(t.item())
    return ms_all, world * T / (ms_all * 1e-3)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


def make_layer(zipf=False):
    """The K3 layer (weights seed 1, router seed 2); zipf=True adds the Zipf(1.1) router
    bias over a seeded permutation of the experts (seed 4)."""
    import synth
    return synth.layer(K3["H"], K3["I"], K3["E"], seed_weights=1, seed_router=2, zipf_seed=4 if zipf else None)


# LatentMoE block at the pages' K3 geometry: hidden 7168, routed latent 3584, 896 experts
# of 3584 x 3072 (18,579,480 B each, the same as the plain K3 layer's), top-16, and the two
# shared experts (bf16) read as one of intermediate 2 x 3072.
KB = dict(H=7168, d=3584, I=3072, E=896, k=16, Is=6144)
KB_DENSE_BYTES = 2 * (2 * KB["d"] * KB["H"]) + 2 * (3 * KB["Is"] * KB["H"])  # bf16 projections + shared


def sweep_point(moe, xs, stream, hbm, bf16, reps, warmup=2, extra_bytes=0, flops_per_token=None):
    """Device time per forward at one batch size (graph replays over the rotating batches
    xs) with the touched experts, the largest bucket and the roofline fractions: bytes =
    touched experts x 18,579,480 (+ extra_bytes read once per forward), FLOPs = 6 T k H I
    (or flops_per_token x T)."""
    Ts = xs[0].shape[0]
    msw, _, _ = time_config(moe, xs, reps, warmup, stream)
    # per-stage times from a separate pass: events between the kernels would break the
    # overlap of programmatic dependent launch in the timed one
    _, prof, _ = time_config(moe, xs, max(4, reps // 4), 1, stream, profile=True)
    tch = [touched(moe, x, K3["E"], K3["k"]) for x in xs]
    dsw = float(np.mean([t[0] for t in tch]))
    byts = dsw * EXPERT_BYTES + extra_bytes
    flops = Ts * (flops_per_token if flops_per_token else 6.0 * K3["k"] * K3["H"] * K3["I"])
    return {"ms": round(msw, 4), "tokens_per_s": round(Ts / (msw * 1e-3), 1), "touched_experts": dsw,
            "largest_bucket": int(max(t[1] for t in tch)), "replays": reps, "batches": len(xs),
            "stage_ms": {k_: round(v[0] / max(1, v[1]), 4) for k_, v in prof.items() if v[1]},
            "hbm_frac": round(byts / (msw * 1e-3) / 1e9 / hbm, 4),
            "tensor_frac": round(flops / (msw * 1e-3) / 1e12 / bf16, 4)}


def cpu_baseline(L, x_bits, n_tokens):
    """The oracle as it stands (fp64, OpenMP) on the first n tokens of a batch."""
    import oracle
    OL = oracle.Layer(L)
    t0 = time.perf_counter()
    oracle.moe_forward(OL, x_bits[:n_tokens], K3["k"])
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"oracle_moe_forward (fp64) on the first {n_tokens} tokens of one K3 decode batch "
                      f"(T={x_bits.shape[0]}), {dt:.1f} s wall"}


def cpu_baseline_bounded(L, batches, min_s=10.0):
    """The oracle on whole decode batches, one after another, until at least min_s of
    CPU work is done (at most all the given batches)."""
    import oracle
    OL = oracle.Layer(L)
    tok, dt = 0, 0.0
    for xb in batches:
        t0 = time.perf_counter()
        oracle.moe_forward(OL, xb, K3["k"])
        dt += time.perf_counter() - t0
        tok += xb.shape[0]
        if dt >= min_s:
            break
    nb = tok // batches[0].shape[0]
    return {"value": tok / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"oracle_moe_forward (fp64) on {nb} whole K3 decode batch(es) of T={batches[0].shape[0]} "
                      f"({tok} tokens), {dt:.1f} s wall"}


def run_reference(args, rank, world):
    """Reference arm: the oracle timed as it stands on the host cores. Each step is
    the oracle on a window of up to 4 tokens of the decode batch (the window moves each
    step), sized from a first untimed call so that K + W steps take a few minutes."""
    if rank != 0:
        return
    import synth
    L = make_layer()
    x = synth.x_bf16(3, args.T, K3["H"])
    n = min(args.cpu_sample or 4, args.T)

    def window(i):
        s0 = (i * n) % max(1, args.T - n + 1)
        return x[s0:s0 + n]
    if not args.cpu_sample:
        # size the window so that all K + W steps take about two and a half minutes
        t0 = time.perf_counter()
        cpu_baseline(L, window(0), n)
        per_token = (time.perf_counter() - t0) / n
        n = max(1, min(n, int(150.0 / (max(1, args.steps + args.warmup) * per_token))))
    for i in range(args.warmup):
        cpu_baseline(L, window(i), n)
    t0 = time.perf_counter()
    for i in range(args.steps):
        cb = cpu_baseline(L, window(args.warmup + i), n)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = n / dt
    cb["sample"] = (f"oracle_moe_forward (fp64) on a moving window of {n} tokens of one K3 decode batch "
                    f"(T={args.T}) per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"k3_decode_T{args.T}", "T": args.T, **K3, "sample_tokens_per_step": n},
            "cpu_baseline": {**cb, "value": value},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def touched(moe, x_dev, E, k):
    import torch
    offs = torch.empty(E + 1, dtype=torch.int32, device=x_dev.device)
    moe.debug_route(x_dev, offsets=offs)
    torch.cuda.synchronize()
    c = np.diff(offs.cpu().numpy())
    return int((c > 0).sum()), int(c.max())


def time_config(moe, xs, steps, warmup, stream, profile=False):
    """Device time per forward: each rotating batch's forward is captured once in a CUDA
    graph and the graphs are replayed in turn; CUDA events on the launching stream bracket
    the timed replays. Returns (ms per forward, per-stage profile, kernels launched)."""
    import torch
    outs = [torch.empty_like(x) for x in xs]
    with torch.cuda.stream(stream):
        for i in range(len(xs)):  # eager first pass (lazy module loading, first touch)
            moe.forward(xs[i], outs[i], stream)
    torch.cuda.synchronize()
    if profile:
        moe.profile_begin(len(xs))  # one set of stage events per captured graph
    n0 = moe.launch_count()
    graphs = []
    for i in range(len(xs)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moe.forward(xs[i], outs[i], stream)
        graphs.append(g)
    per_forward = (moe.launch_count() - n0) / len(xs)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        b.record(stream)
        torch.cuda.synchronize()
    prof = moe.profile_end() if profile else None
    del graphs
    return a.elapsed_time(b) / steps, prof, int(per_forward * steps)


def replay_distribution(moe, xs, stream, n=64):
    """Per-forward device times of n graph replays (CUDA events around each replay on
    the launching stream), outside the timed region: p10 / p50 / p90 in ms. None if
    anything goes wrong (this is a side measurement, never the headline)."""
    try:
        import torch
        outs = [torch.empty_like(x) for x in xs]
        graphs = []
        for i in range(len(xs)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                moe.forward(xs[i], outs[i], stream)
            graphs.append(g)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(len(graphs)):
                graphs[i].replay()
            for i in range(n):
                evs[i][0].record(stream)
                graphs[i % len(graphs)].replay()
                evs[i][1].record(stream)
        torch.cuda.synchronize()
        t = np.array([a.elapsed_time(b) for a, b in evs])
        del graphs
        return {"n": n, "p10_ms": round(float(np.percentile(t, 10)), 5), "p50_ms": round(float(np.percentile(t, 50)), 5),
                "p90_ms": round(float(np.percentile(t, 90)), 5)}
    except Exception as e:  # noqa: BLE001
        return {"error": str(e)[:200]}


def profile_run(args):
    """Forwards of a K3-shaped layer (H=7168, I=1536, k=16) with --experts experts at --T
    tokens: a small case of the same kernels for ncu captures."""
    import torch
    import synth
    import routed_expert_layer_gb300 as rel
    inter = args.inter or K3["I"]
    L = synth.layer(K3["H"], inter, args.experts, seed_weights=1, seed_router=2)
    moe = rel.MoeLayer(K3["H"], inter, args.experts, K3["k"], args.T)
    moe.load(L)
    x = torch.from_numpy(synth.x_bf16(3, args.T, K3["H"]).view(np.int16)).cuda()
    out = torch.empty_like(x)
    for _ in range(args.warmup + args.steps):
        moe.forward(x, out)
    torch.cuda.synchronize()
    d, dmax = touched(moe, x, args.experts, K3["k"])
    print(json.dumps({"profile_run": True, "experts": args.experts, "inter": inter, "T": args.T,
                      "forwards": args.warmup + args.steps, "device_error": moe.get_error(),
                      "kernels": moe.launch_count(), "touched_experts": d, "max_rows": dmax}), flush=True)
    moe.close()


def main():
    args = parse()
    rank, world, local = dist_info()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.profile_run:
        profile_run(args)
        return
    import torch
    import torch.distributed as dist
    import synth
    import routed_expert_layer_gb300 as rel

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    hbm, bf16, bf16_sus, peak_kind = peaks()
    T = args.T
    L = make_layer()
    moe = rel.MoeLayer(K3["H"], K3["I"], K3["E"], K3["k"], max(T, 8192), device=local)
    moe.load(L)
    stream = torch.cuda.Stream()
    xs_host = [synth.x_bf16(3 + 1000 * rank + i, T, K3["H"]) for i in range(N_BATCHES)]
    xs = [torch.from_numpy(x.view(np.int16)).cuda() for x in xs_host]
    tch = [touched(moe, x, K3["E"], K3["k"]) for x in xs]
    d_avg = float(np.mean([t[0] for t in tch]))

    # ---- timed region ---------------------------------------------------------------
    props = torch.cuda.get_device_properties(local)
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(props.uuid) if not str(props.uuid).startswith("GPU-") else str(props.uuid)
    except Exception:
        pass
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id)
    time.sleep(0.4)
    ms, prof, n_launch = time_config(moe, xs, args.steps, args.warmup, stream, profile=True)
    clocks = sampler.stop()
    ms_all, value = job_throughput(ms, T, world, "cuda")
    replays = replay_distribution(moe, xs, stream) if rank == 0 else None

    # ---- end to end through the host-buffer entry point --------------------------------
    xh = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_host]
    oh = torch.empty_like(xh[0]).pin_memory()
    for i in range(5):
        moe.forward_host(xh[i % N_BATCHES], oh, stream)
    n_e2e = max(20, min(args.steps, 200))
    t0 = time.perf_counter()
    for i in range(n_e2e):
        moe.forward_host(xh[i % N_BATCHES], oh, stream)
    e2e_s = (time.perf_counter() - t0) / n_e2e
    e2e_val = world * T / e2e_s  # each replica runs the same loop

    # ---- roofline of the dominant kernel (gate/up) ------------------------------------
    stages = {k_: v[0] / max(1, v[1]) for k_, v in prof.items()}
    dom = max(stages, key=stages.get)
    gu_ms = stages["gateup"]
    # algorithmic bytes of one gate/up launch: the touched experts' gate/up weights, x read
    # once (bf16) and h written once (16-bit)
    gu_bytes = d_avg * GU_BYTES + T * K3["H"] * 2 + T * K3["k"] * K3["I"] * 2
    achieved = gu_bytes / (gu_ms * 1e-3) / 1e9
    step_bytes = d_avg * EXPERT_BYTES + 4 * K3["H"] * K3["E"] + 2 * T * K3["H"] * 2
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            tr = json.load(f).get(f"gateup_T{T}")
            if tr and tr.get("kernel_rev") == rel.KERNEL_REV.get("gateup"):
                traffic = tr["bytes_per_launch"]
    except Exception:
        pass

    sweep = {}
    if not args.no_sweep and rank == 0:
        sweep_sampler = ClockSampler(gpu_id)
        for Ts in (1, 8, 64, 128, 256, 2048, 4096, 8192):
            nb = 4 if Ts >= 2048 else 2
            xsw = [torch.from_numpy(synth.x_bf16(500 + i + Ts, Ts, K3["H"]).view(np.int16)).cuda()
                   for i in range(nb)]
            sweep[f"T{Ts}"] = sweep_point(moe, xsw, stream, hbm, bf16, reps=30 if Ts <= 256 else 20)
            del xsw
        # Zipf(1.1)-skewed routing: the same experts, a router bias making a few experts hot
        zl = dataclasses.replace(L, router_bias=synth.zipf_bias(4, K3["E"], 1.1))
        mz = rel.MoeLayer(K3["H"], K3["I"], K3["E"], K3["k"], 4096, device=local)
        mz.load(zl)
        for Ts in (64, 4096):
            nb = 4 if Ts >= 2048 else 2
            xsw = [torch.from_numpy(synth.x_bf16(700 + i + Ts, Ts, K3["H"]).view(np.int16)).cuda()
                   for i in range(nb)]
            sweep[f"zipf_T{Ts}"] = sweep_point(mz, xsw, stream, hbm, bf16, reps=30 if Ts <= 256 else 20)
            sweep[f"zipf_T{Ts}"]["vs_uniform"] = round(sweep[f"T{Ts}"]["ms"] / sweep[f"zipf_T{Ts}"]["ms"], 4)
            del xsw
        mz.close()
        del zl
        # the LatentMoE block (routed-down projection and shared experts' gate/up, experts in
        # the latent, routed-up projection and shared down)
        bl = synth.block_layer(KB["H"], KB["d"], KB["I"], KB["E"], KB["Is"], seed_weights=1, seed_router=2)
        mb = rel.MoeLayer(KB["H"], KB["I"], KB["E"], KB["k"], 4096, device=local, latent=KB["d"],
                          shared_inter=KB["Is"])
        mb.load(bl)
        del bl
        fpt = 6.0 * KB["k"] * KB["d"] * KB["I"] + 2.0 * 2 * KB["d"] * KB["H"] + 6.0 * KB["Is"] * KB["H"]
        for Ts in (53, 4096):
            nb = 4 if Ts >= 2048 else 2
            xsw = [torch.from_numpy(synth.x_bf16(900 + i + Ts, Ts, KB["H"]).view(np.int16)).cuda()
                   for i in range(nb)]
            sweep[f"block_T{Ts}"] = sweep_point(mb, xsw, stream, hbm, bf16, reps=30 if Ts <= 256 else 20,
                                                extra_bytes=KB_DENSE_BYTES, flops_per_token=fpt)
            del xsw
        mb.close()
        sweep["clocks"] = sweep_sampler.stop()

    cb = None
    if rank == 0:
        if args.cpu_sample:
            cb = cpu_baseline(L, xs_host[0], args.cpu_sample)
        else:
            cb = cpu_baseline_bounded(L, xs_host[:3])

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_all, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; x bf16 N(0,1), router fp32 N(0,1/H), experts N(0,1/fan_in) -> NVFP4)",
            "config": {"workload": f"k3_decode_T{T}", "T": T, **K3, "parallelism": f"replicas{world}",
                       "layer_bytes": K3["E"] * EXPERT_BYTES, "touched_experts_avg": d_avg,
                       "l2": "no flush: touched weights per step (~%.1f GB) exceed the 129 MB L2; %d rotating x batches"
                             % (d_avg * EXPERT_BYTES / 1e9, N_BATCHES)},
            "hbm_frac_step": round(step_bytes / (ms_all * 1e-3) / 1e9 / hbm, 4),
            "roofline": {"bound": "hbm", "kernel": "gateup", "achieved": round(achieved, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": int(gu_bytes),
                         "dominant_stage": dom},
            "stage_ms": {k_: round(v, 5) for k_, v in stages.items()},
            "replay_ms": replays,
            "gpu_launches": int(n_launch),
            "e2e": {"value": round(e2e_val, 2), "unit": "tokens/s", "h2d_bytes_per_step": T * K3["H"] * 2,
                    "d2h_bytes_per_step": T * K3["H"] * 2},
            "clocks": clocks,
            "cpu_baseline": cb,
            "sweep": sweep,
        }
        print(json.dumps(line), flush=True)
    moe.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""The reference arm of bench.py (the oracle on the host cores) prints one JSON line
with the keys the benchmark contract requires; run here on the tiny layer shape so it
takes a second (the real arm uses the K3 shape)."""
import argparse
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

REQUIRED = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"]


def test_reference_arm_line(monkeypatch):
    import bench
    import synth
    tiny = dict(H=256, I=128, E=32, k=4)
    monkeypatch.setattr(bench, "K3", tiny)
    monkeypatch.setattr(bench, "make_layer", lambda zipf=False: synth.layer(256, 128, 32, seed_weights=1,
                                                                            seed_router=2))
    args = argparse.Namespace(T=8, steps=3, warmup=1, cpu_sample=0, gpus=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, 0, 1)
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in REQUIRED:
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith("k3_decode_T")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    import bench
    args = argparse.Namespace(T=8, steps=1, warmup=0, cpu_sample=0, gpus=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, 1, 2)
    assert buf.getvalue() == ""


def test_roofline_constants_match_the_byte_census():
    """The bench's per-expert byte counts follow the page's census of 18,579,480 B per
    expert in 12 tensors (3 x codes, block scales, tensor scale, input scale): gate + up
    are two thirds of the codes and block scales plus their two tensor scales, down the
    rest plus one; the three 4-byte input scales are not read with 16-bit activations."""
    import bench
    H, I = 7168, 1536
    assert bench.EXPERT_BYTES == 18_579_480
    assert bench.GU_BYTES == 2 * I * H // 2 + 2 * I * H // 16 + 8 == 12_386_312
    assert bench.DN_BYTES == H * I // 2 + H * I // 16 + 4 == 6_193_156
    assert bench.GU_BYTES + bench.DN_BYTES + 3 * 4 == bench.EXPERT_BYTES


def test_roofline_byte_constants_match_the_census():
    """The bench's algorithmic bytes per touched expert (the roofline numerator) against the
    pages' byte census: one expert is 18,579,480 B; its gate/up part (two [I][H] tensors of
    E2M1 codes and E4M3 block scales per 16, plus two fp32 tensor scales) and its down part
    (one [H][I] tensor and its scale) add up to it with the three fp32 input scales that
    16-bit activations leave unused."""
    import bench
    with open(os.path.join(ROOT, "tests", "golden", "census.json")) as f:
        census = json.load(f)
    H, I = bench.K3["H"], bench.K3["I"]
    assert bench.EXPERT_BYTES == census["expert_bytes"] == 18_579_480
    assert bench.GU_BYTES == 2 * (H * I // 2 + H * I // 16) + 2 * 4 == 12_386_312
    assert bench.DN_BYTES == H * I // 2 + H * I // 16 + 4 == 6_193_156
    assert bench.GU_BYTES + bench.DN_BYTES + 3 * 4 == bench.EXPERT_BYTES

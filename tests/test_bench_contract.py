"""bench.py on the host: the byte and flop counts its roofline divides by,
against the closed forms of the Xing4 layer, and the reference arm's one
JSON line (the reference arm times the CPU oracle, so it runs without a
GPU)."""
import json
import os
import subprocess
import sys

import bench
from quantized_moe_expert_sigmoid_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_byte_counts_match_the_closed_forms():
    wl = synth.WORKLOADS["decode1"]
    # up + gate + down of one expert: 3 matrices of 1,024 x 3,584 weights at
    # 18 bytes per 32
    assert bench.expert_bytes_of(wl) == 3 * 1024 * 3584 // 32 * 18 == 6_193_152
    # batch 1: four routed experts + the shared one, the fp32 router, x in
    # and out in bf16
    assert bench.algorithmic_bytes(wl, 1, 4) == 5 * 6_193_152 + 64 * 3584 * 4 + 2 * 3584 * 2 == 31_897_600
    # everything a layer holds: 64 + 1 experts and the router
    assert 65 * bench.expert_bytes_of(wl) + wl.E * wl.H * 4 == 403_472_384


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["unit"] == d["e2e"]["unit"] == d["cpu_baseline"]["unit"] == "tokens/s"
    assert d["e2e"]["value"] == d["value"] == d["cpu_baseline"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert "workload" in d["config"]

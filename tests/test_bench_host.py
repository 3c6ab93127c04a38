"""Host-side checks of bench.py's arithmetic and output contract (no GPU):
the per-stage algorithmic FLOPs it divides by add up to the oracle's
per-token formula, and the reference arm prints one JSON line with the keys
the measurement contract asks for."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from efficient_attention_transformer_gb300.synthetic import WORKLOADS  # noqa: E402
from oracle import algorithmic_flops_per_token  # noqa: E402

BF16_STAGES = ("projection", "chunk_state_scan", "chunk_attention", "output")
FP32_STAGES = ("projection", "chunk_state", "prefix_scan", "chunk_attention", "output")


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_stage_flops_add_up_to_the_oracle_formula(name):
    w = WORKLOADS[name]
    work = bench.stage_work(w)
    stages = BF16_STAGES if w["dtype"] == "bf16" else FP32_STAGES
    total = sum(work[n][0] for n in stages)
    M = w["B"] * w["T"]
    # causal with one chunk in bf16: FLASH-Quad, no linear term is formed
    quad = w["causal"] and w["T"] == w["C"] and w["dtype"] == "bf16"
    want = M * algorithmic_flops_per_token(w["d"], w["e"], w["s"], w["C"], w["causal"],
                                           quad_only=quad)
    # the stages also count the scan's additions, B*G*s*e, which the
    # per-token formula leaves out
    extra = 0 if quad else w["B"] * (w["T"] // w["C"]) * w["s"] * w["e"]
    assert total == pytest.approx(want + extra, rel=1e-12)


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_causal_fp32_T256", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["value"] == rec["value"]

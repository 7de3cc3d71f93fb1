"""bench.py's default path end to end on the GPU, on a small batch.

Runs the bench as a child process with every block on (extended entry
points, end-to-end pass, CPU baseline, sustained loop) and parses its one
JSON line, so that an error anywhere in the default path fails the tests.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_default_bench_path_prints_a_complete_line(cuda_lib):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "2", "--warmup", "3",
           "--batch", "1", "--sustain-seconds", "0.3", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-4000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    for key in ("roofline", "roofline_fwd", "roofline_bwd_hbm", "e2e", "cpu_baseline", "clocks",
                "sustained", "extended", "gpu_launches"):
        assert line[key] is not None, key
    assert line["value"] > 0 and line["roofline"]["achieved"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    assert 0 < line["e2e"]["copy_bound"]["frac"] <= 1.5
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["sustained"]["steps"] > 0
    for name in ("graph_step", "bwd_deterministic", "dropout_0.1", "attn_bias", "varlen",
                 "head_dim_96", "head_dim_256", "pages_test", "encoder_dropout", "cross_attn"):
        assert name in line["extended"], name
    for name in ("dropout_0.1", "encoder_dropout", "cross_attn"):
        assert line["extended"][name]["alu_fwd"]["alu_bound_ms"] > 0, name
        assert line["extended"][name]["stored_bits"]["bwd_ms"] > 0, name

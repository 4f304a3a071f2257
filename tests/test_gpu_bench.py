"""The benchmark's own GPU legs at a small size, through the same code the timed runs use:
the single-GPU virtual-rank step and the multi-GPU (rank plan, NCCL exchange) step in a
one-rank group.  Each must print one JSON line that keeps the benchmark contract."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks",
        "e2e")


def _bench(*extra):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--seq", "4096",
                        "--steps", "2", "--warmup", "1", "--no-layer", "--no-ring", "--no-cpu",
                        *extra], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in KEYS:
        assert key in d, key
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 2
    assert d["config"]["seq_len"] == 4096 and d["e2e"]["value"] > 0
    assert d["gpu_launches"] == 12 * 2
    return d


def test_single_gpu_step_line():
    d = _bench()
    assert d["config"]["P"] == 8 and d["roofline"]["kernel"] == "ulysses_attn_bwd"


def test_multi_gpu_code_path_in_a_one_rank_group():
    d = _bench("--sharded")
    assert d["config"]["parallelism"] == "ulysses-sp1" and d["config"]["P"] == 1
    assert set(d["kernels_ms"]) >= {"exchange_qkv", "exchange_o", "exchange_do", "exchange_grads"}

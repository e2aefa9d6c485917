"""bench.py's work model on hand-countable cases (CPU)."""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_dense_flops_closed_form():
    # one head, L = 2: rows see 1 and 2 keys -> 3 (q.k, p.v) pairs of d MACs each
    assert bench.dense_flops([2], 1, d=128) == 4.0 * 128 * 3
    # the 128K Llama layer: 32 heads x 4 d x L(L+1)/2
    assert abs(bench.dense_flops([131072], 32) - 140.739e12) < 0.001e12


def test_causal_tiles_and_executed_flops():
    assert bench.causal_tiles([128], 1) == 1
    assert bench.causal_tiles([129], 2) == 2 * 3          # 2 tiles -> 1 + 2 per head
    assert bench.causal_tiles([131072], 32) == 32 * 1024 * 1025 // 2
    per_tile = 2.0 * 128 * 128 * 128
    # nothing skipped: QK^T and P.V on every causal tile
    assert bench.executed_flops([256], 1, 0) == per_tile * 2 * 3
    # everything but the first tile of each row skipped
    assert bench.executed_flops([256], 1, 1) == per_tile * (3 + 2)


def test_popcount():
    w = np.array([0, 1, 3, 0xFFFFFFFF], np.uint32)
    assert bench.popcount(w) == 0 + 1 + 2 + 32


def test_item_dense_flops_sums_to_layer():
    n = 16
    total = sum(bench.item_dense_flops(i) for i in range(n))
    assert total == bench.dense_flops([n * 128], 1)


def test_reference_arm_prints_one_contract_line():
    """The CPU reference arm (the oracle on a bounded sample) prints one JSON
    line with the contract's keys; the small single-head layer keeps it quick."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "C0", "--steps", "1", "--warmup", "0", "--ref-budget", "0.5"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]

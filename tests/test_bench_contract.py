"""Host-side contract checks: the reference (oracle) arm of bench.py prints one JSON line with
the fields the driver reads, and the sparse-MLA input generator makes well-formed rows."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle as O
from indexer_driven_sparse_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.slow
def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "dtype",
              "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert "workload" in d["config"]


def test_mla_workload_rows_are_well_formed():
    w = I.mla_workload(700, [64, 0, 5, 700], 16, seed=3)
    assert w.kv.shape == (700, 656) and w.kv.dtype == torch.uint8
    assert w.q.shape == (4, 16, 576) and w.q.dtype == torch.bfloat16
    codes = w.kv[:, :512].numpy()
    assert not np.any((codes & 0x7F) == 0x7F)                       # no NaN codes
    lat, rope = O.mla_rows_from_bytes(w.kv.numpy())
    assert np.all(np.isfinite(lat)) and np.all(np.isfinite(rope)) and np.abs(lat).max() < 1.0
    rows, n = w.rows.numpy(), w.n_rows.numpy()
    assert list(n) == [64, 0, 5, 700]
    for b in range(4):
        sel = rows[b, :n[b]]
        assert np.all(np.diff(sel) > 0) and (sel.size == 0 or (sel[0] >= 0 and sel[-1] < 700))
        assert np.all(rows[b, n[b]:] == -1)
    w2 = I.mla_workload(700, [64, 0, 5, 700], 16, seed=3)
    assert torch.equal(w.kv, w2.kv) and torch.equal(w.q, w2.q) and torch.equal(w.rows, w2.rows)

"""bench.py's reference arm (the oracle timed on the host) runs without a GPU:
its JSON line carries the contract's keys, for each workload, and under a
two-rank launch only rank 0 prints."""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT

ENV = dict(os.environ, CUDA_VISIBLE_DEVICES="")


def _line(out: str) -> dict:
    lines = [x for x in out.splitlines() if x.startswith("{")]
    assert len(lines) == 1, out
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["verify", "ngram", "tree_build"])
def test_reference_arm_json_line(workload):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
           "--workload", workload]
    r = subprocess.run(cmd, cwd=ROOT, env=ENV, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = _line(r.stdout)
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 1
    for key in ("metric", "unit", "higher_is_better", "scaling", "dtype", "data", "config"):
        assert key in d, key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_reference_arm_two_ranks_rank0_prints():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=ENV, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    d = _line(r.stdout)
    assert d["impl"] == "reference" and d["n_gpus"] == 2

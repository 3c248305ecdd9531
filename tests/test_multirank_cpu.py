"""The multi-rank path of bench.py without a GPU: two gloo ranks on CPU.

Each rank processes its own batch (weak scaling, no data-path collective);
the only cross-rank step is the host-side maximum of the timed region, and
rank 0 alone prints. The reference arm under torchrun prints one line from
rank 0 and the other ranks exit 0 without work.
"""

import json
import re
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
from rotary_position_embedding_gb300 import workloads as wl
dist.init_process_group("gloo")
rank, world, _ = bench.dist_env()
local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
total = bench.max_over_ranks(local_ms)
w = wl.WORKLOADS[wl.HEADLINE]
v, g = bench.aggregate_throughput(wl.algorithmic_bytes(w), w.numel, 100, total, world)
x0 = wl.make_inputs(w.with_shape(B=1, S=8), shard=rank)["x"]
print(json.dumps({{"rank": rank, "total": total, "value": v, "x00": float(x0.ravel()[0])}}), flush=True)
dist.destroy_process_group()
"""


def _torchrun(args, timeout=600):
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}"] + args
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=env)


def test_two_gloo_ranks_reduce_timing(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER.format(root=ROOT))
    r = _torchrun([str(script)])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [json.loads(m) for m in re.findall(r"\{[^{}]*\}", r.stdout)]
    assert len(lines) == 2
    by_rank = {d["rank"]: d for d in lines}
    assert by_rank[0]["total"] == by_rank[1]["total"] == 15.0       # the slowest rank sets the time
    from rotary_position_embedding_gb300 import workloads as wl
    w = wl.WORKLOADS[wl.HEADLINE]
    exp = 2 * wl.algorithmic_bytes(w) * 100 / 15e-3 / 1e9
    assert abs(by_rank[0]["value"] - exp) < 1e-9 * exp
    assert by_rank[0]["x00"] != by_rank[1]["x00"]                    # each rank has its own batch


def test_reference_arm_under_torchrun_prints_once():
    r = _torchrun(["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "0", "--gpus", "2"])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"

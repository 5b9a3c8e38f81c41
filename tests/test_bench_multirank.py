"""bench.py's multi-rank path (replicas only) with gloo ranks on the CPU.

Each rank times its own replica; rank 0 reports the whole-job rate from the
maximum time over ranks. Runs two real gloo processes on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
world, rank, local = bench.dist_env()
d = bench.init_dist(world, "gloo")
mine = [0.25, 0.75][rank]
mx = bench.max_over_ranks(mine, d)
print(json.dumps({{"rank": rank, "max": mx, "value": bench.aggregate(10, world, mx)}}), flush=True)
dist.destroy_process_group()
"""


def _run_ranks(code, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                   RANK=str(r), LOCAL_RANK=str(r), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_max_over_ranks_and_aggregate_with_gloo():
    outs = _run_ranks(WORKER.format(root=ROOT))
    for o in outs:
        d = json.loads(o.strip().splitlines()[-1])
        assert d["max"] == 0.75
        assert d["value"] == pytest.approx(2 * 10 / 0.75)


def test_reference_arm_prints_only_on_rank0():
    code = ("import sys; sys.path.insert(0, %r); import bench; "
            "bench.main(['--impl', 'reference', '--workload', 'tiny', '--steps', '1', '--warmup', '3', '--gpus', '2'])" % ROOT)
    outs = _run_ranks(code)
    line = json.loads(outs[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert outs[1].strip() == ""

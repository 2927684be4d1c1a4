"""The N>1 bench path on CPU: two gloo ranks, each timing its own replica, agree on the slowest
rank's time (the bench reports the max over ranks), and only rank 0 prints the reference line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


_RANK_SCRIPT = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
mine = 10.0 + 5.0 * rank          # each replica's own elapsed ms
got = bench.dist_max(mine)
bench.barrier()
print(json.dumps({{"rank": rank, "max": got, "env": bench.dist_env()}}), flush=True)
dist.destroy_process_group()
"""


def _launch(script, world=2):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_max_over_ranks_gloo():
    outs = _launch(_RANK_SCRIPT.format(root=ROOT))
    recs = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in recs) == [0, 1]
    for r in recs:
        assert r["max"] == 15.0
        assert r["env"][0] == 2


def test_reference_arm_rank0_only():
    """Under a 2-rank launch only rank 0 runs and prints the oracle (reference) line."""
    script = (
        "import sys, runpy; sys.argv = ['bench.py', '--impl', 'reference', '--config', 'tiny', "
        "'--steps', '1', '--warmup', '1']; sys.path.insert(0, %r); runpy.run_path(%r, run_name='__main__')"
        % (ROOT, os.path.join(ROOT, "bench.py")))
    outs = _launch(script)
    lines = [o.strip() for o in outs]
    printed = [ln for ln in lines if ln]
    assert len(printed) == 1
    rec = json.loads(printed[0].splitlines()[-1])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] == 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0

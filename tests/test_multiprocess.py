"""The multi-rank path of bench.py on CPU: two gloo ranks.

Token rows are independent, so several GPUs run replicas of the workload with
no data-path exchange; the only cross-rank operations are the timing barrier
and the max over ranks of the per-step time.  This checks them with two
processes on the CPU (world size 2, gloo, rendezvous on 127.0.0.1).
"""
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


_WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup()
bench.barrier(world)
t = bench.max_over_ranks(0.5 + rank, world)          # rank 1 is the slower one
total = bench.max_over_ranks(float(world), world)
print(json.dumps({{"rank": rank, "world": world, "max": t, "world_seen": total}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _launch(nproc, code):
    port = _free_port()
    procs = []
    for r in range(nproc):
        env = dict(os.environ, WORLD_SIZE=str(nproc), RANK=str(r), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=180)
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_two_rank_timing_collectives_on_gloo():
    outs = _launch(2, _WORKER.format(root=ROOT))
    lines = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["world"] == 2
        assert l["max"] == 1.5          # every rank reports the slowest rank's time
        assert l["world_seen"] == 2.0


def test_reference_arm_prints_only_on_rank_zero():
    # the reference arm (the CPU oracle) runs on rank 0 only; other ranks exit 0 silently
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); sys.argv = ['bench.py', '--impl', 'reference', "
            f"'--config', 'tiny', '--steps', '1', '--warmup', '1', '--ref-rows', '2']; "
            f"import bench; bench.main()")
    outs = _launch(2, code)
    printed = [o for o in outs if o.strip()]
    assert len(printed) == 1
    line = json.loads(printed[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("M,world", [(4096, 2), (16384, 4), (7, 2)])
def test_rows_split_into_replicas(M, world):
    # weak scaling keeps the per-rank workload fixed: each rank runs the whole
    # configured batch; the job's rows are world * M
    import bench
    cfg = dict(bench.CONFIGS["prefill"], M=M)
    assert bench.flops(cfg) * world == 2.0 * (M * world) * cfg["O"] * (cfg["N"] + cfg["P"])

"""The multi-GPU path of bench.py is replicas only: every rank runs its own copy
of the layer, ranks meet at a barrier before and after the timed region, and
the job time is the maximum over ranks (the optimizer state of different
matrices is independent, so there is no data-path collective).  These checks
run the host logic with two gloo ranks on CPU."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, %(root)r)
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
t = bench.max_over_ranks(10.0 + 5.0 * rank, True)
dist.barrier()
print(json.dumps({"rank": rank, "max": t}), flush=True)
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(WORKER % {"root": ROOT})
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    import json
    vals = sorted(json.loads(o.strip().splitlines()[-1])["max"] for o, _ in outs)
    assert vals == [15.0, 15.0]


def test_reference_arm_prints_only_on_rank_zero():
    import bench
    args = type("A", (), {"steps": 1, "warmup": 3})()
    assert bench.run_reference(args, rank=1, world=2) is None


def test_single_rank_helpers_need_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, False) == 3.5
    # square: P_R G^T then P_L T (two n^3 products)
    assert bench.gemm_flops(2048, 2048) == 2 * (2.0 * 2048 ** 3)
    # tall and wide are mirror images: 2 r L n + 2 r^3 + 2 L n r with r = min, L = max
    assert bench.gemm_flops(8192, 2048) == bench.gemm_flops(2048, 8192) == 4.0 * 8192 * 2048 ** 2 + 2.0 * 2048 ** 3

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


def test_bench_gpus_flag_launches_the_ranks_itself():
    """`bench.py --gpus 2` run as a single process starts two ranks over gloo;
    rank 0 alone prints the line, with n_gpus = 2 and the slower rank's time
    (rank 1 works 30 ms, rank 0 20 ms, in the host-only stand-in)."""
    import json
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run",
                          "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=180,
                         env={k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK")})
    assert res.returncode == 0, res.stderr
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2 and out["dry_run"]
    assert out["ms_per_step"] * out["steps"] >= 30.0
    assert out["value"] == pytest.approx(2 * out["steps"] / (out["ms_per_step"] * out["steps"] * 1e-3))

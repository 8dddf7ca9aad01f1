"""Host-side pieces of bench.py: the byte model, the multi-rank aggregation and the
reference arm (the fp64 oracle on the host's cores, which needs no GPU).

bench.py runs one independent replica per GPU under torchrun (the sparse path
shards by token with no exchange); the only cross-rank step is the max of the
timed values, checked here with two gloo ranks on CPU.
"""
import os

import pytest
import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes_model():
    per_tok = 64 * 576 * 2 + 640 * 4 + 640 * 1152
    assert bench.algorithmic_bytes(1, 1) == per_tok + 64 * 512 + 256
    assert bench.algorithmic_bytes(1, 8, "split") == per_tok + 8 * (131072 + 256)
    assert bench.algorithmic_bytes(1, 8, "call") == per_tok + 2 * 8 * (131072 + 256) + 64 * 512 + 256
    assert bench.algorithmic_bytes(96, 1) == 96 * (per_tok + 32768 + 256)


def test_sweep_point_bytes_use_the_plans_split_count():
    """A swept point's bytes come from the schedule the plan runs: the planner's point
    (requested count 0) counts the partials of the splits it actually uses."""
    per_tok = 64 * 576 * 2 + 640 * 4 + 640 * 1152
    # s_q = 1, the planner's 5 splits: 813,568 + 2 * 5 * 131,328 + 33,024 = 2,159,872 B
    assert bench.point_bytes(1, 5, False, 152) == 2_159_872
    assert bench.point_bytes(1, 5, False, 152) == per_tok + 2 * 5 * (131072 + 256) + 64 * 512 + 256
    assert bench.point_bytes(96, 1, False, 152) == bench.algorithmic_bytes(96, 1)
    assert bench.point_bytes(96, 1, True, 152) == bench.balanced_bytes(96, 152)


def test_single_process_max_is_identity():
    assert bench.max_over_ranks([1.5, 2.0]) == [1.5, 2.0]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = [10.0 + rank, 5.0 - rank]
    out = bench.max_over_ranks(vals)
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 5.0]


def test_reference_arm_line_on_cpu():
    """bench.py --impl reference times the fp64 oracle on the host's cores and prints the contract's
    line (impl, metric, unit, value, cpu_baseline, e2e with no copies); a rank other than 0 prints
    nothing and exits 0."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "us/call" and line["higher_is_better"] is False
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "us/call", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r1 = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root, env=env)
    assert r1.returncode == 0 and r1.stdout.strip() == ""

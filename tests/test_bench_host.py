"""Host logic of bench.py: rank aggregation over 2 gloo ranks on CPU, and the
JSON contract of the reference arm (the oracle, on a small step count)."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.dist_init(world, "gloo")
    bench.barrier(d)
    mx = bench.max_over_ranks(d, 10.0 + rank)
    sm = bench.sum_over_ranks(d, 1.0 + rank)
    bench.barrier(d)
    q.put((rank, mx, sm))
    d.destroy_process_group()


def test_two_gloo_ranks_take_max_and_sum():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 300
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 11.0, 3.0), (1, 11.0, 3.0)]


@pytest.mark.parametrize("seed", [None, 7])
def test_reference_arm_json_line(seed):
    extra = [] if seed is None else ["--seed", str(seed)]
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "1", *extra],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["seed"] == (152 if seed is None else seed)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_unique_kv_bytes_counts_shared_blocks_once():
    """The prefix workload's DRAM-side byte count: a block two tables share is
    counted once, with the most rows any sequence reads from it."""
    sys.path.insert(0, ROOT)
    import bench
    # block 5 is shared (full, 16 rows); blocks 7 and 9 are private tails
    tables = [[5, 7, -1], [5, 9, -1]]
    lens = [20, 30]                      # 16 + 4 rows, 16 + 14 rows
    per_row = 2 * 2 * 128 * 2            # K and V, 2 KV heads, head_dim 128, fp16
    assert bench.unique_kv_bytes(tables, lens, 16, 2, 128) == (16 + 4 + 14) * per_row
    # without sharing it is the logical count
    assert bench.unique_kv_bytes([[1, 2], [3, 4]], lens, 16, 2, 128) == (20 + 30) * per_row

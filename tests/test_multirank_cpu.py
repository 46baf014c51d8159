"""The benchmark's multi-process path on CPU (gloo, world_size 2, 127.0.0.1).

The path shards by sequence with no exchange step: N processes run N
independent replicas, and only the timing and the totals cross ranks (a
barrier, a max of the step times, a sum of the work).  These tests run that
host logic in two processes without a GPU, and the reference arm under
torch.distributed.run, where rank 0 alone times the oracle and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    sys.path.insert(0, ROOT)
    import importlib
    return importlib.import_module("bench")


def _worker(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    bench = _load_bench()
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    res = {"max": bench.max_over_ranks(1.5 + rank, w), "sum": bench.sum_over_ranks(1.0 + rank, w)}
    import torch.distributed as dist
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump(res, f)


def test_rank_collectives_gloo(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert res["max"] == 2.5   # max over ranks of 1.5 + rank
        assert res["sum"] == 3.0   # sum over ranks of 1 + rank


def test_single_rank_helpers_are_identities():
    bench = _load_bench()
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.sum_over_ranks(4.25, 1) == 4.25
    bench.barrier(1)


@pytest.mark.parametrize("name", ["gqa_decode", "long_mqa", "chunked_prefill"])
def test_rank_plans_are_weak_scaling_replicas(name):
    bench = _load_bench()
    p0, p1, p2 = (bench.rank_plan(name, r) for r in range(3))
    for p in (p1, p2):
        assert (p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.page_size) == \
            (p0.batch, p0.num_q_heads, p0.num_kv_heads, p0.head_dim, p0.page_size)
    # each rank draws its own batch (rank 0 is the named workload itself)
    assert not (p0.seq_lens == p1.seq_lens).all() or not (p0.block_table == p1.block_table).all()
    assert not (p1.seq_lens == p2.seq_lens).all() or not (p1.block_table == p2.block_table).all()


def test_reference_arm_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_first_sequences_is_a_compact_prefix_of_the_batch():
    bench = _load_bench()
    full = bench.rank_plan("long_gqa", 0)
    small = bench.rank_plan("long_gqa", 0, batch=16)
    assert small.batch == 16 and (small.seq_lens == full.seq_lens[:16]).all()
    assert (small.num_q_heads, small.num_kv_heads, small.head_dim) == (32, 8, 128)
    used = sum((int(L) + 15) // 16 for L in small.seq_lens)
    assert small.num_pages == used + -(-used // 10)       # its own pool: used pages + 10 % free
    assert bench.rank_plan("gqa_decode", 0, batch=0).batch == 32
    with pytest.raises(ValueError):
        bench.rank_plan("shared_prefix", 0, batch=8)      # shared pages cannot be cut


def test_cpu_baseline_legs_report_all_cores_and_one_thread():
    """The oracle CPU baseline runs in subprocesses with the BLAS thread count
    fixed through the environment: every core, then one thread."""
    bench = _load_bench()
    cpu = bench.cpu_baseline("gqa_decode", 2, 0.05, "decode")
    assert cpu["kind"] == "oracle" and cpu["unit"] == "GB/s" and cpu["value"] > 0
    assert cpu["cores"] == bench.cpu_cores() and cpu["one_thread"]["cores"] == 1
    assert cpu["one_thread"]["value"] > 0 and cpu["full_step_s_extrapolated"] > 0
    assert "first 2/2 sequences" in cpu["sample"]

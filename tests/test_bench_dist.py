"""Multi-rank paths of bench.py on CPU (gloo, world size 2).

The step has no cross-rank exchange: N ranks run N independent replicas, the
slowest rank's time is the job's time and rank 0 alone prints the JSON line.
These tests run the host-side rank logic with the gloo backend (no GPU): the
barrier and max-over-ranks helpers, and the reference arm under torchrun,
where rank 0 prints one line and every other rank exits 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(bench.parse_args([]))
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank's step time differs; the job takes the slowest
    got = bench.max_over_ranks(1.5 + rank, w, "cpu")
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, got))


def test_barrier_and_max_over_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(world))
    assert res == {0: 2.5, 1: 2.5}


def test_single_rank_helpers_need_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(1)
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_reference_arm_under_torchrun_prints_on_rank0_only():
    import oracle
    oracle.build()
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "tiny", "--cpu-seconds", "0.5"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
    # the same workload description as the GPU arm prints, so the two lines compare
    sys.path.insert(0, ROOT)
    import bench
    from block_diffusion_speculative_attn_gb300 import workloads as wl
    assert line["config"] == bench.config_dict(wl.config("tiny"), 2)


def test_accept_bytes_count_the_rows_each_outcome_reads():
    sys.path.insert(0, ROOT)
    import bench
    from block_diffusion_speculative_attn_gb300 import workloads as wl
    cfg = wl.config("qwen3_8b_verify")
    B, V = cfg.B, cfg.V
    small = 4 * (B + (B - 1) + 2) + 4 * (B + 4)
    # a rejection at slot 3 reads 4 pairs and the p and q rows there; a fully
    # accepted row reads B - 1 pairs and the bonus row of p alone
    assert bench.accept_bytes_exact(cfg, [3]) == small + 8 * 4 + 2 * V * 4
    assert bench.accept_bytes_exact(cfg, [B - 1]) == small + 8 * (B - 1) + V * 4
    assert bench.accept_bytes_exact(cfg, [0, B - 1]) == (bench.accept_bytes_exact(cfg, [0]) +
                                                         bench.accept_bytes_exact(cfg, [B - 1]))

"""The benchmark's multi-rank path on the CPU: two gloo ranks (127.0.0.1).
Under torchrun every rank runs its own batch -- weak scaling with no
collective on the data path -- and the job's time is the slowest rank's, its
bytes the sum over ranks; rank 0 alone prints.  No GPU is involved."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, REPO)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, nbytes = bench.reduce_over_ranks(dist, 10.0 + 5.0 * rank, 100.0 * (rank + 1))
        dist.barrier()
        q.put((rank, ms, nbytes))
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_with_two_gloo_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_reduce_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], f"ranks exited with {codes}"
    got = sorted(q.get(timeout=10) for _ in range(2))
    # both ranks see the slowest time and the bytes of both
    assert got == [(0, 15.0, 300.0), (1, 15.0, 300.0)]


def test_single_process_reduction_is_identity():
    sys.path.insert(0, REPO)
    import bench
    assert bench.reduce_over_ranks(None, 3.5, 1e9) == (3.5, 1e9)


def test_each_rank_gets_its_own_batch():
    """Same shapes, different seeded data per rank (weak scaling)."""
    sys.path.insert(0, REPO)
    import bench
    from paged_kv_cache_24_gb300.workloads import make_workload
    specs = [bench.rank_spec("gqa_bf16", r, num_seqs=6) for r in range(2)]
    assert specs[0].seed != specs[1].seed
    ws = [make_workload(s, device="cpu", poison=False) for s in specs]
    for a in ("num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "block_size", "dtype"):
        assert getattr(specs[0], a) == getattr(specs[1], a)
    assert not torch.equal(ws[0].lens_steps, ws[1].lens_steps)
    assert not torch.equal(ws[0].q_steps, ws[1].q_steps)


def test_reference_arm_under_torchrun_rank0_prints_other_ranks_exit(tmp_path):
    """`bench.py --impl reference` as the driver launches it for N = 2: the
    oracle runs on rank 0 only and one JSON line is printed; rank 1 exits 0
    without work."""
    pytest.importorskip("torch.distributed.run")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(REPO, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny_fp32", "--steps", "1", "--warmup", "0",
           "--reference-seconds", "2"]
    r = subprocess.run(cmd, cwd=REPO, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and np.isfinite(line["value"])

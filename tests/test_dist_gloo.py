"""Multi-process paths of bench.py on CPU with the gloo backend (world size 2).

Rows are independent, so N GPUs run N replica batches with no collective on
the data path; the only cross-rank step is the max over ranks of the timed
region.  These tests exercise that host logic without a GPU.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.max_over_ranks(10.0 + 5.0 * rank)
    wl = bench.build_workload("tiny", rank)
    out.put((rank, m, bench.dist_env(), float(wl.q.float().sum())))
    dist.destroy_process_group()


def test_max_over_ranks_and_replica_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]          # slowest rank's time on both
    assert [r[2] for r in res] == [(0, 2, 0), (1, 2, 1)]
    assert res[0][3] != res[1][3]                         # each rank its own replica batch


def test_replica_value_is_whole_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 1000 units in a 2 ms slowest step = 1e6 units/s
    assert bench.replica_value(1000, 2, 2.0) == pytest.approx(1e6)


def test_e2e_staging_views_round_trip():
    # the end-to-end leg stages q, lengths and the page table in one buffer
    # (one copy per step): every view must land on a 256-byte boundary and
    # read back exactly what was written into it
    sys.path.insert(0, ROOT)
    import torch
    import bench
    specs = [((8, 32, 128), torch.bfloat16), ((8,), torch.int32), ((3, 1000), torch.int32)]
    buf = torch.zeros(bench.packed_bytes(specs), dtype=torch.uint8)
    src = [torch.randn(8, 32, 128).to(torch.bfloat16), torch.arange(8, dtype=torch.int32),
           torch.randint(-5, 100, (3, 1000), dtype=torch.int32)]
    for v, t in zip(bench.packed_views(buf, specs), src):
        v.copy_(t)
    views = bench.packed_views(buf, specs)
    for v, t in zip(views, src):
        assert v.is_contiguous() and v.dtype == t.dtype and torch.equal(v, t)
        assert (v.data_ptr() - buf.data_ptr()) % 256 == 0
    assert buf.numel() == 65536 + 256 + 12032  # 32 B and 12000 B pieces padded to 256


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "3",
           "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"

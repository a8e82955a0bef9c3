"""The benchmark's multi-rank plumbing on CPU: two gloo ranks take the
maximum step time over the ranks and report the whole-job throughput; the
reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._DIST["on"] = True
    ms = bench._max_over_ranks(1.5 + rank)          # rank r's step took 1.5 + r ms
    bench._barrier()
    q.put((rank, ms, bench._aggregate_gbs(1_000_000_000, ms, world)))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs in got:
        assert ms == 2.5                               # the slowest rank
        assert abs(gbs - 800.0) < 1e-9                 # 2 x 1 GB in 2.5 ms


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_roofline_traffic_only_from_a_summary_of_the_current_source(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu summary only while its
    recorded source hash matches the kernel source; otherwise it is null."""
    sys.path.insert(0, ROOT)
    import hashlib
    import bench
    t = bench._profiled_traffic()
    cur = hashlib.sha256(open(bench.KERNEL_SRC, "rb").read()).hexdigest()
    recorded = open(bench.PROFILE_SUMMARY).read()
    if f"kernel_source_sha256: {cur}" in recorded:
        # a full launch reads at least its algorithmic KV bytes
        assert t is not None and t >= 16 * 16384 * 8 * 256
    else:
        assert t is None
    changed = tmp_path / "pa_fp8.cu"
    changed.write_bytes(open(bench.KERNEL_SRC, "rb").read() + b"\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", str(changed))
    assert bench._profiled_traffic() is None

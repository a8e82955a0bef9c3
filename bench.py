#!/usr/bin/env python3
"""Benchmark of the quantised paged-attention decode hot path on GB300.

Metric: paged-decode microseconds per step and KV-cache GB/s (as a fraction
of the measured HBM peak) at 1 GPU. A step is one decode over the whole
batch: the partition kernel and the combine kernel of pa_decode_fp8 on the
16 seqs x 16384 tokens, 8 KV heads, group 8, head_dim 128, block 16 workload
with 512-token partitions (P = 32). Inputs are seeded synthetic data, resident
in HBM when the timed region starts; the 537 MB KV stream is larger than L2.

  python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

Prints one JSON line. Under torchrun (N > 1) every rank runs an independent
replica (no collective on the data path) and rank 0 reports the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-decode µs/step and KV-cache GB/s (% of GB300 HBM peak) at 1 GPU"
WORKLOAD = ("fp8 paged decode: 16 seqs x 16384 tokens, 8 KV heads, query group 8 (64 q heads), "
            "head_dim 128, block_size 16, random-permutation block table, P=32 (512-token partitions)")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "pa_fp8_partition_gqa16x16k.md")
KERNEL_SRC = os.path.join(ROOT, "quantized_paged_attention_gb300", "csrc", "pa_fp8.cu")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads' measurements")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile-case", choices=["fp8", "uq", "uq_rand", "idx"], default=None,
                    help="run only this case's kernels (warmup + steps launches) for a profiler; "
                         "fp8: 8 seqs x 16384 (268 MB), uq: 4 seqs x 75000 (173 MB), "
                         "idx: 128 requests (170 MB); prints one status line, not the bench line")
    return ap.parse_args()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        if not sm:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if len(r) > 5 + i and "Active" in r[5 + i] and "Not" not in r[5 + i]:
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ traffic from the committed ncu summary
def _profiled_traffic():
    """Per-launch DRAM bytes of the partition kernel from the committed ncu
    summary, if it was taken on the current kernel source (hash match)."""
    try:
        txt = open(PROFILE_SUMMARY).read()
        h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", txt).group(1)
        t = float(re.search(r"dram_bytes_per_launch_full_workload:\s*([0-9.eE+]+)", txt).group(1))
        cur = hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()
        return t if cur == h else None
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle baseline
def _oracle_unit(args):
    """Oracle on one (seq, kv_head) unit, re-packed as a single-sequence case."""
    import numpy as np
    import oracle
    q_bits, kv_blocks, L, k_scale, v_scale, qg, scale = args
    nb = kv_blocks.shape[0]
    bt = np.arange(nb, dtype=np.int32)[None, :]
    oracle.pa_decode_fp8(q_bits, kv_blocks, bt, np.array([L], dtype=np.int32), k_scale, v_scale, qg, scale)
    return L * 2 * kv_blocks.shape[2] * kv_blocks.shape[4]


def _unit_args(c, s, h):
    import numpy as np
    L = int(c.seq_lens[s])
    nb = (L + c.block_size - 1) // c.block_size
    blocks = c.kv_cache[c.block_table[s, :nb]][:, :, h:h + 1]          # [nb, 2, 1, bs, D]
    qg = c.query_group
    q = c.q_bits[s:s + 1, h * qg:(h + 1) * qg]
    return (np.ascontiguousarray(q), np.ascontiguousarray(blocks), L, c.k_scale, c.v_scale, qg, c.softmax_scale)


class OraclePool:
    """The float64 oracle on (seq, kv_head) units of a workload, spread over a
    spawn-started process pool on the host cores (one worker per core)."""

    def __init__(self, c):
        import multiprocessing as mp
        self.c = c
        self.cores = os.cpu_count() or 1
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"          # one BLAS thread per worker process
        self.pool = mp.get_context("spawn").Pool(self.cores)
        self.units = [(s, h) for s in range(c.num_seqs) for h in range(c.num_kv_heads)]
        self.next = 0
        self.pool.map(_oracle_unit, [_unit_args(c, 0, 0)] * self.cores)     # warm the workers

    def run(self, n):
        """Runs the next n units; returns (KV bytes, seconds)."""
        sel = [self.units[(self.next + i) % len(self.units)] for i in range(n)]
        self.next = (self.next + n) % len(self.units)
        args = [_unit_args(self.c, s, h) for s, h in sel]
        t0 = time.perf_counter()
        b = sum(self.pool.map(_oracle_unit, args, chunksize=1))
        return b, time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


# ------------------------------------------------------------------ GPU timing
def _device_inputs(c, dev):
    import numpy as np
    import torch
    return dict(
        q=torch.from_numpy(c.q_bits.view(np.int16)).view(torch.bfloat16).to(dev),
        kv=torch.from_numpy(c.kv_cache).to(dev),
        bt=torch.from_numpy(c.block_table).to(dev),
        sl=torch.from_numpy(c.seq_lens).to(dev),
        ks=torch.tensor([c.k_scale], dtype=torch.float32, device=dev),
        vs=torch.tensor([c.v_scale], dtype=torch.float32, device=dev))


def time_fp8(c, P, steps, warmup, dev, sampler=None):
    """Times `steps` decode steps (partition then combine) back to back on the
    current stream with CUDA events only at the two ends of the timed region,
    so that the combine kernel's programmatic dependent launch overlaps the
    partition kernel's tail as it does in use (an event recorded between the
    two kernels would serialise them). A second pass of `steps` partition-only
    launches, each between its own pair of CUDA events on the same stream,
    gives the partition kernel's duration for the roofline. Returns (ms per
    step, mean partition-kernel ms, step ms minus partition ms, kernel
    launches in the timed step loop, clocks, total ms of the step loop)."""
    import torch
    import quantized_paged_attention_gb300 as qpa
    x = _device_inputs(c, dev)
    desc = qpa.fp8_desc(x["q"], x["kv"], x["bt"], c.query_group, c.softmax_scale)
    ws = qpa.alloc_workspace(qpa.pa_decode_fp8_workspace_size(desc, P), dev)
    out = torch.empty(x["q"].shape, dtype=torch.float32, device=dev)
    args = (x["q"], x["kv"], x["bt"], x["sl"], x["ks"], x["vs"], P, desc, ws)
    for _ in range(warmup):
        qpa.pa_decode_fp8_partition(*args)
        qpa.pa_decode_fp8_combine(P, out, desc, ws)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.05)
    start.record()
    for i in range(steps):
        qpa.pa_decode_fp8_partition(*args)
        qpa.pa_decode_fp8_combine(P, out, desc, ws)
    end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    _barrier()
    total = start.elapsed_time(end)
    # the partition kernel alone, each launch between its own events
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record()
        qpa.pa_decode_fp8_partition(*args)
        ev[i][1].record()
    torch.cuda.synchronize()
    part = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if qpa.kernel_error() != 0:
        raise RuntimeError("device error word raised during the benchmark")
    return total / steps, part, total / steps - part, 2 * steps, clocks, total


def time_fp8_ext(c, P, steps, warmup, dev):
    """Times `steps` calls of pa_decode_fp8_ext (partition + combine) back to
    back between two CUDA events (the cache, 537 MB, is larger than L2)."""
    import numpy as np
    import torch
    import quantized_paged_attention_gb300 as qpa
    q = torch.from_numpy(c.q_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    kv = torch.from_numpy(c.kv_cache).to(dev)
    bt = torch.from_numpy(c.block_table).to(dev)
    sl = torch.from_numpy(c.seq_lens).to(dev)
    if c.per_token:
        ks = torch.from_numpy(np.ascontiguousarray(c.k_scale)).to(dev)
        vs = torch.from_numpy(np.ascontiguousarray(c.v_scale)).to(dev)
    else:
        ks = torch.tensor([c.k_scale], dtype=torch.float32, device=dev)
        vs = torch.tensor([c.v_scale], dtype=torch.float32, device=dev)
    desc = qpa.fp8_ext_desc(q, kv, bt, c.query_group, c.per_token, c.softmax_scale)
    ws = qpa.alloc_workspace(qpa.pa_decode_fp8_ext_workspace_size(desc, P), dev)
    out = torch.empty(tuple(q.shape), dtype=torch.float32, device=dev)

    def step():
        qpa.pa_decode_fp8_ext(q, kv, bt, sl, ks, vs, P, c.query_group, out=out, workspace=ws, desc=desc)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier()
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    _barrier()
    if qpa.kernel_error() != 0:
        raise RuntimeError("device error word raised during the benchmark")
    return a.elapsed_time(b) / steps


def _time_loop(step_a, step_b, steps, warmup):
    """Times `steps` steps (step_a = partition or whole kernel, step_b =
    combine or None) with L2 flushed before every step: a 256 MB buffer, larger
    than the 129 MB L2, is written and then read back between steps outside the
    timed spans (these workloads are small enough to stay partly cached
    otherwise). The read leaves L2 holding clean lines, so the timed kernel does
    not pay for writing back the flush's dirty lines. A step is timed between
    two CUDA events with nothing between its kernels; with a step_b, a second
    pass times step_a alone the same way. Returns (mean ms per step, mean ms
    of step_a)."""
    import torch
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=torch.cuda.current_device())
    flush_words = flush.view(torch.int32)

    def flush_l2():
        flush.zero_()
        flush_words.sum()

    for _ in range(warmup):
        flush_l2()
        step_a()
        if step_b:
            step_b()
    torch.cuda.synchronize()

    def timed(fns):
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(steps)]
        _barrier()
        torch.cuda.synchronize()
        for i in range(steps):
            flush_l2()
            ev[i][0].record()
            for fn in fns:
                fn()
            ev[i][1].record()
        torch.cuda.synchronize()
        _barrier()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    step = timed([step_a, step_b] if step_b else [step_a])
    return step, (timed([step_a]) if step_b else step)


def time_uq(c, P, steps, warmup, dev, q_haircut=False):
    import numpy as np
    import torch
    import quantized_paged_attention_gb300 as qpa
    q = torch.from_numpy(c.q_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    kv = torch.from_numpy(c.kv_cache).to(dev)
    cent = torch.from_numpy(np.ascontiguousarray(c.centroids, dtype=np.float32)).to(dev)
    bt = torch.from_numpy(c.block_table).to(dev)
    sl = torch.from_numpy(c.seq_lens).to(dev)
    desc = qpa.uq_desc(q, kv, bt, c.query_group, c.softmax_scale, scale_format=c.scale_format,
                       q_haircut=q_haircut, rot_perm=c.rot_perm)
    ws = qpa.alloc_workspace(qpa.uq_decode_hd256_workspace_size(desc, P), dev)
    out = torch.empty((q.shape[0], q.shape[1], 256), dtype=torch.float32, device=dev)
    r = _time_loop(lambda: qpa.uq_decode_hd256_partition(q, kv, cent, bt, sl, P, desc, ws),
                   lambda: qpa.uq_decode_hd256_combine(P, out, desc, ws), steps, warmup)
    if qpa.kernel_error() != 0:
        raise RuntimeError("device error word raised during the benchmark")
    return r


def time_idx(c, steps, warmup, dev, per_token_cols=None):
    import torch
    import quantized_paged_attention_gb300 as qpa
    q = torch.from_numpy(c.q_codes).to(dev)
    pages = torch.from_numpy(c.pages).to(dev)
    bt = torch.from_numpy(c.block_table).to(dev)
    sl = torch.from_numpy(c.seq_lens).to(dev)
    cols = c.num_cols if per_token_cols is None else per_token_cols
    scores = torch.empty((c.num_heads, q.shape[0], cols), dtype=torch.float32, device=dev)
    desc = qpa.idx_desc(q, pages, bt, c.query_len, cols, scores, per_token=per_token_cols is not None)
    r = _time_loop(lambda: qpa.nvfp4_index_score(q, pages, bt, sl, c.query_len, cols, scores=scores,
                                                 desc=desc), None, steps, warmup)
    if qpa.kernel_error() != 0:
        raise RuntimeError("device error word raised during the benchmark")
    return r


def time_e2e(c, P, steps, dev):
    """The same decode through the C ABI from pinned host buffers: every step
    copies all inputs host->device, runs the step and copies the output back."""
    import numpy as np
    import torch
    import quantized_paged_attention_gb300 as qpa
    h = dict(q=torch.from_numpy(c.q_bits.view(np.int16)).view(torch.bfloat16).pin_memory(),
             kv=torch.from_numpy(c.kv_cache).pin_memory(),
             bt=torch.from_numpy(c.block_table).pin_memory(),
             sl=torch.from_numpy(c.seq_lens).pin_memory(),
             ks=torch.tensor([c.k_scale], dtype=torch.float32).pin_memory(),
             vs=torch.tensor([c.v_scale], dtype=torch.float32).pin_memory())
    d = {k: torch.empty_like(v, device=dev) for k, v in h.items()}
    desc = qpa.fp8_desc(d["q"], d["kv"], d["bt"], c.query_group, c.softmax_scale)
    ws = qpa.alloc_workspace(qpa.pa_decode_fp8_workspace_size(desc, P), dev)
    out = torch.empty(d["q"].shape, dtype=torch.float32, device=dev)
    out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = out.numel() * out.element_size()

    def step():
        for k in h:
            d[k].copy_(h[k], non_blocking=True)
        qpa.pa_decode_fp8(d["q"], d["kv"], d["bt"], d["sl"], d["ks"], d["vs"], P, c.query_group, out=out,
                          workspace=ws, desc=desc)
        out_h.copy_(out, non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    _barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        step()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


# ------------------------------------------------------------------ distributed plumbing
_DIST = {"on": False}


def _barrier():
    if _DIST["on"]:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x):
    """The largest x over the ranks (each rank times its own replica; the job
    takes as long as the slowest)."""
    if not _DIST["on"]:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _aggregate_gbs(bytes_per_rank, ms_max, world):
    """Whole-job throughput: the bytes all ranks processed (every rank runs a
    replica of the workload) over the slowest rank's time per step."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def _profile_case(a):
    """Small cases (larger than L2) of each kernel for profiling runs."""
    import numpy as np
    import torch
    import synth
    dev = torch.device("cuda", 0)
    if a.profile_case == "fp8":
        c = synth.make_fp8_case(1001, [16384] * 8, 8, 8, 128, 16, poison=False)
        ms, part, *_ = time_fp8(c, 32, a.steps, a.warmup, dev)
        nbytes = c.kv_bytes
    elif a.profile_case in ("uq", "uq_rand"):
        cent = synth.sorted_random_centroids(5) if a.profile_case == "uq_rand" else None
        c = synth.uq_full(centroids=cent)
        ms, part = time_uq(c, 147, a.steps, a.warmup, dev)
        nbytes = c.kv_bytes
    else:
        r = synth.rng(1104)
        c = synth.make_idx_case(1004, r.integers(4096, 32769, size=128).astype(np.int32), 4, 2,
                                num_cols=256, poison=False)
        ms, part = time_idx(c, a.steps, a.warmup, dev)
        nbytes = c.kv_bytes
    print(f"profile case {a.profile_case}: {ms * 1e3:.1f} us/step, first kernel {part * 1e3:.1f} us, "
          f"{nbytes / 1e6:.1f} MB, {nbytes / (part * 1e-3) / 1e9:.0f} GB/s")


def main():
    a = _args()
    if a.warmup < 3:
        a.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    import synth

    if a.impl == "reference":
        # The reference arm is the float64 CPU oracle, on the host cores, rank 0
        # only; each step is one batch of (seq, kv_head) units of the workload.
        if rank != 0:
            return
        c = synth.fp8_gqa()
        pool = OraclePool(c)
        n = pool.cores
        tot_b, tot_t = 0, 0.0
        for i in range(a.warmup + a.steps):
            b, t = pool.run(n)
            if i >= a.warmup:
                tot_b += b
                tot_t += t
        pool.close()
        val = tot_b / tot_t / 1e9
        sample = (f"{n} (seq, kv_head) units ({n * c.kv_bytes // (c.num_seqs * c.num_kv_heads) / 1e6:.0f} MB "
                  f"of KV) per step, float64 numpy oracle, spawn pool of {pool.cores} workers")
        line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
                "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
                "ms_per_step": round(tot_t / a.steps * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOAD, "reference": "float64 CPU oracle (oracle/), host cores"},
                "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": pool.cores,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    if a.profile_case:
        _profile_case(a)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        _DIST["on"] = True
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peak, peak_kind = _peaks()

    c = synth.fp8_gqa(seed=1001 + rank)
    P = 32
    sampler = ClockSampler(local) if rank == 0 else None
    ms, part_ms, comb_ms, launches, clocks, total_ms = time_fp8(c, P, a.steps, a.warmup, dev, sampler)
    ms_max = _max_over_ranks(ms)
    kv = c.kv_bytes
    value = _aggregate_gbs(kv, ms_max, world)
    part_gbs = kv / (part_ms * 1e-3) / 1e9

    e2e = None
    if not a.no_e2e:
        e_ms, h2d, d2h = time_e2e(c, P, max(3, min(a.steps, 10)), dev)
        e_ms = _max_over_ranks(e_ms)
        e2e = {"value": round(_aggregate_gbs(kv, e_ms, world), 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 4)}

    extra = {}
    if not a.no_extra:
        cr = synth.fp8_ragged(seed=1002 + rank)
        r_ms, r_part, _, _, _, _ = time_fp8(cr, 32, max(20, a.steps // 4), a.warmup, dev)
        r_ms = _max_over_ranks(r_ms)
        extra["fp8_ragged_b128"] = {
            "workload": "fp8 paged decode, 128 seqs, lengths U[1024,16384], 8 KV heads, group 8, block 16, P=32",
            "us_per_step": round(r_ms * 1e3, 2), "partition_us": round(r_part * 1e3, 2),
            "kv_bytes": cr.kv_bytes, "gbs": round(cr.kv_bytes / (r_ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round(cr.kv_bytes / (r_ms * 1e-3) / 1e9 / peak, 4)}
        del cr
        c64 = synth.make_fp8_case(1006 + rank, [16384] * 16, 8, 8, head_dim=64, poison=False)
        h_ms, h_part, _, _, _, _ = time_fp8(c64, 32, max(20, a.steps // 4), a.warmup, dev)
        h_ms = _max_over_ranks(h_ms)
        extra["fp8_b16_16k_hd64"] = {
            "workload": "fp8 paged decode, 16 seqs x 16384 tokens, 8 KV heads, group 8, head_dim 64, block 16, P=32",
            "us_per_step": round(h_ms * 1e3, 2), "partition_us": round(h_part * 1e3, 2),
            "kv_bytes": c64.kv_bytes, "gbs": round(c64.kv_bytes / (h_ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round(c64.kv_bytes / (h_ms * 1e-3) / 1e9 / peak, 4),
            "l2": "no flush: the 268 MB KV stream per step is larger than L2"}
        del c64
        esteps = max(20, a.steps // 4)
        for name, cent, pagefmt in (("uq_hd256_b4_75k_e2m1", None, False),
                                    ("uq_hd256_b4_75k_randtable", "rand", False),
                                    ("uq_hd256_b4_75k_page_formats", None, True)):
            cu = synth.uq_full(seed=1003 + rank, centroids=None if cent is None else synth.sorted_random_centroids(5),
                               scale_format="ue8m0" if pagefmt else "e4m3", rot_perm=pagefmt)
            u_ms, u_part = time_uq(cu, 147, esteps, a.warmup, dev, q_haircut=pagefmt)
            u_ms = _max_over_ranks(u_ms)
            extra[name] = {
                "workload": "4-bit head_dim 256 decode, 4 seqs x 75000 tokens, 2 KV heads, group 8, block 64, "
                            "288-byte slots, P=147, centroid table " + ("e2m1 values" if cent is None else
                                                                         "seeded sorted random")
                            + (", UE8M0 group scales, e4m3 query haircut, column-permuted rotation" if pagefmt
                               else ", e4m3 group scales"),
                "us_per_step": round(u_ms * 1e3, 2), "partition_us": round(u_part * 1e3, 2),
                "l2": "flushed (256 MB write, then read) before every timed step", "kv_bytes": cu.kv_bytes, "gbs": round(cu.kv_bytes / (u_ms * 1e-3) / 1e9, 1),
                "frac_of_peak": round(cu.kv_bytes / (u_ms * 1e-3) / 1e9 / peak, 4)}
            del cu
        for name, ql, qg, pt in (("fp8_ext_b16_16k_ql4_qg4_per_token", 4, 4, True),
                                 ("fp8_ext_b16_16k_ql2_qg8", 2, 8, False)):
            ce = synth.fp8_ext_long(seed=1005 + rank, query_group=qg, query_len=ql, per_token=pt)
            x_ms = _max_over_ranks(time_fp8_ext(ce, 32, esteps, a.warmup, dev))
            extra[name] = {
                "workload": f"fp8 decode of {ql} query tokens per sequence (causal inside the query block), "
                            f"16 seqs x 16384 tokens, 8 KV heads, group {qg}, block 16, P=32, "
                            + ("per-token K/V scales" if pt else "per-tensor K/V scales"),
                "us_per_step": round(x_ms * 1e3, 2), "kv_bytes": ce.kv_bytes,
                "gbs": round(ce.kv_bytes / (x_ms * 1e-3) / 1e9, 1),
                "frac_of_peak": round(ce.kv_bytes / (x_ms * 1e-3) / 1e9 / peak, 4),
                "l2": "no flush: the cache is larger than L2"}
            del ce
        ci = synth.idx_full(seed=1004 + rank)
        i_ms, _ = time_idx(ci, esteps, a.warmup, dev)
        i_ms = _max_over_ranks(i_ms)
        extra["nvfp4_index_score_64req"] = {
            "workload": "NVFP4 paged index scorer, 64 requests, lengths U[4096,32768], query_len 4, 2 heads, "
                        "128-token pages of 72 B/token, S=256",
            "us_per_step": round(i_ms * 1e3, 2), "l2": "flushed (256 MB write, then read) before every timed step",
            "kv_bytes": ci.kv_bytes,
            "gbs": round(ci.kv_bytes / (i_ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round(ci.kv_bytes / (i_ms * 1e-3) / 1e9 / peak, 4)}
        cs = synth.idx_shared_prefix(seed=1007 + rank)
        s_ms, _ = time_idx(cs, esteps, a.warmup, dev)
        s_ms = _max_over_ranks(s_ms)
        extra["nvfp4_index_score_64req_shared_prefix"] = {
            "workload": "NVFP4 paged index scorer, 64 requests, lengths U[16384,32768], the first 16384 tokens "
                        "(128 pages) shared by all requests, query_len 4, 2 heads, S=256",
            "us_per_step": round(s_ms * 1e3, 2), "l2": "flushed (256 MB write, then read) before every timed step",
            "kv_bytes": cs.kv_bytes, "unique_page_bytes": cs.unique_page_bytes,
            "gbs": round(cs.kv_bytes / (s_ms * 1e-3) / 1e9, 1),
            "gbs_unique": round(cs.unique_page_bytes / (s_ms * 1e-3) / 1e9, 1),
            "kv_bytes_is": "pages per (request, block) as the scorer processes them; unique_page_bytes counts a "
                           "shared page once"}
        del cs
        t_ms, _ = time_idx(ci, esteps, a.warmup, dev, per_token_cols=32768)
        t_ms = _max_over_ranks(t_ms)
        out_bytes = ci.num_heads * ci.num_reqs * ci.query_len * 32768 * 4
        extra["nvfp4_index_score_64req_per_token"] = {
            "workload": "NVFP4 paged index scorer, 64 requests, lengths U[4096,32768], query_len 4, 2 heads, "
                        "one score column per token (32768 columns)",
            "us_per_step": round(t_ms * 1e3, 2), "l2": "flushed (256 MB write, then read) before every timed step",
            "kv_bytes": ci.kv_bytes, "score_bytes_written": out_bytes,
            "gbs_kv": round(ci.kv_bytes / (t_ms * 1e-3) / 1e9, 1),
            "gbs_read_plus_written": round((ci.kv_bytes + out_bytes) / (t_ms * 1e-3) / 1e9, 1),
            "frac_of_peak": round((ci.kv_bytes + out_bytes) / (t_ms * 1e-3) / 1e9 / peak, 4)}
        del ci

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu:
        pool = OraclePool(c)
        nbytes, dt, units = 0, 0.0, 0
        while dt < 10.0 and units < len(pool.units):
            b, t = pool.run(pool.cores)
            nbytes += b
            dt += t
            units += pool.cores
        pool.close()
        cpu = {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": pool.cores, "kind": "oracle",
               "sample": f"{units} of {len(pool.units)} (seq, kv_head) units of the workload "
                         f"({nbytes / 1e6:.0f} MB of KV) in {dt:.1f} s, float64 numpy oracle, "
                         f"spawn pool of {pool.cores} workers"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(ms_max, 5), "us_per_step": round(ms_max * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded N(0,1) K/V quantised to e4m3, bf16 Q)",
        "config": {"workload": WORKLOAD, "kv_bytes_per_step": kv,
                   "l2": "no flush: the 537 MB KV stream per step is larger than the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(part_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(part_gbs / peak, 4), "traffic": _profiled_traffic(),
                     "kernel": "pa_fp8_partition_kernel", "peak_kind": peak_kind,
                     "timing": "partition-only pass of the same step count after the step loop, CUDA events "
                               "around each launch on the launching stream",
                     "step_frac": round(value / world / peak, 4)},
        "partition_us": round(part_ms * 1e3, 2), "combine_us": round(comb_ms * 1e3, 2),
        "combine_us_is": "step time minus the partition kernel's own time (the combine overlaps the partition tail)",
        "gpu_launches": launches, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu, "extra": extra,
    }
    print(json.dumps(line))
    if _DIST["on"]:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""The float64 oracle over every unit of a full-size workload, on a
spawn-started process pool of the host cores.

Each unit, a (sequence, KV head) pair for the decodes or a request for the
scorer, is cut out of the case (its query rows and the cache blocks its
block table names, re-packed with an identity table) and handed to a worker
that calls only ``oracle``. The workers also return the unit's max|V|, the
scale of the attention tolerance. Nothing here runs on the GPU or touches the
library; the pool is started with ``spawn`` so that it is safe to create
after the tests have used CUDA."""
from __future__ import annotations

import atexit
import multiprocessing as mp
import os

import numpy as np

_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
        _POOL = mp.get_context("spawn").Pool(max(1, os.cpu_count() or 1))
        atexit.register(_close)
    return _POOL


def _close():
    global _POOL
    if _POOL is not None:
        _POOL.close()
        _POOL.join()
        _POOL = None


# ---------------------------------------------------------------- workers (oracle only)
def _fp8_unit(args):
    import oracle
    q, blocks, L, ks, vs, qg, scale = args
    bt = np.arange(blocks.shape[0], dtype=np.int32)[None, :]
    sl = np.array([L], dtype=np.int32)
    out = oracle.pa_decode_fp8(q, blocks, bt, sl, ks, vs, qg, scale)[0]
    _, v = oracle.attention.dense_kv_fp8(blocks, bt, 0, 0, L, ks, vs)
    return out, (float(np.abs(v).max()) if L else 0.0)


def _fp8_ext_unit(args):
    import oracle
    q, blocks, L, ks, vs, qg, ql, scale = args
    bt = np.arange(blocks.shape[0], dtype=np.int32)[None, :]
    sl = np.array([L], dtype=np.int32)
    out = oracle.pa_decode_fp8_ext(q, blocks, bt, sl, ks, vs, qg, ql, scale)[0]
    if np.ndim(ks) > 0:
        _, v = oracle.attention.dense_kv_fp8_per_token(blocks, bt, 0, 0, L, ks, vs)
    else:
        _, v = oracle.attention.dense_kv_fp8(blocks, bt, 0, 0, L, ks, vs)
    return out, (float(np.abs(v).max()) if L else 0.0)


def _uq_unit(args):
    import oracle
    q, slots, cent, L, qg, scale, fmt, haircut, perm = args
    bt = np.arange(slots.shape[0], dtype=np.int32)[None, :]
    sl = np.array([L], dtype=np.int32)
    out = oracle.uq_decode_hd256(q, slots, cent, bt, sl, qg, scale, scale_format=fmt, q_haircut=haircut,
                                 rot_perm=perm)[0]
    _, v = oracle.uq.dense_kv_uq(slots, cent, bt, 0, 0, L, fmt)
    return out, (float(np.abs(v).max()) if L else 0.0)


def _idx_unit(args):
    import oracle
    q, pages, L, ql, cols, per_token = args
    bt = np.arange(max(1, pages.shape[0]), dtype=np.int32)[None, :]
    sl = np.array([L], dtype=np.int32)
    fn = oracle.nvfp4_index_score_per_token if per_token else oracle.nvfp4_index_score
    return fn(q, pages, bt, sl, ql, cols)


# ---------------------------------------------------------------- unit cutting
def _blocks_of(block_table_row, L, bs):
    nb = max(1, (L + bs - 1) // bs)
    ids = np.asarray(block_table_row[:nb], dtype=np.int64)
    return np.where(ids < 0, 0, ids)


def fp8_reference(c, units=None):
    """{(s, h): (out [QG, D], max|V|)} for the units of an fp8 case."""
    Hk, qg = c.num_kv_heads, c.query_group
    units = units or [(s, h) for s in range(c.num_seqs) for h in range(Hk)]
    args = []
    for s, h in units:
        L = int(c.seq_lens[s])
        blk = c.kv_cache[_blocks_of(c.block_table[s], L, c.block_size)][:, :, h:h + 1]
        q = c.q_bits[s:s + 1, h * qg:(h + 1) * qg]
        args.append((np.ascontiguousarray(q), np.ascontiguousarray(blk), L, c.k_scale, c.v_scale, qg,
                     c.softmax_scale))
    return dict(zip(units, _pool().map(_fp8_unit, args, chunksize=1)))


def fp8_ext_reference(c, units=None):
    """{(s, h): (out [QL, QG, D], max|V|)} for the units of a multi-token case."""
    Hk, qg = c.num_kv_heads, c.query_group
    units = units or [(s, h) for s in range(c.num_seqs) for h in range(Hk)]
    args = []
    for s, h in units:
        L = int(c.seq_lens[s])
        ids = _blocks_of(c.block_table[s], L, c.block_size)
        blk = c.kv_cache[ids][:, :, h:h + 1]
        q = c.q_bits[s:s + 1, :, h * qg:(h + 1) * qg]
        if c.per_token:
            ks = np.ascontiguousarray(np.asarray(c.k_scale)[ids][:, h:h + 1])
            vs = np.ascontiguousarray(np.asarray(c.v_scale)[ids][:, h:h + 1])
        else:
            ks, vs = c.k_scale, c.v_scale
        args.append((np.ascontiguousarray(q), np.ascontiguousarray(blk), L, ks, vs, qg, c.query_len,
                     c.softmax_scale))
    return dict(zip(units, _pool().map(_fp8_ext_unit, args, chunksize=1)))


def uq_reference(c, units=None, q_haircut=False):
    """{(s, h): (out [QG, 256], max|V|)} for the units of an hd256 case."""
    Hk, qg = c.num_kv_heads, c.query_group
    units = units or [(s, h) for s in range(c.num_seqs) for h in range(Hk)]
    args = []
    for s, h in units:
        L = int(c.seq_lens[s])
        slots = c.kv_cache[_blocks_of(c.block_table[s], L, c.block_size)][:, :, h:h + 1]
        q = c.q_bits[s:s + 1, h * qg:(h + 1) * qg]
        args.append((np.ascontiguousarray(q), np.ascontiguousarray(slots), c.centroids, L, qg, c.softmax_scale,
                     c.scale_format, q_haircut, c.rot_perm))
    return dict(zip(units, _pool().map(_uq_unit, args, chunksize=1)))


def idx_reference(c, reqs=None, per_token_cols=None):
    """{r: scores [H, QL, cols]} for the requests of a scorer case."""
    ql = c.query_len
    cols = c.num_cols if per_token_cols is None else per_token_cols
    reqs = list(range(c.num_reqs)) if reqs is None else list(reqs)
    args = []
    for r in reqs:
        L = int(c.seq_lens[r])
        pages = c.pages[_blocks_of(c.block_table[r], L, 128)]
        q = c.q_codes[r * ql:(r + 1) * ql]
        args.append((np.ascontiguousarray(q), np.ascontiguousarray(pages), L, ql, cols, per_token_cols is not None))
    return dict(zip(reqs, _pool().map(_idx_unit, args, chunksize=1)))


def check_units(got, ref, c, what=""):
    """got [B, Hq, D] (or [B, QL, Hq, D]) against the pool's per-unit
    references: max|err| <= 2e-3 * max|V| of each (sequence, KV head); an L = 0
    unit must give exactly 0. Returns the worst err / tol."""
    qg = c.query_group
    worst = 0.0
    for (s, h), (r, vmax) in ref.items():
        rows = slice(h * qg, (h + 1) * qg)
        g = got[s, rows] if got.ndim == 3 else got[s, :, rows]
        assert np.all(np.isfinite(g)), f"{what}: non-finite output at seq {s} head {h}"
        if int(c.seq_lens[s]) == 0:
            assert np.all(g == 0.0), f"{what}: L=0 must give 0 (seq {s})"
            continue
        err = float(np.max(np.abs(g - r)))
        tol = 2e-3 * vmax
        worst = max(worst, err / tol if tol > 0 else 0.0)
        assert err <= tol, f"{what}: seq {s} head {h}: max|err| {err:.3e} > tol {tol:.3e}"
    return worst

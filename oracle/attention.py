"""fp8 paged-attention decode, and the split-KV partition/combine rewrite.

TEST INFRASTRUCTURE (see the package header).

What is computed ([PA] opening description: per-tensor fp8 K/V, query length
1, GQA; [UQ] STEP E..G for the paging and partition mapping):

  for sequence s of length L, KV head h and query row g (query head h*QG+g):
      k_t = e4m3(K code of token t) * k_scale
      v_t = e4m3(V code of token t) * v_scale
      o   = sum_t softmax_t(scale * q . k_t) * v_t,   t = 0 .. L-1

Token t of sequence s lives in physical block ``block_table[s, t // bs]`` at
slot ``t % bs``; the cache is ``[num_blocks][2 (K,V)][Hk][bs][D]``. L = 0
gives 0 ([UQ] STEP G divides by a sum clamped to 1 when it is 0).

The partition rewrite (``partition_partials`` + ``combine_partials``) is the
same result split over P partitions: partition p owns the 256-token tile
groups p, p+P, p+2P, ... ([UQ] STEP F: the tile groups of a partition are strided by P),
keeps (m_p, l_p, O_p) = (max logit, sum of exp(logit - m_p),
sum exp(logit - m_p) v / l_p), an empty partition gives (-inf, 0, 0)
([PA] NaN-guard commit), and the combine takes M = max_p m_p,
w_p = l_p e^(m_p - M), out = sum_p w_p O_p / sum_p w_p ([PA], its
cross-partition reduce kernel).

Pins (tests/test_oracle_attention.py): a 2-token case built so the softmax
weights are exactly 1/4 and 3/4; L = 1 gives v_0; constant V gives the
constant; q = 0 and identical keys give the mean of V; each query head reads
its own KV head (h = head // QG); block-table permutation invariance;
k_scale/softmax_scale trade-off; linearity in v_scale; NaN bytes past the end
of a sequence change nothing; any partition count equals the unsplit result.
"""
import math

import numpy as np

from .formats import decode_bf16, decode_e4m3fn

TILE_GROUP = 256   # tokens per tile group ([UQ] STEP F: 16 tiles of 16)


def attend(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q k^T) v for q_rows [G, D], k [L, Dk], v [L, Dv]."""
    G = q_rows.shape[0]
    if k.shape[0] == 0:
        return np.zeros((G, v.shape[1]))
    logits = scale * (q_rows @ k.T)                  # [G, L]
    m = logits.max(axis=1, keepdims=True)
    w = np.exp(logits - m)
    return (w @ v) / w.sum(axis=1, keepdims=True)


def gather_tokens(cache_kv_head: np.ndarray, block_table_row: np.ndarray, L: int) -> np.ndarray:
    """cache_kv_head: [num_blocks, bs, ...] for one of K/V and one KV head.
    Returns the logical tokens 0..L-1 in order: [L, ...]."""
    bs = cache_kv_head.shape[1]
    nb = (L + bs - 1) // bs
    blocks = np.asarray(block_table_row[:nb], dtype=np.int64)
    dense = cache_kv_head[blocks].reshape((nb * bs,) + cache_kv_head.shape[2:])
    return dense[:L]


def dense_kv_fp8(kv_cache, block_table, seq, kv_head, L, k_scale, v_scale):
    """Dequantised K [L, D] and V [L, D] of one (sequence, KV head)."""
    kc = gather_tokens(kv_cache[:, 0, kv_head], block_table[seq], L)
    vc = gather_tokens(kv_cache[:, 1, kv_head], block_table[seq], L)
    return decode_e4m3fn(kc) * float(k_scale), decode_e4m3fn(vc) * float(v_scale)


def pa_decode_fp8(q_bits, kv_cache, block_table, seq_lens, k_scale, v_scale,
                  query_group: int, softmax_scale: float | None = None,
                  units=None) -> np.ndarray:
    """Reference output [B, Hq, D] (float64).

    q_bits [B, Hq, D] uint16 bf16 bits; kv_cache [NB, 2, Hk, bs, D] uint8;
    block_table [B, max_blocks] int32; seq_lens [B] int32. ``units`` is an
    optional list of (seq, kv_head) pairs to compute (others stay 0)."""
    q = decode_bf16(q_bits)
    B, Hq, D = q.shape
    Hk = kv_cache.shape[2]
    assert Hq == Hk * query_group
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, Hq, D))
    if units is None:
        units = [(s, h) for s in range(B) for h in range(Hk)]
    for s, h in units:
        L = int(seq_lens[s])
        k, v = dense_kv_fp8(kv_cache, block_table, s, h, L, k_scale, v_scale)
        rows = slice(h * query_group, (h + 1) * query_group)
        out[s, rows] = attend(q[s, rows], k, v, softmax_scale)
    return out


def dense_kv_fp8_per_token(kv_cache, block_table, seq, kv_head, L, k_scales, v_scales):
    """Dequantised K and V [L, D] of one (sequence, KV head) with per-token
    scales: k_scales / v_scales [num_blocks, Hk, bs] float, gathered through the
    block table exactly like the codes."""
    kc = gather_tokens(kv_cache[:, 0, kv_head], block_table[seq], L)
    vc = gather_tokens(kv_cache[:, 1, kv_head], block_table[seq], L)
    ks = gather_tokens(np.asarray(k_scales, dtype=np.float64)[:, kv_head], block_table[seq], L)
    vs = gather_tokens(np.asarray(v_scales, dtype=np.float64)[:, kv_head], block_table[seq], L)
    return decode_e4m3fn(kc) * ks[:, None], decode_e4m3fn(vc) * vs[:, None]


def pa_decode_fp8_ext(q_bits, kv_cache, block_table, seq_lens, k_scale, v_scale,
                      query_group: int, query_len: int, softmax_scale: float | None = None,
                      units=None) -> np.ndarray:
    """Decode of query_len new tokens per sequence ([PA] "per_token_kv" and MTP
    query_length 1..4 commits): reference output [B, QL, Hq, D] (float64).

    q_bits [B, QL, Hq, D] bf16 bits. Query position qoff of a sequence of
    length L (L counts the QL new tokens) sees the tokens t <= L - QL + qoff
    (causal inside the query block); a row that sees no token gives 0.
    k_scale / v_scale are floats (per-tensor, as in ``pa_decode_fp8``) or
    arrays [num_blocks, Hk, bs] (one scale per cached token and KV head)."""
    q = decode_bf16(q_bits)
    B, QL, Hq, D = q.shape
    assert QL == query_len
    Hk = kv_cache.shape[2]
    assert Hq == Hk * query_group
    per_token = np.ndim(k_scale) > 0
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, QL, Hq, D))
    if units is None:
        units = [(s, h) for s in range(B) for h in range(Hk)]
    for s, h in units:
        L = int(seq_lens[s])
        if per_token:
            k, v = dense_kv_fp8_per_token(kv_cache, block_table, s, h, L, k_scale, v_scale)
        else:
            k, v = dense_kv_fp8(kv_cache, block_table, s, h, L, k_scale, v_scale)
        heads = slice(h * query_group, (h + 1) * query_group)
        for qoff in range(QL):
            n = max(0, L - QL + 1 + qoff)
            out[s, qoff, heads] = attend(q[s, qoff, heads], k[:n], v[:n], softmax_scale)
    return out


# ----------------------------------------------------------------------------
# split-KV partitions and their flash-combine
# ----------------------------------------------------------------------------
def tile_groups_of_partition(L: int, p: int, P: int, tg: int = TILE_GROUP):
    """Tile groups owned by partition p of P: p, p+P, ... below ceil(L/tg)."""
    return list(range(p, (L + tg - 1) // tg, P))


def partition_partials(q_rows, k, v, scale, P: int, tg: int = TILE_GROUP):
    """(m [P, G], l [P, G], O [P, G, Dv]) for one (sequence, KV head).

    m is in natural-log units of the scaled logits."""
    G = q_rows.shape[0]
    L = k.shape[0]
    m = np.full((P, G), -np.inf)
    l = np.zeros((P, G))
    O = np.zeros((P, G, v.shape[1]))
    for p in range(P):
        toks = [t for g in tile_groups_of_partition(L, p, P, tg)
                for t in range(g * tg, min((g + 1) * tg, L))]
        if not toks:
            continue
        logits = scale * (q_rows @ k[toks].T)
        m[p] = logits.max(axis=1)
        w = np.exp(logits - m[p][:, None])
        l[p] = w.sum(axis=1)
        O[p] = (w @ v[toks]) / l[p][:, None]
    return m, l, O


def combine_partials(m, l, O):
    """Merge (m [P, G], l [P, G], O [P, G, D]) into [G, D]."""
    M = m.max(axis=0)                                   # [G]
    out = np.zeros(O.shape[1:])
    live = np.isfinite(M)
    if not live.any():
        return out
    w = np.where(np.isfinite(m), l * np.exp(np.where(np.isfinite(m), m - M, 0.0)), 0.0)
    den = w.sum(axis=0)
    num = np.einsum("pg,pgd->gd", w, O)
    out[live] = num[live] / den[live][:, None]
    return out

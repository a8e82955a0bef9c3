"""NVFP4 paged index scorer: per-block max of causal-masked dot products.

TEST INFRASTRUCTURE (see the package header).

Page ([IDX] ``load_tile``: codes of token t of a page at byte 64 t, scales
after ``PAGE_CODES`` = 8192 at byte 8 t): a 9216-byte page holds 128 tokens;
bytes 0..8191 are the e2m1 codes (64 B per token, dim 2i in the low nibble of
byte i) and bytes 8192..9215 the e4m3 scales (8 per token, one per 16 dims).

  k[t, d]          = e2m1(code[t, d]) * e4m3(scale[t, d // 16])
  dot[h, row, t]   = sum_d q[row, h, d] * k[t, d]         (q is e4m3)
  visible(row, t)  : t <= L - QL + qoff,  row = req * QL + qoff
                     ([IDX] ``score_cgs`` limit seq - QL + qoff - b*BLK)
  score[h, row, b] = max of dot over visible t of block b, else -inf
                     ([IDX] ``frag_max``: the max of a column's scores over
                     the page); blocks at or past ceil(L / 128) get -inf.

Per-token output (``nvfp4_index_score_per_token``): the same dots before the
block max, one column per token, -inf where the token is not visible.

Readings: no scale, weight or activation is applied to the dot (none is
shown); the per-block sentinels ``init``/``local`` are taken as 0, which
makes the page's skip predicate false everywhere; columns the page never
writes (b >= ceil(L/128)) are written as -inf.

Pins (tests/test_oracle_scorer.py): a scalar brute force over single tokens
and nibbles on tiny inputs; query_len 1 with a fully visible block gives the
max of the dots; a fully masked block gives -inf; every score is >= each
visible dot of its block and equal to one of them. Per-token output: the
same scalar brute force token by token; its block max equals the block score.
"""
import numpy as np

from .formats import decode_e2m1, decode_e4m3fn, unpack_nibbles

BLK = 128
D = 128
PAGE_CODES = 8192
PAGE_BYTES = 9216


def decode_page(page: np.ndarray) -> np.ndarray:
    """[9216] uint8 -> K [128, 128] float64."""
    codes = unpack_nibbles(page[:PAGE_CODES].reshape(BLK, D // 2))
    scales = decode_e4m3fn(page[PAGE_CODES:PAGE_BYTES].reshape(BLK, D // 16))
    return decode_e2m1(codes) * np.repeat(scales, 16, axis=1)


def nvfp4_token_dots(q_codes, pages, block_table, seq_lens, query_len: int, req: int):
    """dot [H, QL, L] for one request (no masking)."""
    L = int(seq_lens[req])
    nblk = (L + BLK - 1) // BLK
    if nblk == 0:
        H = q_codes.shape[1]
        return np.zeros((H, query_len, 0))
    k = np.concatenate([decode_page(pages[int(block_table[req, b])]) for b in range(nblk)])[:L]
    q = decode_e4m3fn(q_codes[req * query_len:(req + 1) * query_len])   # [QL, H, D]
    return np.einsum("qhd,td->hqt", q, k)


def nvfp4_index_score(q_codes, pages, block_table, seq_lens, query_len: int,
                      num_cols: int, reqs=None) -> np.ndarray:
    """Reference scores [H, R*QL, S] (float64, -inf where nothing is
    visible). ``reqs`` optionally limits the requests computed (the other
    rows stay NaN)."""
    R = seq_lens.shape[0]
    H = q_codes.shape[1]
    out = np.full((H, R * query_len, num_cols), np.nan)
    if reqs is None:
        reqs = range(R)
    for r in reqs:
        L = int(seq_lens[r])
        dots = nvfp4_token_dots(q_codes, pages, block_table, seq_lens, query_len, r)
        rows = slice(r * query_len, (r + 1) * query_len)
        res = np.full((H, query_len, num_cols), -np.inf)
        for qoff in range(query_len):
            last = L - query_len + qoff          # last visible token index
            for b in range(num_cols):
                lo, hi = b * BLK, min((b + 1) * BLK, L, last + 1)
                if hi > lo:
                    res[:, qoff, b] = dots[:, qoff, lo:hi].max(axis=1)
        out[:, rows] = res
    return out


def nvfp4_index_score_per_token(q_codes, pages, block_table, seq_lens, query_len: int,
                                num_cols: int, reqs=None) -> np.ndarray:
    """Per-token scores [H, R*QL, num_cols] (float64): column t holds
    dot[h, row, t] where token t is visible to the row (t < L and
    t <= L - QL + qoff), else -inf. The block score above is the max of these
    columns over a block. ``reqs`` as for nvfp4_index_score."""
    R = seq_lens.shape[0]
    H = q_codes.shape[1]
    out = np.full((H, R * query_len, num_cols), np.nan)
    if reqs is None:
        reqs = range(R)
    for r in reqs:
        L = int(seq_lens[r])
        dots = nvfp4_token_dots(q_codes, pages, block_table, seq_lens, query_len, r)
        res = np.full((H, query_len, num_cols), -np.inf)
        for qoff in range(query_len):
            n = max(0, min(L - query_len + qoff + 1, L, num_cols))   # visible tokens 0 .. n-1
            res[:, qoff, :n] = dots[:, qoff, :n]
        out[:, r * query_len:(r + 1) * query_len] = res
    return out

"""Pins of the NVFP4 index-scorer oracle: scalar brute force on tiny inputs,
closed forms and invariants."""
import math

import numpy as np
import pytest

import oracle
import synth

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _scalar_e2m1(n):
    v = E2M1[n & 7]
    return -v if n & 8 else v


def _scalar_e4m3(b):
    s = -1.0 if b & 0x80 else 1.0
    e = (b >> 3) & 0xF
    m = b & 7
    if e == 0xF and m == 7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (8 + m) * 2.0 ** (e - 10)


def _brute(c, per_token_cols=None):
    """Token-by-token, nibble-by-nibble scalar scoring; with per_token_cols,
    the per-token dots in that many columns instead of the block max."""
    R, QL, H, S = c.num_reqs, c.query_len, c.num_heads, c.num_cols
    if per_token_cols is not None:
        S = per_token_cols
    out = [[[-math.inf] * S for _ in range(R * QL)] for _ in range(H)]
    for r in range(R):
        L = int(c.seq_lens[r])
        for t in range(L):
            page = c.pages[int(c.block_table[r, t // 128])]
            tt = t % 128
            k = []
            for d in range(128):
                byte = int(page[64 * tt + d // 2])
                nib = byte & 0xF if d % 2 == 0 else byte >> 4
                k.append(_scalar_e2m1(nib) * _scalar_e4m3(int(page[8192 + 8 * tt + d // 16])))
            for qoff in range(QL):
                if t > L - QL + qoff:
                    continue
                row = r * QL + qoff
                for h in range(H):
                    dot = sum(_scalar_e4m3(int(c.q_codes[row, h, d])) * k[d] for d in range(128))
                    if per_token_cols is not None:
                        if t < S:
                            out[h][row][t] = dot
                        continue
                    b = t // 128
                    if b < S and dot > out[h][row][b]:
                        out[h][row][b] = dot
    return np.array(out)


def _run(c):
    return oracle.nvfp4_index_score(c.q_codes, c.pages, c.block_table, c.seq_lens,
                                    c.query_len, c.num_cols)


@pytest.mark.parametrize("lens", [[130], [3, 257]])
def test_brute_force_tiny(lens):
    c = synth.make_idx_case(31, lens, query_len=4, num_heads=2, num_cols=4)
    ref = _brute(c)
    got = _run(c)
    assert np.array_equal(np.isinf(ref), np.isinf(got))
    fin = np.isfinite(ref)
    assert np.max(np.abs(got[fin] - ref[fin]) / np.maximum(np.abs(ref[fin]), 1.0)) < 1e-12


def test_all_ones_closed_form():
    c = synth.make_idx_case(1, [128], query_len=1, num_heads=1, num_cols=1)
    c.pages[:, :8192] = 0x22          # every code e2m1 1.0
    c.pages[:, 8192:] = 0x38          # every scale 1.0
    c.q_codes[:] = 0x40               # every q element 2.0
    assert _run(c)[0, 0, 0] == 256.0


def test_query_len_one_full_block_is_max_dot():
    c = synth.make_idx_case(2, [300], query_len=1, num_heads=2, num_cols=3)
    dots = oracle.nvfp4_token_dots(c.q_codes, c.pages, c.block_table, c.seq_lens, 1, 0)
    s = _run(c)
    for h in range(2):
        assert s[h, 0, 0] == dots[h, 0, :128].max()
        assert s[h, 0, 1] == dots[h, 0, 128:256].max()
        assert s[h, 0, 2] == dots[h, 0, 256:300].max()


def test_masking_and_bounds():
    # L = 129: row qoff sees t <= 125 + qoff, so block 1 (token 128 only) is
    # visible only for qoff = 3; blocks past ceil(L/128) are -inf.
    c = synth.make_idx_case(4, [129], query_len=4, num_heads=2, num_cols=4)
    s = _run(c)
    dots = oracle.nvfp4_token_dots(c.q_codes, c.pages, c.block_table, c.seq_lens, 4, 0)
    for qoff in range(4):
        last = 125 + qoff
        assert np.all(s[:, qoff, 0] == dots[:, qoff, :min(last + 1, 128)].max(axis=1))
        if qoff < 3:
            assert np.all(s[:, qoff, 1] == -np.inf)
        else:
            assert np.all(s[:, qoff, 1] == dots[:, qoff, 128])
    assert np.all(s[:, :, 2:] == -np.inf)


def test_score_dominates_visible_dots():
    c = synth.make_idx_case(6, [700, 1], query_len=4, num_heads=2, num_cols=6)
    s = _run(c)
    for r in range(2):
        L = int(c.seq_lens[r])
        dots = oracle.nvfp4_token_dots(c.q_codes, c.pages, c.block_table, c.seq_lens, 4, r)
        for qoff in range(4):
            row = r * 4 + qoff
            for b in range(6):
                vis = [t for t in range(b * 128, min(b * 128 + 128, L)) if t <= L - 4 + qoff]
                if not vis:
                    assert np.all(s[:, row, b] == -np.inf)
                    continue
                assert np.all(s[:, row, b][:, None] >= dots[:, qoff, vis])
                assert all(s[h, row, b] in dots[h, qoff, vis] for h in range(2))


def test_tail_poison_ignored():
    c = synth.make_idx_case(7, [200], query_len=4, num_heads=2, num_cols=2)
    s = _run(c)
    assert not np.any(np.isnan(s))


# ---- per-token output
@pytest.mark.parametrize("lens,cols", [([130], 200), ([3, 257], 300), ([5], 2)])
def test_per_token_brute_force_tiny(lens, cols):
    c = synth.make_idx_case(41, lens, query_len=4, num_heads=2, num_cols=4)
    ref = _brute(c, per_token_cols=cols)
    got = oracle.nvfp4_index_score_per_token(c.q_codes, c.pages, c.block_table, c.seq_lens, 4, cols)
    assert np.array_equal(np.isinf(ref), np.isinf(got))
    fin = np.isfinite(ref)
    assert np.max(np.abs(got[fin] - ref[fin]) / np.maximum(np.abs(ref[fin]), 1.0)) < 1e-12


def test_per_token_block_max_is_block_score():
    c = synth.make_idx_case(43, [1, 127, 128, 129, 700, 1000], query_len=3, num_heads=2, num_cols=8)
    blk = oracle.nvfp4_index_score(c.q_codes, c.pages, c.block_table, c.seq_lens, 3, 8)
    tok = oracle.nvfp4_index_score_per_token(c.q_codes, c.pages, c.block_table, c.seq_lens, 3, 8 * 128)
    assert np.array_equal(tok.reshape(2, -1, 8, 128).max(axis=3), blk)
    # visible columns per row: min(L - QL + qoff + 1, L), never negative
    for r, L in enumerate(c.seq_lens.tolist()):
        for qoff in range(3):
            n = int(np.isfinite(tok[0, 3 * r + qoff]).sum())
            assert n == max(0, min(L - 3 + qoff + 1, L, 1024))

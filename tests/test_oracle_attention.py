"""Pins of the fp8 attention oracle: closed forms and invariants."""
import math

import numpy as np
import pytest

import oracle
import synth
from oracle.attention import attend, combine_partials, partition_partials, dense_kv_fp8


def _e4m3(x):
    return synth.round_to_e4m3_bytes(np.asarray(x, dtype=np.float32))


def _single_seq_case(L, D=128, Hk=1, QG=8, bs=16, seed=5, k_scale=0.05, v_scale=0.04):
    return synth.make_fp8_case(seed, [L], Hk, QG, D, bs, k_scale=k_scale, v_scale=v_scale)


def _run(c, **kw):
    args = dict(softmax_scale=c.softmax_scale)
    args.update(kw)
    return oracle.pa_decode_fp8(c.q_bits, c.kv_cache, c.block_table, c.seq_lens,
                                c.k_scale, c.v_scale, c.query_group, **args)


def test_two_token_weights_quarter_three_quarters():
    # k_0 = 0, k_1 = e_0 * c; q = e_0 * q0. Choose the softmax scale so that the
    # logit gap is ln 3: weights are exactly 1/4 and 3/4, o = (v0 + 3 v1) / 4.
    c = _single_seq_case(2, QG=1)
    kc = c.kv_cache
    blk = c.block_table[0, 0]
    kc[blk, 0, 0, :, :] = 0
    kc[blk, 0, 0, 1, 0] = _e4m3([8.0])[0]              # k_1[0] = 8 * k_scale
    q = np.zeros((1, 1, 128), dtype=np.float32)
    q[0, 0, 0] = 1.5
    c.q_bits = synth.round_to_bf16_bits(q)
    scale = math.log(3.0) / (1.5 * 8.0 * c.k_scale)
    out = _run(c, softmax_scale=scale)[0, 0]
    v = oracle.decode_e4m3fn(kc[blk, 1, 0, :2, :]) * c.v_scale
    expect = (v[0] + 3.0 * v[1]) / 4.0
    assert np.max(np.abs(out - expect)) < 1e-12


def test_single_token_returns_v0():
    c = _single_seq_case(1)
    out = _run(c)[0]
    v0 = oracle.decode_e4m3fn(c.kv_cache[c.block_table[0, 0], 1, 0, 0]) * c.v_scale
    assert np.allclose(out, np.broadcast_to(v0, out.shape), rtol=0, atol=1e-15)


def test_constant_v_returns_constant():
    c = _single_seq_case(77)
    for b in c.block_table[0][c.block_table[0] >= 0]:
        c.kv_cache[b, 1] = _e4m3([3.0])[0]
    out = _run(c)
    assert np.allclose(out, 3.0 * c.v_scale, rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_v():
    c = _single_seq_case(53)
    c.q_bits[:] = 0
    out = _run(c)[0]
    k, v = dense_kv_fp8(c.kv_cache, c.block_table, 0, 0, 53, c.k_scale, c.v_scale)
    assert np.allclose(out, v.mean(axis=0)[None, :], rtol=0, atol=1e-13)


def test_identical_keys_give_mean_of_v():
    c = _single_seq_case(40)
    row = c.kv_cache[c.block_table[0, 0], 0, 0, 0].copy()
    for b in c.block_table[0][c.block_table[0] >= 0]:
        c.kv_cache[b, 0, 0, :, :] = row
    out = _run(c)[0]
    _, v = dense_kv_fp8(c.kv_cache, c.block_table, 0, 0, 40, c.k_scale, c.v_scale)
    assert np.allclose(out, v.mean(axis=0)[None, :], rtol=0, atol=1e-13)


def test_each_query_head_reads_its_kv_head():
    # Constant V per KV head (value 1 + h): query head j must output 1 + j // QG.
    Hk, QG = 3, 4
    c = synth.make_fp8_case(11, [33, 5], Hk, QG, 128, 16, k_scale=1.0, v_scale=1.0)
    for h in range(Hk):
        c.kv_cache[:, 1, h] = _e4m3([1.0 + h])[0]
    out = _run(c)
    for j in range(Hk * QG):
        assert np.allclose(out[:, j], 1.0 + j // QG, rtol=0, atol=1e-13)


def test_block_table_permutation_invariance():
    c = synth.fp8_tiny()
    ref = _run(c)
    # move every block to a new physical slot
    rng = np.random.default_rng(3)
    NB = c.kv_cache.shape[0]
    perm = rng.permutation(NB)
    new_cache = np.empty_like(c.kv_cache)
    new_cache[perm] = c.kv_cache
    bt = np.where(c.block_table >= 0, perm[np.maximum(c.block_table, 0)], -1).astype(np.int32)
    out = oracle.pa_decode_fp8(c.q_bits, new_cache, bt, c.seq_lens, c.k_scale, c.v_scale,
                               c.query_group, c.softmax_scale)
    assert np.array_equal(out, ref)


def test_contiguous_equals_paged():
    c = synth.fp8_tiny()
    ref = _run(c)
    # re-lay each sequence contiguously in block order 0, 1, 2, ...
    nblk = (c.seq_lens + 15) // 16
    new_cache = np.full_like(c.kv_cache, 0x7F)
    bt = np.full_like(c.block_table, -1)
    o = 0
    for s in range(c.num_seqs):
        for j in range(nblk[s]):
            new_cache[o] = c.kv_cache[c.block_table[s, j]]
            bt[s, j] = o
            o += 1
    out = oracle.pa_decode_fp8(c.q_bits, new_cache, bt, c.seq_lens, c.k_scale, c.v_scale,
                               c.query_group, c.softmax_scale)
    assert np.allclose(out, ref, rtol=0, atol=1e-14)


def test_kscale_softmax_scale_tradeoff():
    c = synth.fp8_tiny()
    a = _run(c)
    b = oracle.pa_decode_fp8(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, c.k_scale * 4.0,
                             c.v_scale, c.query_group, c.softmax_scale / 4.0)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_linear_in_v_scale():
    c = synth.fp8_tiny()
    a = _run(c)
    b = oracle.pa_decode_fp8(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, c.k_scale,
                             c.v_scale * 3.0, c.query_group, c.softmax_scale)
    assert np.allclose(3.0 * a, b, rtol=0, atol=1e-12)


def test_tail_poison_is_ignored_and_masking_is_by_length():
    c = synth.fp8_tiny()
    a = _run(c)
    assert np.all(np.isfinite(a))
    # changing bytes past the end of sequence 0 changes nothing
    L = int(c.seq_lens[0])
    blk = c.block_table[0, L // 16]
    c.kv_cache[blk, :, :, L % 16:, :] = 0x55
    assert np.array_equal(_run(c), a)
    # but extending the length by one token does change the output
    c.seq_lens = c.seq_lens.copy()
    c.seq_lens[0] += 1
    assert not np.allclose(_run(c)[0], a[0])


def test_empty_sequence_gives_zero():
    c = synth.make_fp8_case(9, [0, 20], 2, 8)
    out = _run(c)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out[1]))


@pytest.mark.parametrize("P", [1, 2, 3, 7, 32, 100])
@pytest.mark.parametrize("L", [1, 255, 256, 257, 1000, 2049])
def test_any_partition_count_equals_unsplit(P, L):
    rng = np.random.default_rng(L * 131 + P)
    q = rng.standard_normal((8, 128))
    k = rng.standard_normal((L, 128))
    v = rng.standard_normal((L, 128))
    ref = attend(q, k, v, 0.088)
    m, l, O = partition_partials(q, k, v, 0.088, P)
    assert np.max(np.abs(combine_partials(m, l, O) - ref)) < 1e-12
    # a partition past the tile groups is empty: (-inf, 0, 0)
    ntg = (L + 255) // 256
    for p in range(ntg, P):
        assert np.all(m[p] == -np.inf) and np.all(l[p] == 0) and np.all(O[p] == 0)


def test_partition_map_is_strided_tile_groups():
    assert oracle.tile_groups_of_partition(16384, 0, 32) == [0, 32]
    assert oracle.tile_groups_of_partition(16384, 31, 32) == [31, 63]
    assert oracle.tile_groups_of_partition(1024, 5, 32) == []
    assert oracle.tile_groups_of_partition(1025, 4, 32) == [4]


# ---------------------------------------------------------------- multi-token queries, per-token scales
def _ext(c):
    return oracle.pa_decode_fp8_ext(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, c.k_scale,
                                    c.v_scale, c.query_group, c.query_len, c.softmax_scale)


def test_ext_single_query_token_is_plain_decode():
    c = synth.make_fp8_ext_case(31, [0, 1, 37, 300], 2, 4, 1, False)
    ref = oracle.pa_decode_fp8(c.q_bits[:, 0], c.kv_cache, c.block_table, c.seq_lens, c.k_scale,
                               c.v_scale, c.query_group, c.softmax_scale)
    assert np.max(np.abs(_ext(c)[:, 0] - ref)) < 1e-12


def test_ext_query_rows_are_prefix_decodes():
    """Query position qoff of a length-L sequence decodes the prefix of
    length L - QL + 1 + qoff: the plain decode on that shorter length."""
    c = synth.make_fp8_ext_case(32, [2, 5, 40, 257], 2, 4, 3, False)
    out = _ext(c)
    for qoff in range(3):
        lens = np.maximum(0, c.seq_lens - 3 + 1 + qoff).astype(np.int32)
        ref = oracle.pa_decode_fp8(c.q_bits[:, qoff], c.kv_cache, c.block_table, lens, c.k_scale,
                                   c.v_scale, c.query_group, c.softmax_scale)
        assert np.max(np.abs(out[:, qoff] - ref)) < 1e-12
    # the first row of the 2-token sequence sees nothing
    assert np.all(out[0, 0] == 0.0)


def test_ext_constant_per_token_scales_equal_per_tensor():
    c = synth.make_fp8_ext_case(33, [1, 100, 333], 2, 8, 2, False, poison=False)
    NB, Hk, bs = c.kv_cache.shape[0], c.num_kv_heads, c.block_size
    ks = np.full((NB, Hk, bs), c.k_scale, dtype=np.float32)
    vs = np.full((NB, Hk, bs), c.v_scale, dtype=np.float32)
    per_token = oracle.pa_decode_fp8_ext(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, ks, vs,
                                         c.query_group, c.query_len, c.softmax_scale)
    # (the per-tensor scalars rounded to float32 like the arrays)
    per_tensor = oracle.pa_decode_fp8_ext(c.q_bits, c.kv_cache, c.block_table, c.seq_lens,
                                          float(np.float32(c.k_scale)), float(np.float32(c.v_scale)),
                                          c.query_group, c.query_len, c.softmax_scale)
    assert np.max(np.abs(per_token - per_tensor)) < 1e-12


def test_ext_per_token_brute_force():
    """Scalar loops over a tiny case: every logit and output element written
    out from the decoded bytes and each token's own scales."""
    c = synth.make_fp8_ext_case(34, [5, 3], 1, 2, 2, True, head_dim=128, block_size=16)
    out = _ext(c)
    q = oracle.decode_bf16(c.q_bits)
    kc = oracle.decode_e4m3fn(c.kv_cache[:, 0])
    vc = oracle.decode_e4m3fn(c.kv_cache[:, 1])
    bs = c.block_size
    for s in range(c.num_seqs):
        L = int(c.seq_lens[s])
        for qoff in range(2):
            n = L - 2 + 1 + qoff
            for g in range(2):
                logits = []
                for t in range(n):
                    blk, sl = int(c.block_table[s, t // bs]), t % bs
                    dot = 0.0
                    for d in range(128):
                        dot += float(q[s, qoff, g, d]) * float(kc[blk, 0, sl, d]) * float(c.k_scale[blk, 0, sl])
                    logits.append(dot * c.softmax_scale)
                mx = max(logits)
                w = [math.exp(x - mx) for x in logits]
                den = sum(w)
                for d in range(0, 128, 17):
                    num = 0.0
                    for t in range(n):
                        blk, sl = int(c.block_table[s, t // bs]), t % bs
                        num += w[t] * float(vc[blk, 0, sl, d]) * float(c.v_scale[blk, 0, sl])
                    assert abs(out[s, qoff, g, d] - num / den) < 1e-12


def test_head_dim_64_is_the_zero_padded_128_case():
    """The decode at head_dim 64 equals the head_dim 128 decode of the same
    tokens with the extra 64 dims of q and K zero and V's extra dims dropped,
    at the same softmax scale."""
    c = synth.make_fp8_case(77, [5, 130], 2, 4, head_dim=64)
    out64 = oracle.pa_decode_fp8(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, c.k_scale, c.v_scale, 4,
                                 c.softmax_scale)
    q = np.zeros(c.q_bits.shape[:2] + (128,), dtype=np.uint16)
    q[..., :64] = c.q_bits
    kv = np.zeros(c.kv_cache.shape[:4] + (128,), dtype=np.uint8)
    kv[..., :64] = c.kv_cache
    out128 = oracle.pa_decode_fp8(q, kv, c.block_table, c.seq_lens, c.k_scale, c.v_scale, 4, c.softmax_scale)
    assert c.softmax_scale == 1 / 8
    assert np.max(np.abs(out128[..., :64] - out64)) < 1e-13
    assert np.all(out128[..., 64:] == 0)

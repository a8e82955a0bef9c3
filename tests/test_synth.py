"""The seeded input generators keep the recipes the workloads are stated with:
shapes, block-table structure, scale ranges and formats, tail poison, shared
prefixes, and determinism per seed."""
import math

import numpy as np

import oracle
import synth


def test_fp8_tiny_recipe():
    c = synth.fp8_tiny()
    assert c.kv_cache.shape == (32, 2, 1, 16, 128) and c.q_bits.shape == (2, 8, 128)
    assert list(c.seq_lens) == [37, 200]
    used = np.concatenate([c.block_table[0, :3], c.block_table[1, :13]])
    assert len(set(used.tolist())) == 16 and used.min() >= 0 and used.max() < 32
    # tail slots of the last block of seq 0 (37 = 2 * 16 + 5) hold NaN codes
    tail = c.kv_cache[c.block_table[0, 2], :, 0, 5:]
    assert np.all(np.isnan(oracle.decode_e4m3fn(tail)))


def test_fp8_gqa_block_table_is_a_permutation():
    c = synth.make_fp8_case(1001, [256] * 4, 2, 8, poison=False)     # small copy of the GQA recipe
    bt = c.block_table[:, :16]
    assert sorted(bt.ravel().tolist()) == list(range(c.kv_cache.shape[0]))


def test_seeds_are_deterministic_and_distinct():
    a, b = synth.make_fp8_case(5, [100], 1, 8), synth.make_fp8_case(5, [100], 1, 8)
    assert np.array_equal(a.kv_cache, b.kv_cache) and np.array_equal(a.q_bits, b.q_bits)
    c = synth.make_fp8_case(6, [100], 1, 8)
    assert not np.array_equal(a.kv_cache, c.kv_cache)


def test_ragged_lengths_in_range():
    c = synth.fp8_ragged(batch=16)
    assert c.seq_lens.min() >= 1024 and c.seq_lens.max() <= 16384
    assert c.block_table.shape[1] == 1024


def test_per_token_scales_log_uniform_and_float32():
    c = synth.make_fp8_ext_case(11, [300, 700], 2, 4, 2, True, poison=False)
    for s in (c.k_scale, c.v_scale):
        assert s.dtype == np.float32 and s.shape == (c.kv_cache.shape[0], 2, 16)
        assert s.min() >= 0.01 * (1 - 1e-6) and s.max() <= 0.2 * (1 + 1e-6)
        # log-uniform: about half the draws below the geometric mean
        frac = float(np.mean(s < math.sqrt(0.01 * 0.2)))
        assert 0.4 < frac < 0.6


def test_uq_scale_formats():
    e = synth.make_uq_case(12, [200], 1, 8, 64, 288, poison=False)
    u = synth.make_uq_case(12, [200], 1, 8, 64, 288, poison=False, scale_format="ue8m0")
    ub = np.concatenate([u.kv_cache[..., 128:136].ravel(), u.kv_cache[..., 264:272].ravel()])
    assert ub.min() >= 1 and ub.max() <= 254
    assert e.kv_cache.shape == u.kv_cache.shape and e.scale_format == "e4m3" and u.scale_format == "ue8m0"
    # a UE8M0 group scale is the smallest power of two that keeps the group inside the e2m1 range
    k_e, _ = oracle.uq.dense_kv_uq(u.kv_cache, u.centroids, u.block_table, 0, 0, 200, "ue8m0")
    amax = np.abs(k_e.reshape(200, 8, 32)).max(axis=2)
    t = np.arange(200)
    sbytes = u.kv_cache[u.block_table[0, t // 64], t % 64, 0, 128:136]      # token t's K scale bytes
    scale = np.exp2(sbytes.astype(np.int64) - 127)
    assert np.all(amax <= 6 * scale)


def test_uq_rotated_domain_recipe():
    # K_r decoded from the slots, rotated back by the (permuted) rotation, is
    # close to N(0,1) data: the quantisation error is small against unit scale
    for perm in (False, True):
        c = synth.make_uq_case(13, [128], 1, 8, 64, 288, poison=False, rot_perm=perm)
        k_r, _ = oracle.uq.dense_kv_uq(c.kv_cache, c.centroids, c.block_table, 0, 0, 128)
        k = k_r @ oracle.rotation_matrix(perm).T
        assert 0.8 < float(k.std()) < 1.2


def test_scorer_shared_prefix_layout():
    c = synth.make_idx_case(14, [300, 1000, 129, 700], 4, 2, num_cols=8, shared_prefix_blocks=2)
    assert np.all(c.block_table[:, :2] == c.block_table[0, :2])
    nblk = [3, 8, 2, 6]
    own = np.concatenate([c.block_table[s, 2:n] for s, n in enumerate(nblk)])
    assert len(set(own.tolist())) == own.size and not set(own.tolist()) & set(c.block_table[0, :2].tolist())
    assert c.unique_page_bytes == (2 + own.size) * 9216
    assert c.kv_bytes == sum(nblk) * 9216
    # no NaN scales were written into a shared page (request 2 ends inside one)
    for b in c.block_table[0, :2]:
        assert not np.any(c.pages[b, 8192:] == 0x7F)


def test_uq_ue8m0_window_cases_cover_their_windows():
    """The byte-level UE8M0 generator draws every K and V scale byte from its
    window (plus 0 sentinels), codes uniform over all 16 codes, and NaN-class
    bytes (0xFF) only past a sequence's end."""
    c = synth.make_uq_ue8m0_window_case(13, [300, 65], (1, 45), (200, 252), poison=True)
    nb = -(-c.seq_lens.astype(np.int64) // c.block_size)
    for s, L in enumerate(c.seq_lens):
        t = np.arange(int(L))
        slots = c.kv_cache[c.block_table[s, t // c.block_size], t % c.block_size]     # [L, Hk, slot]
        kb, vb = slots[..., 128:136], slots[..., 264:272]
        assert kb.max() <= 45 and vb.max() <= 252
        assert set(np.unique(kb[kb > 0])) <= set(range(1, 46))
        assert vb[vb > 0].min() >= 200
        assert 0 < np.mean(kb == 0) < 0.1 and 0 < np.mean(vb == 0) < 0.1
    codes = c.kv_cache[..., :128].ravel()
    assert len(np.unique(codes & 0xF)) == 16 and len(np.unique(codes >> 4)) == 16
    assert c.scale_format == "ue8m0" and int(nb.sum()) == c.kv_cache.shape[0]

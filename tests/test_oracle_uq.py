"""Pins of the UltraQuant hd256 oracle: rotation, slot decode, byte count,
and the rotated pipeline against logical-domain attention."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle.attention import attend
from oracle.uq import decode_uq_slots, dense_kv_uq


def _read_sections(path):
    sec, out = None, {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line in ("bytes", "K", "V"):
                sec = line
                out[sec] = []
                continue
            a, b = line.split()
            out[sec].append((int(a), int(b, 16) if sec == "bytes" else float(b)))
    return out


def _facts(golden_dir):
    d = {}
    with open(os.path.join(golden_dir, "page_facts.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                d[k] = float(v)
    return d


def test_wht_orthonormal_symmetric_involution():
    R = oracle.wht_matrix(256)
    I = np.eye(256)
    assert np.max(np.abs(R @ R.T - I)) < 1e-13
    assert np.array_equal(R, R.T)
    assert np.max(np.abs(R @ R - I)) < 1e-13
    assert np.allclose(np.abs(R), 1.0 / 16.0, rtol=0, atol=0)


def test_wht_matches_recursive_sylvester():
    # H_1 = [1]; H_2n = [[H, H], [H, -H]] (independent construction)
    h = np.array([[1.0]])
    while h.shape[0] < 256:
        h = np.block([[h, h], [h, -h]])
    assert np.array_equal(oracle.wht_matrix(256) * 16.0, h)


def test_butterfly_vs_matrix_within_page_bound(golden_dir):
    # An 8-stage in-place butterfly in fp32 (the page's STEP B' computes the
    # rotation this way) against the float64 matrix.
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    y = x.copy()
    n, st = 256, 1
    while st < n:
        y = y.reshape(64, n // (2 * st), 2, st)
        a, b = y[:, :, 0, :].copy(), y[:, :, 1, :].copy()
        y[:, :, 0, :], y[:, :, 1, :] = a + b, a - b
        y = y.reshape(64, n)
        st *= 2
    y = y * np.float32(1.0 / 16.0)
    ref = x.astype(np.float64) @ oracle.wht_matrix(256)
    assert np.max(np.abs(y - ref)) <= _facts(golden_dir)["wht_butterfly_vs_matmul_fp32_max_abs"]


def test_slot_decode_hand_example(golden_dir):
    ex = _read_sections(os.path.join(golden_dir, "uq_slot_example.txt"))
    slot = np.zeros(288, dtype=np.uint8)
    for off, val in ex["bytes"]:
        slot[off] = val
    K, V = decode_uq_slots(slot, synth.e2m1_table())
    expK, expV = np.zeros(256), np.zeros(256)
    for d, v in ex["K"]:
        expK[d] = v
    for d, v in ex["V"]:
        expV[d] = v
    assert np.array_equal(K, expK)
    assert np.array_equal(V, expV)


def test_slot_ignores_padding_bytes():
    c = synth.make_uq_case(3, [70], 1, 8, 64, 288)
    s = c.kv_cache[0, :, 0].copy()
    a = decode_uq_slots(s, c.centroids)
    s[:, 272:] ^= 0xA5
    b = decode_uq_slots(s, c.centroids)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_byte_count_matches_page(golden_dir):
    c = synth.UqCase(None, None, None, None, np.array([75000] * 4, dtype=np.int32),
                     1, 8, 64, 288, 1 / 16)
    assert c.kv_bytes == int(_facts(golden_dir)["uq_kv_bytes_b4_seq75k_one_head"])


@pytest.mark.parametrize("QG", [8, 6])
def test_rotated_pipeline_equals_logical_attention(QG):
    c = synth.make_uq_case(21, [150, 64, 1], 2, QG, 64, 288)
    out = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens,
                                 QG, c.softmax_scale)
    R = oracle.wht_matrix(256)
    q = oracle.decode_bf16(c.q_bits)
    for s in range(3):
        for h in range(2):
            L = int(c.seq_lens[s])
            k_r, v_r = dense_kv_uq(c.kv_cache, c.centroids, c.block_table, s, h, L)
            rows = slice(h * QG, (h + 1) * QG)
            ref = attend(q[s, rows], k_r @ R, v_r @ R, 1.0 / 16.0)
            assert np.max(np.abs(out[s, rows] - ref)) < 1e-11


def test_single_token_returns_unrotated_v():
    c = synth.make_uq_case(5, [1], 1, 8, 64, 288)
    out = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 8)
    _, v_r = decode_uq_slots(c.kv_cache[c.block_table[0, 0], 0, 0], c.centroids)
    v = v_r @ oracle.wht_matrix(256)
    assert np.max(np.abs(out[0] - v[None, :])) < 1e-13


def test_poisoned_tail_ignored():
    c = synth.make_uq_case(8, [100], 1, 8, 64, 288)
    out = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 8)
    assert np.all(np.isfinite(out))


def test_ue8m0_variant_is_powers_of_two():
    slot = np.zeros(288, dtype=np.uint8)
    slot[0] = 0x22                     # dims 0, 1 = 1.0
    slot[128] = 127 + 3                # K scale 2^3 for dims 0..31
    K, _ = decode_uq_slots(slot, synth.e2m1_table(), scale_format="ue8m0")
    assert K[0] == 8.0 and K[1] == 8.0 and np.all(K[2:] == 0)


def test_rotate_q_fp32_exact_on_small_integers():
    # integer inputs keep every butterfly sum exact in float32, so the result
    # is exactly x H with the Sylvester matrix built here by recursion
    h = np.array([[1.0]])
    while h.shape[0] < 256:
        h = np.block([[h, h], [h, -h]])
    x = np.random.default_rng(4).integers(-50, 51, size=(5, 256)).astype(np.float32)
    assert np.array_equal(oracle.rotate_q_fp32(x).astype(np.float64), x.astype(np.float64) @ h)


def test_rotate_q_fp32_within_page_bound(golden_dir):
    x = np.random.default_rng(6).standard_normal((64, 256)).astype(np.float32)
    y = oracle.rotate_q_fp32(x).astype(np.float64) / 16.0
    ref = x.astype(np.float64) @ oracle.wht_matrix(256)
    assert np.max(np.abs(y - ref)) <= _facts(golden_dir)["wht_butterfly_vs_matmul_fp32_max_abs"]


def _bf16_bits(x):
    return synth.round_to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_haircut_is_identity_on_e4m3_exact_rotated_queries():
    # q = (a e_i + b e_j) R has entries +-(a +- b)/16: with a/16, b/16 on the
    # e4m3 grid and few mantissa bits the query is exact in bf16, its rotation
    # is exactly 16 (a e_i + b e_j), and q_r / 16 is already e4m3, so the
    # haircut changes nothing and the logits keep the single softmax scale.
    c = synth.make_uq_case(31, [40, 7], 1, 2, 64, 288)
    R = oracle.wht_matrix(256)
    q = np.zeros((2, 2, 256))
    for s in range(2):
        for g in range(2):
            e = np.zeros(256)
            e[3 + 17 * g + s] = 5.0 * (1 + g)       # q_r entries 5 or 10 and -3: 5/16, 10/16, -3/16 are e4m3
            e[200 - g] = -3.0
            q[s, g] = e @ R
    qb = _bf16_bits(q)
    assert np.array_equal(oracle.decode_bf16(qb), q)
    a = oracle.uq_decode_hd256(qb, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 2, 1 / 16)
    b = oracle.uq_decode_hd256(qb, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 2, 1 / 16,
                               q_haircut=True)
    assert np.max(np.abs(a - b)) < 1e-13


def test_haircut_against_torch_cast_and_softmax():
    # The haircut query built another way (float64 matrix rotation, torch's
    # e4m3 cast), then softmax attention written out over the decoded tokens.
    c = synth.make_uq_case(33, [90, 5], 2, 4, 64, 288)
    sc = 1 / 16
    out = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 4, sc,
                                 q_haircut=True)
    R = oracle.wht_matrix(256)
    q = oracle.decode_bf16(c.q_bits)
    for s in range(2):
        for h in range(2):
            rows = slice(4 * h, 4 * h + 4)
            qr = (q[s, rows] @ R * sc).astype(np.float32)
            qh = torch.from_numpy(np.clip(qr, -448, 448)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
            k_r, v_r = dense_kv_uq(c.kv_cache, c.centroids, c.block_table, s, h, int(c.seq_lens[s]))
            logits = qh @ k_r.T
            w = np.exp(logits - logits.max(axis=1, keepdims=True))
            ref = (w / w.sum(axis=1, keepdims=True)) @ v_r @ R
            assert np.max(np.abs(out[s, rows] - ref)) < 1e-11
    plain = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 4, sc)
    assert np.max(np.abs(out - plain)) > 1e-2          # the haircut is visible at this size


@pytest.mark.parametrize("QG", [8, 3])
def test_ue8m0_case_pipeline_equals_logical_attention(QG):
    c = synth.make_uq_case(35, [130, 64, 1], 2, QG, 64, 288, scale_format="ue8m0")
    slots = c.kv_cache.reshape(-1, 288)
    for off in (128, 264):
        sb = slots[:, off:off + 8]
        live = sb[sb != 0xFF]
        assert live.min() >= 1 and live.max() <= 254
    out = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens,
                                 QG, c.softmax_scale, scale_format="ue8m0")
    assert np.all(np.isfinite(out))
    R = oracle.wht_matrix(256)
    q = oracle.decode_bf16(c.q_bits)
    for s in range(3):
        for h in range(2):
            L = int(c.seq_lens[s])
            k_r, v_r = dense_kv_uq(c.kv_cache, c.centroids, c.block_table, s, h, L, "ue8m0")
            # a power-of-two scale keeps the e2m1 mantissas: every nonzero K
            # value is 1 or 1.5 times a power of two
            nz = np.abs(k_r[k_r != 0])
            mant = nz / np.exp2(np.floor(np.log2(nz)))
            assert np.all((mant == 1.0) | (mant == 1.5))
            rows = slice(h * QG, (h + 1) * QG)
            ref = attend(q[s, rows], k_r @ R, v_r @ R, 1.0 / 16.0)
            assert np.max(np.abs(out[s, rows] - ref)) < 1e-11


# ---- the page's column permutation of the rotation
def test_perm_dest_agrees_with_the_pages_per_lane_split():
    # the page gives the permutation twice: as one formula on the dim, and as
    # a sum of a part in the element t and a part in the 32-dim chunk c
    for c in range(8):
        for t in range(32):
            ct = (t & 0x0F) | ((t & 0x10) << 1)
            rt = ((c & 2) << 3) | ((c & 1) << 6) | ((c & 4) << 5)
            assert int(oracle.perm_dest(32 * c + t)) == ct | rt


def test_perm_is_a_bit_permutation_and_inverse():
    d = np.arange(256)
    p = oracle.perm_dest(d)
    assert sorted(p.tolist()) == list(range(256))
    assert np.array_equal(oracle.perm_source(p), d)
    for b in range(8):                      # a single set bit goes to a single set bit
        assert bin(int(oracle.perm_dest(1 << b))).count("1") == 1
    assert np.array_equal(p & 0x8F, d & 0x8F)


def test_permuted_rotation_orthonormal_and_a_column_permutation():
    M = oracle.rotation_matrix(True)
    R = oracle.wht_matrix(256)
    assert np.max(np.abs(M @ M.T - np.eye(256))) < 1e-13
    q = np.random.default_rng(8).standard_normal((3, 256))
    qr = q @ R
    assert np.allclose((q @ M)[:, oracle.perm_dest(np.arange(256))], qr, atol=1e-13, rtol=0)
    # M is no longer symmetric, so the output needs M^T, not M
    assert not np.array_equal(M, M.T)


@pytest.mark.parametrize("haircut", [False, True])
def test_permuted_pipeline_equals_logical_attention(haircut):
    c = synth.make_uq_case(37, [120, 9], 2, 4, 64, 288, rot_perm=True)
    out = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 4,
                                 c.softmax_scale, rot_perm=True, q_haircut=haircut)
    M = oracle.rotation_matrix(True)
    q = oracle.decode_bf16(c.q_bits)
    for s in range(2):
        for h in range(2):
            k_r, v_r = dense_kv_uq(c.kv_cache, c.centroids, c.block_table, s, h, int(c.seq_lens[s]))
            rows = slice(4 * h, 4 * h + 4)
            if haircut:
                # q M rounded to e4m3 after the scale, built from the float64 matrix and torch's cast
                qr = (q[s, rows] @ M * (1 / 16)).astype(np.float32)
                qh = torch.from_numpy(qr).to(torch.float8_e4m3fn).to(torch.float64).numpy()
                lg = qh @ k_r.T
                w = np.exp(lg - lg.max(axis=1, keepdims=True))
                ref = (w / w.sum(axis=1, keepdims=True)) @ v_r @ M.T
            else:
                ref = attend(q[s, rows], k_r @ M.T, v_r @ M.T, 1.0 / 16.0)     # logical domain
            assert np.max(np.abs(out[s, rows] - ref)) < 1e-11
    plain = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 4,
                                   c.softmax_scale, q_haircut=haircut)
    assert np.max(np.abs(out - plain)) > 1e-2        # the permutation matters on this cache

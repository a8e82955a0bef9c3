"""Pins of the UltraQuant hd256 oracle: rotation, slot decode, byte count,
and the rotated pipeline against logical-domain attention."""
import os

import numpy as np
import pytest

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

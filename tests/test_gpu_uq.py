"""GPU parity of uq_decode_hd256 (4-bit head_dim=256 slot cache, in-kernel
WHT rotation of Q, un-rotated output) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_attention_gb300 as qpa
import synth
from _gpu import UqDev, check_attention, uq_v_absmax
from _oracle_pool import check_units, uq_reference

# the partition count the benchmark runs the full hd256 workload with
UQ_BENCH_P = 38

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _check(c, got, units=None, what="", q_haircut=False):
    ref = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens,
                                 c.query_group, c.softmax_scale, units=units, scale_format=c.scale_format,
                                 q_haircut=q_haircut, rot_perm=c.rot_perm)
    return check_attention(got, ref, lambda s, h: uq_v_absmax(c, s, h), c, units, what)


LENS = [0, 1, 15, 63, 64, 65, 255, 256, 257, 777, 1500]


@pytest.mark.parametrize("P", [1, 3, 7])
def test_e2m1_centroids_partitions(P):
    c = synth.make_uq_case(200 + P, LENS, 2, 8, 64, 288)
    out, _, _ = UqDev(c).run(P)
    _check(c, out.cpu().double().numpy(), what=f"e2m1 P={P}")


@pytest.mark.parametrize("P", [1, 4])
def test_random_sorted_centroids(P):
    c = synth.make_uq_case(210 + P, LENS, 2, 8, 64, 288, centroids=synth.sorted_random_centroids(5))
    out, _, _ = UqDev(c).run(P)
    _check(c, out.cpu().double().numpy(), what=f"lut P={P}")


@pytest.mark.parametrize("qg", [6, 8, 3])
def test_query_groups(qg):
    c = synth.make_uq_case(220 + qg, [70, 500], 2, qg, 64, 288)
    out, _, _ = UqDev(c).run(2)
    _check(c, out.cpu().double().numpy(), what=f"qg={qg}")


@pytest.mark.parametrize("bs", [16, 32, 128, 256])
def test_block_sizes(bs):
    c = synth.make_uq_case(230 + bs, [1, bs - 1, bs + 1, 700], 2, 8, bs, 288)
    out, _, _ = UqDev(c).run(3)
    _check(c, out.cpu().double().numpy(), what=f"bs={bs}")


@pytest.mark.parametrize("slot", [272, 320])
def test_slot_padding(slot):
    c = synth.make_uq_case(240 + slot, [100, 333], 1, 8, 64, slot,
                           centroids=synth.sorted_random_centroids(6))
    out, _, _ = UqDev(c).run(2)
    _check(c, out.cpu().double().numpy(), what=f"slot={slot}")


def test_bf16_output_and_determinism():
    c = synth.make_uq_case(250, [300, 64], 2, 8, 64, 288)
    d = UqDev(c)
    a, ws, _ = d.run(3)
    b, _, _ = d.run(3, workspace=ws)
    assert torch.equal(a, b)
    o16, _, _ = d.run(3, out_dtype=torch.bfloat16)
    assert o16.dtype == torch.bfloat16
    assert torch.max(torch.abs(o16.float() - a)).item() <= torch.max(torch.abs(a)).item() * 2 ** -8 + 1e-6


def _plan(hk, qg):
    """The launcher's split: heads per item HG (the largest of 8, 4, 2, 1
    dividing Hk with HG * halves <= 8), the 8-row halves of the query group,
    and J = 8 / (HG * halves) partial slots per item and head."""
    nh = -(-qg // 8)
    for hg in (8, 4, 2, 1):
        if hk % hg == 0 and hg * nh <= 8:
            return hg, nh, 8 // (hg * nh)


@pytest.mark.parametrize("hk,qg,P", [
    (1, 8, 3),      # one head per item, every 8th slice per warp
    (1, 16, 2),     # two row halves, J = 4
    (2, 16, 5),     # J = 2
    (4, 16, 1),     # eight (head, half) pairs, J = 1
    (8, 8, 2),      # eight heads per item, J = 1
    (4, 12, 3),     # query group 12: the second half has 4 live rows
    (2, 3, 4),
])
def test_head_groups_and_row_halves(hk, qg, P):
    """Every way the launcher splits a launch over its eight consumer warps,
    with sequences shorter than J slices (warps left without a slice write
    empty slots)."""
    hg, nh, j = _plan(hk, qg)
    c = synth.make_uq_case(260 + 10 * hk + qg + P, [1, 31, 33, 64, 200, 257, 1300], hk, qg, 64, 288,
                           centroids=synth.sorted_random_centroids(hk + qg))
    out, ws, desc = UqDev(c).run(P)
    assert qpa.uq_decode_hd256_workspace_size(desc, P) >= c.num_seqs * hk * P * j * qg * 256 * 4
    _check(c, out.cpu().double().numpy(), what=f"Hk={hk} qg={qg} (HG={hg}, halves={nh}, J={j}) P={P}")


def test_query_group_16_long():
    """Query group 16 (the builder's largest group) on 2 x 20000 tokens."""
    c = synth.make_uq_case(275, [20000, 7777], 2, 16, 64, 288)
    out, _, _ = UqDev(c).run(9)
    check_units(out.cpu().double().numpy(), uq_reference(c), c, what="qg16 long")


# ---- UE8M0 group scales over the whole byte range, window by window
UE8_WINDOWS = [
    ((1, 45), (1, 45), 1.0),
    ((40, 90), (40, 90), 1.0),
    ((85, 125), (85, 125), 1.0),
    ((118, 140), (118, 140), 1.0),
    ((135, 180), (135, 180), 1.0),
    ((175, 215), (175, 215), 1.0),
    # the top bytes: the query is scaled down so that the largest logits stay
    # inside float32, and V stops at 248 so that the un-rotated output (up to
    # 16 times the largest rotated value) does too
    ((210, 254), (210, 248), 2.0 ** -12),
]


@pytest.mark.parametrize("kb,vb,gain", UE8_WINDOWS)
@pytest.mark.parametrize("lut", [False, True])
def test_ue8m0_byte_windows(kb, vb, gain, lut):
    """Scale bytes drawn uniformly from each window (with 0 sentinels), codes
    uniform over all 16 codes: together the windows cover bytes 0..254 of K
    and 0..248 of V (the last V bytes: next test)."""
    cent = synth.sorted_random_centroids(11) if lut else None
    c = synth.make_uq_ue8m0_window_case(700 + kb[0] + (1 if lut else 0), [1, 63, 200, 700], kb, vb,
                                        q_gain=gain, centroids=cent)
    out, _, _ = UqDev(c).run(3)
    _check(c, out.cpu().double().numpy(), what=f"ue8m0 K{kb} V{vb} lut={lut}")


def test_ue8m0_top_v_bytes_with_small_centroids():
    """V scale bytes up to 254 (2^127) with a centroid table below 2^-6, so
    that every V value and the un-rotated output are float32 values."""
    cent = (synth.sorted_random_centroids(13) * np.float32(2.0 ** -7)).astype(np.float32)
    c = synth.make_uq_ue8m0_window_case(760, [1, 63, 200, 700], (200, 254), (230, 254), q_gain=2.0 ** -12,
                                        centroids=cent)
    out, _, _ = UqDev(c).run(3)
    _check(c, out.cpu().double().numpy(), what="ue8m0 top V bytes")


def test_ue8m0_byte_255_raises_the_range_error_word():
    """0xFF is not a power of two of the format (the OCP encoding's NaN): a
    live token with that K scale byte raises error word 5."""
    c = synth.make_uq_ue8m0_window_case(790, [100], (120, 130), (120, 130))
    t = 37
    c.kv_cache[c.block_table[0, t // 64], t % 64, 0, 128 + 3] = 0xFF
    d = UqDev(c)
    desc = d.desc()
    ws = qpa.alloc_workspace(qpa.uq_decode_hd256_workspace_size(desc, 2), d.q.device)
    qpa.uq_decode_hd256(d.q, d.kv, d.cent, d.bt, d.sl, 2, 8, workspace=ws, desc=desc)
    assert qpa.kernel_error() == 5
    assert qpa.kernel_error() == 0


@pytest.mark.parametrize("gain,v_gain", [(1000.0, 1000.0 * 200), (1e-5, 1e-5 / 200)])
def test_centroid_tables_of_any_magnitude(gain, v_gain):
    """Centroid tables whose products with the e4m3 group scales (here near
    200 and near 1/200) lie far outside f16 (|c| * scale > 65504, or below
    f16's smallest subnormal): the kernel's table is normalised and the
    output scaled back."""
    cent = (synth.sorted_random_centroids(12) * np.float32(gain)).astype(np.float32)
    c = synth.make_uq_case(795 + int(gain > 1), [1, 100, 900], 2, 8, 64, 288, centroids=cent, v_gain=v_gain)
    out, _, _ = UqDev(c).run(2)
    _check(c, out.cpu().double().numpy(), what=f"centroids x{gain}")


@pytest.mark.parametrize("qg", [8, 6])
def test_full_config_all_units(qg):
    """4 seqs x 75000 tokens, 2 KV heads, block 64, 288-byte slots, with the
    benchmark's partition count; all 8 (seq, head) units against the oracle."""
    c = synth.uq_full(query_group=qg)
    out, _, _ = UqDev(c).run(UQ_BENCH_P)
    check_units(out.cpu().double().numpy(), uq_reference(c), c, what=f"uq-full qg={qg}")


# ---- page formats: UE8M0 group scales and the e4m3 query haircut
@pytest.mark.parametrize("haircut", [False, True])
@pytest.mark.parametrize("fmt", ["e4m3", "ue8m0"])
@pytest.mark.parametrize("P", [1, 5])
def test_scale_format_and_haircut(fmt, haircut, P):
    c = synth.make_uq_case(260 + P + (3 if haircut else 0), LENS, 2, 8, 64, 288, scale_format=fmt)
    out, _, _ = UqDev(c).run(P, q_haircut=haircut)
    _check(c, out.cpu().double().numpy(), what=f"{fmt} haircut={haircut} P={P}", q_haircut=haircut)


def test_haircut_result_differs_from_plain():
    """The haircut test above discriminates: the oracle's plain result misses
    the kernel's haircut result by more than the tolerance."""
    c = synth.make_uq_case(270, [5, 40], 2, 8, 64, 288, scale_format="ue8m0")
    out, _, _ = UqDev(c).run(3, q_haircut=True)
    got = out.cpu().double().numpy()
    plain = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 8,
                                   c.softmax_scale, scale_format="ue8m0")
    tol = max(uq_v_absmax(c, s, h) for s in range(2) for h in range(2)) * 2e-3
    assert np.max(np.abs(got - plain)) > 3 * tol
    _check(c, got, what="ue8m0 haircut", q_haircut=True)


@pytest.mark.parametrize("qg,bs", [(6, 16), (3, 256)])
def test_page_formats_with_lut_groups_and_blocks(qg, bs):
    c = synth.make_uq_case(280 + qg, [1, bs + 1, 900], 2, qg, bs, 288,
                           centroids=synth.sorted_random_centroids(7), scale_format="ue8m0")
    out, _, _ = UqDev(c).run(4, q_haircut=True)
    _check(c, out.cpu().double().numpy(), what=f"ue8m0 haircut lut qg={qg} bs={bs}", q_haircut=True)


def test_page_formats_full_config_all_units():
    """4 seqs x 75000 tokens with UE8M0 scales and the query haircut, with the
    benchmark's partition count; all 8 (seq, head) units against the oracle."""
    c = synth.make_uq_case(1013, [75000] * 4, 2, 8, 64, 288, poison=False, scale_format="ue8m0")
    out, _, _ = UqDev(c).run(UQ_BENCH_P, q_haircut=True)
    check_units(out.cpu().double().numpy(), uq_reference(c, q_haircut=True), c, what="uq-full ue8m0 haircut")


# ---- the page's column-permuted rotation
@pytest.mark.parametrize("fmt,haircut", [("e4m3", False), ("ue8m0", True)])
@pytest.mark.parametrize("P", [1, 4])
def test_rotation_permutation(fmt, haircut, P):
    c = synth.make_uq_case(290 + P + (5 if haircut else 0), LENS, 2, 8, 64, 288, scale_format=fmt, rot_perm=True)
    out, _, _ = UqDev(c).run(P, q_haircut=haircut)
    got = out.cpu().double().numpy()
    _check(c, got, what=f"perm {fmt} haircut={haircut} P={P}", q_haircut=haircut)


def test_rotation_permutation_matters_and_bf16_output():
    c = synth.make_uq_case(299, [7, 40], 2, 6, 32, 288, rot_perm=True,
                           centroids=synth.sorted_random_centroids(8))
    d = UqDev(c)
    out, _, _ = d.run(2)
    got = out.cpu().double().numpy()
    _check(c, got, what="perm lut qg=6 bs=32")
    plain = oracle.uq_decode_hd256(c.q_bits, c.kv_cache, c.centroids, c.block_table, c.seq_lens, 6,
                                   c.softmax_scale)
    tol = max(uq_v_absmax(c, s, h) for s in range(2) for h in range(2)) * 2e-3
    assert np.max(np.abs(got - plain)) > 3 * tol
    o16, _, _ = d.run(2, out_dtype=torch.bfloat16)
    assert torch.max(torch.abs(o16.float() - out)).item() <= torch.max(torch.abs(out)).item() * 2 ** -8 + 1e-6

"""GPU parity of uq_decode_hd256 (4-bit head_dim=256 slot cache, in-kernel
WHT rotation of Q, un-rotated output) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import UqDev, check_attention, uq_v_absmax
from _oracle_pool import check_units, uq_reference

# the partition count the benchmark runs the full hd256 workload with
UQ_BENCH_P = 147

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


def _warps_per_item(items, max_tokens, P, sms):
    """The launcher's choice of warps per item: the smallest W among those with
    the fewest slices per warp (rounds x slices of an item / W) on one
    8-warp CTA per SM."""
    tiles_per_item = max(1, -(-(-(-max_tokens // 256)) // P))
    best_w, best = 4, None
    for w in (1, 2, 4):
        slots = sms * (8 // w)
        cost = -(-items // slots) * tiles_per_item * 8 // w
        if best is None or cost < best:
            best, best_w = cost, w
    return best_w


@pytest.mark.parametrize("lens,P,want_w,rand", [
    ([64000, 9000], 250, 1, False),     # 1000 items: one warp per item on 152 SMs
    ([64000, 9000], 250, 1, True),
    ([30720, 7000], 120, 2, False),     # 480 items: two warps per item
    ([30720, 7000], 40, 4, False),      # 160 items: four warps per item
])
def test_warps_per_item(lens, P, want_w, rand):
    """Item groups of 1, 2 and 4 warps (the launcher picks W from the item
    count); ragged lengths leave most partitions of the short sequence empty."""
    cent = synth.sorted_random_centroids(7) if rand else None
    c = synth.make_uq_case(260 + P + int(rand), lens, 2, 8, 64, 288, centroids=cent)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    max_tokens = c.block_table.shape[1] * c.block_size
    w = _warps_per_item(c.num_seqs * c.num_kv_heads * P, max_tokens, P, sms)
    if sms == 152:
        assert w == want_w
    out, _, _ = UqDev(c).run(P)
    _check(c, out.cpu().double().numpy(), what=f"W={w} P={P}")


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

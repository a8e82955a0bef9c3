"""GPU parity of pa_decode_fp8 against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import quantized_paged_attention_gb300 as qpa
import synth
from _gpu import Fp8Dev, check_attention, fp8_v_absmax
from _oracle_pool import check_units, fp8_reference
from oracle.attention import dense_kv_fp8, partition_partials

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _oracle(c, units=None):
    return oracle.pa_decode_fp8(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, c.k_scale, c.v_scale,
                                c.query_group, c.softmax_scale, units=units)


def _check(c, got, units=None, what=""):
    ref = _oracle(c, units)
    return check_attention(got, ref, lambda s, h: fp8_v_absmax(c, s, h), c, units, what)


def test_tiny_config():
    """2 seqs (37, 200), 1 KV head, group 8, block 16, 32 permuted blocks, P=2."""
    c = synth.fp8_tiny()
    out, _, _ = Fp8Dev(c).run(2)
    _check(c, out.cpu().double().numpy(), what="tiny")


def _check_slots_cover(c, O, m, l, s, h, P, what):
    """The slots of (sequence s, head h) hold the softmax states of
    consecutive runs of 256-token tile groups that cover the sequence, in slot
    order; every other slot is empty (m = -inf, l = 0)."""
    QG = c.query_group
    L = int(c.seq_lens[s])
    q = oracle.decode_bf16(c.q_bits)[s, h * QG:(h + 1) * QG]
    k, v = dense_kv_fp8(c.kv_cache, c.block_table, s, h, L, c.k_scale, c.v_scale)
    T = -(-L // 256)
    live = [pp for pp in range(P) if l[s, h, pp].max() > 0]
    for pp in range(P):
        if pp not in live:
            assert np.all(np.isneginf(m[s, h, pp])) and np.all(l[s, h, pp] == 0), f"{what}: slot {pp} not empty"
    vmax = float(np.abs(v).max()) if L else 0.0
    b = 0
    for idx, pp in enumerate(live):
        ends = [T] if idx == len(live) - 1 else range(b + 1, T)
        hit = None
        for e in ends:
            t1 = min(e * 256, L)
            rm, rl, rO = partition_partials(q, k[b * 256:t1], v[b * 256:t1], c.softmax_scale, 1)
            if np.max(np.abs(m[s, h, pp] - rm[0])) < 1e-3 and np.max(np.abs(l[s, h, pp] / rl[0] - 1)) < 2e-3:
                hit = e
                break
        assert hit is not None, f"{what}: slot {pp} is no run of tile groups starting at {b}"
        assert np.max(np.abs(O[s, h, pp] - rO[0])) <= 2e-3 * vmax, f"{what}: slot {pp} O"
        b = hit
    assert b == T, f"{what}: runs end at tile group {b} of {T}"


def test_tiny_partials_cover_the_sequence():
    c = synth.fp8_tiny()
    P = 2
    out, ws, desc = Fp8Dev(c).run(P)
    O, m, l = [t.cpu().double().numpy() for t in qpa.fp8_workspace_views(ws, desc, P)]
    for s in range(c.num_seqs):
        _check_slots_cover(c, O, m, l, s, 0, P, "tiny")


@pytest.mark.parametrize("P", [1, 2, 3, 7, 32])
def test_partials_cover_ragged(P):
    """Runs of tile groups per slot, on sequences of 0..9 tile groups, with
    one to 32 slots."""
    c = synth.make_fp8_case(70 + P, [0, 1, 255, 256, 257, 700, 1500, 2304, 40, 900], 2, 8)
    out, ws, desc = Fp8Dev(c).run(P)
    O, m, l = [t.cpu().double().numpy() for t in qpa.fp8_workspace_views(ws, desc, P)]
    for s in range(c.num_seqs):
        for h in range(2):
            _check_slots_cover(c, O, m, l, s, h, P, f"P={P} seq {s} head {h}")
    _check(c, out.cpu().double().numpy(), what=f"cover P={P}")


@pytest.mark.parametrize("P", [1, 2, 3, 7, 32, 100, 300])
def test_partition_counts_ragged(P):
    # P = 300 takes two rounds of the combine kernel's partition loads
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 255, 256, 257, 1000, 2049]
    c = synth.make_fp8_case(40 + P, lens, 2, 8, 128, 16)
    out, _, _ = Fp8Dev(c).run(P)
    _check(c, out.cpu().double().numpy(), what=f"P={P}")


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
def test_block_sizes(bs):
    lens = [1, bs - 1, bs, bs + 1, 300, 777]
    c = synth.make_fp8_case(60 + bs, lens, 2, 8, 128, bs)
    out, _, _ = Fp8Dev(c).run(3)
    _check(c, out.cpu().double().numpy(), what=f"bs={bs}")


@pytest.mark.parametrize("qg", [1, 4, 6, 8, 12, 16, 24, 32, 64])
def test_query_groups(qg):
    c = synth.make_fp8_case(80 + qg, [5, 129, 600], 2, qg, 128, 16)
    out, _, _ = Fp8Dev(c).run(2)
    _check(c, out.cpu().double().numpy(), what=f"qg={qg}")


def test_strided_query_from_fused_qkv():
    c = synth.make_fp8_case(91, [100, 300], 2, 8, 128, 16)
    d = Fp8Dev(c)
    B, Hq, D = c.q_bits.shape
    Hk = c.num_kv_heads
    qkv = torch.randn(B, Hq + 2 * Hk, D, device=d.q.device).to(torch.bfloat16)
    qkv[:, :Hq] = d.q
    out, _, _ = d.run(4, q=qkv[:, :Hq])
    _check(c, out.cpu().double().numpy(), what="strided q")


def test_bf16_output():
    c = synth.make_fp8_case(92, [50, 513], 1, 8, 128, 16)
    out, _, _ = Fp8Dev(c).run(2, out_dtype=torch.bfloat16)
    assert out.dtype == torch.bfloat16
    got = out.float().cpu().double().numpy()
    ref = _oracle(c)
    # bf16 output rounding adds up to 2^-8 |o| on top of the kernel error
    for s in range(2):
        vmax = fp8_v_absmax(c, s, 0)
        assert np.max(np.abs(got[s] - ref[s])) <= 2e-3 * vmax + np.max(np.abs(ref[s])) * 2 ** -8


def test_scales_and_softmax_scale():
    c = synth.make_fp8_case(93, [333], 1, 8, 128, 16, k_scale=0.3, v_scale=2.5, softmax_scale=0.02)
    out, _, _ = Fp8Dev(c).run(2)
    _check(c, out.cpu().double().numpy(), what="scales")


def test_repeat_is_deterministic():
    c = synth.make_fp8_case(94, [1000, 37], 2, 8, 128, 16)
    d = Fp8Dev(c)
    a, ws, _ = d.run(5)
    b, _, _ = d.run(5, workspace=ws)
    assert torch.equal(a, b)


def test_bounded_wait_runs_out_and_the_next_call_is_clean():
    """The timeout path: with the test-only flag, copy warp 0 withholds its
    arrival on its CTA's first tile, so the roles waiting for that tile run
    into their time limit. The call returns, the error word reports a timeout
    (1 or 2), and a normal call in the same process then passes parity."""
    import time
    c = synth.make_fp8_case(96, [700, 300, 5000], 2, 8, 128, 16)
    d = Fp8Dev(c)
    desc = d.desc()
    desc.test_flags = qpa.QPA_TEST_WITHHOLD_ARRIVAL
    ws = qpa.alloc_workspace(qpa.pa_decode_fp8_workspace_size(desc, 3), d.q.device)
    t0 = time.time()
    qpa.pa_decode_fp8(d.q, d.kv, d.bt, d.sl, d.ks, d.vs, 3, 8, workspace=ws, desc=desc)
    assert qpa.kernel_error() in (1, 2)
    assert time.time() - t0 < 60
    assert qpa.kernel_error() == 0                      # reading cleared it
    out, _, _ = d.run(3)                                # a normal call: error word stays 0 (checked in run)
    _check(c, out.cpu().double().numpy(), what="after the timeout")


def test_invalid_block_id_raises_error_word():
    c = synth.make_fp8_case(95, [40], 1, 8, 128, 16)
    c.block_table[0, 1] = c.kv_cache.shape[0] + 5       # past the cache
    d = Fp8Dev(c)
    desc = d.desc()
    ws = qpa.alloc_workspace(qpa.pa_decode_fp8_workspace_size(desc, 1), d.q.device)
    qpa.pa_decode_fp8(d.q, d.kv, d.bt, d.sl, d.ks, d.vs, 1, 8, workspace=ws, desc=desc)
    assert qpa.kernel_error() == 3
    assert qpa.kernel_error() == 0                      # reading clears it


def test_full_gqa_config_all_units():
    """16 seqs x 16384, 8 KV heads, group 8, P=32 (512-token partitions), as
    the benchmark runs it; every one of the 128 (seq, head) units against the
    oracle, element by element."""
    c = synth.fp8_gqa()
    out, _, _ = Fp8Dev(c).run(32)
    check_units(out.cpu().double().numpy(), fp8_reference(c), c, what="gqa-full")


def test_full_ragged_config_all_units():
    """128 seqs, lengths U[1024, 16384], P=32; all 1024 (seq, head) units."""
    c = synth.fp8_ragged()
    out, _, _ = Fp8Dev(c).run(32)
    check_units(out.cpu().double().numpy(), fp8_reference(c), c, what="ragged-full")


# ---- head_dim 64 ([PA]: head_dim 64 or 128)
@pytest.mark.parametrize("P", [1, 3, 32])
@pytest.mark.parametrize("qg", [8, 16, 5, 48])
def test_head_dim_64(P, qg):
    c = synth.make_fp8_case(900 + P + qg, [0, 1, 127, 128, 129, 255, 256, 257, 1000, 3000], 2, qg, head_dim=64)
    out, _, _ = Fp8Dev(c).run(P)
    _check(c, out.cpu().double().numpy(), what=f"hd64 P={P} qg={qg}")


@pytest.mark.parametrize("bs", [32, 64, 256])
def test_head_dim_64_block_sizes_and_bf16(bs):
    c = synth.make_fp8_case(930 + bs, [1, bs - 1, bs + 1, 2000], 2, 8, head_dim=64, block_size=bs)
    d = Fp8Dev(c)
    out, _, _ = d.run(4)
    _check(c, out.cpu().double().numpy(), what=f"hd64 bs={bs}")
    o16, _, _ = d.run(4, out_dtype=torch.bfloat16)
    assert torch.max(torch.abs(o16.float() - out)).item() <= torch.max(torch.abs(out)).item() * 2 ** -8 + 1e-6


@pytest.mark.parametrize("qg,P", [(1, 1), (3, 2), (8, 1), (8, 7), (5, 40)])
def test_head_dim_64_packed_halves(qg, P):
    """head_dim 64 with at most 8 query rows takes a 256-token tile group per
    pass as two 128-token halves: sequences ending inside the first half, at
    its end, one token into the second half and inside it, over block size 16
    (a half spans several blocks), with partition counts from 1 to above the
    tile groups of a sequence; all (seq, head) units against the oracle."""
    lens = [0, 1, 100, 128, 129, 200, 256, 257, 383, 384, 385, 511, 700, 1500]
    c = synth.make_fp8_case(990 + 10 * qg + P, lens, 3, qg, head_dim=64, block_size=16)
    out, _, _ = Fp8Dev(c).run(P)
    _check(c, out.cpu().double().numpy(), what=f"hd64 packed qg={qg} P={P}")


@pytest.mark.parametrize("P", [1, 5, 32])
def test_wide_group_partition_counts(P):
    """Query group 32 (two blocks of 16 rows over one KV head's pages) with
    ragged lengths and several partition counts."""
    c = synth.make_fp8_case(970 + P, [0, 1, 255, 257, 1500, 4000], 3, 32, 128, 16)
    out, _, _ = Fp8Dev(c).run(P)
    _check(c, out.cpu().double().numpy(), what=f"qg32 P={P}")


def test_head_dim_64_long_all_units():
    """16 seqs x 16384 tokens, 8 KV heads, group 8, head_dim 64, P = 32 (the
    benchmark's head_dim 64 line); all 128 (seq, head) units."""
    c = synth.make_fp8_case(960, [16384] * 16, 8, 8, head_dim=64, poison=False)
    out, _, _ = Fp8Dev(c).run(32)
    check_units(out.cpu().double().numpy(), fp8_reference(c), c, what="hd64 long")


@pytest.mark.parametrize("qg", [8, 16])
def test_query_rows_with_a_wide_dynamic_range(qg):
    """Query rows with one outlier (+-64) and the other elements log-uniform
    in 2^-24 .. 1 (massive-activation rows): the query enters as e4m3 terms (4
    with up to 8 rows per KV head, 2 with 16), exact down to 2^-22 resp. 2^-14
    of the row maximum; many elements fall below the 2-term bound, and the
    result still matches the float64 oracle within the tolerance."""
    c = synth.make_fp8_case(720 + qg, [300, 2049, 5000], 2, qg, 128, 16)
    r = np.random.default_rng(720 + qg)
    shape = c.q_bits.shape
    q = np.where(r.random(shape) < 0.5, -1.0, 1.0) * 2.0 ** r.uniform(-24.0, 0.0, shape)
    q[..., 0] = np.where(r.random(shape[:-1]) < 0.5, -64.0, 64.0)
    c.q_bits = synth.round_to_bf16_bits(q.astype(np.float32))
    out, _, _ = Fp8Dev(c).run(3)
    _check(c, out.cpu().double().numpy(), what=f"wide-range q, group {qg}")

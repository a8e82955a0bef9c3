"""GPU parity of pa_decode_fp8_ext (query_len new tokens per sequence with
the causal mask inside the query block; per-tensor or per-token K/V scales)
against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_paged_attention_gb300 as qpa
from _gpu import ATT_TOL, bf16_tensor, dev
from _oracle_pool import check_units, fp8_ext_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _run(c, P, out_dtype=torch.float32):
    d = dev()
    q = bf16_tensor(c.q_bits, d)
    kv = torch.from_numpy(c.kv_cache).to(d)
    bt = torch.from_numpy(c.block_table).to(d)
    sl = torch.from_numpy(c.seq_lens).to(d)
    if c.per_token:
        ks = torch.from_numpy(np.ascontiguousarray(c.k_scale, dtype=np.float32)).to(d)
        vs = torch.from_numpy(np.ascontiguousarray(c.v_scale, dtype=np.float32)).to(d)
    else:
        ks = torch.tensor([c.k_scale], dtype=torch.float32, device=d)
        vs = torch.tensor([c.v_scale], dtype=torch.float32, device=d)
    out = qpa.pa_decode_fp8_ext(q, kv, bt, sl, ks, vs, P, c.query_group, softmax_scale=c.softmax_scale,
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert qpa.kernel_error() == 0
    return out.float().cpu().double().numpy()


def _v_absmax(c, s, h):
    L = int(c.seq_lens[s])
    if L == 0:
        return 0.0
    if c.per_token:
        _, v = oracle.attention.dense_kv_fp8_per_token(c.kv_cache, c.block_table, s, h, L, c.k_scale, c.v_scale)
    else:
        _, v = oracle.attention.dense_kv_fp8(c.kv_cache, c.block_table, s, h, L, c.k_scale, c.v_scale)
    return float(np.abs(v).max())


def _check(c, got, units=None, what=""):
    ref = oracle.pa_decode_fp8_ext(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, c.k_scale, c.v_scale,
                                   c.query_group, c.query_len, c.softmax_scale, units=units)
    QG, QL = c.query_group, c.query_len
    if units is None:
        units = [(s, h) for s in range(c.num_seqs) for h in range(c.num_kv_heads)]
    for s, h in units:
        g = got[s, :, h * QG:(h + 1) * QG]
        r = ref[s, :, h * QG:(h + 1) * QG]
        assert np.all(np.isfinite(g)), f"{what} non-finite output at seq {s} head {h}"
        L = int(c.seq_lens[s])
        for qoff in range(QL):
            if L - QL + 1 + qoff <= 0:
                assert np.all(g[qoff] == 0.0), f"{what} a row with no visible token must give 0"
        tol = ATT_TOL * _v_absmax(c, s, h)
        err = float(np.max(np.abs(g - r)))
        assert err <= tol, f"{what} seq {s} head {h}: max|err| {err:.3e} > tol {tol:.3e}"


LENS = [0, 1, 2, 3, 15, 16, 17, 63, 64, 65, 255, 256, 257, 1000, 2049]


@pytest.mark.parametrize("per_token", [False, True])
@pytest.mark.parametrize("ql,qg", [(1, 8), (2, 8), (3, 4), (4, 4), (1, 16), (4, 2),
                                   # above 16 rows: blocks of 16 query rows
                                   (3, 8), (4, 8), (2, 16), (4, 16), (1, 24), (3, 7)])
def test_query_len_and_scales(ql, qg, per_token):
    c = synth.make_fp8_ext_case(500 + 10 * ql + qg + (7 if per_token else 0), LENS, 2, qg, ql, per_token)
    _check(c, _run(c, 3), what=f"ql={ql} qg={qg} per_token={per_token}")


@pytest.mark.parametrize("per_token", [False, True])
@pytest.mark.parametrize("ql,qg,P", [(1, 8, 2), (4, 4, 3), (2, 8, 1), (4, 8, 7), (3, 16, 2)])
def test_head_dim_64(ql, qg, P, per_token):
    """head_dim 64 with several query tokens and per-token scales ([PA]'s
    phase-split head_dim 64 commit times per_token MTP shapes)."""
    c = synth.make_fp8_ext_case(620 + 10 * ql + qg + P + (5 if per_token else 0), LENS, 2, qg, ql, per_token,
                                head_dim=64)
    _check(c, _run(c, P), what=f"hd64 ql={ql} qg={qg} P={P} per_token={per_token}")


@pytest.mark.parametrize("P", [1, 2, 7, 32, 300])
def test_partition_counts(P):
    c = synth.make_fp8_ext_case(540 + P, LENS, 1, 4, 4, True)
    _check(c, _run(c, P), what=f"P={P}")


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
def test_block_sizes(bs):
    c = synth.make_fp8_ext_case(560 + bs, [1, 4, bs - 1, bs, bs + 1, 700], 2, 8, 2, True, block_size=bs)
    _check(c, _run(c, 3), what=f"bs={bs}")


def test_single_query_token_matches_plain_decode():
    """query_len 1 with per-tensor scales is the plain decode's operation."""
    c = synth.make_fp8_ext_case(580, [5, 300, 1025], 2, 8, 1, False)
    got = _run(c, 4)[:, 0]
    ref = oracle.pa_decode_fp8(c.q_bits[:, 0], c.kv_cache, c.block_table, c.seq_lens, c.k_scale, c.v_scale,
                               c.query_group, c.softmax_scale)
    for s in range(c.num_seqs):
        for h in range(c.num_kv_heads):
            tol = ATT_TOL * _v_absmax(c, s, h)
            assert np.max(np.abs(got[s, h * 8:(h + 1) * 8] - ref[s, h * 8:(h + 1) * 8])) <= tol


def test_bf16_output():
    c = synth.make_fp8_ext_case(590, [100, 333], 2, 4, 4, True)
    a = _run(c, 2)
    b = _run(c, 2, out_dtype=torch.bfloat16)
    assert np.max(np.abs(a - b)) <= np.max(np.abs(a)) * 2 ** -8 + 1e-6


def test_long_group8_four_tokens_all_units():
    """16 seqs x 16384 tokens, 8 KV heads, group 8, 4 query tokens (32 rows:
    two row blocks), per-token scales, P = 32 (the benchmark's line); all 128
    units against the oracle."""
    c = synth.make_fp8_ext_case(610, [16384] * 16, 8, 8, 4, True, poison=False)
    check_units(_run(c, 32), fp8_ext_reference(c), c, what="long ql4 qg8")


def test_long_sequences_all_units():
    """16 seqs x 16384 tokens, 8 KV heads, group 4, 4 query tokens, per-token
    scales, P = 32; all 128 (seq, head) units against the oracle."""
    c = synth.make_fp8_ext_case(600, [16384] * 16, 8, 4, 4, True, poison=False)
    check_units(_run(c, 32), fp8_ext_reference(c), c, what="long")

"""GPU parity of nvfp4_index_score against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import IdxDev, check_scores
from _oracle_pool import idx_reference

pytestmark = pytest.mark.gpu

# page strides: the dense 9216 bytes and 9232 (pages in a wider buffer)
KERNELS = {"dense": 0, "stride9232": 16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _ref(c, reqs=None):
    return oracle.nvfp4_index_score(c.q_codes, c.pages, c.block_table, c.seq_lens, c.query_len, c.num_cols,
                                    reqs=reqs)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("ql,h", [(4, 2), (1, 1), (2, 4), (3, 2), (4, 4), (1, 16), (8, 2)])
def test_small_ragged(ql, h, kernel):
    lens = [0, 1, 3, 4, 5, 127, 128, 129, 255, 256, 257, 1000]
    c = synth.make_idx_case(300 + ql * 10 + h, lens, query_len=ql, num_heads=h, num_cols=12)
    got = IdxDev(c, stride_pad=KERNELS[kernel]).run().cpu().double().numpy()
    check_scores(got, _ref(c), what=f"{kernel} ql={ql} h={h}")


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_many_short_requests_and_table_entries(kernel):
    """300 requests of 0..700 tokens (most CTAs take pages of several
    requests, so the query operand changes many times per CTA) and a table
    wider than the columns."""
    r = np.random.default_rng(9)
    lens = [int(x) for x in r.integers(0, 700, 300)]
    c = synth.make_idx_case(309, lens, query_len=2, num_heads=4, num_cols=5)
    got = IdxDev(c, stride_pad=KERNELS[kernel]).run().cpu().double().numpy()
    check_scores(got, _ref(c), what=f"{kernel} many requests")


def test_columns_beyond_blocks_and_table_width():
    c = synth.make_idx_case(320, [300, 900], query_len=4, num_heads=2, num_cols=20)
    got = IdxDev(c).run().cpu().double().numpy()
    check_scores(got, _ref(c), what="wide")
    assert np.all(np.isneginf(got[:, :, 8:]))


def test_strided_scores_output():
    c = synth.make_idx_case(321, [500, 40, 1300], query_len=4, num_heads=2, num_cols=11)
    d = IdxDev(c)
    big = torch.full((2, 12, 16), 7.0, device=d.q.device)
    view = big[:, :, :11]
    d.run(scores=view)
    got = big.cpu().double().numpy()
    check_scores(got[:, :, :11], _ref(c), what="strided")
    assert np.all(got[:, :, 11:] == 7.0)      # nothing written outside the view


def test_repeat_is_deterministic():
    c = synth.make_idx_case(322, [4000, 2500], query_len=4, num_heads=2, num_cols=32)
    d = IdxDev(c)
    a = d.run().clone()
    b = d.run()
    assert torch.equal(a, b)


def _check_all_requests(c, got, per_token_cols=None, what=""):
    """Every request's score rows against the oracle (one pool task per
    request)."""
    ref = idx_reference(c, per_token_cols=per_token_cols)
    ql = c.query_len
    full = np.stack([ref[r] for r in range(c.num_reqs)], axis=1)      # [H, R, QL, cols]
    full = full.reshape(full.shape[0], c.num_reqs * ql, full.shape[-1])
    check_scores(got, full, what=what)


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_full_config_all_requests(kernel):
    """64 requests, lengths U[4096, 32768], query_len 4, 2 heads, S=256 (as
    the benchmark runs it); all 64 requests against the oracle."""
    c = synth.idx_full()
    _check_all_requests(c, IdxDev(c, stride_pad=KERNELS[kernel]).run().cpu().double().numpy(),
                        what=f"idx-full {kernel}")


# ---- per-token output
def _ref_tok(c, cols, reqs=None):
    return oracle.nvfp4_index_score_per_token(c.q_codes, c.pages, c.block_table, c.seq_lens, c.query_len, cols,
                                              reqs=reqs)


@pytest.mark.parametrize("ql,h", [(4, 2), (1, 1), (3, 4)])
@pytest.mark.parametrize("cols", [1536, 1000, 77])
def test_per_token_small_ragged(ql, h, cols):
    """Token columns past the table (1536 > 12 blocks), ending inside a block
    (1000) and short of most requests (77); both kernels."""
    lens = [0, 1, 3, 4, 5, 127, 128, 129, 255, 256, 257, 1000]
    c = synth.make_idx_case(330 + ql * 10 + h, lens, query_len=ql, num_heads=h, num_cols=12)
    for kernel, pad in KERNELS.items():
        got = IdxDev(c, stride_pad=pad).run(per_token_cols=cols).cpu().double().numpy()
        check_scores(got, _ref_tok(c, cols), what=f"{kernel} per-token ql={ql} h={h} cols={cols}")


def test_per_token_strided_and_block_max():
    c = synth.make_idx_case(340, [500, 40, 1300], query_len=4, num_heads=2, num_cols=11)
    d = IdxDev(c)
    big = torch.full((2, 12, 1500), 7.0, device=d.q.device)
    view = big[:, :, :1408]
    d.run(scores=view, per_token_cols=1408)
    got = big.cpu().double().numpy()
    check_scores(got[:, :, :1408], _ref_tok(c, 1408), what="per-token strided")
    assert np.all(got[:, :, 1408:] == 7.0)
    blk = d.run().cpu().double().numpy()                 # the block max of the same dots
    assert np.array_equal(got[:, :, :1408].reshape(2, 12, 11, 128).max(axis=3), blk)


def test_per_token_full_config_all_requests():
    """64 requests, lengths U[4096, 32768], query_len 4, 2 heads, 32768 token
    columns; all 64 requests against the oracle."""
    c = synth.idx_full()
    got = IdxDev(c).run(per_token_cols=32768).cpu().double().numpy()
    _check_all_requests(c, got, per_token_cols=32768, what="idx-full per-token")


def test_shared_prefix_pages():
    """Requests whose first blocks map the same physical pages (a shared
    prefix): every request's scores against the oracle."""
    c = synth.make_idx_case(350, [300, 700, 1000, 256, 129, 900], query_len=4, num_heads=2, num_cols=9,
                            shared_prefix_blocks=2)
    assert np.all(c.block_table[:, :2] == c.block_table[0, :2])
    got = IdxDev(c).run().cpu().double().numpy()
    check_scores(got, _ref(c), what="shared prefix")


def test_shared_prefix_full_all_requests():
    """64 requests, lengths U[16384, 32768], 128 shared prefix pages (the
    benchmark's shared-prefix line); all 64 requests against the oracle."""
    c = synth.idx_shared_prefix()
    _check_all_requests(c, IdxDev(c).run().cpu().double().numpy(), what="shared prefix full")


# ---- page-by-page dedup of shared pages (QPA_IDX_SHARED_PAGES)
@pytest.mark.parametrize("ql,h", [(4, 2), (1, 1), (3, 4), (2, 4)])
@pytest.mark.parametrize("shared", [0, 2, 5])
def test_shared_pages_flag_small(ql, h, shared):
    """The dedup split against the oracle and bit for bit against the
    request-by-request split (the same dequantisation and MMA tiles), with and without a shared prefix, on ragged lengths (requests
    shorter than the prefix, empty requests, a group of 8 cut short)."""
    lens = [0, 1, 130, 300, 700, 1000, 256, 129, 900, 5, 640, 777, 3]
    c = synth.make_idx_case(400 + 10 * ql + h + shared, lens, query_len=ql, num_heads=h, num_cols=9,
                            shared_prefix_blocks=shared)
    got = IdxDev(c).run(shared_pages=True)
    check_scores(got.cpu().double().numpy(), _ref(c), what=f"shared flag ql={ql} h={h} prefix={shared}")
    assert torch.equal(got, IdxDev(c, stride_pad=KERNELS["stride9232"]).run())


@pytest.mark.parametrize("cols", [1536, 700])
def test_shared_pages_flag_per_token(cols):
    c = synth.make_idx_case(430, [300, 700, 1000, 256, 129, 900, 64, 1100, 33], query_len=4, num_heads=2,
                            num_cols=9, shared_prefix_blocks=3)
    got = IdxDev(c).run(per_token_cols=cols, shared_pages=True)
    check_scores(got.cpu().double().numpy(), _ref_tok(c, cols), what=f"shared flag per-token cols={cols}")
    assert torch.equal(got, IdxDev(c, stride_pad=KERNELS["stride9232"]).run(per_token_cols=cols))


def test_shared_pages_flag_full_prefix_workload_all_requests():
    """The benchmark's shared-prefix workload (64 requests sharing 128 prefix
    pages) through the dedup split: all requests against the oracle."""
    c = synth.idx_shared_prefix()
    got = IdxDev(c).run(shared_pages=True)
    _check_all_requests(c, got.cpu().double().numpy(), what="shared prefix dedup")
    assert torch.equal(got, IdxDev(c, stride_pad=KERNELS["stride9232"]).run())


def test_shared_pages_flag_unshared_full_workload():
    """The unshared 64-request workload through the dedup split (every page
    has one mapper): identical to the request-by-request split."""
    c = synth.idx_full()
    assert torch.equal(IdxDev(c).run(shared_pages=True), IdxDev(c, stride_pad=KERNELS["stride9232"]).run())

"""The allocation-free fp8 entry point, pa_decode_fp8_static, called through
the C ABI. It exists for callers that cannot allocate device memory (their
host framework owns every allocation, or all device memory is reserved up
front), so it keeps its partials in the library's static device array
instead of a caller workspace.

Checked: two calls in a row give the same output as pa_decode_fp8, bit for
bit and within the attention tolerance of the parity tests (2e-3 * max|V|
of each sequence) of the float64 oracle, after a larger call with more
partitions has left its partials in the array; and a request larger than
the array is refused without a launch.

This file is collected last, so a failing run that stops at the first
failure has already run every other test; it also passes on its own in a
fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_paged_attention_gb300 as qpa
import synth
from _gpu import Fp8Dev, fp8_v_absmax

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return qpa.load_library()


def _static_call(lib, d, P, out, desc):
    return lib.pa_decode_fp8_static(qpa._ptr(d.q), qpa._ptr(d.kv), qpa._ptr(d.bt), qpa._ptr(d.sl),
                                    qpa._ptr(d.ks), qpa._ptr(d.vs), P, qpa._ptr(out), ctypes.byref(desc),
                                    qpa._stream(None))


@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_static_matches_workspace_entry_point_twice(lib, case):
    if case == "tiny":
        c, P = synth.fp8_tiny(), 2
    else:
        c, P = synth.make_fp8_case(7, [1000, 37, 0, 333, 2049], 2, 8, 128, 16), 5
    # a larger call first, with more partitions and another shape, so that the
    # shared array holds stale partials where the checked calls put theirs
    big = synth.make_fp8_case(8, [3000, 2500, 700, 64, 5000], 4, 8, 128, 16)
    bd = Fp8Dev(big)
    bout = torch.empty(bd.q.shape, dtype=torch.float32, device=bd.q.device)
    assert _static_call(lib, bd, 40, bout, bd.desc()) == 0
    torch.cuda.synchronize()
    assert qpa.kernel_error() == 0

    d = Fp8Dev(c)
    ref_t, _, desc = d.run(P)                      # pa_decode_fp8 with a workspace
    ref = ref_t.cpu().double().numpy()
    want = oracle.pa_decode_fp8(c.q_bits, c.kv_cache, c.block_table, c.seq_lens, c.k_scale, c.v_scale,
                                c.query_group, c.softmax_scale)
    for _ in range(2):                             # two calls in a row share the static array
        out = torch.full(d.q.shape, float("nan"), dtype=torch.float32, device=d.q.device)
        assert _static_call(lib, d, P, out, desc) == 0
        torch.cuda.synchronize()
        assert qpa.kernel_error() == 0
        assert torch.equal(out, ref_t)             # the same kernels on the same inputs
        got = out.cpu().double().numpy()
        for s in range(c.num_seqs):
            for h in range(c.num_kv_heads):
                rows = slice(h * c.query_group, (h + 1) * c.query_group)
                tol = 2e-3 * fp8_v_absmax(c, s, h)
                assert np.max(np.abs(got[s, rows] - ref[s, rows])) <= tol
                assert np.max(np.abs(got[s, rows] - want[s, rows])) <= tol


def test_static_refuses_requests_larger_than_the_array(lib):
    desc = qpa.Fp8Desc()
    desc.num_seqs, desc.num_kv_heads, desc.query_group, desc.head_dim = 16, 8, 8, 128
    desc.block_size, desc.num_blocks, desc.max_blocks_per_seq = 16, 16384, 1024
    need = lib.pa_decode_fp8_workspace_size(ctypes.byref(desc), 32)
    assert need > (8 << 20)
    fake = ctypes.c_void_p(0x100000)     # never dereferenced: the call is refused on the host
    st = lib.pa_decode_fp8_static(fake, fake, fake, fake, fake, fake, 32, fake, ctypes.byref(desc), None)
    assert st == -4                      # QPA_ERR_WORKSPACE

"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_paged_attention_gb300 as qpa
    return qpa.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "qpa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = "\n".join(l for l in src.splitlines() if not l.lstrip().startswith("#"))
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\([^;{]*\)\s*;", src)
    return sorted(set(n for n in names if n not in ("sizeof",)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "pa_decode_fp8" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_header():
    import quantized_paged_attention_gb300 as qpa
    assert set(_declared_functions()) <= set(qpa.declared_symbols())


def test_status_strings(lib):
    assert lib.qpa_status_string(0) == b"ok"
    assert b"partitions" in lib.qpa_status_string(-5)


def _desc(**kw):
    import quantized_paged_attention_gb300 as qpa
    d = qpa.Fp8Desc()
    d.num_seqs, d.num_kv_heads, d.query_group, d.head_dim = 2, 1, 8, 128
    d.block_size, d.num_blocks, d.max_blocks_per_seq, d.out_dtype = 16, 32, 13, 0
    for k, v in kw.items():
        setattr(d, k, v)
    return d


FAKE = ctypes.c_void_p(0x100000)      # never dereferenced: every call below fails validation


def _call(lib, d, P=2, ws_bytes=1 << 20, q=FAKE, ws=FAKE):
    return lib.pa_decode_fp8(q, FAKE, FAKE, FAKE, FAKE, FAKE, P, FAKE, ctypes.byref(d), ws, ws_bytes, None)


def test_host_validation(lib):
    assert _call(lib, _desc(), P=0) == -5
    assert _call(lib, _desc(head_dim=96)) == -2
    assert _call(lib, _desc(block_size=24)) == -2
    assert _call(lib, _desc(query_group=65)) == -2               # up to 64 query rows per KV head
    assert _call(lib, _desc(), q=ctypes.c_void_p(0)) == -1
    assert _call(lib, _desc(), q=ctypes.c_void_p(0x100008)) == -3
    assert _call(lib, _desc(q_stride_head=100)) == -3
    assert _call(lib, _desc(), ws_bytes=16) == -4
    assert lib.pa_decode_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, FAKE, None, FAKE, 1, None) == -1


def test_workspace_size(lib):
    d = _desc()
    n = lib.pa_decode_fp8_workspace_size(ctypes.byref(d), 2)
    rows = 2 * 1 * 2 * 8
    assert n >= rows * 130 * 4 and n % 256 == 0
    assert lib.pa_decode_fp8_workspace_size(ctypes.byref(_desc(head_dim=96)), 2) == 0
    # head_dim 64 with a group of at most 8 keeps both 64-dim halves of each
    # partial row (the packed kernel): as many floats per row as head_dim 128
    n64 = lib.pa_decode_fp8_workspace_size(ctypes.byref(_desc(head_dim=64)), 2)
    assert n64 >= rows * 130 * 4
    n64w = lib.pa_decode_fp8_workspace_size(ctypes.byref(_desc(head_dim=64, query_group=16)), 2)
    n128w = lib.pa_decode_fp8_workspace_size(ctypes.byref(_desc(query_group=16)), 2)
    assert 2 * rows * 66 * 4 <= n64w < n128w


def _ext_desc(query_len=2, per_token=1, **kw):
    import quantized_paged_attention_gb300 as qpa
    d = qpa.Fp8ExtDesc()
    d.base = _desc(**kw)
    d.query_len = query_len
    d.kv_scale_per_token = per_token
    return d


def _call_ext(lib, d, P=2, ws_bytes=1 << 20, ks=FAKE):
    return lib.pa_decode_fp8_ext(FAKE, FAKE, FAKE, FAKE, ks, FAKE, P, FAKE, ctypes.byref(d), FAKE, ws_bytes, None)


def test_ext_host_validation(lib):
    assert _call_ext(lib, _ext_desc(), P=0) == -5
    assert _call_ext(lib, _ext_desc(query_len=5)) == -2
    assert _call_ext(lib, _ext_desc(query_len=4, query_group=17)) == -2     # 68 rows > 64
    assert _call_ext(lib, _ext_desc(query_len=4, query_group=4), ws_bytes=16) == -4
    assert _call_ext(lib, _ext_desc(per_token=2)) == -2
    assert _call_ext(lib, _ext_desc(), ks=ctypes.c_void_p(0x100004)) == -3    # per-token scales need 16 B
    assert _call_ext(lib, _ext_desc(per_token=0), ks=ctypes.c_void_p(0x100004), ws_bytes=16) == -4
    assert _call_ext(lib, _ext_desc(), ks=ctypes.c_void_p(0)) == -1


def test_ext_workspace_size(lib):
    n = lib.pa_decode_fp8_ext_workspace_size(ctypes.byref(_ext_desc(query_len=2, query_group=8)), 3)
    rows = 2 * 1 * 3 * 16
    assert n >= rows * 130 * 4 and n % 256 == 0
    n24 = lib.pa_decode_fp8_ext_workspace_size(ctypes.byref(_ext_desc(query_len=3, query_group=8)), 3)
    assert n24 >= 2 * 1 * 3 * 24 * 130 * 4                       # 24 rows: two row blocks
    assert lib.pa_decode_fp8_ext_workspace_size(ctypes.byref(_ext_desc(query_len=4, query_group=17)), 3) == 0
    # query_len 0 means one query token
    one = lib.pa_decode_fp8_ext_workspace_size(ctypes.byref(_ext_desc(query_len=0)), 2)
    assert one == lib.pa_decode_fp8_workspace_size(ctypes.byref(_desc()), 2)
    # head_dim 64: rows of 64 partial values
    n64 = lib.pa_decode_fp8_ext_workspace_size(ctypes.byref(_ext_desc(query_len=2, head_dim=64)), 2)
    assert n64 >= 2 * 1 * 2 * 16 * 66 * 4 and n64 < lib.pa_decode_fp8_ext_workspace_size(
        ctypes.byref(_ext_desc(query_len=2)), 2)


def _uq_desc(**kw):
    import quantized_paged_attention_gb300 as qpa
    d = qpa.UqDesc()
    d.num_seqs, d.num_kv_heads, d.query_group, d.head_dim = 2, 2, 8, 256
    d.block_size, d.num_blocks, d.max_blocks_per_seq, d.padded_slot = 64, 8, 4, 288
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_idx_flags_validation(lib):
    import quantized_paged_attention_gb300 as qpa
    assert qpa.IdxDesc.flags.offset == 28
    d = qpa.IdxDesc()
    d.num_reqs, d.query_len, d.num_heads, d.head_dim = 2, 4, 2, 128
    d.num_blocks, d.max_blocks_per_seq, d.num_cols = 8, 4, 512
    for f, want in ((4, -2), (-1, -2)):
        d.flags = f
        assert lib.nvfp4_index_score(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(d), None) == want
    for f in (1, 2, 3):        # per-token output, shared-page split, both
        d.flags = f
        assert lib.nvfp4_index_score(ctypes.c_void_p(0), FAKE, FAKE, FAKE, FAKE, ctypes.byref(d), None) == -1


def test_uq_flags_validation(lib):
    import quantized_paged_attention_gb300 as qpa
    assert qpa.UqDesc.flags.offset == 36 and ctypes.sizeof(qpa.UqDesc) == 64
    for f in range(8):
        assert lib.uq_decode_hd256_workspace_size(ctypes.byref(_uq_desc(flags=f)), 3) > 0
    for f in (8, 16, -1):
        assert lib.uq_decode_hd256_workspace_size(ctypes.byref(_uq_desc(flags=f)), 3) == 0
        st = lib.uq_decode_hd256(FAKE, FAKE, FAKE, FAKE, FAKE, 3, FAKE, ctypes.byref(_uq_desc(flags=f)), FAKE,
                                 1 << 20, None)
        assert st == -2

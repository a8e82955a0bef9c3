"""Quantised paged-attention decode for GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``libqpa.so`` (declared in
``include/qpa.h``). It only marshals arguments: every step of the decode runs
in the library's CUDA kernels. PyTorch supplies device memory and streams.
There is no CPU fallback: if the library is missing or a tensor is not on a
CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqpa.so")

QPA_OK = 0
QPA_OUT_F32 = 0
QPA_OUT_BF16 = 1
QPA_UQ_UE8M0_SCALES = 1
QPA_UQ_Q_HAIRCUT = 2
QPA_UQ_ROT_PERM = 4
QPA_IDX_PER_TOKEN = 1
QPA_IDX_SHARED_PAGES = 2
QPA_TEST_WITHHOLD_ARRIVAL = 1
_lib = None


class QpaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = _lib.qpa_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {msg} ({status})")


class Fp8Desc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("query_group", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("q_stride_seq", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
                ("softmax_scale", ctypes.c_float), ("test_flags", ctypes.c_int32)]


class Fp8ExtDesc(ctypes.Structure):
    _fields_ = [("base", Fp8Desc), ("query_len", ctypes.c_int32), ("kv_scale_per_token", ctypes.c_int32),
                ("q_stride_tok", ctypes.c_int64)]


class UqDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("query_group", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("padded_slot", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("q_stride_seq", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
                ("softmax_scale", ctypes.c_float)]


class IdxDesc(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("query_len", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_cols", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("page_stride", ctypes.c_int64), ("q_stride_tok", ctypes.c_int64),
                ("q_stride_head", ctypes.c_int64), ("s_stride_head", ctypes.c_int64),
                ("s_stride_row", ctypes.c_int64)]


_P = ctypes.c_void_p
_SIGS = {
    "qpa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qpa_version": (ctypes.c_int, []),
    "qpa_kernel_error": (ctypes.c_int, [_P]),
    "pa_decode_fp8_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(Fp8Desc), ctypes.c_int]),
    "pa_decode_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, _P,
                                     ctypes.POINTER(Fp8Desc), _P, ctypes.c_size_t, _P]),
    "pa_decode_fp8_partition": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int,
                                               ctypes.POINTER(Fp8Desc), _P, ctypes.c_size_t, _P]),
    "pa_decode_fp8_combine": (ctypes.c_int, [ctypes.c_int, _P, ctypes.POINTER(Fp8Desc), _P,
                                             ctypes.c_size_t, _P]),
    "pa_decode_fp8_static": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, _P,
                                            ctypes.POINTER(Fp8Desc), _P]),
    "pa_decode_fp8_ext_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(Fp8ExtDesc), ctypes.c_int]),
    "pa_decode_fp8_ext": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, _P,
                                         ctypes.POINTER(Fp8ExtDesc), _P, ctypes.c_size_t, _P]),
    "uq_decode_hd256_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(UqDesc), ctypes.c_int]),
    "uq_decode_hd256": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.POINTER(UqDesc), _P,
                                       ctypes.c_size_t, _P]),
    "uq_decode_hd256_partition": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int, ctypes.POINTER(UqDesc),
                                                 _P, ctypes.c_size_t, _P]),
    "uq_decode_hd256_combine": (ctypes.c_int, [ctypes.c_int, _P, ctypes.POINTER(UqDesc), _P,
                                               ctypes.c_size_t, _P]),
    "nvfp4_index_score": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.POINTER(IdxDesc), _P]),
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqpa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libqpa.so not found at {path}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def declared_symbols():
    return list(_SIGS)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("qpa runs on CUDA tensors only (no CPU path)")


def _check(fn, st):
    if st != QPA_OK:
        raise QpaError(fn, st)


def kernel_error(stream=None) -> int:
    """Synchronise the stream and return/clear the device error word."""
    return load_library().qpa_kernel_error(_stream(stream))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------- fp8
def fp8_desc(q, kv_cache, block_table, query_group, softmax_scale=None, out_dtype=torch.float32):
    B, Hq, D = q.shape
    NB, two, Hk, bs, D2 = kv_cache.shape
    assert two == 2 and D2 == D and Hq == Hk * query_group
    d = Fp8Desc()
    d.num_seqs, d.num_kv_heads, d.query_group, d.head_dim = B, Hk, query_group, D
    d.block_size, d.num_blocks, d.max_blocks_per_seq = bs, NB, block_table.shape[1]
    d.out_dtype = QPA_OUT_BF16 if out_dtype == torch.bfloat16 else QPA_OUT_F32
    if q.stride(2) != 1:
        raise ValueError("q must be contiguous along head_dim")
    d.q_stride_seq, d.q_stride_head = q.stride(0), q.stride(1)
    d.softmax_scale = 0.0 if softmax_scale is None else float(softmax_scale)
    return d


def pa_decode_fp8_workspace_size(desc: Fp8Desc, num_partitions: int) -> int:
    return int(load_library().pa_decode_fp8_workspace_size(ctypes.byref(desc), num_partitions))


def pa_decode_fp8(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions: int,
                  query_group: int, out=None, workspace=None, softmax_scale=None,
                  out_dtype=torch.float32, stream=None, desc=None):
    """fp8 paged-attention decode. q bf16 [B, Hq, 128]; kv_cache uint8
    [NB, 2, Hk, bs, 128]; block_table int32 [B, maxb]; seq_lens int32 [B];
    k_scale / v_scale float32 [1] on the device. Returns out [B, Hq, 128]."""
    lib = load_library()
    _need_cuda(q, kv_cache, block_table, seq_lens, k_scale, v_scale)
    if desc is None:
        desc = fp8_desc(q, kv_cache, block_table, query_group, softmax_scale, out_dtype)
    if out is None:
        odt = torch.bfloat16 if desc.out_dtype == QPA_OUT_BF16 else torch.float32
        out = torch.empty((q.shape[0], q.shape[1], q.shape[2]), dtype=odt, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(pa_decode_fp8_workspace_size(desc, num_partitions), q.device)
    st = lib.pa_decode_fp8(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), _ptr(k_scale),
                           _ptr(v_scale), num_partitions, _ptr(out), ctypes.byref(desc),
                           _ptr(workspace), workspace.numel(), _stream(stream))
    _check("pa_decode_fp8", st)
    return out


def pa_decode_fp8_partition(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions,
                            desc, workspace, stream=None):
    st = load_library().pa_decode_fp8_partition(
        _ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), _ptr(k_scale), _ptr(v_scale),
        num_partitions, ctypes.byref(desc), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("pa_decode_fp8_partition", st)


def pa_decode_fp8_combine(num_partitions, out, desc, workspace, stream=None):
    st = load_library().pa_decode_fp8_combine(num_partitions, _ptr(out), ctypes.byref(desc),
                                              _ptr(workspace), workspace.numel(), _stream(stream))
    _check("pa_decode_fp8_combine", st)


def fp8_ext_desc(q, kv_cache, block_table, query_group, per_token, softmax_scale=None,
                 out_dtype=torch.float32):
    """Descriptor of pa_decode_fp8_ext for q bf16 [B, QL, Hq, 128]."""
    B, QL, Hq, D = q.shape
    NB, two, Hk, bs, D2 = kv_cache.shape
    assert two == 2 and D2 == D and Hq == Hk * query_group
    if q.stride(3) != 1:
        raise ValueError("q must be contiguous along head_dim")
    d = Fp8ExtDesc()
    b = d.base
    b.num_seqs, b.num_kv_heads, b.query_group, b.head_dim = B, Hk, query_group, D
    b.block_size, b.num_blocks, b.max_blocks_per_seq = bs, NB, block_table.shape[1]
    b.out_dtype = QPA_OUT_BF16 if out_dtype == torch.bfloat16 else QPA_OUT_F32
    b.q_stride_seq, b.q_stride_head = q.stride(0), q.stride(2)
    b.softmax_scale = 0.0 if softmax_scale is None else float(softmax_scale)
    d.query_len = QL
    d.kv_scale_per_token = 1 if per_token else 0
    d.q_stride_tok = q.stride(1)
    return d


def pa_decode_fp8_ext_workspace_size(desc: Fp8ExtDesc, num_partitions: int) -> int:
    return int(load_library().pa_decode_fp8_ext_workspace_size(ctypes.byref(desc), num_partitions))


def pa_decode_fp8_ext(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions: int,
                      query_group: int, out=None, workspace=None, softmax_scale=None,
                      out_dtype=torch.float32, stream=None, desc=None):
    """fp8 decode of QL query tokens per sequence. q bf16 [B, QL, Hq, 128];
    k_scale / v_scale float32 [1] (per-tensor) or [NB, Hk, bs] (per-token) on
    the device. Returns out [B, QL, Hq, 128]."""
    lib = load_library()
    _need_cuda(q, kv_cache, block_table, seq_lens, k_scale, v_scale)
    per_token = k_scale.numel() > 1 or k_scale.dim() == 3
    if desc is None:
        desc = fp8_ext_desc(q, kv_cache, block_table, query_group, per_token, softmax_scale, out_dtype)
    if out is None:
        odt = torch.bfloat16 if desc.base.out_dtype == QPA_OUT_BF16 else torch.float32
        out = torch.empty(tuple(q.shape), dtype=odt, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(pa_decode_fp8_ext_workspace_size(desc, num_partitions), q.device)
    st = lib.pa_decode_fp8_ext(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), _ptr(k_scale),
                               _ptr(v_scale), num_partitions, _ptr(out), ctypes.byref(desc),
                               _ptr(workspace), workspace.numel(), _stream(stream))
    _check("pa_decode_fp8_ext", st)
    return out


def fp8_workspace_views(workspace, desc: Fp8Desc, num_partitions: int):
    """(O, m, l) float32 views of the partition partials in a workspace."""
    rows = desc.num_seqs * desc.num_kv_heads * num_partitions * desc.query_group
    up = lambda x: (x + 255) // 256 * 256
    m_off = up(rows * desc.head_dim * 4)
    l_off = up(m_off + rows * 4)
    f = workspace.view(torch.uint8)
    shp = (desc.num_seqs, desc.num_kv_heads, num_partitions, desc.query_group)
    O = f[:rows * desc.head_dim * 4].view(torch.float32).view(*shp, desc.head_dim)
    m = f[m_off:m_off + rows * 4].view(torch.float32).view(*shp)
    l = f[l_off:l_off + rows * 4].view(torch.float32).view(*shp)
    return O, m, l


def pa_decode_fp8_static(q, kv_cache, block_table, seq_lens, k_scale, v_scale, num_partitions: int,
                         query_group: int, out=None, softmax_scale=None, out_dtype=torch.float32,
                         stream=None, desc=None):
    """pa_decode_fp8 without a workspace: for callers that cannot allocate
    device memory. The partials go to the library's static device array
    (8 MiB per GPU); calls that overlap on the GPU race on it."""
    lib = load_library()
    _need_cuda(q, kv_cache, block_table, seq_lens, k_scale, v_scale, out)
    if desc is None:
        desc = fp8_desc(q, kv_cache, block_table, query_group, softmax_scale, out_dtype)
    if out is None:
        raise ValueError("pa_decode_fp8_static writes into a caller-provided `out` tensor")
    st = lib.pa_decode_fp8_static(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
                                  _ptr(k_scale), _ptr(v_scale), num_partitions, _ptr(out),
                                  ctypes.byref(desc), _stream(stream))
    _check("pa_decode_fp8_static", st)
    return out


# --------------------------------------------------------------------- uq hd256
def uq_desc(q, kv_cache, block_table, query_group, softmax_scale=None, out_dtype=torch.float32,
            scale_format="e4m3", q_haircut=False, rot_perm=False):
    """scale_format: "e4m3" or "ue8m0" group scale bytes; q_haircut: round
    softmax_scale * q_r to e4m3 before the QK product; rot_perm: the cache is
    in the domain of the column-permuted rotation."""
    if scale_format not in ("e4m3", "ue8m0"):
        raise ValueError(f"scale_format {scale_format!r}")
    B, Hq, D = q.shape
    NB, bs, Hk, slot = kv_cache.shape
    assert D == 256 and Hq == Hk * query_group
    if q.stride(2) != 1:
        raise ValueError("q must be contiguous along head_dim")
    d = UqDesc()
    d.num_seqs, d.num_kv_heads, d.query_group, d.head_dim = B, Hk, query_group, D
    d.block_size, d.num_blocks, d.max_blocks_per_seq, d.padded_slot = bs, NB, block_table.shape[1], slot
    d.out_dtype = QPA_OUT_BF16 if out_dtype == torch.bfloat16 else QPA_OUT_F32
    d.q_stride_seq, d.q_stride_head = q.stride(0), q.stride(1)
    d.softmax_scale = 0.0 if softmax_scale is None else float(softmax_scale)
    d.flags = ((QPA_UQ_UE8M0_SCALES if scale_format == "ue8m0" else 0) | (QPA_UQ_Q_HAIRCUT if q_haircut else 0)
               | (QPA_UQ_ROT_PERM if rot_perm else 0))
    return d


def uq_decode_hd256_workspace_size(desc: UqDesc, num_partitions: int) -> int:
    return int(load_library().uq_decode_hd256_workspace_size(ctypes.byref(desc), num_partitions))


def uq_decode_hd256(q, kv_cache, centroids, block_table, seq_lens, num_partitions: int, query_group: int,
                    out=None, workspace=None, softmax_scale=None, out_dtype=torch.float32, stream=None,
                    desc=None, scale_format="e4m3", q_haircut=False, rot_perm=False):
    """4-bit head_dim=256 decode. q bf16 [B, Hq, 256] (not rotated); kv_cache
    uint8 [NB, bs, Hk, padded_slot]; centroids float32 [16]; returns the
    un-rotated out [B, Hq, 256]. scale_format / q_haircut / rot_perm as in uq_desc."""
    lib = load_library()
    _need_cuda(q, kv_cache, centroids, block_table, seq_lens)
    if desc is None:
        desc = uq_desc(q, kv_cache, block_table, query_group, softmax_scale, out_dtype, scale_format, q_haircut,
                       rot_perm)
    if out is None:
        odt = torch.bfloat16 if desc.out_dtype == QPA_OUT_BF16 else torch.float32
        out = torch.empty((q.shape[0], q.shape[1], 256), dtype=odt, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(uq_decode_hd256_workspace_size(desc, num_partitions), q.device)
    st = lib.uq_decode_hd256(_ptr(q), _ptr(kv_cache), _ptr(centroids), _ptr(block_table), _ptr(seq_lens),
                             num_partitions, _ptr(out), ctypes.byref(desc), _ptr(workspace), workspace.numel(),
                             _stream(stream))
    _check("uq_decode_hd256", st)
    return out


def uq_decode_hd256_partition(q, kv_cache, centroids, block_table, seq_lens, num_partitions, desc, workspace,
                              stream=None):
    st = load_library().uq_decode_hd256_partition(
        _ptr(q), _ptr(kv_cache), _ptr(centroids), _ptr(block_table), _ptr(seq_lens), num_partitions,
        ctypes.byref(desc), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("uq_decode_hd256_partition", st)


def uq_decode_hd256_combine(num_partitions, out, desc, workspace, stream=None):
    st = load_library().uq_decode_hd256_combine(num_partitions, _ptr(out), ctypes.byref(desc), _ptr(workspace),
                                                workspace.numel(), _stream(stream))
    _check("uq_decode_hd256_combine", st)


# --------------------------------------------------------------------- nvfp4 index scorer
def idx_desc(q_codes, pages, block_table, query_len, num_cols, scores=None, per_token=False, shared_pages=False):
    """num_cols counts blocks, or tokens with per_token (one column per token);
    shared_pages: score page by page over groups of 8 requests, loading a page
    that several requests map once (for requests that share pages)."""
    RQ, H, D = q_codes.shape
    assert D == 128 and RQ % query_len == 0
    d = IdxDesc()
    d.num_reqs, d.query_len, d.num_heads, d.head_dim = RQ // query_len, query_len, H, D
    d.num_blocks, d.max_blocks_per_seq, d.num_cols = pages.shape[0], block_table.shape[1], num_cols
    d.page_stride = pages.stride(0) * pages.element_size()
    d.q_stride_tok, d.q_stride_head = q_codes.stride(0), q_codes.stride(1)
    if scores is not None:
        d.s_stride_head, d.s_stride_row = scores.stride(0), scores.stride(1)
    d.flags = (QPA_IDX_PER_TOKEN if per_token else 0) | (QPA_IDX_SHARED_PAGES if shared_pages else 0)
    return d


def nvfp4_index_score(q_codes, pages, block_table, seq_lens, query_len: int, num_cols: int, scores=None,
                      stream=None, desc=None, per_token=False, shared_pages=False):
    """Paged NVFP4 index scores. q_codes uint8 (e4m3) [R*QL, H, 128]; pages
    uint8 [NB, 9216]; returns float32 scores [H, R*QL, num_cols] (columns are
    blocks, or tokens with per_token)."""
    lib = load_library()
    _need_cuda(q_codes, pages, block_table, seq_lens, scores)
    if scores is None:
        scores = torch.empty((q_codes.shape[1], q_codes.shape[0], num_cols), dtype=torch.float32,
                             device=q_codes.device)
    if desc is None:
        desc = idx_desc(q_codes, pages, block_table, query_len, num_cols, scores, per_token, shared_pages)
    st = lib.nvfp4_index_score(_ptr(q_codes), _ptr(pages), _ptr(block_table), _ptr(seq_lens), _ptr(scores),
                               ctypes.byref(desc), _stream(stream))
    _check("nvfp4_index_score", st)
    return scores

"""Seeded synthetic inputs for the three decode entry points.

This module is shared by the tests, the benchmark and the oracle checks. It
only *produces* inputs: random draws, rounding of those draws into the stored
formats (e4m3fn bytes, e2m1 nibbles, bf16 bits), and page/slot packing. It
holds none of the decode arithmetic (no dequantisation of stored codes, no
rotation of queries, no attention, no scoring), so neither the oracle nor the
CUDA path can borrow its results.

Every generator takes an explicit seed and uses numpy's PCG64, so the same
call returns the same bytes on x86 and on Arm.

Workload shapes follow the five configurations of the decode study:
  fp8 tiny       2 seqs (37, 200 tokens), 1 KV head, group 8, D 128, block 16
  fp8 GQA        16 seqs x 16384 tokens, 8 KV heads, group 8, D 128, block 16
  fp8 ragged     128 seqs, lengths U[1024, 16384], 8 KV heads, group 8
  uq hd256       4 seqs x 75000 tokens, 2 KV heads, group 8 or 6, block 64,
                 288-byte slots (272 used); UE8M0 caches also drawn byte
                 by byte over windows of the scale-byte range
  nvfp4 scorer   64 requests, lengths U[4096, 32768], query_len 4,
                 2 index heads, D 128, 128-token pages of 72 B/token
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

E4M3_MAX = 448.0
# The eight non-negative e2m1 magnitudes in code order 0..7 (OCP MX spec).
_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
_E2M1_MID = (_E2M1_POS[1:] + _E2M1_POS[:-1]) / 2.0


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# ----------------------------------------------------------------------------
# rounding of random draws into stored formats (producer side only)
# ----------------------------------------------------------------------------
def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bit patterns (uint16), round-to-nearest-even via torch."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def round_to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """float -> e4m3fn bytes, RNE, saturating to +-448 (torch's cast of an
    out-of-range value would give NaN)."""
    x = np.clip(np.asarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def e4m3_bytes_to_float(b: np.ndarray) -> np.ndarray:
    """Producer-side read-back of e4m3 bytes (used only to pick group scales
    while quantising). Goes through torch, not through either decoder."""
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy()


def round_to_e2m1_codes(x: np.ndarray) -> np.ndarray:
    """float (already divided by its group scale) -> e2m1 code 0..15, nearest
    magnitude (ties toward the smaller one), sign in bit 3."""
    a = np.minimum(np.abs(x), 6.0)
    mag = np.searchsorted(_E2M1_MID, a, side="left").astype(np.uint8)
    sign = (np.signbit(x) & (mag != 0)).astype(np.uint8)
    return (mag | (sign << 3)).astype(np.uint8)


def round_to_centroid_codes(x: np.ndarray, centroids: np.ndarray) -> np.ndarray:
    """float -> index of the nearest centroid (ties toward the lower index)."""
    c = np.asarray(centroids, dtype=np.float64)
    order = np.argsort(c, kind="stable")
    cs = c[order]
    mids = (cs[1:] + cs[:-1]) / 2.0
    pos = np.searchsorted(mids, x, side="left")
    return order[pos].astype(np.uint8)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., 2n] codes -> [..., n] bytes, element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def group_scales_e4m3(x: np.ndarray, group: int, qmax: float) -> np.ndarray:
    """Per-group e4m3 scale bytes for x[..., D]: e4m3(absmax / qmax), never 0."""
    shp = x.shape[:-1] + (x.shape[-1] // group, group)
    amax = np.abs(x.reshape(shp)).max(axis=-1)
    s = round_to_e4m3_bytes(np.maximum(amax / qmax, 2.0 ** -9))
    return s


def group_scales_ue8m0(x: np.ndarray, group: int, qmax: float) -> np.ndarray:
    """Per-group UE8M0 scale bytes for x[..., D]: the smallest power of two
    2^(byte-127) with absmax / 2^(byte-127) <= qmax (bytes 1..254; an
    all-zero group gets the smallest power, byte 1)."""
    shp = x.shape[:-1] + (x.shape[-1] // group, group)
    amax = np.abs(x.reshape(shp)).max(axis=-1).astype(np.float64)
    e = np.ceil(np.log2(np.maximum(amax / qmax, 2.0 ** -126)))
    return np.clip(127 + e, 1, 254).astype(np.uint8)


def e2m1_table() -> np.ndarray:
    """16-entry e2m1 value table in code order (a centroid table choice)."""
    return np.concatenate([_E2M1_POS, -_E2M1_POS]).astype(np.float32)


# ----------------------------------------------------------------------------
# paged fp8 cache: kv_cache[num_blocks][2 (K,V)][Hk][block_size][D] uint8
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Fp8Case:
    q_bits: np.ndarray        # [B, Hq, D] uint16 (bf16 bits)
    kv_cache: np.ndarray      # [NB, 2, Hk, bs, D] uint8 (e4m3fn)
    block_table: np.ndarray   # [B, max_blocks] int32 (unused entries -1)
    seq_lens: np.ndarray      # [B] int32
    k_scale: float
    v_scale: float
    num_kv_heads: int
    query_group: int
    head_dim: int
    block_size: int
    softmax_scale: float

    @property
    def num_seqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def kv_bytes(self) -> int:
        """KV bytes the decode must read once: every stored token of every
        sequence, K and V, for all KV heads."""
        return int(self.seq_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_dim


def _assign_blocks(r, nblk_per_seq, num_blocks, max_blocks):
    perm = r.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(nblk_per_seq), max_blocks), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(nblk_per_seq):
        bt[s, :n] = perm[off:off + n]
        off += n
    return bt


def _fill_e4m3_normal(r, shape, inv_scale, chunk=1 << 24):
    """e4m3 bytes of N(0,1) * inv_scale, generated in chunks."""
    out = np.empty(int(np.prod(shape)), dtype=np.uint8)
    for o in range(0, out.size, chunk):
        n = min(chunk, out.size - o)
        out[o:o + n] = round_to_e4m3_bytes(r.standard_normal(n, dtype=np.float32) * inv_scale)
    return out.reshape(shape)


def make_fp8_case(seed: int, seq_lens, num_kv_heads: int, query_group: int,
                  head_dim: int = 128, block_size: int = 16, num_blocks: int | None = None,
                  max_blocks: int | None = None, k_scale: float = 0.05, v_scale: float = 0.04,
                  softmax_scale: float | None = None, poison: bool = True) -> Fp8Case:
    r = rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.shape[0]
    nblk = [int(math.ceil(int(L) / block_size)) for L in seq_lens]
    if max_blocks is None:
        max_blocks = max(1, max(nblk) if nblk else 1)
    if num_blocks is None:
        num_blocks = max(1, sum(nblk))
    assert num_blocks >= sum(nblk)
    Hq = num_kv_heads * query_group
    q = r.standard_normal((B, Hq, head_dim), dtype=np.float32)
    q_bits = round_to_bf16_bits(q)
    shape = (num_blocks, 2, num_kv_heads, block_size, head_dim)
    cache = np.empty(shape, dtype=np.uint8)
    cache[:, 0] = _fill_e4m3_normal(r, (num_blocks, num_kv_heads, block_size, head_dim), 1.0 / k_scale)
    cache[:, 1] = _fill_e4m3_normal(r, (num_blocks, num_kv_heads, block_size, head_dim), 1.0 / v_scale)
    bt = _assign_blocks(r, nblk, num_blocks, max_blocks)
    if poison:
        # Slots past each sequence's end in its last block hold NaN codes
        # (0x7F / 0xFF); a kernel that reads them unmasked poisons its output.
        for s in range(B):
            L = int(seq_lens[s])
            if L % block_size and nblk[s]:
                blk = bt[s, nblk[s] - 1]
                cache[blk, :, :, L % block_size:, :] = r.choice(
                    np.array([0x7F, 0xFF], dtype=np.uint8),
                    size=cache[blk, :, :, L % block_size:, :].shape)
        used = set(int(b) for b in bt[bt >= 0].ravel())
        spare = [b for b in range(num_blocks) if b not in used]
        if spare:
            cache[spare] = 0x7F
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    return Fp8Case(q_bits, cache, bt, seq_lens, float(k_scale), float(v_scale),
                   num_kv_heads, query_group, head_dim, block_size, float(softmax_scale))


@dataclasses.dataclass
class Fp8ExtCase:
    q_bits: np.ndarray        # [B, QL, Hq, D] uint16 (bf16 bits)
    kv_cache: np.ndarray      # [NB, 2, Hk, bs, D] uint8 (e4m3fn)
    block_table: np.ndarray   # [B, max_blocks] int32 (unused entries -1)
    seq_lens: np.ndarray      # [B] int32 (including the QL query tokens)
    k_scale: object           # float, or [NB, Hk, bs] float32 per token
    v_scale: object
    num_kv_heads: int
    query_group: int
    query_len: int
    head_dim: int
    block_size: int
    softmax_scale: float

    @property
    def num_seqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def per_token(self):
        return np.ndim(self.k_scale) > 0

    @property
    def kv_bytes(self):
        """Cache bytes read: 2 x 128 code bytes per (token, KV head), plus the
        two 4-byte scales per (token, KV head) with per-token scales."""
        tok = int(np.sum(self.seq_lens.astype(np.int64)))
        return tok * self.num_kv_heads * (2 * self.head_dim + (8 if self.per_token else 0))


def make_fp8_ext_case(seed: int, seq_lens, num_kv_heads: int, query_group: int, query_len: int,
                      per_token: bool, head_dim: int = 128, block_size: int = 16,
                      max_blocks: int | None = None, poison: bool = True) -> Fp8ExtCase:
    """As make_fp8_case with query_len query tokens per sequence. With
    per_token, every (token, KV head) has its own K and V scale, drawn
    log-uniform in [0.01, 0.2] and rounded to float32, and its codes are the
    e4m3 of N(0,1) / scale."""
    r = rng(seed)
    base = make_fp8_case(seed, seq_lens, num_kv_heads, query_group, head_dim, block_size,
                         max_blocks=max_blocks, poison=poison)
    B = base.num_seqs
    Hq = num_kv_heads * query_group
    q = r.standard_normal((B, query_len, Hq, head_dim), dtype=np.float32)
    q_bits = round_to_bf16_bits(q)
    cache = base.kv_cache
    if per_token:
        NB = cache.shape[0]
        ks = np.exp(r.uniform(np.log(0.01), np.log(0.2), size=(NB, num_kv_heads, block_size))).astype(np.float32)
        vs = np.exp(r.uniform(np.log(0.01), np.log(0.2), size=(NB, num_kv_heads, block_size))).astype(np.float32)
        cache = cache.copy()
        cache[:, 0] = round_to_e4m3_bytes(
            r.standard_normal(cache[:, 0].shape, dtype=np.float32) / ks[..., None])
        cache[:, 1] = round_to_e4m3_bytes(
            r.standard_normal(cache[:, 1].shape, dtype=np.float32) / vs[..., None])
        if poison:
            for s in range(B):
                L = int(base.seq_lens[s])
                nb = (L + block_size - 1) // block_size
                if L % block_size and nb:
                    blk = base.block_table[s, nb - 1]
                    cache[blk, :, :, L % block_size:, :] = 0x7F
                    ks[blk, :, L % block_size:] = np.nan
                    vs[blk, :, L % block_size:] = np.nan
        k_scale, v_scale = ks, vs
    else:
        k_scale, v_scale = base.k_scale, base.v_scale
    return Fp8ExtCase(q_bits, cache, base.block_table, base.seq_lens, k_scale, v_scale,
                      num_kv_heads, query_group, query_len, head_dim, block_size, base.softmax_scale)


def fp8_ext_long(seed: int = 1005, batch: int = 16, seq_len: int = 16384, query_group: int = 4,
                 query_len: int = 4, per_token: bool = True) -> Fp8ExtCase:
    """Throughput workload of the multi-token decode: 16 seqs x 16384 tokens, 8
    KV heads, group 4, 4 query tokens. The codes are the per-tensor draw of
    fp8_gqa (e4m3 of N(0,1)/0.05 and N(0,1)/0.04); with per_token, the K and V
    scales of every (token, head) are drawn log-uniform in [0.01, 0.2]
    independently of the codes (a throughput input, not a quantisation of a
    common logical cache)."""
    r = rng(seed)
    base = make_fp8_case(seed, [seq_len] * batch, 8, query_group, 128, 16, poison=False)
    Hq = 8 * query_group
    q_bits = round_to_bf16_bits(r.standard_normal((batch, query_len, Hq, 128), dtype=np.float32))
    if per_token:
        NB = base.kv_cache.shape[0]
        ks = np.exp(r.uniform(np.log(0.01), np.log(0.2), size=(NB, 8, 16))).astype(np.float32)
        vs = np.exp(r.uniform(np.log(0.01), np.log(0.2), size=(NB, 8, 16))).astype(np.float32)
    else:
        ks, vs = base.k_scale, base.v_scale
    return Fp8ExtCase(q_bits, base.kv_cache, base.block_table, base.seq_lens, ks, vs, 8, query_group,
                      query_len, 128, 16, base.softmax_scale)


def fp8_tiny(seed: int = 1000) -> Fp8Case:
    """2 seqs (37, 200), 1 KV head, group 8, D 128, block 16, 32 blocks in a
    seeded random permutation."""
    return make_fp8_case(seed, [37, 200], 1, 8, 128, 16, num_blocks=32)


def fp8_gqa(seed: int = 1001, batch: int = 16, seq_len: int = 16384) -> Fp8Case:
    """Llama-style GQA: 16 seqs x 16384, 8 KV heads, group 8, D 128, block 16;
    the block table is a permutation of all blocks. No spare blocks."""
    return make_fp8_case(seed, [seq_len] * batch, 8, 8, 128, 16, poison=False)


def fp8_ragged(seed: int = 1002, batch: int = 128, lo: int = 1024, hi: int = 16384) -> Fp8Case:
    """Ragged high batch: 128 seqs with lengths uniform in [1024, 16384]."""
    r = rng(seed + 7)
    lens = r.integers(lo, hi + 1, size=batch).astype(np.int32)
    return make_fp8_case(seed, lens, 8, 8, 128, 16, max_blocks=int(math.ceil(hi / 16)),
                         poison=False)


# ----------------------------------------------------------------------------
# 4-bit head_dim=256 slot cache: cache[num_blocks][bs][Hk][padded_slot] uint8
#   bytes   0..127  K e2m1 codes (dim 2i low nibble, 2i+1 high nibble)
#   bytes 128..135  K e4m3 scale per 32 dims
#   bytes 136..263  V centroid codes (same nibble order)
#   bytes 264..271  V e4m3 scale per 32 dims
# ----------------------------------------------------------------------------
UQ_D = 256
UQ_CONTENT = 272


@dataclasses.dataclass
class UqCase:
    q_bits: np.ndarray        # [B, Hq, 256] uint16 (bf16 bits), NOT rotated
    kv_cache: np.ndarray      # [NB, bs, Hk, padded_slot] uint8
    centroids: np.ndarray     # [16] float32
    block_table: np.ndarray   # [B, max_blocks] int32
    seq_lens: np.ndarray      # [B] int32
    num_kv_heads: int
    query_group: int
    block_size: int
    padded_slot: int
    softmax_scale: float
    scale_format: str = "e4m3"   # group scale bytes: "e4m3" (e4m3fn) or "ue8m0" (2^(b-127))
    rot_perm: bool = False       # K/V rotated with the page's column-permuted rotation

    @property
    def num_seqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def kv_bytes(self) -> int:
        """Slot content bytes read once (272 per token and KV head)."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.num_kv_heads * UQ_CONTENT


def page_rotation_perm() -> np.ndarray:
    """The dim each butterfly position d = 32 c + t of the rotation lands on
    when the page's column permutation is folded in, from the page's per-lane
    split of it: (t & 0x0F) | ((t & 0x10) << 1) | ((c & 2) << 3) |
    ((c & 1) << 6) | ((c & 4) << 5). Producer side: used only to put the
    synthetic K/V into the permuted rotated domain."""
    c = np.arange(256) // 32
    t = np.arange(256) % 32
    return (t & 0x0F) | ((t & 0x10) << 1) | ((c & 2) << 3) | ((c & 1) << 6) | ((c & 4) << 5)


def sylvester_pm1(n: int) -> np.ndarray:
    """+-1 Sylvester Hadamard matrix (producer-side copy used only to put the
    synthetic logical K/V into the rotated domain before quantising)."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def make_uq_case(seed: int, seq_lens, num_kv_heads: int = 2, query_group: int = 8,
                 block_size: int = 64, padded_slot: int = 288, centroids=None,
                 num_blocks: int | None = None, softmax_scale: float | None = None,
                 poison: bool = True, chunk_tokens: int = 1 << 15,
                 scale_format: str = "e4m3", rot_perm: bool = False, v_gain: float = 1.0) -> UqCase:
    """v_gain multiplies the logical V draws (so that a centroid table of
    another magnitude still quantises a spread of values)."""
    if scale_format not in ("e4m3", "ue8m0"):
        raise ValueError(scale_format)
    r = rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.shape[0]
    nblk = [int(math.ceil(int(L) / block_size)) for L in seq_lens]
    max_blocks = max(1, max(nblk))
    if num_blocks is None:
        num_blocks = max(1, sum(nblk))
    if centroids is None:
        centroids = e2m1_table()
    centroids = np.asarray(centroids, dtype=np.float32)
    cmax = float(np.abs(centroids).max())
    Hq = num_kv_heads * query_group
    q_bits = round_to_bf16_bits(r.standard_normal((B, Hq, UQ_D), dtype=np.float32))
    rot = (sylvester_pm1(UQ_D) / 16.0).astype(np.float32)
    if rot_perm:
        prm = np.empty_like(rot)
        prm[:, page_rotation_perm()] = rot
        rot = prm
    ntok = num_blocks * block_size * num_kv_heads
    cache = np.zeros((ntok, padded_slot), dtype=np.uint8)
    for o in range(0, ntok, chunk_tokens):
        n = min(chunk_tokens, ntok - o)
        kl = r.standard_normal((n, UQ_D), dtype=np.float32) @ rot
        vl = (r.standard_normal((n, UQ_D), dtype=np.float32) * np.float32(v_gain)) @ rot
        if scale_format == "e4m3":
            ks = group_scales_e4m3(kl, 32, 6.0)
            vs = group_scales_e4m3(vl, 32, cmax)
            ksf = np.repeat(e4m3_bytes_to_float(ks), 32, axis=1)
            vsf = np.repeat(e4m3_bytes_to_float(vs), 32, axis=1)
        else:
            ks = group_scales_ue8m0(kl, 32, 6.0)
            vs = group_scales_ue8m0(vl, 32, cmax)
            ksf = np.repeat(np.ldexp(1.0, ks.astype(np.int32) - 127), 32, axis=1)
            vsf = np.repeat(np.ldexp(1.0, vs.astype(np.int32) - 127), 32, axis=1)
        cache[o:o + n, 0:128] = pack_nibbles(round_to_e2m1_codes(kl / ksf))
        cache[o:o + n, 128:136] = ks
        cache[o:o + n, 136:264] = pack_nibbles(round_to_centroid_codes(vl / vsf, centroids))
        cache[o:o + n, 264:272] = vs
        if padded_slot > UQ_CONTENT:
            cache[o:o + n, UQ_CONTENT:] = r.integers(0, 256, size=(n, padded_slot - UQ_CONTENT),
                                                     dtype=np.uint8)
    cache = cache.reshape(num_blocks, block_size, num_kv_heads, padded_slot)
    bt = _assign_blocks(r, nblk, num_blocks, max_blocks)
    if poison:
        for s in range(B):
            L = int(seq_lens[s])
            if L % block_size and nblk[s]:
                blk = bt[s, nblk[s] - 1]
                # NaN (e4m3) / 2^128 (ue8m0) scale bytes and random codes past
                # the end of the sequence.
                cache[blk, L % block_size:, :, 128:136] = 0x7F if scale_format == "e4m3" else 0xFF
                cache[blk, L % block_size:, :, 264:272] = 0xFF
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(UQ_D)
    return UqCase(q_bits, cache, centroids, bt, seq_lens, num_kv_heads, query_group,
                  block_size, padded_slot, float(softmax_scale), scale_format, rot_perm)


def sorted_random_centroids(seed: int) -> np.ndarray:
    """A seeded, sorted 16-entry centroid table (the second table of the
    hd256 runs)."""
    return np.sort(rng(seed).standard_normal(16).astype(np.float32) * 2.0)


def make_uq_ue8m0_window_case(seed: int, seq_lens, k_bytes, v_bytes, num_kv_heads: int = 2,
                              query_group: int = 8, block_size: int = 64, padded_slot: int = 288,
                              centroids=None, q_gain: float = 1.0, zero_frac: float = 0.03,
                              poison: bool = True) -> UqCase:
    """A UE8M0 slot cache drawn byte by byte: every K and V code uniform over
    the 16 codes, every K group-scale byte uniform in k_bytes = (lo, hi), every
    V group-scale byte in v_bytes, and a zero_frac share of the scale bytes
    set to the 0 sentinel (a zero group). q = q_gain * N(0, 1) in bf16. Used to
    cover the whole UE8M0 byte range window by window (a case's scales span at
    most a few dozen binades, so its tolerance, 2e-3 * max|V|, still sees the
    small ones)."""
    r = rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.shape[0]
    nblk = [int(math.ceil(int(L) / block_size)) for L in seq_lens]
    max_blocks = max(1, max(nblk))
    num_blocks = max(1, sum(nblk))
    if centroids is None:
        centroids = e2m1_table()
    Hq = num_kv_heads * query_group
    q_bits = round_to_bf16_bits(r.standard_normal((B, Hq, UQ_D), dtype=np.float32) * np.float32(q_gain))
    ntok = num_blocks * block_size * num_kv_heads
    cache = r.integers(0, 256, size=(ntok, padded_slot), dtype=np.uint8)   # codes (and padding) uniform
    ks = r.integers(k_bytes[0], k_bytes[1] + 1, size=(ntok, 8)).astype(np.uint8)
    vs = r.integers(v_bytes[0], v_bytes[1] + 1, size=(ntok, 8)).astype(np.uint8)
    ks[r.random((ntok, 8)) < zero_frac] = 0
    vs[r.random((ntok, 8)) < zero_frac] = 0
    cache[:, 128:136] = ks
    cache[:, 264:272] = vs
    cache = cache.reshape(num_blocks, block_size, num_kv_heads, padded_slot)
    bt = _assign_blocks(r, nblk, num_blocks, max_blocks)
    if poison:
        for s in range(B):
            L = int(seq_lens[s])
            if L % block_size and nblk[s]:
                blk = bt[s, nblk[s] - 1]
                cache[blk, L % block_size:, :, 128:136] = 0xFF
                cache[blk, L % block_size:, :, 264:272] = 0xFF
    return UqCase(q_bits, cache, np.asarray(centroids, dtype=np.float32), bt, seq_lens, num_kv_heads,
                  query_group, block_size, padded_slot, 1.0 / math.sqrt(UQ_D), "ue8m0", False)


def uq_full(seed: int = 1003, query_group: int = 8, centroids=None, scale_format: str = "e4m3",
            rot_perm: bool = False) -> UqCase:
    """4 seqs x 75000 tokens, 2 KV heads, block 64, 288-byte slots."""
    return make_uq_case(seed, [75000] * 4, 2, query_group, 64, 288, centroids=centroids,
                        poison=False, scale_format=scale_format, rot_perm=rot_perm)


# ----------------------------------------------------------------------------
# NVFP4 index pages: pages[num_blocks][9216] uint8
#   bytes 0..8191    128 tokens x 64 B of e2m1 codes (dim 2i low nibble)
#   bytes 8192..9215 128 tokens x 8 e4m3 scales (one per 16 dims)
# ----------------------------------------------------------------------------
IDX_BLK = 128
IDX_D = 128
IDX_PAGE = IDX_BLK * 72


@dataclasses.dataclass
class IdxCase:
    q_codes: np.ndarray       # [R*QL, H, 128] uint8 (e4m3fn)
    pages: np.ndarray         # [NB, 9216] uint8
    block_table: np.ndarray   # [R, max_blocks] int32
    seq_lens: np.ndarray      # [R] int32
    query_len: int
    num_heads: int
    num_cols: int             # S, score columns per row

    @property
    def num_reqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def kv_bytes(self) -> int:
        """Page bytes read once: whole 9216-byte pages of every request."""
        nblk = (self.seq_lens.astype(np.int64) + IDX_BLK - 1) // IDX_BLK
        return int(nblk.sum()) * IDX_PAGE

    @property
    def unique_page_bytes(self) -> int:
        """Bytes of the distinct physical pages the requests map."""
        nblk = (self.seq_lens.astype(np.int64) + IDX_BLK - 1) // IDX_BLK
        ids = np.concatenate([self.block_table[s, :n] for s, n in enumerate(nblk)]) if len(nblk) else []
        return int(np.unique(ids).size) * IDX_PAGE


def make_idx_case(seed: int, seq_lens, query_len: int = 4, num_heads: int = 2,
                  num_blocks: int | None = None, num_cols: int | None = None,
                  poison: bool = True, chunk_pages: int = 512, shared_prefix_blocks: int = 0) -> IdxCase:
    """shared_prefix_blocks: the first that many blocks of every request map
    to the same physical pages (a prefix shared by all requests); the other
    blocks get pages of their own."""
    r = rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    R = seq_lens.shape[0]
    nblk = [int(math.ceil(int(L) / IDX_BLK)) for L in seq_lens]
    max_blocks = max(1, max(nblk))
    SP = int(shared_prefix_blocks)
    if num_blocks is None:
        num_blocks = max(1, SP + sum(max(0, n - SP) for n in nblk) if SP else sum(nblk))
    if num_cols is None:
        num_cols = max_blocks
    q_codes = round_to_e4m3_bytes(r.standard_normal((R * query_len, num_heads, IDX_D),
                                                    dtype=np.float32))
    pages = np.empty((num_blocks, IDX_PAGE), dtype=np.uint8)
    for o in range(0, num_blocks, chunk_pages):
        n = min(chunk_pages, num_blocks - o)
        k = r.standard_normal((n * IDX_BLK, IDX_D), dtype=np.float32)
        sc = group_scales_e4m3(k, 16, 6.0)
        scf = np.repeat(e4m3_bytes_to_float(sc), 16, axis=1)
        codes = pack_nibbles(round_to_e2m1_codes(k / scf))
        pages[o:o + n, :8192] = codes.reshape(n, 8192)
        pages[o:o + n, 8192:] = sc.reshape(n, 1024)
    if SP:
        perm = r.permutation(num_blocks).astype(np.int32)
        bt = np.full((R, max_blocks), -1, dtype=np.int32)
        off = SP
        for s, n in enumerate(nblk):
            k = min(n, SP)
            bt[s, :k] = perm[:k]
            bt[s, k:n] = perm[off:off + n - k]
            off += n - k
    else:
        bt = _assign_blocks(r, nblk, num_blocks, max_blocks)
    if poison:
        for s in range(R):
            L = int(seq_lens[s])
            if L % IDX_BLK and nblk[s] > SP:          # never poison a shared page
                blk = bt[s, nblk[s] - 1]
                t0 = L % IDX_BLK
                pages[blk, 8192 + 8 * t0:] = 0x7F   # NaN scales past the end
    return IdxCase(q_codes, pages, bt, seq_lens, query_len, num_heads, num_cols)


def idx_full(seed: int = 1004) -> IdxCase:
    """64 requests, lengths U[4096, 32768], query_len 4, 2 index heads."""
    r = rng(seed + 7)
    lens = r.integers(4096, 32768 + 1, size=64).astype(np.int32)
    return make_idx_case(seed, lens, 4, 2, num_cols=256, poison=False)


def idx_shared_prefix(seed: int = 1007) -> IdxCase:
    """64 requests, lengths U[16384, 32768], query_len 4, 2 index heads, the
    first 16384 tokens (128 pages) shared by all requests."""
    r = rng(seed + 7)
    lens = r.integers(16384, 32768 + 1, size=64).astype(np.int32)
    return make_idx_case(seed, lens, 4, 2, num_cols=256, poison=False, shared_prefix_blocks=128)

"""UltraQuant head_dim=256 4-bit decode: slot decode, Q rotation, attention,
un-rotation.

TEST INFRASTRUCTURE (see the package header).

Slot ([UQ] builder docstring and STEP F addressing): the cache is
``[num_blocks][bs][Hk][padded_slot]`` uint8; per (token, KV head) the slot
holds K e2m1 codes in bytes 0..127, K scales in 128..135 (one per 32 dims),
V codes in 136..263 and V scales in 264..271. Dim 2i is the low nibble of
code byte i.

Dequantisation (readings of the pages, listed in the design notes):
  K[d] = e2m1(code) * e4m3(kscale[d // 32])
  V[d] = centroid[code] * e4m3(vscale[d // 32])     (16-entry fp32 table)
The page prints UE8M0 scales and an e2m1 V convert; the e2m1 table as the
centroid table reproduces that V path, and ``scale_format='ue8m0'`` selects
the page's scale decode.

Rotation ([UQ] STEP B'): the cached K and V live in the domain rotated by
the orthonormal Sylvester-Hadamard matrix R = H_256 / 16, H[i][j] =
(-1)^popcount(i & j); R is symmetric and its own inverse. Q is rotated with
the same R, attention runs in the rotated domain with scale 1/sqrt(256)
(the builder's default softmax scale), and the output is rotated back:
o = softmax(scale q_r K_r^T) V_r R.

Column permutation ([UQ] STEP B', the permutation folded into the rotation
constant): with ``rot_perm`` the rotation is M, R with its columns permuted
so that the value at butterfly position d lands at dim perm_dest(d); K_r, V_r
are in that domain and the output is o_r M^T.

Query haircut (the e4m3 rounding that closes [UQ] STEP B'), the
``q_haircut`` option: q_h = e4m3(scale * q_r), rounded to nearest even and
saturating at +-448, and the logits are q_h K_r^T with no further scale. The
rotation feeding this rounding is computed in float32 by butterfly stages of
strides 1, 2, ..., 128 (``rotate_q_fp32``), so that the rounding decision is
taken on the same float32 value as in the kernel.

Pins (tests/test_oracle_uq.py): R R^T = I, R = R^T, R R = I, the +-1 entries
against the recursive Sylvester construction, a fast butterfly transform
against R to within the fp32 difference the page reports (1.8e-6); a
hand-built slot against its expected dequantised vector (tests/golden); the
page's 81.6 MB slot byte count at B=4, seq 75k, one KV head; the whole
rotated pipeline against plain attention on the logical K = K_r R,
V = V_r R (e4m3 and UE8M0 scales). The float32 rotation exactly against
x H on integer inputs and within the page's fp32 bound on random ones; the
haircut as the identity on queries whose scaled rotation is already e4m3, and
against torch's e4m3 cast plus a written-out softmax. The permutation against
the page's second, per-lane form of it; a bijection moving single bits; the
permuted rotation orthonormal and a column permutation of R; the permuted
pipeline (with and without the haircut) against logical-domain attention.
"""
import math

import numpy as np

from .attention import attend, gather_tokens
from .formats import decode_bf16, decode_e2m1, decode_e4m3fn, decode_ue8m0, round_e4m3, unpack_nibbles

HEAD = 256
K_CODES, K_SCALES, V_CODES, V_SCALES, CONTENT = 0, 128, 136, 264, 272
GROUP = 32


def wht_matrix(n: int = HEAD) -> np.ndarray:
    """Orthonormal Sylvester-Hadamard matrix, entry (i, j) = (-1)^popcount(i&j)
    / sqrt(n)."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    x = i & j
    parity = np.zeros_like(x)
    while np.any(x):
        parity ^= x & 1
        x = x >> 1
    return np.where(parity == 1, -1.0, 1.0) / math.sqrt(n)


def perm_dest(d):
    """The page's column permutation of the rotation ([UQ] STEP B', the
    inverse query permutation): the rotated value at butterfly position d is
    stored at dim (d & 0x8F) | ((d >> 2) & 0x10) | ((d << 1) & 0x60), i.e.
    bits 4, 5, 6 of the index move to 5, 6, 4."""
    d = np.asarray(d)
    return (d & 0x8F) | ((d >> 2) & 0x10) | ((d << 1) & 0x60)


def perm_source(j):
    """Inverse of perm_dest: the butterfly position whose value lands at dim j."""
    j = np.asarray(j)
    return (j & 0x8F) | ((j & 0x10) << 2) | ((j >> 1) & 0x30)


def rotation_matrix(rot_perm: bool = False) -> np.ndarray:
    """q_r = q M. Without the permutation M = R = H/16; with it, column
    perm_dest(d) of M is column d of R (q_r[perm_dest(d)] = (q R)[d])."""
    R = wht_matrix(HEAD)
    if not rot_perm:
        return R
    M = np.empty_like(R)
    M[:, perm_dest(np.arange(HEAD))] = R
    return M


def rotate_q_fp32(q: np.ndarray) -> np.ndarray:
    """q [..., 256] -> q H in float32 by butterfly stages of strides 1, 2, ...,
    128 (x, y) -> (x + y, x - y), i.e. 16 q R rounded as the kernel computes
    it. Only the query haircut uses it: there the e4m3 rounding decision has to
    be taken on the same float32 value the kernel rounds."""
    v = np.asarray(q, dtype=np.float32).copy()
    st = 1
    while st < HEAD:
        v = v.reshape(v.shape[:-1] + (HEAD // (2 * st), 2, st))
        x, y = v[..., 0, :].copy(), v[..., 1, :].copy()
        v[..., 0, :] = x + y
        v[..., 1, :] = x - y
        v = v.reshape(v.shape[:-3] + (HEAD,))
        st *= 2
    return v


def decode_uq_slots(slots: np.ndarray, centroids, scale_format: str = "e4m3"):
    """slots [..., >=272] uint8 -> (K [..., 256], V [..., 256]) float64."""
    s = np.asarray(slots, dtype=np.uint8)
    dec = decode_e4m3fn if scale_format == "e4m3" else decode_ue8m0
    kcode = unpack_nibbles(s[..., K_CODES:K_SCALES])
    vcode = unpack_nibbles(s[..., V_CODES:V_SCALES])
    ks = np.repeat(dec(s[..., K_SCALES:V_CODES]), GROUP, axis=-1)
    vs = np.repeat(dec(s[..., V_SCALES:CONTENT]), GROUP, axis=-1)
    cent = np.asarray(centroids, dtype=np.float32).astype(np.float64)
    return decode_e2m1(kcode) * ks, cent[vcode] * vs


def dense_kv_uq(kv_cache, centroids, block_table, seq, kv_head, L, scale_format="e4m3"):
    slots = gather_tokens(kv_cache[:, :, kv_head], block_table[seq], L)
    return decode_uq_slots(slots, centroids, scale_format)


def uq_decode_hd256(q_bits, kv_cache, centroids, block_table, seq_lens, query_group: int,
                    softmax_scale: float | None = None, units=None,
                    scale_format: str = "e4m3", q_haircut: bool = False,
                    rot_perm: bool = False) -> np.ndarray:
    """Reference output [B, Hq, 256] in the un-rotated (logical) domain.

    q_bits [B, Hq, 256] uint16 bf16 bits (un-rotated); kv_cache [NB, bs, Hk,
    padded_slot] uint8; centroids [16] float32. With q_haircut (the e4m3
    rounding that closes [UQ] STEP B'), the rotated query times the
    softmax scale is rounded to e4m3 (float32 rotation, as the kernel) and the
    logits are that rounded query times K_r, with no further scale. With
    rot_perm the rotation is M = R with the page's column permutation
    (rotation_matrix) and the output is o_r M^T."""
    q = decode_bf16(q_bits)
    B, Hq, D = q.shape
    assert D == HEAD
    Hk = kv_cache.shape[2]
    assert Hq == Hk * query_group
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(HEAD)
    M = rotation_matrix(rot_perm)
    out = np.zeros((B, Hq, D))
    if units is None:
        units = [(s, h) for s in range(B) for h in range(Hk)]
    for s, h in units:
        L = int(seq_lens[s])
        k_r, v_r = dense_kv_uq(kv_cache, centroids, block_table, s, h, L, scale_format)
        rows = slice(h * query_group, (h + 1) * query_group)
        if q_haircut:
            # q M = (q permuted by perm_source) R, since the permutation only
            # moves index bits: the float32 butterfly runs on the permuted q
            qin = q[s, rows][:, perm_source(np.arange(HEAD))] if rot_perm else q[s, rows]
            q16 = rotate_q_fp32(qin)                                           # 16 q M in float32
            qs = (q16 * np.float32(0.0625)) * np.float32(softmax_scale)         # float32 products
            q_h = round_e4m3(qs.astype(np.float64))
            o_r = attend(q_h, k_r, v_r, 1.0)
        else:
            q_r = q[s, rows] @ M
            o_r = attend(q_r, k_r, v_r, softmax_scale)
        out[s, rows] = o_r @ M.T
    return out

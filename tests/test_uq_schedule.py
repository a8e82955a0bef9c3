"""The hd256 partition kernel's work split, restated on the host.

A sequence of L tokens is ns = ceil(L / 32) slices of 32 tokens; partition p
owns the slices p, p+P, p+2P, ... (the ultraquant_decode_hd256 page's strided
partition map, STEP F, at a 32-token granule). A work item (sequence, head
group, partition) is streamed through the CTA's ring by two producer warps
taking alternate stages, and its slices go to the consumer warps of each
(head, 8-row half) pair in turn: warp jr of a pair takes the item's slices
k = jr, jr+J, ... and writes partial slot p*J + jr, an empty slot when the
item has no slice for it. The plan takes the largest head group HG of 8, 4,
2, 1 that divides the KV heads with at most 8 (head, half) pairs and a ring
of at least J + 2 stages, J = 8 / (HG * halves).

These tests check that integer arithmetic (the same formulas as the kernel)
and that the library's workspace size, which is callable without a GPU,
holds exactly the P * J slots per (sequence, head) that the plan gives. The
kernel itself is checked against the oracle on the GPU (test_gpu_uq.py)."""
import ctypes
import random

import pytest

SLICE = 32
NC, NPW = 8, 2                     # consumer warps, producer warps
CONTENT = 272
HEAD_SLICE = SLICE * CONTENT
LUT_BYTES = 256 * 16 * 4
QF_BYTES = NC * 32 * 32 * 4
MAX_DEPTH = 12
SMEM_LIMIT = 232448
TAIL_BYTES = 2 * MAX_DEPTH * 8 + 16 + 128


def uq_slices(L, p, P):
    ns = (L + SLICE - 1) // SLICE
    return (ns - 1 - p) // P + 1 if p < ns else 0


def uq_plan(hk, qg):
    nh = (qg + 7) // 8
    for hg in (8, 4, 2, 1):
        if hk % hg or hg * nh > NC:
            continue
        j = NC // (hg * nh)
        depth = min(MAX_DEPTH, (SMEM_LIMIT - LUT_BYTES - QF_BYTES - TAIL_BYTES) // (hg * HEAD_SLICE))
        if depth < j + 2:
            continue
        return hg, nh, j, depth
    return None


def _lens(rng):
    return [rng.choice([0, 1, 31, 32, 33, 64, 255, 256, 257]) if rng.random() < 0.3 else rng.randint(0, 80000)
            for _ in range(rng.randint(1, 6))]


@pytest.mark.parametrize("seed", range(40))
def test_every_slice_once_and_partitions_balanced(seed):
    rng = random.Random(seed)
    for L in _lens(rng):
        P = rng.choice([1, 2, 3, 7, 38, 64, 300, 3000])
        ns = (L + SLICE - 1) // SLICE
        seen = []
        counts = []
        for p in range(P):
            n = uq_slices(L, p, P)
            counts.append(n)
            seen += [p + P * k for k in range(n)]
        assert sorted(seen) == list(range(ns)), (L, P)
        assert max(counts) - min(counts) <= 1
        # the last slice of a partition is the last one below ns
        for p in range(min(P, ns)):
            assert p + P * (counts[p] - 1) < ns <= p + P * counts[p]


@pytest.mark.parametrize("seed", range(20))
def test_consumer_warps_and_producer_stages_cover_each_slice_once(seed):
    rng = random.Random(100 + seed)
    for hk in (1, 2, 3, 4, 6, 8, 16):
        for qg in (1, 6, 8, 9, 16):
            hg, nh, J, depth = uq_plan(hk, qg)
            C = hg * nh
            assert C * J == NC and depth >= J + 2
            P = rng.choice([1, 5, 38])
            lens = _lens(rng)
            g = 0                                      # the CTA's stage count before an item
            for L in lens:
                for part in range(P):
                    nsl = uq_slices(L, part, P)
                    # consumers: every (head, half) pair's J warps split the item's slices
                    for pair in range(C):
                        taken = []
                        empty_slots = []
                        for jr in range(J):
                            ks = list(range(jr, nsl, J))
                            if nsl <= jr:
                                assert not ks
                                empty_slots.append(part * J + jr)
                            taken += ks
                        assert sorted(taken) == list(range(nsl))
                        assert all(part * J <= s < (part + 1) * J for s in empty_slots)
                    # producers: warp pw issues stage g + k when (g + k) % NPW == pw
                    issued = []
                    for pw in range(NPW):
                        k0 = (pw - g % NPW + NPW) % NPW
                        for k in range(k0, nsl, NPW):
                            assert (g + k) % NPW == pw
                            issued.append(k)
                    assert sorted(issued) == list(range(nsl))
                    g += nsl


def test_plan_on_the_benchmark_shapes():
    # 2 KV heads, group 8: both heads in one item, 4 warps per pair, 10 stages
    assert uq_plan(2, 8) == (2, 1, 4, 10)
    assert uq_plan(2, 6) == (2, 1, 4, 10)
    # group 16: two 8-row halves per head
    assert uq_plan(2, 16) == (2, 2, 2, 10)
    assert uq_plan(1, 16) == (1, 2, 4, 12)
    # 8 heads of group 8: a ring of two 69.6 KB stages is too short for J = 1,
    # so the items hold 4 heads (5 stages of 34.8 KB)
    assert uq_plan(8, 8) == (4, 1, 2, 5)
    assert uq_plan(3, 8) == (1, 1, 8, 12)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_paged_attention_gb300 as qpa
    return qpa.load_library()


def _uq_desc(B, hk, qg):
    import quantized_paged_attention_gb300 as qpa
    d = qpa.UqDesc()
    d.num_seqs, d.num_kv_heads, d.query_group, d.head_dim = B, hk, qg, 256
    d.block_size, d.num_blocks, d.max_blocks_per_seq, d.padded_slot = 64, 8, 4, 288
    return d


def _round256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("hk,qg", [(1, 8), (2, 6), (2, 8), (2, 16), (3, 8), (4, 1), (8, 8), (16, 16)])
@pytest.mark.parametrize("P", [1, 3, 38])
def test_workspace_holds_p_times_j_slots(lib, hk, qg, P):
    B = 3
    _, _, J, _ = uq_plan(hk, qg)
    rows = B * hk * P * J * qg
    m_off = _round256(rows * 256 * 4)
    l_off = _round256(m_off + rows * 4)
    want = _round256(l_off + rows * 4)
    assert lib.uq_decode_hd256_workspace_size(ctypes.byref(_uq_desc(B, hk, qg)), P) == want

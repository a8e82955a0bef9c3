"""The fp8 partition kernel's work split, restated on the host: the CTAs form
groups of Hk, the groups cut every head's tile groups (in sequence order) into
equal contiguous ranges, a sequence's part inside a range goes to the next
slot of that (sequence, head), and the range count is lowered until every
range holds at least ceil(Tmax / max(1, P - 2)) tile groups. These tests check
the integer arithmetic of that rule (the same formulas as the kernel's copy
warps): every tile group is covered once, slots are 0, 1, ... below P, the
slots marked empty are exactly the rest, and the ranges are balanced. The
kernel itself is checked on the GPU by the slot-cover tests of
test_gpu_fp8.py."""
import random

import pytest

TG = 256


def _schedule(lens, Hk, P, G):
    Ts = [(max(0, L) + TG - 1) // TG for L in lens]
    B, W, Tmax = len(lens), sum(Ts), max(Ts, default=0)
    cover, empties, work = {}, {}, [0] * G
    for blk in range(G):
        if G >= Hk:
            NG, g, h0, hstep = G // Hk, blk // Hk, blk % Hk, Hk
        else:
            NG, g, h0, hstep = 1, 0, blk, G
        NGe = NG
        if P >= 2 and W > 0:
            rreq = -(-Tmax // max(1, P - 2))
            NGe = max(1, min(NG, W // rreq))
        active = W > 0 and g < NGe
        rs, re = (W * g // NGe, W * (g + 1) // NGe) if active else (0, 0)
        rng_of = lambda x: ((x + 1) * NGe + W - 1) // W - 1  # noqa: E731
        for pr in range(blk, B * Hk, G):                       # pairs with no tokens
            if Ts[pr // Hk] == 0:
                empties.setdefault((pr // Hk, pr % Hk), set()).update(range(P))
        if not active:
            continue
        off, first = 0, None
        for s in range(B):
            if Ts[s] > 0 and ((off + Ts[s] > rs) if P >= 2 else (off >= rs)):
                first = (s, off)
                break
            off += Ts[s]
        if first is None:
            continue
        for h in range(h0, Hk, hstep):
            s, off = first
            while s < B and off < re:
                T = Ts[s]
                if T:
                    b, e, slot, nc = 0, T, 0, 1
                    if P >= 2:
                        b, e = max(rs, off) - off, min(re, off + T) - off
                        slot, nc = g - rng_of(off), rng_of(off + T - 1) - rng_of(off) + 1
                    assert 0 <= slot < nc <= P and b < e
                    cover.setdefault((s, h), []).append((slot, b, e))
                    work[blk] += e - b
                    if slot == 0 and nc < P:
                        empties.setdefault((s, h), set()).update(range(nc, P))
                off += T
                s += 1
    return Ts, cover, empties, work


def _check(lens, Hk, P, G):
    Ts, cover, empties, work = _schedule(lens, Hk, P, G)
    for s, T in enumerate(Ts):
        for h in range(Hk):
            runs = sorted(cover.get((s, h), []))
            slots = [r[0] for r in runs]
            assert slots == list(range(len(slots)))
            pos = 0
            for _, b, e in runs:
                assert b == pos
                pos = e
            assert pos == T
            assert set(slots) | empties.get((s, h), set()) == set(range(P))
            assert not set(slots) & empties.get((s, h), set())
    return work


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes(seed):
    r = random.Random(seed)
    for _ in range(150):
        B = r.choice([1, 2, 3, 16, 40, 128])
        lens = [r.choice([0, 1, 255, 256, 257, r.randint(1, 20000)]) for _ in range(B)]
        _check(lens, r.choice([1, 2, 3, 8, 16, 200]), r.choice([1, 2, 3, 7, 32, 300]), r.choice([1, 7, 64, 152]))


def test_benchmark_shapes_are_balanced():
    # 16 x 16384 tokens, 8 heads, P = 32 on 152 SMs: 19 ranges of 53 or 54 tile groups
    work = _check([16384] * 16, 8, 32, 152)
    live = [w for w in work if w]
    assert len(live) == 152 and max(live) - min(live) <= 1
    # the ragged batch: the same balance
    r = random.Random(1)
    work = _check([r.randint(1024, 16384) for _ in range(128)], 8, 32, 152)
    assert max(work) - min(work) <= 1


@pytest.mark.parametrize("seed", range(3))
def test_row_blocks_share_their_heads_slots(seed):
    """Above 16 query rows per KV head the kernel schedules Hk * RB virtual
    heads (virtual head vh reads KV head vh // RB and writes rows 16 (vh % RB)
    .. of it): every row block of a head must get the same runs in the same
    slots, or its rows would be combined with another block's state."""
    r = random.Random(100 + seed)
    for _ in range(60):
        B = r.choice([1, 3, 16, 40])
        lens = [r.choice([0, 1, 257, r.randint(1, 20000)]) for _ in range(B)]
        Hk, RB = r.choice([1, 2, 8]), r.choice([2, 3, 4])
        P, G = r.choice([1, 2, 7, 32]), r.choice([5, 64, 152])
        Ts, cover, empties, _ = _schedule(lens, Hk * RB, P, G)
        _check(lens, Hk * RB, P, G)
        for s in range(B):
            for h in range(Hk):
                runs = [sorted(cover.get((s, h * RB + rb), [])) for rb in range(RB)]
                assert all(x == runs[0] for x in runs)
                emp = [empties.get((s, h * RB + rb), set()) for rb in range(RB)]
                assert all(x == emp[0] for x in emp)

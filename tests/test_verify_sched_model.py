"""The arithmetic of the persistent verify's work schedule, checked on the host.

The schedule lays the batch's key tiles end to end (unit u = b * n_kv_heads +
kvh holds ceil(len_b / 128) tiles), gives CTA c the run [c * chunk, (c + 1) *
chunk), cuts each run into one segment per unit it touches, stores segment
(c, u) in partial slot c + u, and merges unit u from slots c0(u) + u ..
c1(u) + u.  This is a plain restatement of those rules (the CUDA kernels
carry them out on the device); the properties below are what makes them
correct: every tile is streamed exactly once, no two segments share a slot,
every slot lies inside the workspace, and the merge reads exactly the slots
of the unit's own segments.  The GPU tests check the kernels themselves
against the oracle.
"""
import math
import random

import pytest

TILE = 128


def schedule(lens, n_kv_heads, n_cta):
    nt = [math.ceil(max(0, n) / TILE) for n in lens]
    prefix = [0]
    for x in nt:
        prefix.append(prefix[-1] + x)
    total = prefix[-1] * n_kv_heads
    chunk = -(-total // n_cta) if total > 0 else 1
    starts = []
    for c in range(n_cta):
        t0 = c * chunk
        if t0 >= total:
            starts.append((0, 0, 0, 0))
            continue
        lo, hi = 0, len(lens) - 1
        while lo < hi:  # first b with n_kv_heads * prefix[b + 1] > t0
            mid = (lo + hi) // 2
            if n_kv_heads * prefix[mid + 1] > t0:
                hi = mid
            else:
                lo = mid + 1
        n_b = prefix[lo + 1] - prefix[lo]
        within = t0 - n_kv_heads * prefix[lo]
        kvh = within // n_b
        starts.append((lo, kvh, within - kvh * n_b, min(chunk, total - t0)))
    return prefix, chunk, total, starts


def walk(start, prefix, n_kv_heads):
    b, kvh, t_off, left = start
    batch = len(prefix) - 1
    segs = []
    while left > 0 and b < batch:
        nt = prefix[b + 1] - prefix[b]
        if nt <= 0:
            b, kvh, t_off = b + 1, 0, 0
            continue
        if t_off < nt:
            take = min(nt - t_off, left)
            segs.append((b, kvh, t_off, take))
            left -= take
            t_off += take
            if t_off >= nt:
                t_off = 0
                kvh += 1
                if kvh == n_kv_heads:
                    kvh, b = 0, b + 1
            continue
        t_off = 0
        kvh += 1
        if kvh == n_kv_heads:
            kvh, b = 0, b + 1
    return segs


def merge_slots(b, kvh, prefix, chunk, n_kv_heads):
    nt = prefix[b + 1] - prefix[b]
    if nt == 0:
        return []
    start = n_kv_heads * prefix[b] + kvh * nt
    c0, c1 = start // chunk, (start + nt - 1) // chunk
    u = b * n_kv_heads + kvh
    return list(range(c0 + u, c1 + u + 1))


def check(lens, n_kv_heads, n_cta):
    prefix, chunk, total, starts = schedule(lens, n_kv_heads, n_cta)
    units = len(lens) * n_kv_heads
    n_slots = n_cta + units - 1
    covered = {}
    slots = {}
    for c, st in enumerate(starts):
        segs = walk(st, prefix, n_kv_heads)
        assert sum(n for *_, n in segs) == st[3]
        for b, kvh, t0, n in segs:
            u = b * n_kv_heads + kvh
            slot = c + u
            assert 0 <= slot < n_slots
            assert slot not in slots, "two segments share a partial slot"
            slots[slot] = (b, kvh)
            for t in range(t0, t0 + n):
                assert (b, kvh, t) not in covered, "a tile streamed twice"
                covered[(b, kvh, t)] = c
    for b in range(len(lens)):
        nt = prefix[b + 1] - prefix[b]
        for kvh in range(n_kv_heads):
            for t in range(nt):
                assert (b, kvh, t) in covered, "a tile never streamed"
            want = sorted(s for s, unit in slots.items() if unit == (b, kvh))
            assert merge_slots(b, kvh, prefix, chunk, n_kv_heads) == want
    assert len(covered) == total
    # every run but the last holds the same number of tiles
    runs = [st[3] for st in starts if st[3] > 0]
    assert all(r == chunk for r in runs[:-1])


@pytest.mark.parametrize("n_cta", [1, 7, 152, 304])
def test_schedule_on_fixed_mixes(n_cta):
    check([4000, 0, 130, 128, 1, 2500, 777, 3, 256, 1900], 2, n_cta)
    check([0, 0, 0], 2, n_cta)
    check([9000, 9000, 9000], 4, n_cta)
    check([40000] + [5] * 63, 2, n_cta)
    check([1] * 500, 3, n_cta)


def test_schedule_on_random_mixes():
    rng = random.Random(7)
    for _ in range(200):
        B = rng.randint(1, 40)
        hi = rng.choice([1, 200, 5000, 300000])
        lens = [rng.randint(0, hi) for _ in range(B)]
        check(lens, rng.choice([1, 2, 8]), rng.choice([1, 3, 152, 304, 1000]))

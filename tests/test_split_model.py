"""A CPU model of the decode kernel's balanced split in cost order, checked on
seeded random batches (host logic: no GPU).

The kernel (pa_decode.cuh, frag_balanced / ring_of / MergeSlots) lays the
attended units out segment by segment, (sequence, KV head) in order, each
segment charged its units plus `frag_cost` positions of overhead, and gives
ring g the positions [g*U/nw, (g+1)*U/nw).  A ring owns the units whose
positions fall in its range; a range that ends inside a segment's leading
overhead gives the whole segment to the next ring.  Split segments write one
partial record per fragment into slot 2*ring + (0 for the ring's first
fragment, 1 otherwise), and the merging warp recomputes, from the segment
alone, how many fragments it has (the rings of its first and last unit) and
where each record lives.  This model restates those rules and checks that:
  * every attended unit is assigned to exactly one ring;
  * the fragment count and record slots the merge recomputes are the ones the
    fragments wrote, and no two records share a slot;
  * the forward scan from the previous fragment's sequence (the kernel's
    fragment transition) finds the same sequence as a binary search;
  * a fragment the kernel treats as its ring's last (its end reaches the end
    of the ring's range, where it arrives with an acquire) has no successor.
"""

import numpy as np
import pytest


def _binary_seq(prefix, S, u):
    lo, hi = 0, S - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if prefix[mid] <= u:
            lo = mid
        else:
            hi = mid - 1
    return lo


def _split(lens, Hkv, UR, beta, nw_total, window=0, q_len=1, min_units=2):
    S = len(lens)
    segs = []  # (attended units, first attended unit) per sequence
    for T in lens:
        first = T - q_len + 1
        lo = first - window if (window > 0 and first > window) else 0
        segs.append((((T + UR - 1) // UR) - (lo // UR), lo // UR))
    prefix = [0]
    for nu, _ in segs:
        prefix.append(prefix[-1] + ((nu + beta) * Hkv if nu > 0 else 0))
    U = prefix[-1]
    if U == 0:
        return 0
    want = (U + min_units + beta - 1) // (min_units + beta)
    nw = max(1, min(want, nw_total))
    covered, frags = {}, {}
    for g in range(nw):
        u, u1 = g * U // nw, (g + 1) * U // nw
        s = _binary_seq(prefix, S, u)
        ring_frags = []
        while u < u1:
            while s + 1 < S and prefix[s + 1] <= u:  # forward scan
                s += 1
            assert s == _binary_seq(prefix, S, u)
            seg = (prefix[s + 1] - prefix[s]) // Hkv
            assert seg > 0
            r = u - prefix[s]
            kvh, off = r // seg, r % seg
            seg_start = prefix[s] + kvh * seg
            fend = min(u1, seg_start + seg)
            ja, jb = max(0, off - beta), fend - seg_start - beta
            if jb <= ja:  # the range ends inside this segment's overhead
                u = fend
                continue
            nu = seg - beta
            slot = -1 if (ja == 0 and jb == nu) else 2 * g + (0 if not ring_frags else 1)
            for j in range(ja, jb):
                assert (s, kvh, j) not in covered
                covered[(s, kvh, j)] = g
            ring_frags.append((fend, u1))
            frags.setdefault((s, kvh), []).append((g, slot))
            u = fend
        for i, (fend, end) in enumerate(ring_frags):
            if fend >= end:
                assert i == len(ring_frags) - 1
    assert len(covered) == sum(nu for nu, _ in segs) * Hkv

    def ring_of(x):
        return ((x + 1) * nw - 1) // U

    for (s, kvh), fr in frags.items():
        seg = (prefix[s + 1] - prefix[s]) // Hkv
        seg_start = prefix[s] + kvh * seg
        first_w = ring_of(seg_start + beta)
        nfr = ring_of(seg_start + seg - 1) - first_w + 1
        assert nfr == len(fr)
        if nfr == 1:
            assert fr[0][1] == -1
            continue
        for f, (g, slot) in enumerate(fr):
            w = first_w + f
            assert g == w
            assert slot == 2 * w + (1 if w * U // nw < seg_start else 0)
    slots = [sl for fr in frags.values() for _, sl in fr if sl >= 0]
    assert len(slots) == len(set(slots))
    return len(slots)


@pytest.mark.parametrize("kind", ["uniform", "lognormal", "equal", "short"])
def test_balanced_split_covers_every_unit_and_merge_slots_agree(kind):
    rng = np.random.default_rng({"uniform": 1, "lognormal": 2, "equal": 3, "short": 4}[kind])
    records = 0
    for _ in range(250):
        S = int(rng.integers(1, 60))
        if kind == "uniform":
            lens = rng.integers(0, 300, size=S)
        elif kind == "lognormal":
            lens = np.clip(np.round(rng.lognormal(5, 1.2, size=S)), 0, 3000).astype(int)
        elif kind == "equal":
            lens = np.full(S, int(rng.integers(1, 2000)))
        else:
            lens = rng.integers(0, 40, size=S)
        records += _split([int(x) for x in lens], Hkv=int(rng.choice([1, 2, 8])), UR=int(rng.choice([32, 64])),
                          beta=int(rng.integers(0, 5)), nw_total=int(rng.choice([1, 3, 17, 912])),
                          window=int(rng.choice([0, 0, 50, 300])), q_len=int(rng.choice([1, 1, 3])))
    assert records > 0  # the batches do split segments


def test_workload_batches_split_as_the_kernel_does():
    """The bench's GQA and FP8 batches on 152 SMs x 6 rings, with the kernel's fragment charge of 3."""
    import workloads
    for name, ur in (("gqa_32x4k", 32), ("fp8_mix", 64), ("long_32k", 32)):
        b = workloads.make_batch(name, seed=0)
        assert _split([int(x) for x in b.seq_lens], b.num_kv_heads, ur, 3, 152 * 6) > 0


@pytest.mark.parametrize("GM,D", [(4, 64), (4, 128), (8, 64), (8, 128), (16, 64), (16, 128)])
def test_merge_output_staging_is_a_bijection_read_back_by_rows(GM, D):
    """The split merge's output staging: lane l folds row l % GM, element l + 32 j of a record being
    (column (l + 32 j) // GM, row l % GM); it stores that element at row * D + ((col // 4) ^ (row % 8)) * 4
    + col % 4, and the rows are then read 16 bytes per lane, lane c taking physical chunk c ^ (row % 8).
    Every element lands once, inside GM * D words, and every row reads back its own columns in order."""
    per = GM * D // 32
    where = {}
    for lane in range(32):
        g = lane % GM
        for j in range(per):
            d = (lane + 32 * j) // GM
            assert (lane + 32 * j) % GM == g
            addr = g * D + ((((d >> 2) ^ (g & 7)) << 2) | (d & 3))
            assert 0 <= addr < GM * D and addr not in where.values()
            where[(g, d)] = addr
    assert len(where) == GM * D
    inv = {a: k for k, a in where.items()}
    for r in range(GM):
        for c in range(D // 4):
            base = r * D + ((c ^ (r & 7)) << 2)
            assert [inv[base + k] for k in range(4)] == [(r, 4 * c + k) for k in range(4)]

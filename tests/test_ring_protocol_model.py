"""A CPU model of one decode ring's handshakes, run under random schedules
(host logic: no GPU).

A ring has NS stages and NC consumer warps (NC > 1: several queries per
sequence, 16 rows per warp).  The producer issues the ring's units in order:
unit i goes to stage i % NS once every consumer has released the unit NS
before it on that stage (the stage's empty barrier counts NC arrivals).  With
several queries the query rows of a fragment live in one buffer per ring: the
producer copies them with the fragment's first unit, and only once every
consumer has read the previous fragment's rows (the q_empty barrier, NC
arrivals per phase).  A consumer waits for each unit's stage to be full, reads
the query rows at its fragment's first unit and arrives on q_empty, computes,
then releases the stage.  The model checks, over many random interleavings and
fragment lengths (down to one unit), that every consumer reads the rows of its
own fragment (never a later fragment's or a half-written buffer), that every
stage holds the unit a consumer expects, and that the ring always finishes.
"""

import numpy as np
import pytest


def _run(frag_lens, NS, NC, rng):
    units = [f for f, n in enumerate(frag_lens) for _ in range(n)]  # fragment of each unit, in order
    first = {}
    for i, f in enumerate(units):
        first.setdefault(f, i)
    N = len(units)
    stage = [None] * NS            # unit held by each stage (None: free for the producer)
    released = [[0] * NS for _ in range(NC)]  # per consumer: releases of each stage so far
    qbuf = None                    # fragment whose rows the query buffer holds
    q_loads = 0                    # query loads issued
    q_reads = [0] * NC             # per consumer: query reads done (one per fragment)
    issued = 0
    pos = [0] * NC                 # next unit of each consumer
    phase = [0] * NC               # 0: wait for the stage; 1: computing (stage held)
    steps = 0
    while min(pos) < N:
        steps += 1
        assert steps < 100000, "no progress: the protocol deadlocked"
        actors = ["p"] + list(range(NC))
        who = actors[int(rng.integers(0, len(actors)))]
        if who == "p":
            if issued == N:
                continue
            st = issued % NS
            # the stage is free once every consumer has released the unit NS before
            if issued >= NS and min(released[c][st] for c in range(NC)) < issued // NS:
                continue
            if issued == first[units[issued]] and q_loads > 0 and min(q_reads) < q_loads:
                continue  # the query buffer is still being read
            stage[st] = issued
            if issued == first[units[issued]]:
                qbuf = units[issued]
                q_loads += 1
            issued += 1
        else:
            c = who
            i = pos[c]
            if i >= N:
                continue
            st = i % NS
            if phase[c] == 0:
                if stage[st] != i:
                    continue  # not full yet
                assert stage[st] == i
                if i == first[units[i]]:
                    assert qbuf == units[i], "a consumer read another fragment's query rows"
                    q_reads[c] += 1
                phase[c] = 1
            else:
                released[c][st] += 1
                phase[c] = 0
                pos[c] += 1
    assert issued == N and q_reads == [len(frag_lens)] * NC


@pytest.mark.parametrize("NC", [1, 2, 3, 4])
@pytest.mark.parametrize("NS", [2, 3, 8])
def test_query_buffer_and_stage_handshakes_under_random_schedules(NS, NC):
    rng = np.random.default_rng(100 * NS + NC)
    for _ in range(60):
        nfrag = int(rng.integers(1, 12))
        frag_lens = [int(x) for x in rng.choice([1, 1, 2, 3, 7], size=nfrag)]
        _run(frag_lens, NS, NC, rng)

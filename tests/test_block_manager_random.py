"""Random operation sequences on the host block manager (the copy-on-write
decision of the PagedAttention explainer's "Copy-on-Write（CoW）によるメモリ共有"
section), checked three ways after every operation:
  * content: a simulated pool receives every token write at the slot the
    manager returns, and every copy pair as a whole-block copy (what
    pa_copy_blocks does); each live sequence must read back exactly its own
    history (inherited at fork time, then its own appends) through its table;
  * reference counts equal the number of table entries naming each block, and
    the free list holds exactly the unreferenced blocks;
  * tables, counts and copy pairs equal a mirror driven by the oracle's
    refcount primitives (allocate / share / release / copy_on_write).
"""

import numpy as np
import pytest

import oracle
import paged_kv_cache_144_gb300 as pa


class _Mirror:
    def __init__(self, free, B):
        self.om = oracle.RefcountBlockManager(free)
        self.t, self.n, self.B = {}, {}, B

    def append(self, s):
        pos = self.n[s]
        j = pos // self.B
        if j == len(self.t[s]):
            self.t[s].append(self.om.allocate())
        else:
            oracle.copy_on_write(self.t, s, j, self.om)
        self.n[s] = pos + 1

    def fork(self, p, c):
        self.t[c], self.n[c] = list(self.t[p]), self.n[p]
        for b in self.t[c]:
            self.om.share(b)

    def free(self, s):
        for b in self.t.pop(s):
            self.om.release(b)
        del self.n[s]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("B", [1, 4, 16])
def test_random_operations_keep_every_sequence_isolated(seed, B):
    rng = np.random.default_rng(seed * 31 + B)
    NB = 48
    free = [int(x) for x in rng.permutation(NB)]
    bm = pa.BlockManager(NB, B, free_order=free)
    mir = _Mirror(free, B)
    pool = {}            # slot -> value
    hist = {}            # sequence -> values it must read back
    next_id, next_val = 0, 1
    for _ in range(300):
        live = sorted(hist)
        op = rng.choice(["add", "fork", "append", "append", "append", "free"]) if live else "add"
        try:
            if op == "add":
                n = int(rng.integers(0, 3 * B + 1))
                mir.t[next_id], mir.n[next_id] = [], 0
                try:
                    slots = bm.add_sequence(next_id, n)
                except MemoryError:
                    # the manager reserved blocks until the pool ran out: the mirror does the same, then
                    # both give them back (in table order, so the free lists stay in step)
                    try:
                        for _k in range(n):
                            mir.append(next_id)
                    except MemoryError:
                        pass
                    bm.free(next_id)
                    mir.free(next_id)
                    next_id += 1
                    raise
                for _k in range(n):
                    mir.append(next_id)
                hist[next_id] = []
                for sl in slots:
                    pool[sl] = next_val
                    hist[next_id].append(next_val)
                    next_val += 1
                next_id += 1
            elif op == "fork":
                p = live[int(rng.integers(len(live)))]
                bm.fork(p, next_id)
                mir.fork(p, next_id)
                hist[next_id] = list(hist[p])
                next_id += 1
            elif op == "append":
                s = live[int(rng.integers(len(live)))]
                copies_before = len(mir.om.copies)
                mir.append(s)
                sl, pair = bm.append_slot(s)
                want_pair = mir.om.copies[copies_before] if len(mir.om.copies) > copies_before else None
                assert pair == want_pair
                if pair is not None:          # the device copy of the whole block, before the write
                    src, dst = pair
                    for r in range(B):
                        if src * B + r in pool:
                            pool[dst * B + r] = pool[src * B + r]
                pool[sl] = next_val
                hist[s].append(next_val)
                next_val += 1
            else:
                s = live[int(rng.integers(len(live)))]
                bm.free(s)
                mir.free(s)
                del hist[s]
        except MemoryError:
            # pool exhausted (an append raises before either side changes): free the longest sequence
            if hist:
                s = max(hist, key=lambda k: len(hist[k]))
                bm.free(s)
                mir.free(s)
                del hist[s]
            continue
        # content: every live sequence reads back its own history
        for s, vals in hist.items():
            assert [pool[bm.slot(s, p)] for p in range(len(vals))] == vals
        # reference counts and the free list
        refs = {}
        for t in bm.tables.values():
            for b in t:
                refs[b] = refs.get(b, 0) + 1
        assert bm.refcount == refs
        assert sorted(bm._free) == sorted(set(range(NB)) - set(refs))
        # the oracle-driven mirror
        assert bm.tables == mir.t and bm.refcount == mir.om.refcount

"""Reference-counted block sharing and the copy-on-write decision.

Test infrastructure (see ``oracle/__init__``).

[P1] §"Copy-on-Write（CoW）によるメモリ共有": sequences that share a prompt point
their block tables at the same physical blocks, and every physical block
carries a reference count.  Before a sequence writes into one of its blocks:
if more than one table references that block, a fresh block is taken from
the allocator, the old block's contents are copied into it, the old block's
count drops by one and this sequence's table entry is redirected to the
fresh block, which is then written; if the sequence is the only holder, it
writes in place.  [P2] §"prefix共有とcopy-on-write" and [P3] §"KV Cache 共享机制"
describe the same rule (share while reading, copy at the first write).

This module records the decisions (the (src, dst) copy list and the final
tables); the byte copy itself is ``cache_ops.copy_blocks``.  It is the oracle
for the library's host-side block manager.

Pins: the isolation property (after the copies no sequence sees another's
private writes) and the reference-count invariants
(``tests/test_oracle_pins.py::test_cow_*``).
"""

from __future__ import annotations


class RefcountBlockManager:
    """Physical block ids handed out from a given free-list order, with refcounts."""

    def __init__(self, free_order):
        self.free = list(int(b) for b in free_order)
        self.refcount: dict[int, int] = {}
        self.copies: list[tuple[int, int]] = []

    def allocate(self) -> int:
        if not self.free:
            raise MemoryError("block pool exhausted")
        b = self.free.pop(0)
        self.refcount[b] = 1
        return b

    def share(self, block: int) -> None:
        self.refcount[block] += 1

    def release(self, block: int) -> None:
        self.refcount[block] -= 1
        if self.refcount[block] == 0:
            del self.refcount[block]
            self.free.append(block)


def copy_on_write(tables: dict, seq_id, logical_block: int, manager: RefcountBlockManager) -> int:
    """Physical block that ``seq_id`` may write for ``logical_block``; copies if shared."""
    current = tables[seq_id][logical_block]
    if manager.refcount[current] <= 1:
        return current
    fresh = manager.allocate()
    manager.copies.append((current, fresh))
    manager.refcount[current] -= 1
    tables[seq_id][logical_block] = fresh
    return fresh

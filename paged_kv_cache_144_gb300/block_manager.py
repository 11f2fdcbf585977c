"""Host-side block manager: allocation, sharing and the copy-on-write decision.

The PagedAttention explainer (0h-n0.github.io), §"Copy-on-Write（CoW）による
メモリ共有", splits copy-on-write into a host decision and a device copy:
sequences that share a prompt reference the same physical blocks, each block
has a reference count, and a sequence about to write into a block that other
sequences still reference first receives a fresh block holding a copy (the
count of the old block drops by one); a sole holder writes in place.
"KVキャッシュとPagedAttention" (youngju.dev), §"PagedAttention: OS仮想メモリ式の
管理", adds that blocks are handed out one at a time as tokens accumulate.

This class makes those decisions and returns the slot numbers and (src, dst)
copy pairs that ``pa_reshape_and_cache`` and ``pa_copy_blocks`` consume.
Slot encoding: slot = physical_block * block_size + position % block_size.
"""

from __future__ import annotations


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.block_size = int(block_size)
        self.num_blocks = int(num_blocks)
        order = range(num_blocks) if free_order is None else free_order
        self._free = [int(b) for b in order]
        self.refcount: dict[int, int] = {}
        self.tables: dict[object, list[int]] = {}
        self.lengths: dict[object, int] = {}

    # -- allocation -------------------------------------------------------
    def allocate(self) -> int:
        if not self._free:
            raise MemoryError("no free KV block")
        b = self._free.pop(0)
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            del self.refcount[b]
            self._free.append(b)

    @property
    def num_free(self) -> int:
        return len(self._free)

    # -- sequences --------------------------------------------------------
    def add_sequence(self, seq, num_tokens: int = 0) -> list[int]:
        """Register a sequence and reserve slots for its first tokens."""
        if seq in self.tables:
            raise KeyError(f"sequence {seq!r} exists")
        self.tables[seq] = []
        self.lengths[seq] = 0
        return [self.append_slot(seq)[0] for _ in range(num_tokens)]

    def fork(self, parent, child) -> None:
        """The child shares every block of the parent (reference counts +1)."""
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def free(self, seq) -> None:
        for b in self.tables.pop(seq):
            self._release(b)
        del self.lengths[seq]

    def copy_on_write(self, seq, logical_block: int):
        """Make ``logical_block`` of ``seq`` private; returns (src, dst) or None."""
        table = self.tables[seq]
        old = table[logical_block]
        if self.refcount[old] <= 1:
            return None
        new = self.allocate()
        self.refcount[old] -= 1
        table[logical_block] = new
        return (old, new)

    def append_slot(self, seq):
        """Slot for the next token of ``seq``; opens a block or copies a shared one.

        Returns (slot, cow_pair_or_None).
        """
        pos = self.lengths[seq]
        table = self.tables[seq]
        j = pos // self.block_size
        pair = None
        if j == len(table):
            table.append(self.allocate())
        else:
            pair = self.copy_on_write(seq, j)
        self.lengths[seq] = pos + 1
        return table[j] * self.block_size + pos % self.block_size, pair

    def slot(self, seq, position: int) -> int:
        return self.tables[seq][position // self.block_size] * self.block_size + position % self.block_size

    def block_table(self, seq, width: int | None = None, pad: int = -1) -> list[int]:
        t = list(self.tables[seq])
        if width is not None:
            t = t + [pad] * (width - len(t))
        return t

"""Reference block manager: allocation, sharing, copy-on-write and slot mapping.

TEST INFRASTRUCTURE ONLY.  A plain, slow restatement of the host-side block
bookkeeping the pages describe, used by the tests to check the library's C++
block manager operation by operation.  The product path never imports it.

Sources (web pages, cited by title and section):
  [GAO]  "PagedAttention & Continuous Batching": §1.3 a physical block holds
         block_size tokens and a reference count (prefix sharing), §1.4 each
         request keeps a block table (logical index -> physical block), blocks
         need not be contiguous, §1.5 slot = table[pos // bs] * bs + pos % bs.
  [FEI]  "vLLM 架构详解": "Block Table 实现" (blocks are allocated on demand;
         appending a token whose block is full allocates a new block),
         "共享前缀的 Block 复用" (tables of requests with a common prefix name
         the same physical blocks; those blocks' reference counts count the
         tables naming them).
  [LAKE] "vLLM源码解析(二)": §3.2 copy-on-write -- a sequence about to modify
         a block that other sequences share allocates a new physical block,
         copies the old block's contents into it, points its table at the new
         block and drops one reference to the old one; §4.2 a block comes from
         the free blocks, and an exhausted pool is an out-of-memory condition.
  [P1]   "vLLM核心机制": §3.1 a finished request's blocks return to the pool;
         parallel samples of one prompt share its blocks.

Readings where the pages are silent:
  - Which free block is taken: the lowest-numbered free block.
  - A sequence "modifies" a block when a token is appended into it; only a
    partially filled last block can receive one, so copy-on-write happens on
    the first token of an append whose last block is shared.
  - Fork (parallel samples / a shared prefix): the child gets the parent's
    table and token count; every block gains one reference.
  - An append that cannot get every block it needs (new blocks and a
    copy-on-write copy) fails and changes nothing.  A table longer than
    max_blocks_per_seq is refused the same way.
  - The FEI sketch's token count (`len(blocks) * block_size`, "近似值") is
    not used: the count is the number of tokens appended.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple


class OutOfBlocks(Exception):
    """No free physical block for an allocation ([LAKE] §4.2)."""


class TableFull(Exception):
    """A sequence would need more than max_blocks_per_seq blocks."""


def slot_for_position(table: Sequence[int], position: int, block_size: int) -> int:
    """[GAO] §1.5."""
    return table[position // block_size] * block_size + position % block_size


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.max_blocks_per_seq = max_blocks_per_seq
        self.ref: List[int] = [0] * num_blocks       # [GAO] §1.3 reference counts
        self.tables: Dict[int, List[int]] = {}       # [GAO] §1.4 block tables
        self.lengths: Dict[int, int] = {}            # tokens appended per sequence

    # -- the free pool ------------------------------------------------------
    def free_blocks(self) -> List[int]:
        return [b for b in range(self.num_blocks) if self.ref[b] == 0]

    def num_free(self) -> int:
        return len(self.free_blocks())

    def _allocate(self) -> int:
        free = self.free_blocks()
        if not free:
            raise OutOfBlocks()
        b = min(free)
        self.ref[b] = 1
        return b

    # -- sequences ----------------------------------------------------------
    def add_sequence(self, seq: int) -> None:
        if seq in self.tables or seq < 0:
            raise KeyError(seq)
        self.tables[seq] = []
        self.lengths[seq] = 0

    def fork(self, parent: int, child: int) -> None:
        """[FEI] shared blocks, [P1] §3.1 parallel samples: the child names
        the parent's blocks, each gaining a reference."""
        if parent not in self.tables or child in self.tables or child < 0:
            raise KeyError((parent, child))
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_sequence(self, seq: int) -> None:
        """[P1] §3.1: a finished request's blocks go back to the pool once no
        table names them."""
        for b in self.tables.pop(seq):
            self.ref[b] -= 1
        del self.lengths[seq]

    def blocks_needed(self, seq: int, n: int) -> int:
        length, bs = self.lengths[seq], self.block_size
        new = (length + n + bs - 1) // bs - (length + bs - 1) // bs
        cow = 0
        if n > 0 and length % bs != 0 and self.ref[self.tables[seq][-1]] > 1:
            cow = 1
        return new + cow

    def append_tokens(self, seq: int, n: int) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Slots of n new tokens of `seq` and the copy-on-write (src, dst)
        pairs the engine must copy before writing them."""
        table, bs = self.tables[seq], self.block_size
        length = self.lengths[seq]
        if (length + n + bs - 1) // bs > self.max_blocks_per_seq:
            raise TableFull()
        if self.blocks_needed(seq, n) > self.num_free():
            raise OutOfBlocks()
        slots, pairs = [], []
        for _ in range(n):
            pos = length
            if pos % bs == 0:
                # [FEI] the last block is full (or there is none): a new block
                table.append(self._allocate())
            else:
                last = table[pos // bs]
                if self.ref[last] > 1:
                    # [LAKE] §3.2: allocate, copy contents, remap, drop a reference
                    new = self._allocate()
                    pairs.append((last, new))
                    self.ref[last] -= 1
                    table[pos // bs] = new
            slots.append(slot_for_position(table, pos, bs))
            length += 1
        self.lengths[seq] = length
        return slots, pairs

    def append_batch(self, seqs: Sequence[int], counts: Sequence[int]
                     ) -> Tuple[List[int], List[Tuple[int, int]]]:
        """One step's appends: the appends of `seqs` in order, applied all or
        nothing.  Refusals are checked in this order: an unknown or repeated
        sequence (KeyError), a table past max_blocks_per_seq (TableFull),
        then running out of blocks part-way (OutOfBlocks)."""
        if len(set(seqs)) != len(seqs) or any(s not in self.tables for s in seqs):
            raise KeyError(seqs)
        bs = self.block_size
        for s, n in zip(seqs, counts):
            if n < 0:
                raise KeyError(s)
            if (self.lengths[s] + n + bs - 1) // bs > self.max_blocks_per_seq:
                raise TableFull()
        saved = (list(self.ref), {k: list(v) for k, v in self.tables.items()},
                 dict(self.lengths))
        slots, pairs = [], []
        try:
            for s, n in zip(seqs, counts):
                sl, pr = self.append_tokens(s, n)
                slots += sl
                pairs += pr
        except OutOfBlocks:
            self.ref, self.tables, self.lengths = saved
            raise
        return slots, pairs

    # -- step inputs ------------------------------------------------------------
    def build_batch(self, seqs: Sequence[int], max_blocks: int,
                    pad_block: int) -> Tuple[List[List[int]], List[int]]:
        tables, lens = [], []
        for s in seqs:
            row = list(self.tables[s]) + [pad_block] * (max_blocks - len(self.tables[s]))
            tables.append(row[:max_blocks])
            lens.append(self.lengths[s])
        return tables, lens

    def table(self, seq: int) -> List[int]:
        return list(self.tables[seq])

    def length(self, seq: int) -> Optional[int]:
        return self.lengths.get(seq)

"""Paged KV block pool policy (host side) -- TEST INFRASTRUCTURE.

"One forward per step", §What changed: the engine keeps a KV pool of fixed-size
blocks and reserves a request's blocks when it is admitted.  "33. Removing
overhead", §CUDA graphs for a changing batch: a scratch block that the block
manager never hands out absorbs the writes of padding rows.

The pages give no allocation order.  Reading taken: the free list starts as
0, 1, ..., num_blocks - 1; allocation takes from the front and freeing appends
to the back (first in, first out).  Block ``num_blocks`` is the scratch block.
This policy is deterministic, so block tables are compared bit for bit.
Pins: the pool tests check the policy on hand-worked sequences.
"""
from __future__ import annotations

from collections import deque


class PoolExhausted(RuntimeError):
    pass


def blocks_needed(tokens: int, block_size: int = 16) -> int:
    """Blocks a request reserves on admission to hold ``tokens`` positions."""
    return -(-int(tokens) // block_size)


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int = 16):
        if num_blocks <= 0:
            raise ValueError("num_blocks must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.scratch = num_blocks
        self._free: deque[int] = deque(range(num_blocks))
        self._used: set[int] = set()

    @property
    def free_count(self) -> int:
        return len(self._free)

    def alloc(self, n: int) -> list[int]:
        if n < 0:
            raise ValueError("negative block count")
        if n > len(self._free):
            raise PoolExhausted(f"need {n} blocks, {len(self._free)} free")
        out = [self._free.popleft() for _ in range(n)]
        self._used.update(out)
        return out

    def free(self, ids) -> None:
        ids = [int(i) for i in ids]
        for i in ids:
            if i not in self._used:
                raise ValueError(f"block {i} is not allocated")
        for i in ids:
            self._used.remove(i)
            self._free.append(i)

"""Plain-Python model of the fixed-block K/V allocator -- TEST INFRASTRUCTURE.

Semantics follow lucebox PR #555 (Summary): "an exact fixed-block paged K/V
allocator (transactional allocation, stale-handle detection, immediate
release)".  Readings where the page is silent:

  * A handle is ``(generation << 32) | index``.  Every block starts at
    generation 1; releasing a block bumps its generation, so any handle to it
    taken before the release is stale afterwards.
  * ``alloc(n)`` is all-or-nothing: with fewer than n free blocks it fails
    with OOM and changes nothing.  Free blocks are handed out from a LIFO
    stack that initially yields indices 0, 1, 2, ... in order; a released
    block is pushed on top, so it is the next one handed out (immediate
    release).
  * ``release(handles)`` is all-or-nothing too: if any handle is out of
    range, not currently allocated, of the wrong generation, or repeated in
    the same call, it fails with STALE and releases nothing.  Blocks are
    pushed in the order given.

The library's C++ allocator must match this model handle for handle.
"""
from __future__ import annotations

OK, INVALID, UNSUPPORTED, OOM, STALE = 0, 1, 2, 3, 4


class AllocatorModel:
    def __init__(self, n_blocks: int):
        if n_blocks <= 0 or n_blocks >= 2**31:
            raise ValueError("n_blocks")
        self.n = n_blocks
        self.gen = [1] * n_blocks
        self.live = [False] * n_blocks
        self.stack = list(range(n_blocks - 1, -1, -1))  # top = end of list = block 0

    def free_count(self) -> int:
        return len(self.stack)

    @staticmethod
    def handle(gen: int, idx: int) -> int:
        return ((gen & 0xFFFFFFFF) << 32) | (idx & 0xFFFFFFFF)

    def alloc(self, n: int):
        if n > len(self.stack):
            return OOM, []
        out = []
        for _ in range(n):
            idx = self.stack.pop()
            self.live[idx] = True
            out.append(self.handle(self.gen[idx], idx))
        return OK, out

    def _valid(self, h: int) -> bool:
        idx, gen = h & 0xFFFFFFFF, h >> 32
        return idx < self.n and self.live[idx] and self.gen[idx] == gen

    def release(self, handles):
        seen = set()
        for h in handles:
            if not self._valid(h) or h in seen:
                return STALE
            seen.add(h)
        for h in handles:
            idx = h & 0xFFFFFFFF
            self.live[idx] = False
            self.gen[idx] = (self.gen[idx] + 1) & 0xFFFFFFFF or 1
            self.stack.append(idx)
        return OK

    def block_index(self, h: int):
        if not self._valid(h):
            return STALE, -1
        return OK, h & 0xFFFFFFFF

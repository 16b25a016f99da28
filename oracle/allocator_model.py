"""Plain-Python model of the fixed-block K/V allocator -- TEST INFRASTRUCTURE.

Semantics follow lucebox PR #555: its Summary asks for an exact fixed-block
allocator whose allocations are transactional, whose stale handles are
detected and whose releases take effect at once; its roadmap (item 6) adds
prefix caching, sharing prefix blocks by reference count with copy-on-write.
Readings where the page is silent:

  * A handle is ``(generation << 32) | index``.  Every block starts at
    generation 1; a block's generation is bumped when it returns to the free
    list, so any handle to it taken before then is stale afterwards.
  * Every allocated block carries a reference count, 1 after ``alloc``.
  * ``alloc(n)`` is all-or-nothing: with fewer than n free blocks it fails
    with OOM and changes nothing.  Free blocks are handed out from a LIFO
    stack that initially yields indices 0, 1, 2, ... in order; a block that
    becomes free is pushed on top, so it is the next one handed out.
  * ``share(handles)`` takes one more reference per occurrence of a handle;
    any stale handle fails the call with STALE and nothing changes.
  * ``release(handles)`` drops one reference per occurrence; a block whose
    count reaches 0 is freed at that occurrence (pushed in that order).  It
    is all-or-nothing: a handle that is out of range, not allocated, of the
    wrong generation, or that occurs more often than its reference count
    fails the call with STALE and releases nothing.
  * ``cow(handles)`` prepares blocks for writing.  Taking the handles in
    order: a block held once is returned as it is; a shared block gets a
    fresh block in its place (the old one loses the caller's reference) and
    a copy (old index, new index) is listed for the caller to perform on the
    device.  All-or-nothing: a stale handle gives STALE, too few free blocks
    for the copies gives OOM, and nothing changes.

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
        self.ref = [0] * n_blocks
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
            self.ref[idx] = 1
            out.append(self.handle(self.gen[idx], idx))
        return OK, out

    def _valid(self, h: int) -> bool:
        idx, gen = h & 0xFFFFFFFF, h >> 32
        return idx < self.n and self.ref[idx] > 0 and self.gen[idx] == gen

    def _free(self, idx: int) -> None:
        self.ref[idx] = 0
        self.gen[idx] = (self.gen[idx] + 1) & 0xFFFFFFFF or 1
        self.stack.append(idx)

    def share(self, handles):
        if not all(self._valid(h) for h in handles):
            return STALE
        for h in handles:
            self.ref[h & 0xFFFFFFFF] += 1
        return OK

    def release(self, handles):
        count = {}
        for h in handles:
            if not self._valid(h):
                return STALE
            count[h] = count.get(h, 0) + 1
            if count[h] > self.ref[h & 0xFFFFFFFF]:
                return STALE
        for h in handles:
            idx = h & 0xFFFFFFFF
            self.ref[idx] -= 1
            if self.ref[idx] == 0:
                self._free(idx)
        return OK

    def refcount(self, h: int):
        if not self._valid(h):
            return STALE, 0
        return OK, self.ref[h & 0xFFFFFFFF]

    def cow(self, handles):
        if not all(self._valid(h) for h in handles):
            return STALE, [], []
        # how many copies the sequence of handles needs
        left = {}
        copies = 0
        for h in handles:
            idx = h & 0xFFFFFFFF
            r = left.get(idx, self.ref[idx])
            if r > 1:
                copies += 1
                left[idx] = r - 1
            else:
                left[idx] = r
        if copies > len(self.stack):
            return OOM, [], []
        out, pairs = [], []
        for h in handles:
            idx = h & 0xFFFFFFFF
            if self.ref[idx] > 1:
                self.ref[idx] -= 1
                new = self.stack.pop()
                self.ref[new] = 1
                out.append(self.handle(self.gen[new], new))
                pairs.append((idx, new))
            else:
                out.append(h)
        return OK, out, pairs

    def block_index(self, h: int):
        if not self._valid(h):
            return STALE, -1
        return OK, h & 0xFFFFFFFF

"""Pins for the allocator model against the semantics the pages state:
transactional allocation, stale-handle detection and immediate release
(lucebox PR #555, Summary)."""
import numpy as np

from oracle.allocator_model import OK, OOM, STALE, AllocatorModel


def _state(a):
    return (list(a.gen), list(a.ref), list(a.stack))


def test_fresh_pool_hands_out_blocks_in_order():
    a = AllocatorModel(5)
    rc, hs = a.alloc(3)
    assert rc == OK and [h & 0xFFFFFFFF for h in hs] == [0, 1, 2]
    assert all(h >> 32 == 1 for h in hs)
    assert a.free_count() == 2


def test_alloc_is_all_or_nothing():
    a = AllocatorModel(4)
    a.alloc(3)
    before = _state(a)
    rc, hs = a.alloc(2)
    assert rc == OOM and hs == [] and _state(a) == before


def test_release_is_immediate_and_bumps_generation():
    a = AllocatorModel(4)
    _, hs = a.alloc(2)
    assert a.release([hs[1]]) == OK
    rc, again = a.alloc(1)
    assert rc == OK and again[0] & 0xFFFFFFFF == hs[1] & 0xFFFFFFFF
    assert again[0] >> 32 == (hs[1] >> 32) + 1
    assert a.block_index(hs[1])[0] == STALE       # the old handle is stale
    assert a.block_index(again[0]) == (OK, hs[1] & 0xFFFFFFFF)


def test_stale_release_changes_nothing():
    a = AllocatorModel(6)
    _, hs = a.alloc(4)
    a.release([hs[0]])
    before = _state(a)
    for bad in ([hs[1], hs[0]], [hs[2], hs[2]], [hs[3], (1 << 32) | 99]):
        assert a.release(bad) == STALE and _state(a) == before


def test_random_sequences_keep_invariants():
    rng = np.random.default_rng(0)
    for trial in range(20):
        n = int(rng.integers(1, 40))
        a = AllocatorModel(n)
        held = []
        for _ in range(300):
            if rng.random() < 0.5:
                k = int(rng.integers(0, n + 2))
                before = _state(a)
                rc, hs = a.alloc(k)
                if k > n - len(held):
                    assert rc == OOM and _state(a) == before
                else:
                    assert rc == OK and len(hs) == k
                    held += hs
            elif held:
                k = int(rng.integers(1, len(held) + 1))
                idx = rng.choice(len(held), size=k, replace=False)
                rel = [held[i] for i in idx]
                assert a.release(rel) == OK
                held = [h for i, h in enumerate(held) if i not in set(idx.tolist())]
                assert a.release(rel[:1]) == STALE
            live_idx = [h & 0xFFFFFFFF for h in held]
            assert len(set(live_idx)) == len(live_idx)
            assert a.free_count() + len(held) == n
            assert all(a.block_index(h)[0] == OK for h in held)


def test_shared_blocks_free_at_last_reference():
    """A shared block is freed (and its generation bumped) only when its last
    reference is released; releasing more references than held changes
    nothing."""
    a = AllocatorModel(3)
    _, (h,) = a.alloc(1)
    assert a.share([h, h]) == OK and a.refcount(h) == (OK, 3)
    before = _state(a)
    assert a.release([h, h, h, h]) == STALE and _state(a) == before
    assert a.release([h]) == OK and a.refcount(h) == (OK, 2) and a.free_count() == 2
    assert a.release([h, h]) == OK and a.refcount(h) == (STALE, 0) and a.free_count() == 3
    assert a.alloc(1) == (OK, [AllocatorModel.handle(2, 0)])


def test_cow_copies_only_shared_blocks_and_is_all_or_nothing():
    a = AllocatorModel(4)
    _, (x, y) = a.alloc(2)
    a.share([x])
    rc, out, pairs = a.cow([x, y, x])
    # x shared twice: the first occurrence copies (x keeps one reference), the
    # second finds it held once and keeps it; y is private
    assert rc == OK and out[1] == y and out[2] == x and pairs == [(0, 2)]
    assert a.refcount(x) == (OK, 1) and a.refcount(out[0]) == (OK, 1)
    b = AllocatorModel(2)
    _, (u, v) = b.alloc(2)
    b.share([u, v])
    before = _state(b)
    assert b.cow([u, v])[0] == OOM and _state(b) == before
    assert b.cow([u, (9 << 32) | 1])[0] == STALE and _state(b) == before

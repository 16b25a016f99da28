"""Sharding a decode batch across GPUs: host logic, no device code.

The (sequence, KV head) segments of a decode batch are independent -- the
split-K decode of one never reads another's rows or partials (llama.cpp fork
PR #2, split-K decode commit: every KV head's six query heads attend to that
head's rows only; lucebox PR #555, Summary: ragged requests decode side by
side over one pool).  A batch therefore shards across GPUs with no exchange
at all: each rank holds the pages of its share, runs pa_decode on it, and the
outputs are put back in batch order.  Two ways to cut:

  * by sequence: whole sequences per rank, balanced by the K/V bytes a step
    reads (longest first onto the least-loaded rank);
  * by KV head: every rank holds all sequences but only some KV heads (their
    pools are built with n_kv_heads / n_ranks heads) and answers the query
    heads of those KV heads.

Splitting one sequence's context across GPUs would need one exchange of the
split partials (out, lse) and the same log-sum-exp merge; the pages measure
only single-device decode, so it is not offered here.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from . import row_bytes

GQA = 6  # query heads per KV head


def kv_bytes_per_sequence(seq_lens, k_type: int, v_type: int, n_kv_heads: int = 4, head_dim: int = 256) -> np.ndarray:
    """K/V bytes one decode step reads for each sequence (every live row of
    every KV head once)."""
    per_row = n_kv_heads * (row_bytes(k_type, head_dim) + row_bytes(v_type, head_dim))
    return np.asarray(seq_lens, dtype=np.int64) * per_row


def balance_by_sequence(weights: Sequence[int], n_ranks: int) -> list[list[int]]:
    """Assign whole sequences to ranks, balancing the summed weight.

    Longest-processing-time order: sequences by decreasing weight (ties by
    index), each onto the rank with the smallest load so far (ties: the lower
    rank).  Deterministic; each rank's list is in increasing sequence order.
    Every sequence lands on exactly one rank."""
    if n_ranks < 1:
        raise ValueError("n_ranks must be >= 1")
    w = np.asarray(weights, dtype=np.int64)
    order = sorted(range(len(w)), key=lambda i: (-int(w[i]), i))
    load = [0] * n_ranks
    parts: list[list[int]] = [[] for _ in range(n_ranks)]
    for i in order:
        r = min(range(n_ranks), key=lambda k: (load[k], k))
        parts[r].append(i)
        load[r] += int(w[i])
    return [sorted(p) for p in parts]


def split_kv_heads(n_kv_heads: int, n_ranks: int) -> list[range]:
    """Contiguous KV-head ranges, one per rank; n_ranks must divide the head
    count (each rank's pools then hold n_kv_heads / n_ranks heads)."""
    if n_ranks < 1 or n_kv_heads % n_ranks:
        raise ValueError(f"{n_ranks} ranks do not divide {n_kv_heads} KV heads")
    k = n_kv_heads // n_ranks
    return [range(r * k, (r + 1) * k) for r in range(n_ranks)]


def assemble_by_sequence(parts: list[list[int]], outs: list[np.ndarray], n_seq: int) -> np.ndarray:
    """Put the ranks' outputs ([len(part)][...] each, in their part's order)
    back in batch order.  Raises if a sequence is missing or repeated."""
    seen = np.zeros(n_seq, np.int32)
    for p in parts:
        seen[p] += 1
    if not (seen == 1).all():
        raise ValueError("the parts do not cover every sequence exactly once")
    shape = outs[0].shape[1:]
    full = np.empty((n_seq,) + shape, dtype=outs[0].dtype)
    for p, o in zip(parts, outs):
        if len(p):
            full[np.asarray(p)] = o
    return full


def assemble_by_kv_head(ranges: list[range], outs: list[np.ndarray]) -> np.ndarray:
    """Concatenate the ranks' outputs along the query-head axis (axis 2 of
    [n_seq][n_qtok][heads][...]): rank r answers query heads
    6 * ranges[r].start .. 6 * ranges[r].stop - 1."""
    for r, (rg, o) in enumerate(zip(ranges, outs)):
        if o.shape[2] != GQA * len(rg):
            raise ValueError(f"rank {r}: {o.shape[2]} query heads for {len(rg)} KV heads")
    return np.concatenate(outs, axis=2)

"""Seeded synthetic inputs for paged GQA decode attention.

This module only *produces input bytes*: random sources, per-block quantisers
that turn float sources into ggml F16/Q4_0/Q8_0 row bytes, block tables and
sequence lengths.  It holds none of the decode arithmetic (no dequantisation,
no gather, no softmax) so that both the float64 oracle and the CUDA library
can consume the same inputs without sharing any of the method's code.

Shapes follow the Qwen attention dims every benchmark of lucebox PR #555
(Benchmark results) uses: head size D=256, 24 query heads, 4 KV heads (GQA 6).

Quantiser (a reading: the pages name the formats but not a quantiser; any
deterministic quantiser is valid because both sides consume the same bytes):
  * Q8_0: d = max|x| / 127 over a 32-block, q = round-half-away(x / d) as int8,
    block = fp16 d (little endian) followed by 32 int8 quants (34 bytes).
  * Q4_0: m = the block element of largest magnitude (signed, first on ties),
    d = m / -8, q = min(15, trunc(x / d + 8.5)), block = fp16 d followed by 16
    bytes where byte j holds quant j in its low nibble and quant j+16 in its
    high nibble (18 bytes).
  * F16: IEEE binary16, round to nearest even.
The fp16 scale is rounded to nearest even; quants are computed from the
unrounded scale.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

D = 256
HQ = 24
HKV = 4
GQA = HQ // HKV
SCALE = 1.0 / 16.0  # 1/sqrt(256), exact in binary

# ggml type numbering (format identifiers only)
TYPE_F16 = 1
TYPE_Q4_0 = 2
TYPE_Q8_0 = 8
TYPE_NAMES = {TYPE_F16: "f16", TYPE_Q4_0: "q4_0", TYPE_Q8_0: "q8_0"}
BLOCK_BYTES = {TYPE_Q4_0: 18, TYPE_Q8_0: 34}

_GEN_CHUNK = 1 << 15  # tokens per random-generation chunk (fixes the stream layout)


def row_bytes(t: int, d: int = D) -> int:
    """Bytes of one stored K or V row of `d` values in format `t`."""
    if t == TYPE_F16:
        return 2 * d
    return (d // 32) * BLOCK_BYTES[t]


# ---------------------------------------------------------------- quantisers

def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """float32 [..., d] -> uint8 [..., d/32*34] ggml Q8_0 blocks."""
    lead = x.shape[:-1]
    xb = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, 32)
    amax = np.abs(xb).max(axis=1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    v = xb * inv[:, None]
    q = np.trunc(v + np.copysign(np.float32(0.5), v))
    q = np.clip(q, -127, 127).astype(np.int8)
    out = np.empty((xb.shape[0], 34), np.uint8)
    out[:, 0:2] = d.astype("<f2").view(np.uint8).reshape(-1, 2)
    out[:, 2:] = q.view(np.uint8)
    return out.reshape(*lead, x.shape[-1] // 32 * 34)


def quantize_q4_0(x: np.ndarray) -> np.ndarray:
    """float32 [..., d] -> uint8 [..., d/32*18] ggml Q4_0 blocks."""
    lead = x.shape[:-1]
    xb = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, 32)
    idx = np.argmax(np.abs(xb), axis=1)
    m = xb[np.arange(xb.shape[0]), idx]
    d = (m / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    q = np.trunc(xb * inv[:, None] + np.float32(8.5))
    q = np.clip(q, 0, 15).astype(np.uint8)
    out = np.empty((xb.shape[0], 18), np.uint8)
    out[:, 0:2] = d.astype("<f2").view(np.uint8).reshape(-1, 2)
    out[:, 2:] = q[:, :16] | (q[:, 16:] << 4)
    return out.reshape(*lead, x.shape[-1] // 32 * 18)


def encode_f16(x: np.ndarray) -> np.ndarray:
    """float32 [..., d] -> uint8 [..., 2d] little-endian IEEE binary16."""
    lead = x.shape[:-1]
    h = np.ascontiguousarray(x, dtype=np.float32).astype("<f2")
    return h.view(np.uint8).reshape(*lead, x.shape[-1] * 2)


def encode_rows(x: np.ndarray, t: int) -> np.ndarray:
    if t == TYPE_F16:
        return encode_f16(x)
    if t == TYPE_Q4_0:
        return quantize_q4_0(x)
    if t == TYPE_Q8_0:
        return quantize_q8_0(x)
    raise ValueError(f"unsupported type {t}")


def random_rows(rng: np.random.Generator, n_tokens: int, t: int,
                hkv: int = HKV, d: int = D) -> np.ndarray:
    """n_tokens x hkv rows from N(0,1) sources, stored in format t.

    Returns uint8 [n_tokens][hkv][row_bytes(t)].  Generated in fixed chunks so
    memory stays bounded at large sizes.
    """
    out = np.empty((n_tokens, hkv, row_bytes(t, d)), np.uint8)
    for a in range(0, n_tokens, _GEN_CHUNK):
        b = min(n_tokens, a + _GEN_CHUNK)
        x = rng.standard_normal((b - a, hkv, d), dtype=np.float32)
        out[a:b] = encode_rows(x, t)
    return out


# ---------------------------------------------------------------- tables

def pages_needed(length: int, ps: int) -> int:
    return (int(length) + ps - 1) // ps


def interleaved_blocks(lengths, ps: int) -> list[list[int]]:
    """Blocks handed out round-robin while a sequence still needs pages, the
    way a shared pool fills when requests arrive and grow concurrently."""
    need = [pages_needed(L, ps) for L in lengths]
    got: list[list[int]] = [[] for _ in lengths]
    nxt = 0
    while True:
        progressed = False
        for s, n in enumerate(need):
            if len(got[s]) < n:
                got[s].append(nxt)
                nxt += 1
                progressed = True
        if not progressed:
            return got


def table_from_lists(lists: list[list[int]], max_pages: int | None = None) -> np.ndarray:
    mp = max_pages if max_pages is not None else max(1, max(len(l) for l in lists))
    tab = np.full((len(lists), mp), -1, np.int32)
    for s, l in enumerate(lists):
        tab[s, :len(l)] = l
    return tab


# ---------------------------------------------------------------- workloads

@dataclass
class Workload:
    """One decode problem: logical K/V rows plus where each page lives."""
    name: str
    seq_lens: np.ndarray          # int32 [n_seq]
    n_qtok: int
    page_size: int
    n_blocks: int
    k_type: int
    v_type: int
    table: np.ndarray             # int32 [n_seq][max_pages]; unused entries -1
    k_rows: np.ndarray            # uint8 [total_tokens][HKV][row_bytes(k_type)], seq-major
    v_rows: np.ndarray            # uint8 [total_tokens][HKV][row_bytes(v_type)]
    q: np.ndarray                 # float32 [n_seq][n_qtok][HQ][D]
    scale: float = SCALE
    meta: dict = field(default_factory=dict)

    @property
    def n_seq(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.sum())

    @property
    def row_seq(self) -> np.ndarray:
        return np.repeat(np.arange(self.n_seq, dtype=np.int32), self.seq_lens)

    @property
    def row_pos(self) -> np.ndarray:
        return np.concatenate([np.arange(L, dtype=np.int32) for L in self.seq_lens]) \
            if self.total_tokens else np.zeros(0, np.int32)

    @property
    def seq_offsets(self) -> np.ndarray:
        o = np.zeros(self.n_seq + 1, np.int64)
        np.cumsum(self.seq_lens, out=o[1:])
        return o

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode step reads: every live row of every
        KV head, once."""
        return self.total_tokens * HKV * (row_bytes(self.k_type) + row_bytes(self.v_type))

    def with_table(self, table: np.ndarray, n_blocks: int, name: str | None = None) -> "Workload":
        return Workload(name or self.name, self.seq_lens, self.n_qtok, self.page_size, n_blocks,
                        self.k_type, self.v_type, table, self.k_rows, self.v_rows, self.q,
                        self.scale, dict(self.meta))

    def with_q(self, q: np.ndarray, n_qtok: int) -> "Workload":
        return Workload(self.name, self.seq_lens, n_qtok, self.page_size, self.n_blocks,
                        self.k_type, self.v_type, self.table, self.k_rows, self.v_rows, q,
                        self.scale, dict(self.meta))

    def subset(self, seq_ids) -> "Workload":
        """The batch made of sequences seq_ids (in that order, repeats
        allowed): their rows, queries and pages.  Block numbers are renumbered
        compactly, keeping their relative order (so the placement pattern
        survives); a repeated sequence gets its own copy of its pages."""
        ids = [int(i) for i in seq_ids]
        offs = self.seq_offsets
        lens = self.seq_lens[ids].astype(np.int32)
        k_rows = np.concatenate([self.k_rows[offs[i]:offs[i + 1]] for i in ids]) if ids else self.k_rows[:0]
        v_rows = np.concatenate([self.v_rows[offs[i]:offs[i + 1]] for i in ids]) if ids else self.v_rows[:0]
        pages = [self.table[i, :pages_needed(self.seq_lens[i], self.page_size)] for i in ids]
        keys = sorted((int(b), n, j) for n, pg in enumerate(pages) for j, b in enumerate(pg))
        new = {(n, j): r for r, (_, n, j) in enumerate(keys)}
        lists = [[new[(n, j)] for j in range(len(pg))] for n, pg in enumerate(pages)]
        return Workload(self.name, lens, self.n_qtok, self.page_size, len(keys), self.k_type, self.v_type,
                        table_from_lists(lists), k_rows, v_rows, np.ascontiguousarray(self.q[ids]), self.scale,
                        dict(self.meta))

    def contiguous(self, slots_per_seq: int | None = None) -> "Workload":
        """Same rows through an identity table: sequence s owns blocks
        [s*P, (s+1)*P) in order, P = slots_per_seq / page_size."""
        ps = self.page_size
        slots = slots_per_seq if slots_per_seq is not None else int(self.seq_lens.max())
        P = pages_needed(slots, ps)
        tab = np.full((self.n_seq, P), -1, np.int32)
        for s in range(self.n_seq):
            tab[s] = np.arange(s * P, (s + 1) * P, dtype=np.int32)
        return self.with_table(tab, self.n_seq * P, self.name + "/contiguous")


def make_workload(name: str, seed: int, lengths, ps: int, k_type: int, v_type: int,
                  n_qtok: int = 1, layout: str = "interleaved", pool_blocks: int | None = None,
                  ) -> Workload:
    """Build a workload.

    layout: 'interleaved'  - round-robin arrival order, blocks numbered 0..n-1;
            'shuffled'     - interleaved, then the pool's block ids permuted;
            'permuted'     - every page's block drawn from a seeded permutation
                             of a pool of `pool_blocks` blocks (holes allowed);
            'identity'     - sequence s owns a run of consecutive blocks.
    """
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    lists = interleaved_blocks(lengths, ps)
    n_pages = sum(len(l) for l in lists)
    n_blocks = n_pages
    if layout == "interleaved":
        pass
    elif layout == "shuffled":
        perm = rng.permutation(n_pages)
        lists = [[int(perm[b]) for b in l] for l in lists]
    elif layout == "permuted":
        n_blocks = int(pool_blocks) if pool_blocks is not None else n_pages
        assert n_blocks >= n_pages
        perm = rng.permutation(n_blocks)[:n_pages]
        it = iter(perm.tolist())
        lists = [[next(it) for _ in l] for l in lists]
    elif layout == "identity":
        nxt = 0
        lists = []
        for L in lengths:
            n = pages_needed(L, ps)
            lists.append(list(range(nxt, nxt + n)))
            nxt += n
    else:
        raise ValueError(layout)
    table = table_from_lists(lists)
    total = int(lengths.sum())
    k_rows = random_rows(rng, total, k_type)
    v_rows = random_rows(rng, total, v_type)
    q = rng.standard_normal((len(lengths), n_qtok, HQ, D), dtype=np.float32)
    return Workload(name, lengths, n_qtok, ps, n_blocks, k_type, v_type, table,
                    k_rows, v_rows, q, SCALE, {"seed": seed, "layout": layout})


# The five workloads, shaped like the pages' benchmarks.

RAGGED_LENGTHS = [131072] + [8192] * 7
VERIFY_LENGTHS = [32768, 20000, 9000, 513]


def lognormal_lengths(seed: int, n: int = 64) -> np.ndarray:
    rng = np.random.default_rng(seed)
    L = np.rint(rng.lognormal(mean=np.log(4096.0), sigma=1.2, size=n))
    return np.clip(L, 1, 65536).astype(np.int32)


def config(idx: int, n_qtok: int | None = None, variant: str = "") -> Workload:
    """Workload `idx` (1-based) with seed = idx.

    1 tiny    : 1 x 300 tokens, ps 16, 19 pages in a 32-block pool (seeded
                permutation), F16 K/V, 1 query token.
    2 uniform : 8 x 4096, ps 16, interleaved then shuffled pool, Q4_0.
    3 ragged  : 131072 + 7 x 8192, ps 16, interleaved (concurrent arrivals),
                Q4_0.  variant='contiguous' gives the identity table padded
                to 131072 slots per sequence.
    4 verify  : 32768/20000/9000/513, ps 256, shuffled pool, Q8_0, n_qtok 1..4.
    5a long   : 1 x 262144, F16, ps 64.
    5b many   : 64 sequences, lognormal(ln 4096, 1.2) lengths clipped to
                [1, 65536], ps 16, Q8_0.
    """
    if idx == 1:
        return make_workload("tiny", 1, [300], 16, TYPE_F16, TYPE_F16, 1, "permuted", 32)
    if idx == 2:
        return make_workload("uniform", 2, [4096] * 8, 16, TYPE_Q4_0, TYPE_Q4_0, 1, "shuffled")
    if idx == 3:
        w = make_workload("ragged", 3, RAGGED_LENGTHS, 16, TYPE_Q4_0, TYPE_Q4_0, 1, "interleaved")
        if variant == "contiguous":
            w = w.contiguous(131072)
        return w
    if idx == 4:
        return make_workload("verify", 4, VERIFY_LENGTHS, 256, TYPE_Q8_0, TYPE_Q8_0,
                             n_qtok or 4, "shuffled")
    if idx == 5 and variant in ("", "a", "long"):
        return make_workload("long", 5, [262144], 64, TYPE_F16, TYPE_F16, 1, "identity")
    if idx == 5 and variant in ("b", "many"):
        return make_workload("many", 5, lognormal_lengths(5), 16, TYPE_Q8_0, TYPE_Q8_0, 1,
                             "interleaved")
    raise ValueError((idx, variant))


def shared_prefix(n_seq: int = 8, prefix: int = 32768, own: int = 1024, ps: int = 16, k_type: int = TYPE_Q4_0,
                  v_type: int = TYPE_Q4_0, n_qtok: int = 1, seed: int = 7) -> Workload:
    """Prefix sharing (lucebox PR #555, roadmap item 6): n_seq sequences forked
    from one prompt of `prefix` rows (a multiple of ps) whose pages they all
    share, each followed by `own` rows of its own.  The prefix pages are
    blocks 0 .. prefix/ps - 1; the own pages follow, interleaved across
    sequences.  Logical rows are stored per sequence, so the prefix rows repeat
    (identical bytes) in k_rows / v_rows."""
    assert prefix % ps == 0
    rng = np.random.default_rng(seed)
    n_pre = prefix // ps
    pre_k = random_rows(rng, prefix, k_type)
    pre_v = random_rows(rng, prefix, v_type)
    own_k = [random_rows(rng, own, k_type) for _ in range(n_seq)]
    own_v = [random_rows(rng, own, v_type) for _ in range(n_seq)]
    own_lists = interleaved_blocks([own] * n_seq, ps)
    lists = [list(range(n_pre)) + [n_pre + b for b in own_lists[s]] for s in range(n_seq)]
    lengths = np.full(n_seq, prefix + own, np.int32)
    k_rows = np.concatenate([np.concatenate([pre_k, own_k[s]]) for s in range(n_seq)])
    v_rows = np.concatenate([np.concatenate([pre_v, own_v[s]]) for s in range(n_seq)])
    q = rng.standard_normal((n_seq, n_qtok, HQ, D), dtype=np.float32)
    n_blocks = n_pre + sum(len(l) for l in own_lists)
    return Workload(f"shared-prefix-{n_seq}x{prefix // 1024}k+{own}", lengths, n_qtok, ps, n_blocks, k_type, v_type,
                    table_from_lists(lists), k_rows, v_rows, q, SCALE, {"seed": seed, "layout": "shared prefix"})


PERCALL_LENGTHS = (32768, 131072, 262144)


def percall(length: int, n_qtok: int) -> Workload:
    """The per-call shape of the llama.cpp fork's RDNA4 table (PR #2, Q8_0 K
    scale-read commit): one sequence of 32k / 131k / 262k tokens, Q8_0 K with
    Q4_0 V, 1 / 3 / 4 query tokens.  The table gives no page size; 256-row
    pages (the fork's stream pages) in a shuffled pool are a reading."""
    assert length in PERCALL_LENGTHS and n_qtok in (1, 3, 4)
    return make_workload(f"percall-{ {32768: 32, 131072: 131, 262144: 262}[length]}k-{n_qtok}", 6, [length], 256, TYPE_Q8_0, TYPE_Q4_0,
                         n_qtok, "shuffled")


ROWS_CONTEXTS = (4096, 16384, 65536)
ROWS_QTOK = (17, 65, 96)


def rows_workload(context: int, n_qtok: int) -> Workload:
    """The shape of the llama.cpp fork's row-tile table (PR #2, the commit on
    ubatches of more than 8 tokens: chunked prefill against row tiles per
    attention layer): one sequence of 4k / 16k / 64k cached tokens, of which
    the last 17 / 65 / 96 are the query tokens.  The table gives no formats or
    page size; the fork's production pair (Q8_0 K, Q4_0 V) in 256-row pages of
    a shuffled pool is a reading, as for the per-call workload."""
    return make_workload(f"rows-{context // 1024}k-{n_qtok}", 7, [context], 256, TYPE_Q8_0, TYPE_Q4_0, n_qtok,
                         "shuffled")


def _table_for(rng: np.random.Generator, lengths, ps: int, layout: str):
    """Block table of `lengths` for the 'interleaved' / 'shuffled' / 'identity'
    layouts of make_workload; returns (table, n_blocks)."""
    lists = interleaved_blocks(lengths, ps)
    n_pages = sum(len(l) for l in lists)
    if layout == "shuffled":
        perm = rng.permutation(n_pages)
        lists = [[int(perm[b]) for b in l] for l in lists]
    elif layout == "identity":
        nxt, lists = 0, []
        for L in lengths:
            n = pages_needed(L, ps)
            lists.append(list(range(nxt, nxt + n)))
            nxt += n
    elif layout != "interleaved":
        raise ValueError(layout)
    return table_from_lists(lists), n_pages


STRESS_KINDS = ("rising", "late", "bigq", "scales")


def stress_workload(kind: str, seed: int, lengths, ps: int, k_type: int, v_type: int, n_qtok: int,
                    layout: str = "shuffled") -> Workload:
    """Inputs that push the online softmax's running maximum up after the
    first keys of a sequence, so that a decoder must rescale an accumulator
    that already holds weight (plus blocks with zero and subnormal scales).
    Only the K / V sources and Q are shaped; they are then stored exactly as
    make_workload stores them.

    kind 'rising': each KV head's key sources drift towards the last query
        token's first query head of its group, K_j = N(0,1) + 3 (j+1)/L q,
        so that head's logits grow along the sequence (to about 48) and the
        others' spread grows with it.
    kind 'late':   N(0,1) keys except two dominant ones, 2 q at 0.8 L and
        1.5 q at 0.55 L (q as above), far past the first tiles; the pieces of
        a split sequence then carry maxima tens of units apart.
    kind 'bigq':   N(0,1) K/V and Q = 16 N(0,1) rounded to binary16 values
        (so Q itself carries no rounding): logits of standard deviation 16.
    kind 'scales': N(0,1) K/V sources whose 32-value blocks are, at random,
        zero (scale 0), multiplied by 2^-14 (binary16 scales and values in the
        subnormal range) or left as they are; Q as in 'rising'.
    """
    assert kind in STRESS_KINDS, kind
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    table, n_blocks = _table_for(rng, lengths, ps, layout)
    q = rng.standard_normal((len(lengths), n_qtok, HQ, D), dtype=np.float32)
    if kind == "bigq":
        q = (q * np.float32(16.0)).astype(np.float16).astype(np.float32)
    ks, vs = [], []
    for s, L in enumerate(lengths.tolist()):
        qhat = q[s, n_qtok - 1, ::GQA, :]  # [HKV][D]: the first query head of each group
        for a in range(0, L, _GEN_CHUNK):
            b = min(L, a + _GEN_CHUNK)
            xk = rng.standard_normal((b - a, HKV, D), dtype=np.float32)
            xv = rng.standard_normal((b - a, HKV, D), dtype=np.float32)
            if kind == "rising":
                ramp = (np.arange(a, b, dtype=np.float32) + 1) * np.float32(3.0 / L)
                xk += ramp[:, None, None] * qhat[None]
            elif kind == "late":
                for pos, c in ((int(0.8 * L), 2.0), (int(0.55 * L), 1.5)):
                    if a <= pos < b and L > 64:
                        xk[pos - a] = np.float32(c) * qhat
            elif kind == "scales":
                for x in (xk, xv):
                    cat = rng.integers(0, 5, size=(b - a, HKV, D // 32))
                    f = np.where(cat == 0, np.float32(0.0), np.where(cat == 1, np.float32(2.0 ** -14), np.float32(1.0)))
                    x *= np.repeat(f, 32, axis=2).astype(np.float32)
            ks.append(encode_rows(xk, k_type))
            vs.append(encode_rows(xv, v_type))
    k_rows = np.concatenate(ks) if ks else np.zeros((0, HKV, row_bytes(k_type)), np.uint8)
    v_rows = np.concatenate(vs) if vs else np.zeros((0, HKV, row_bytes(v_type)), np.uint8)
    return Workload(f"stress-{kind}", lengths, n_qtok, ps, n_blocks, k_type, v_type, table, k_rows, v_rows, q,
                    SCALE, {"seed": seed, "layout": layout, "stress": kind})


def small_workload(seed: int, lengths, ps: int, k_type: int, v_type: int | None = None,
                   n_qtok: int = 1, layout: str = "shuffled") -> Workload:
    """Oracle-sized variants for parity tests (same recipe, smaller lengths)."""
    return make_workload(f"small-{seed}", seed, lengths, ps, k_type,
                         k_type if v_type is None else v_type, n_qtok, layout)

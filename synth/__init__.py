"""Seeded synthetic inputs for row-indexed attention over a unified KV pool.

This module is shared by the oracle's tests, the CUDA-path tests and the
benchmark.  It only draws random numbers and lays out index lists; it holds
none of the attention, quantisation or page-expansion arithmetic.  Every
floating-point tensor is returned as raw 16-bit patterns (``uint16``) so that
each side widens them with its own code.

Workloads follow the shapes of the pages' benchmark ("llama.cpp 0.9.0
inference boundaries", section 1: 4 sequences x 99,936 prompt tokens, context
400,000, batch = ubatch = 2,048) and the v100llm article (sections 1-2:
64-token paged KV in INT8, anchor + recent + sink sparse prefill).  Values are
N(0,1) drawn as float32 and rounded to nearest-even into the storage dtype.

Randomness: numpy's Philox counter-based bit generator keyed by the seed, so
the same seed gives the same bytes on any host.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

SEED_BASE = 0x5EED0000

# ---------------------------------------------------------------------------
# raw sampling


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=int(seed)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to IEEE half (nearest, ties to even); returns uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


PARALLEL_CHUNK = 1 << 24


def normal_bits(g: np.random.Generator, shape, dtype: str, chunk: int = 1 << 26) -> np.ndarray:
    """N(0,1) float32 samples rounded into ``dtype`` ('bf16' or 'f16'), as uint16 bits.

    Small tensors are drawn from ``g`` directly.  Tensors of at least
    ``chunk`` elements are drawn in blocks of PARALLEL_CHUNK elements: one
    64-bit key is taken from ``g`` and block i comes from Philox(key) jumped
    i + 1 times (independent streams), so the bytes depend on the seed alone
    while the blocks are generated on a thread pool and no float32 copy of the
    whole tensor is ever held.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    conv = f32_to_bf16_bits if dtype == "bf16" else f32_to_f16_bits
    if n < chunk:
        out[:] = conv(g.standard_normal(n, dtype=np.float32))
        return out.reshape(shape)
    key = int(g.integers(0, 1 << 63))
    base = np.random.Philox(key=key)
    blocks = range(0, n, PARALLEL_CHUNK)

    def fill(i):
        m = min(PARALLEL_CHUNK, n - i)
        gi = np.random.Generator(base.jumped(i // PARALLEL_CHUNK + 1))
        out[i:i + m] = conv(gi.standard_normal(m, dtype=np.float32))

    import concurrent.futures as cf
    import os
    with cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1))) as ex:
        list(ex.map(fill, blocks))
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# one attention problem


@dataclasses.dataclass
class Problem:
    """One row-indexed attention problem, all arrays on the host.

    q      uint16 bits [S, Nq, Hq, D]
    k, v   uint16 bits [R, Hkv, D]  (the unified pool; for the INT8 workload
           these are the bf16 values that each side quantises itself)
    kv_rows int32 [S, L]; negative = padding
    """
    name: str
    dtype: str                   # 'bf16' or 'f16' (Q, and K/V before quantisation)
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    kv_rows: Optional[np.ndarray]            # None for the paged workload (expanded by each side)
    scale: float
    causal: bool = False
    kv_len: Optional[np.ndarray] = None        # int32 [S] or None
    mask: Optional[np.ndarray] = None          # float32 [S, Nq, L] or None
    kv_int8: bool = False                      # K/V to be stored as int8 + fp16 scales
    page_table: Optional[np.ndarray] = None    # int32 [S, max_pages] (paged workload)
    seq_len: Optional[np.ndarray] = None       # int32 [S] (paged workload)
    page_size: int = 64
    list_len: int = 0                          # padded list length when kv_rows is None

    @property
    def S(self): return self.q.shape[0]
    @property
    def Nq(self): return self.q.shape[1]
    @property
    def Hq(self): return self.q.shape[2]
    @property
    def D(self): return self.q.shape[3]
    @property
    def R(self): return self.k.shape[0]
    @property
    def Hkv(self): return self.k.shape[1]
    @property
    def L(self): return self.kv_rows.shape[1] if self.kv_rows is not None else self.list_len

    def n_valid(self) -> int:
        """Number of listed (non-negative) entries, counting only positions < kv_len."""
        if self.kv_rows is None:
            return int(self.seq_len.sum())
        r = self.kv_rows
        if self.kv_len is not None:
            pos = np.arange(self.L)[None, :]
            return int(((r >= 0) & (pos < self.kv_len[:, None])).sum())
        return int((r >= 0).sum())


# ---------------------------------------------------------------------------
# the five workloads


def decode_fp16_small(seed: int = SEED_BASE + 1) -> Problem:
    """Decode, fp16: 4096-row pool, 8 q / 2 KV heads, D 128; 2 sequences of 1000
    rows at random pool positions, list in random order, padded with -1 to 1024."""
    g = rng(seed)
    R, Hq, Hkv, D, S, n, L = 4096, 8, 2, 128, 2, 1000, 1024
    perm = g.permutation(R)[: S * n].astype(np.int32)
    rows = np.full((S, L), -1, dtype=np.int32)
    for s in range(S):
        rows[s, :n] = perm[s * n:(s + 1) * n]
    q = normal_bits(g, (S, 1, Hq, D), "f16")
    k = normal_bits(g, (R, Hkv, D), "f16")
    v = normal_bits(g, (R, Hkv, D), "f16")
    return Problem("decode-f16 2x1000 of 4096, GQA 8/2, D128", "f16", q, k, v, rows, 1.0 / math.sqrt(D))


def decode_bf16_large(seed: int = SEED_BASE + 2, seq_rows: int = 16384, n_seq: int = 4) -> Problem:
    """Decode, bf16: n_seq x seq_rows rows filling a shuffled unified pool,
    32 q / 8 KV heads, D 128, one query token each, lists sorted ascending."""
    g = rng(seed)
    Hq, Hkv, D = 32, 8, 128
    R = n_seq * seq_rows
    perm = g.permutation(R).astype(np.int32)
    rows = np.sort(perm.reshape(n_seq, seq_rows), axis=1).astype(np.int32)
    q = normal_bits(g, (n_seq, 1, Hq, D), "bf16")
    k = normal_bits(g, (R, Hkv, D), "bf16")
    v = normal_bits(g, (R, Hkv, D), "bf16")
    return Problem(f"decode-bf16 {n_seq}x{seq_rows} shuffled pool, GQA 32/8, D128", "bf16", q, k, v, rows,
                   1.0 / math.sqrt(D))


def prefill_runs_layout(n_seq: int, seq_rows: int, run: int) -> np.ndarray:
    """Pool rows of each sequence when ubatches of ``run`` tokens are written
    round-robin across sequences; the partial last runs are packed at the end.

    Returns int32 [n_seq, seq_rows] of pool rows in position order.
    """
    full = seq_rows // run
    tail = seq_rows - full * run
    rows = np.empty((n_seq, seq_rows), dtype=np.int64)
    for s in range(n_seq):
        for r in range(full):
            base = (r * n_seq + s) * run
            rows[s, r * run:(r + 1) * run] = np.arange(base, base + run)
        if tail:
            base = full * n_seq * run + s * tail
            rows[s, full * run:] = np.arange(base, base + tail)
    return rows.astype(np.int32)


def prefill_bf16(seed: int = SEED_BASE + 3, n_seq: int = 4, seq_rows: int = 99936, pool_rows: int = 400000,
                 n_query: int = 2048, run: int = 2048, Hq: int = 32, Hkv: int = 8, D: int = 128,
                 shuffled: bool = False, dtype: str = "bf16") -> Problem:
    """Prefill chunk (bf16 unless ``dtype`` says f16): n_seq sequences of
    seq_rows prompt tokens in a pool_rows unified pool; one ubatch of n_query
    query rows per sequence at the prompt's end, causal within each sequence's
    rows (bottom-right aligned).

    The pool is written in ``run``-row ubatch runs, round-robin across
    sequences; with ``shuffled`` every row is placed at a random pool slot.
    """
    assert n_seq * seq_rows <= pool_rows
    g = rng(seed)
    if shuffled:
        perm = g.permutation(pool_rows)[: n_seq * seq_rows].astype(np.int32)
        rows = perm.reshape(n_seq, seq_rows)
    else:
        rows = prefill_runs_layout(n_seq, seq_rows, run)
    q = normal_bits(g, (n_seq, n_query, Hq, D), dtype)
    k = normal_bits(g, (pool_rows, Hkv, D), dtype)
    v = normal_bits(g, (pool_rows, Hkv, D), dtype)
    layout = "shuffled" if shuffled else f"{run}-row runs"
    return Problem(f"prefill-{dtype} {n_seq}x{seq_rows} in {pool_rows} ({layout}), {n_query} q rows, "
                   f"GQA {Hq}/{Hkv}, D{D}", dtype, q, k, v, rows, 1.0 / math.sqrt(D), causal=True)


def relabel_rows(p: Problem, seed: int, name: str) -> Problem:
    """The same problem with every listed row moved to a random pool slot: a
    seeded permutation of the pool applied to ``kv_rows`` (padding stays -1).
    The pool bytes are shared, so a fully shuffled variant of a large pool
    costs no second draw."""
    perm = rng(seed).permutation(p.R).astype(np.int32)
    rows = np.where(p.kv_rows >= 0, perm[np.maximum(p.kv_rows, 0)], p.kv_rows).astype(np.int32)
    return dataclasses.replace(p, kv_rows=rows, name=name)


def paged_int8(seed: int = SEED_BASE + 4, n_seq: int = 32, lo: int = 1024, hi: int = 131072,
               page: int = 64, Hq: int = 32, Hkv: int = 8, D: int = 128) -> Problem:
    """Paged decode with INT8 KV: sequence lengths log-uniform in [lo, hi],
    64-token pages whose ids are a random permutation over the whole pool.

    K/V are drawn as bf16 N(0,1); the INT8 pool is made by each side's own
    quantiser, and each side expands the page table into ``kv_rows`` itself
    (``kv_rows`` is None here; the padded list length is max_pages * page).
    """
    g = rng(seed)
    lens = np.floor(np.exp(g.uniform(math.log(lo), math.log(hi), size=n_seq))).astype(np.int64)
    lens = np.clip(lens, 1, hi).astype(np.int32)
    pages = (lens + page - 1) // page
    total_pages = int(pages.sum())
    perm = g.permutation(total_pages).astype(np.int32)
    max_pages = int(pages.max())
    pt = np.full((n_seq, max_pages), -1, dtype=np.int32)
    off = 0
    for s in range(n_seq):
        pt[s, :pages[s]] = perm[off:off + pages[s]]
        off += int(pages[s])
    R = total_pages * page
    L = max_pages * page
    q = normal_bits(g, (n_seq, 1, Hq, D), "bf16")
    k = normal_bits(g, (R, Hkv, D), "bf16")
    v = normal_bits(g, (R, Hkv, D), "bf16")
    return Problem(f"paged-int8 {n_seq} seqs len log-U[{lo},{hi}], 64-token pages, GQA {Hq}/{Hkv}, D{D}", "bf16",
                   q, k, v, None, 1.0 / math.sqrt(D), kv_int8=True, page_table=pt, seq_len=lens,
                   page_size=page, list_len=L)


def sparse_bf16(seed: int = SEED_BASE + 5, R: int = 262144, sinks: int = 4, recent: int = 512,
                selected: int = 1532, Hq: int = 16, Hkv: int = 2, D: int = 256) -> Problem:
    """Sparse long-context decode, bf16: 1 sequence whose pool row = position;
    list = sink rows + most recent rows + distinct uniform draws in between, sorted."""
    g = rng(seed)
    lo, hi = sinks, R - recent
    chosen = g.choice(hi - lo, size=selected, replace=False) + lo
    rows = np.concatenate([np.arange(sinks), np.sort(chosen), np.arange(hi, R)]).astype(np.int32)[None, :]
    q = normal_bits(g, (1, 1, Hq, D), "bf16")
    k = normal_bits(g, (R, Hkv, D), "bf16")
    v = normal_bits(g, (R, Hkv, D), "bf16")
    return Problem(f"sparse-bf16 {sinks}+{selected}+{recent} of {R}, GQA {Hq}/{Hkv}, D{D}", "bf16", q, k, v, rows,
                   1.0 / math.sqrt(D))


WORKLOADS = {
    "decode_f16_small": decode_fp16_small,
    "decode_bf16": decode_bf16_large,
    "prefill_bf16": prefill_bf16,
    "paged_int8": paged_int8,
    "sparse_bf16": sparse_bf16,
}


# ---------------------------------------------------------------------------
# small random problems for parity sweeps


def random_problem(seed: int, *, S=2, Nq=1, Hq=4, Hkv=2, D=128, R=300, L=77, dtype="bf16",
                   pad_frac=0.1, distinct=True, causal=False, with_mask=False, kv_len=False,
                   int8=False, neg_inf_frac=0.0) -> Problem:
    """A small problem with ragged lists, interior padding and optional extras."""
    g = rng(seed)
    if distinct:
        rows = np.stack([g.permutation(R)[:L] for _ in range(S)]).astype(np.int32)
    else:
        rows = g.integers(0, R, size=(S, L)).astype(np.int32)
    if pad_frac > 0:
        pad = g.random((S, L)) < pad_frac
        rows[pad] = -1 - g.integers(0, 3, size=int(pad.sum()))  # any negative value is padding
    q = normal_bits(g, (S, Nq, Hq, D), dtype)
    k = normal_bits(g, (R, Hkv, D), dtype)
    v = normal_bits(g, (R, Hkv, D), dtype)
    mask = None
    if with_mask:
        mask = g.standard_normal((S, Nq, L), dtype=np.float32)
        if neg_inf_frac > 0:
            mask[g.random((S, Nq, L)) < neg_inf_frac] = -np.inf
    kl = None
    if kv_len:
        kl = g.integers(0, L + 1, size=S).astype(np.int32)
    return Problem(f"random seed={seed}", dtype, q, k, v, rows, 1.0 / math.sqrt(D), causal=causal, kv_len=kl,
                   mask=mask, kv_int8=int8)

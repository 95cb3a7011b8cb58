"""Seeded synthetic inputs for one block-diffusion denoising round.

This module is shared by the tests, the benchmark and the oracle's callers.  It only
draws random numbers and lays them out; it holds none of the round's arithmetic
(no attention, no projection, no softmax, no commit rule).

Shapes follow the SDAR model family (SDAR page, "Available Models"; SDAR-4B: 32 query
heads, 8 KV heads, head dim 128, hidden 2560; SDAR-8B: hidden 4096; vocabulary 151936)
served by JetEngine at batch 128 with block length 4 (SDAR page, "High-performance batch
inference with JetEngine"; JetEngine README, "Quick start").  Values are drawn as float32
from numpy's PCG64 generator and rounded once, round-to-nearest-even, to bfloat16 bits.

Every array that stands for bf16 data is a ``numpy.uint16`` array of raw bf16 bits.
"""
from __future__ import annotations

import dataclasses
import math
import os
from typing import Optional

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
VOCAB = 151936
PAGE = 16


# --------------------------------------------------------------------------- bf16 bits
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); NaN -> 0x7FC0."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.reshape(-1)
    flat_out = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_in.size, step):
        u = flat_in[s:s + step].view(np.uint32)
        r = (u + (((u >> 16) & 1) + np.uint32(0x7FFF))) >> 16
        r = r.astype(np.uint16)
        r[np.isnan(flat_in[s:s + step])] = BF16_NAN
        flat_out[s:s + step] = r
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """N(0, std^2) drawn in float32, rounded once to bf16 bits.

    One 63-bit seed is drawn from ``rng``; chunk k of 2^22 values then comes from its own
    PCG64 stream seeded with (seed, k), so large arrays are drawn by several threads and
    the result depends only on ``rng``'s state, never on the thread count."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    seed = int(rng.integers(0, 2**63 - 1))
    step = 1 << 22

    def chunk(k):
        s = k * step
        m = min(step, n - s)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, k])))
        v = g.standard_normal(m, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        u = v.view(np.uint32)
        u += (u >> 16) & 1
        u += np.uint32(0x7FFF)
        out[s:s + m] = (u >> 16).astype(np.uint16)

    nchunks = (n + step - 1) // step
    if nchunks <= 1:
        for k in range(nchunks):
            chunk(k)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(chunk, range(nchunks)))
    return out.reshape(shape)


# --------------------------------------------------------------------------- attention
@dataclasses.dataclass
class AttnInputs:
    """Inputs of block attention over a paged KV cache.

    ``k_ref``/``v_ref`` hold only the pages the batch references, in page-table order
    (sequence 0's pages first).  ``page_table`` holds pool page ids (a shuffled pool of
    ``pool_pages`` pages; unused entries -1); ``page_table_ref`` holds the same entries
    as indices into ``k_ref``.  ``ref_page_ids[j]`` is the pool page holding ``k_ref[j]``.
    Slots of the last page past ``prefix_len + L`` hold bf16 NaN when ``poison`` is set.
    """
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    P: int
    pool_pages: int
    max_pages: int
    q: np.ndarray            # [B, L, Hq, D] bf16 bits
    k_ref: np.ndarray        # [n_ref, P, Hkv, D] bf16 bits
    v_ref: np.ndarray        # [n_ref, P, Hkv, D] bf16 bits
    page_table: np.ndarray   # [B, max_pages] int32, pool ids
    page_table_ref: np.ndarray  # [B, max_pages] int32, indices into k_ref
    ref_page_ids: np.ndarray    # [n_ref] int32
    prefix_lens: np.ndarray  # [B] int32

    @property
    def kv_lens(self) -> np.ndarray:
        return self.prefix_lens.astype(np.int64) + self.L


def make_attention(rng: np.random.Generator, B: int, L: int, Hq: int, Hkv: int, D: int,
                   prefix_range=(0, 0), P: int = PAGE, pool_pages: Optional[int] = None,
                   pool_factor: float = 1.25, identity_pages: bool = False,
                   prefix_lens: Optional[np.ndarray] = None, poison: bool = True,
                   qkv_std: float = 0.5) -> AttnInputs:
    if prefix_lens is None:
        lo, hi = prefix_range
        prefix_lens = rng.integers(lo, hi + 1, size=B, dtype=np.int64)
    prefix_lens = np.asarray(prefix_lens, dtype=np.int32)
    kv = prefix_lens.astype(np.int64) + L
    pages_per_seq = (kv + P - 1) // P
    n_ref = int(pages_per_seq.sum())
    max_pages = int(pages_per_seq.max()) if B else 0
    if pool_pages is None:
        pool_pages = n_ref if identity_pages else int(math.ceil(n_ref * pool_factor))
    if pool_pages < n_ref:
        raise ValueError("pool too small")
    if identity_pages:
        perm = np.arange(pool_pages, dtype=np.int64)
    else:
        perm = rng.permutation(pool_pages)
    page_table = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
    page_table_ref = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
    ref_ids = perm[:n_ref].astype(np.int32)
    c = 0
    for b in range(B):
        n = int(pages_per_seq[b])
        page_table[b, :n] = ref_ids[c:c + n]
        page_table_ref[b, :n] = np.arange(c, c + n, dtype=np.int32)
        c += n
    q = _normal_bf16(rng, (B, L, Hq, D), qkv_std)
    k_ref = _normal_bf16(rng, (n_ref, P, Hkv, D), qkv_std)
    v_ref = _normal_bf16(rng, (n_ref, P, Hkv, D), qkv_std)
    if poison:
        c = 0
        for b in range(B):
            n = int(pages_per_seq[b])
            used = int(kv[b] - (n - 1) * P)
            if used < P:
                k_ref[c + n - 1, used:] = BF16_NAN
                v_ref[c + n - 1, used:] = BF16_NAN
            c += n
    return AttnInputs(B, L, Hq, Hkv, D, P, pool_pages, max(max_pages, 1), q, k_ref, v_ref,
                      page_table, page_table_ref, ref_ids, prefix_lens)


# --------------------------------------------------------------------------- logits/mask
def make_mask_fixed_fraction(rng: np.random.Generator, B: int, L: int, frac) -> np.ndarray:
    """Per block exactly max(1, round(f*L)) masked positions, chosen without replacement.

    ``frac`` is a scalar or a per-block array; a block whose fraction is 0 gets no masked
    position (a SAVING block)."""
    mask = np.zeros((B, L), dtype=np.uint8)
    fr = np.broadcast_to(np.asarray(frac, dtype=np.float64), (B,))
    for b in range(B):
        if fr[b] <= 0:
            continue
        n = max(1, int(round(fr[b] * L)))
        mask[b, rng.choice(L, size=min(n, L), replace=False)] = 1
    return mask


def make_logits(rng: np.random.Generator, rows: int, V: int, std: float = 2.0,
                peak_rows=None, peak_height=None, peak_index: str = "uniform",
                zipf_a: float = 1.1) -> np.ndarray:
    """Background N(0, std^2) logits plus one planted peak per selected row.

    ``peak_height``: a number (fixed height) or a (lo, hi) pair (uniform height).
    ``peak_index``: "uniform" over the vocabulary or "zipf" (Zipf(a) rank k <= V drawn by
    rejection, token k - 1).  The peak is added to the background value at that token."""
    x = np.empty((rows, V), dtype=np.float32)
    for r0 in range(0, rows, 64):
        r1 = min(rows, r0 + 64)
        x[r0:r1] = rng.standard_normal((r1 - r0, V), dtype=np.float32) * np.float32(std)
    if peak_height is not None:
        sel = range(rows) if peak_rows is None else peak_rows
        for r in sel:
            if peak_index == "zipf":
                while True:
                    k = int(rng.zipf(zipf_a))
                    if k <= V:
                        break
                t = k - 1
            else:
                t = int(rng.integers(0, V))
            if isinstance(peak_height, tuple):
                h = float(rng.uniform(peak_height[0], peak_height[1]))
            else:
                h = float(peak_height)
            x[r, t] += np.float32(h)
    return f32_to_bf16_bits(x)


def poison_unmasked_rows(logits: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """Logits rows of positions that are not masked are never read: fill them with NaN."""
    out = logits.copy()
    out[mask.reshape(-1) == 0] = BF16_NAN
    return out


# --------------------------------------------------------------------------- configs
# The five workloads: shapes, distributions and seeds.  Seed = 1000 + config number.
CONFIGS = {
    1: dict(name="B1-L4-prefix60-Hq16", B=1, L=4, Hq=16, Hkv=8, D=128, prefix=(60, 60),
            identity_pages=True, V=VOCAB, threshold=0.9, temperature=1.0),
    2: dict(name="B128-L4-SDAR4B-shape", B=128, L=4, Hq=32, Hkv=8, D=128, prefix=(512, 4096),
            pool_pages=140_000, V=VOCAB, threshold=0.75, temperature=1.0),
    3: dict(name="B64-L16/32-SDAR4B-lmhead", B=64, L=16, Hq=32, Hkv=8, D=128,
            prefix=(1024, 8192), V=VOCAB, H=2560, threshold=0.9, temperature=1.0),
    4: dict(name="B16-L64-long-prefix", B=16, L=64, Hq=32, Hkv=8, D=128, prefix=(8192, 16384),
            V=VOCAB, threshold=0.75, temperature=1.0),
    5: dict(name="B128-L4-4step-chain-SDAR8B", B=128, L=4, Hq=32, Hkv=8, D=128,
            prefix=(256, 4096), V=VOCAB, H=4096, steps=4, threshold=0.75, temperature=1.0),
}


def seed_for(config: int, extra: int = 0) -> int:
    return 1000 + int(config) + 7919 * int(extra)


@dataclasses.dataclass
class CommitInputs:
    B: int
    L: int
    V: int
    logits: np.ndarray   # [B*L, V] bf16 bits (unmasked rows NaN when poisoned)
    mask: np.ndarray     # [B, L] uint8
    threshold: float
    temperature: float


def commit_inputs(config: int, rng: np.random.Generator, B: int, L: int, V: int,
                  peak_height=None, mask_frac=None, poison: bool = True,
                  supplementary: bool = False) -> CommitInputs:
    c = CONFIGS[config]
    rows = B * L
    if config == 1:
        mask = np.zeros((B, L), dtype=np.uint8)
        mask[:, [1, 3]] = 1
        peak_rows = [r for r in range(rows) if r % L in (0, 1, 2)]
        logits = make_logits(rng, rows, V, peak_rows=peak_rows,
                             peak_height=(8.0, 24.0) if supplementary else 8.0)
    elif config == 4:
        mask = make_mask_fixed_fraction(rng, B, L, rng.uniform(0.1, 0.9, size=B)
                                        if mask_frac is None else mask_frac)
        logits = make_logits(rng, rows, V, peak_height=(8.0, 24.0) if supplementary
                             else (0.0, 10.0), peak_index="zipf")
    else:
        mask = make_mask_fixed_fraction(rng, B, L, 0.5 if mask_frac is None else mask_frac)
        logits = make_logits(rng, rows, V, peak_height=(8.0, 24.0) if supplementary
                             else (peak_height or (0.0, 10.0)))
    if poison:
        logits = poison_unmasked_rows(logits, mask)
    return CommitInputs(B, L, V, logits, mask, c["threshold"], c["temperature"])


@dataclasses.dataclass
class LmHeadInputs:
    n_rows: int
    H: int
    V: int
    hidden: np.ndarray       # [n_rows, H] bf16 bits
    w: np.ndarray            # [V, H] bf16 bits
    active_idx: np.ndarray   # [n_act] int32, ascending


def lm_head_inputs(rng: np.random.Generator, n_rows: int, H: int, V: int,
                   active_idx: np.ndarray, w: Optional[np.ndarray] = None) -> LmHeadInputs:
    hidden = _normal_bf16(rng, (n_rows, H), 1.0)
    if w is None:
        w = _normal_bf16(rng, (V, H), 0.02)
    return LmHeadInputs(n_rows, H, V, hidden, w, np.ascontiguousarray(active_idx, dtype=np.int32))


def denoising_sequences(rng: np.random.Generator, B: int, frac: float = 0.75) -> np.ndarray:
    """A random ``frac`` of the sequences are DENOISING (1), the rest SAVING (0)."""
    n = int(round(frac * B))
    d = np.zeros(B, dtype=np.uint8)
    d[rng.choice(B, size=n, replace=False)] = 1
    return d


def rows_of_sequences(seq_flags: np.ndarray, L: int) -> np.ndarray:
    """Row ids b*L+i of every position of the flagged sequences, ascending."""
    seqs = np.nonzero(seq_flags)[0]
    return (seqs[:, None] * L + np.arange(L)[None, :]).reshape(-1).astype(np.int32)

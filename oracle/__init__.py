"""fp64 CPU oracle of one block-diffusion denoising round.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()`` and by
the CPU-baseline leg of ``bench.py``.  The CUDA library never imports, links or calls it,
and it shares no code with the CUDA library.

``bdlm_oracle.cpp`` holds the definitions (plain loops in fp64); this module compiles it
with g++ and wraps it with ctypes.  ``brute.py`` holds independent NumPy formulations used
only to pin the oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bdlm_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (g++, OpenMP, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_block_attention.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P,
                                                   ctypes.c_double, P, I, P]
            lib.oracle_block_attention.restype = I
            lib.oracle_attention_probs.argtypes = [I, I, I, I, I, I, I, P, P, P, P,
                                                   ctypes.c_double, I, I, I, P]
            lib.oracle_attention_probs.restype = I
            lib.oracle_lm_head.argtypes = [I, I, I, P, P, P, I, P, I, P]
            lib.oracle_lm_head.restype = I
            lib.oracle_confidence_commit.argtypes = [I, I, I, P, P, ctypes.c_double,
                                                     ctypes.c_double, P, I, P, P, P, P, P]
            lib.oracle_confidence_commit.restype = I
            lib.oracle_confidence_commit_rule.argtypes = [I, I, I, P, P, I, I, ctypes.c_double,
                                                          ctypes.c_double, P, I, P, P, P, P, P,
                                                          P, P]
            lib.oracle_confidence_commit_rule.restype = I
            lib.oracle_apply_commit.argtypes = [I, P, P]
            lib.oracle_apply_commit.restype = None
            lib.oracle_num_threads.restype = I
            lib.oracle_set_num_threads.argtypes = [I]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """OpenMP threads for later oracle calls."""
    _load().oracle_set_num_threads(int(n))


def block_attention(q, k_pages, v_pages, page_table, prefix_lens, L, Hq, Hkv, D, P,
                    sm_scale=None, seqs=None) -> np.ndarray:
    """fp64 attention output [B, L, Hq, D]; rows of sequences not in ``seqs`` stay NaN."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
    v_pages = np.ascontiguousarray(v_pages, dtype=np.uint16)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    prefix_lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    B = prefix_lens.shape[0]
    max_pages = page_table.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    out = np.full((B, L, Hq, D), np.nan, dtype=np.float64)
    sl = None if seqs is None else np.ascontiguousarray(seqs, dtype=np.int32)
    rc = lib.oracle_block_attention(B, L, Hq, Hkv, D, P, max_pages, k_pages.shape[0], _ptr(q),
                                    _ptr(k_pages),
                                    _ptr(v_pages), _ptr(page_table), _ptr(prefix_lens),
                                    float(sm_scale), _ptr(sl), 0 if sl is None else len(sl),
                                    _ptr(out))
    if rc != 0:
        raise ValueError("oracle_block_attention: bad arguments")
    return out


def attention_probs(q, k_pages, page_table, prefix_lens, L, Hq, Hkv, D, P, b, i, h,
                    sm_scale=None) -> np.ndarray:
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pages = np.ascontiguousarray(k_pages, dtype=np.uint16)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    prefix_lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    out = np.zeros(int(prefix_lens[b]) + L, dtype=np.float64)
    rc = lib.oracle_attention_probs(L, Hq, Hkv, D, P, page_table.shape[1], k_pages.shape[0],
                                    _ptr(q), _ptr(k_pages), _ptr(page_table), _ptr(prefix_lens),
                                    float(sm_scale), b, i, h, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_attention_probs: bad arguments")
    return out


def lm_head(hidden, w, rows, cols=None) -> np.ndarray:
    """fp64 logits [len(rows), len(cols) or V] of the listed hidden rows."""
    lib = _load()
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    n_rows, H = hidden.shape
    V = w.shape[0]
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int32)
    nc = V if c is None else len(c)
    out = np.empty((len(rows), nc), dtype=np.float64)
    rc = lib.oracle_lm_head(n_rows, H, V, _ptr(hidden), _ptr(w), _ptr(rows), len(rows), _ptr(c),
                            0 if c is None else len(c), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_lm_head: bad arguments")
    return out


class CommitResult:
    def __init__(self, tok, conf, conf32, commit, near, ent, ent32):
        self.tok, self.conf, self.conf32, self.commit, self.near = tok, conf, conf32, commit, near
        self.ent, self.ent32 = ent, ent32


# Commit rules (JetEngine notes, "Remasking Strategies"): threshold = low_confidence_dynamic,
# top-k = low_confidence_static, sequential / anti-sequential = left-to-right / right-to-left,
# entropy-bounded = lowest entropies first within an entropy budget (eb_threshold).
RULE_THRESHOLD, RULE_TOPK, RULE_SEQUENTIAL, RULE_ANTI_SEQUENTIAL = 0, 1, 2, 3
RULE_ENTROPY_BOUNDED = 4


def confidence_commit(logits, mask, threshold, temperature, blocks=None, rule=RULE_THRESHOLD,
                      k=1) -> CommitResult:
    """Per-position argmax token, confidence and entropy (nats), and the per-block commit
    decision by `rule` (k positions per block for the top-k and sequential rules; `threshold`
    is the entropy budget of the entropy-bounded rule)."""
    lib = _load()
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    B, L = mask.shape
    logits = np.ascontiguousarray(logits, dtype=np.uint16).reshape(B * L, -1)
    V = logits.shape[1]
    tok = np.full((B, L), -1, dtype=np.int32)
    conf = np.full((B, L), -np.inf, dtype=np.float64)
    conf32 = np.full((B, L), -np.inf, dtype=np.float32)
    commit = np.zeros((B, L), dtype=np.uint8)
    near = np.zeros((B, L), dtype=np.uint8)
    ent = np.full((B, L), np.inf, dtype=np.float64)
    ent32 = np.full((B, L), np.inf, dtype=np.float32)
    bl = None if blocks is None else np.ascontiguousarray(blocks, dtype=np.int32)
    rc = lib.oracle_confidence_commit_rule(B, L, V, _ptr(logits), _ptr(mask), int(rule), int(k),
                                           float(threshold), float(temperature), _ptr(bl),
                                           0 if bl is None else len(bl), _ptr(tok), _ptr(conf),
                                           _ptr(conf32), _ptr(commit), _ptr(near), _ptr(ent),
                                           _ptr(ent32))
    if rc != 0:
        raise ValueError("oracle_confidence_commit: bad arguments")
    return CommitResult(tok, conf, conf32, commit, near, ent, ent32)


def apply_commit(mask, commit) -> np.ndarray:
    lib = _load()
    m = np.ascontiguousarray(mask, dtype=np.uint8).copy()
    c = np.ascontiguousarray(commit, dtype=np.uint8)
    lib.oracle_apply_commit(m.size, _ptr(m), _ptr(c))
    return m


def round_logits_to_bf16(x64: np.ndarray) -> np.ndarray:
    """Store fp64 logits as bf16 bits: one round-to-nearest-even (via exact float32 for
    values whose float32 rounding does not straddle a bf16 tie; ties are resolved on the
    fp64 value)."""
    x64 = np.asarray(x64, dtype=np.float64)
    # Exact RNE from fp64 to bf16: pick the two bf16 neighbours and compare distances.
    f = x64.astype(np.float32)  # nearest float32 (RNE)
    u = f.view(np.uint32).astype(np.uint64)
    lo = (u & 0xFFFF0000).astype(np.uint32)
    lo_f = lo.view(np.float32).astype(np.float64)
    hi = (lo.astype(np.uint64) + 0x10000).astype(np.uint32)
    hi_f = hi.view(np.float32).astype(np.float64)
    # for negative numbers "lo" (truncated magnitude) is the larger value; distances work
    # on magnitudes either way
    d_lo = np.abs(x64 - lo_f)
    d_hi = np.abs(x64 - hi_f)
    lo_even = ((lo >> 16) & 1) == 0
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ~lo_even)
    out = np.where(pick_hi, hi, lo) >> 16
    return out.astype(np.uint16)


def active_rows(mask, denoising=None) -> np.ndarray:
    """Rows b*L+i with mask[b, i] != 0 and (no flags or denoising[b] != 0), increasing: the
    rows a step's selective LM head computes (JetEngine notes, "ModelRunner")."""
    mask = np.asarray(mask)
    keep = mask != 0
    if denoising is not None:
        keep &= (np.asarray(denoising) != 0)[:, None]
    return np.nonzero(keep.reshape(-1))[0].astype(np.int32)


def write_block_kv(k_pages, v_pages, page_table, prefix_lens, k_new, v_new, P=16):
    """Copies of the K/V pools with k_new/v_new [B, L, Hkv, D] written to the slots
    prefix_lens[b] .. prefix_lens[b]+L-1 of sequence b (token j: page page_table[b][j // P],
    slot j % P)."""
    k = np.array(k_pages, copy=True)
    v = np.array(v_pages, copy=True)
    B, L = k_new.shape[:2]
    for b in range(B):
        for i in range(L):
            j = int(prefix_lens[b]) + i
            page = int(page_table[b][j // P])
            k[page, j % P] = k_new[b, i]
            v[page, j % P] = v_new[b, i]
    return k, v


def prefill_attention(q, k_new, v_new, k_pages, v_pages, page_table, prefix_lens, L, Hq, Hkv, D,
                      P=16, sm_scale=None):
    """Block prefill: the prompt's K/V written after each sequence's cached prefix, then every
    prompt block j attends to the cache up to the end of block j (prefix + (j+1)*L tokens).
    q [B, n, Hq, D], k_new/v_new [B, n, Hkv, D] with n a multiple of L.  Returns the fp64
    output [B, n, Hq, D] and the updated pools."""
    q = np.asarray(q)
    B, n = q.shape[:2]
    k, v = write_block_kv(k_pages, v_pages, page_table, prefix_lens, k_new, v_new, P)
    out = np.empty((B, n, Hq, D), dtype=np.float64)
    for j in range(n // L):
        pre = np.asarray(prefix_lens, dtype=np.int32) + j * L
        qj = np.ascontiguousarray(q[:, j * L:(j + 1) * L])
        out[:, j * L:(j + 1) * L] = block_attention(qj, k, v, page_table, pre, L, Hq, Hkv, D, P,
                                                    sm_scale=sm_scale)
    return out, k, v

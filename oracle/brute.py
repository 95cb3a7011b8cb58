"""Independent NumPy formulations used only to pin the oracle (test infrastructure).

These restate the round from a different angle than ``bdlm_oracle.cpp``: attention as a
dense masked matrix product over a whole multi-block sequence, the LM head as a BLAS
matrix product, confidence through ``scipy.special.softmax``.
"""
from __future__ import annotations

import numpy as np

from workloads import bf16_bits_to_f32


def dense_block_causal_attention(q_seq, k_seq, v_seq, block_len, Hq, Hkv, sm_scale=None):
    """Attention over a whole sequence of ``n`` tokens split into blocks of ``block_len``.

    q_seq [n, Hq, D], k_seq/v_seq [n, Hkv, D] (float arrays).  Token i may attend to token
    j when block(j) <= block(i) (block-causal: bidirectional inside a block, causal across
    blocks).  Returns [n, Hq, D] fp64."""
    q = np.asarray(q_seq, dtype=np.float64)
    k = np.asarray(k_seq, dtype=np.float64)
    v = np.asarray(v_seq, dtype=np.float64)
    n, _, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    blk = np.arange(n) // block_len
    allowed = blk[None, :] <= blk[:, None]            # [query, key]
    G = Hq // Hkv
    out = np.empty((n, Hq, D), dtype=np.float64)
    for h in range(Hq):
        s = (q[:, h, :] @ k[:, h // G, :].T) * sm_scale  # [n, n]
        s = np.where(allowed, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        e = np.exp(s)
        p = e / e.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, h // G, :]
    return out


def lm_head_matmul(hidden_bits, w_bits, rows):
    h = bf16_bits_to_f32(hidden_bits).astype(np.float64)[np.asarray(rows)]
    w = bf16_bits_to_f32(w_bits).astype(np.float64)
    return h @ w.T


def confidence_scipy(logits_f64, temperature):
    """(argmax token, max softmax probability) per row via scipy."""
    from scipy.special import softmax
    x = np.asarray(logits_f64, dtype=np.float64)
    p = softmax(x / temperature, axis=-1)
    return np.argmax(x, axis=-1), p.max(axis=-1)

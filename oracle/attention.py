"""Attention of verify rows over a KV cache (test infrastructure).

The TensorFold pages speak of the KV cache only through its guarantees: by
the README's note on drafting, a run with drafts and a run without them emit
the same tokens when they start from one cache; the 0.3.4.1 release note
("TensorFold: the contract is what it does not change", section "The
regression it published against itself") keeps prompt caches only at points
of a fixed grid, so that cached bits do not depend on where a conversation
resumed.  The pages do not write out the attention itself, so the oracle
takes the textbook definition of causal scaled dot-product attention with grouped key/value
heads (Vaswani et al. 2017, section 3.2.1; Ainslie et al. 2023 for the
grouping):

* head dimension D = 128; query head h reads key/value head h // group;
* verify row r sits at position p = pos0 + r and sees cache positions
  0 .. p (its own entry included);
* s_t = (q . k_t) / sqrt(D);  w_t = exp(s_t - max_t s_t);
  out = sum_t w_t v_t / sum_t w_t.

Everything is evaluated in fp64 from the bf16 inputs.  The cache arrays here
are in the plain layout ``[n_kv][L][D]``; the device's storage order is not
the oracle's concern.
"""

from __future__ import annotations

import math

import numpy as np

from .linear import bf16_to_f64

HEAD_DIM = 128


def attention_row(q_f64: np.ndarray, k_f64: np.ndarray, v_f64: np.ndarray, p: int) -> np.ndarray:
    """fp64 attention of one query vector over cache positions 0..p of one head.

    q_f64 [D]; k_f64, v_f64 [L][D] (fp64).  Returns [D].
    """
    D = q_f64.shape[0]
    scores = (k_f64[: p + 1] @ q_f64) / math.sqrt(D)
    w = np.exp(scores - scores.max())
    return (w @ v_f64[: p + 1]) / w.sum()


def attention_verify(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, pos0: int, group: int,
                     heads=None) -> np.ndarray:
    """fp64 outputs [R][n_q][D] of R verify rows at positions pos0 .. pos0 + R - 1.

    q_bits bf16 bits [R][n_q][D]; k_bits, v_bits bf16 bits [n_kv][L][D].
    ``heads``: optional list of (row, query head) pairs; only those outputs are
    computed (the rest stay NaN), for spot checks at full size.
    """
    q_bits = np.asarray(q_bits)
    R, n_q, D = q_bits.shape
    n_kv = k_bits.shape[0]
    if n_q != n_kv * group:
        raise ValueError("n_q must equal n_kv * group")
    out = np.full((R, n_q, D), np.nan)
    pairs = heads if heads is not None else [(r, h) for r in range(R) for h in range(n_q)]
    kv_cache = {}
    for r, h in pairs:
        j = h // group
        p = pos0 + r
        if j not in kv_cache:
            hi = pos0 + R
            kv_cache[j] = (bf16_to_f64(k_bits[j, :hi]), bf16_to_f64(v_bits[j, :hi]))
        k, v = kv_cache[j]
        out[r, h] = attention_row(bf16_to_f64(q_bits[r, h]), k, v, p)
    return out

"""Synthetic decoder with an attention sub-block per block (test infrastructure).

The attention-free decoder of ``decoder.py`` with, before each MLP block, an
attention sub-block over a KV cache.  The pages name the guarantee, not the
layer: by the README's note on drafting, a run with drafts and a run without
them emit the same tokens when they start from one cache.  Each block
computes, on fp64 rows x:

    n   = bf16(rms_norm(x))
    qkv = n Wqkv                       (queries n_q x 128, keys n_kv x 128, values n_kv x 128)
    q, k, v = bf16(qkv)                (round to nearest even)
    cache[pos_r] = (k_r, v_r)          for every row r of the pass, before any row reads
    o_r = attention(q_r, cache[0..pos_r])          (attention.attention_verify)
    x   = x + bf16(o) Wo
    x   = decoder.block_forward(x, mlp block)

then logits = fp32(bf16(rms_norm(x)) Wlm).  A pass of R rows at position p
(the next position to sample) feeds the last committed token and R - 1 drafts
at cache positions p - 1 .. p + R - 2 and samples positions p .. p + R - 1.
Entries written for rejected rows stay in the cache; the next pass starts at
the first of them and rewrites it before anything reads it.
"""

from __future__ import annotations

import numpy as np

from .linear import w4_linear, bf16_to_f64
from .numerics import bf16_round, bf16_bits_of, rms_norm
from . import attention, sampling, accept as acc
from .decoder import block_forward, final_input, EPS

D = attention.HEAD_DIM


def new_cache(model, max_len: int):
    """Per block: K and V bf16 bits [n_kv][max_len][128], zero."""
    n_kv = model["n_kv"]
    return [dict(k=np.zeros((n_kv, max_len, D), np.uint16), v=np.zeros((n_kv, max_len, D), np.uint16))
            for _ in model["blocks"]]


def pass_rows(model, cache, tokens, pos_first: int):
    """Rows tokens[i] at cache positions pos_first + i through every block;
    returns the final fp64 residual rows [R][H]."""
    G, n_kv, grp = model["group"], model["n_kv"], model["attn_group"]
    n_q = n_kv * grp
    toks = np.asarray(tokens, dtype=np.int64)
    R = len(toks)
    x = bf16_to_f64(model["emb"][toks])
    for blk, att, c in zip(model["blocks"], model["attn"], cache):
        n_bits = bf16_bits_of(bf16_round(rms_norm(x, EPS)))
        qkv = bf16_bits_of(bf16_round(w4_linear(att["qkv_codes"], att["qkv_scales"], n_bits, G)))
        q = qkv[:, : n_q * D].reshape(R, n_q, D)
        k = qkv[:, n_q * D: (n_q + n_kv) * D].reshape(R, n_kv, D)
        v = qkv[:, (n_q + n_kv) * D:].reshape(R, n_kv, D)
        c["k"][:, pos_first: pos_first + R] = k.transpose(1, 0, 2)
        c["v"][:, pos_first: pos_first + R] = v.transpose(1, 0, 2)
        o = attention.attention_verify(q, c["k"], c["v"], pos_first, grp).reshape(R, n_q * D)
        x = x + w4_linear(att["o_codes"], att["o_scales"], bf16_bits_of(bf16_round(o)), G)
        x = block_forward(x, blk, G)
    return x


def logits_of(model, x):
    return w4_linear(model["lm_codes"], model["lm_scales"], final_input(x), model["group"]).astype(np.float32)


def prefill(model, cache, prompt):
    """Cache entries of the prompt tokens at positions 0 .. len - 1 (one pass)."""
    pass_rows(model, cache, prompt, 0)


def serial_decode(model, cache, last: int, pos: int, n_tokens: int, temperature, top_k, top_p, seed):
    """One row per pass; ``last`` is the committed token at position pos - 1."""
    out = []
    for _ in range(n_tokens):
        l = logits_of(model, pass_rows(model, cache, [last], pos - 1))
        t, _ = sampling.sample_row(l[0], temperature, top_k, top_p, seed, pos)
        out.append(t)
        last, pos = t, pos + 1
    return out


def drafted_decode(model, cache, last: int, pos: int, n_tokens: int, R: int, temperature, top_k, top_p, seed,
                   draft_fn):
    """R rows per pass; ``draft_fn(pos0, n)`` gives drafts for positions pos0 ..
    pos0 + n - 1.  Returns (tokens, accepted lengths per pass)."""
    out, lens = [], []
    while len(out) < n_tokens:
        d = [int(t) for t in draft_fn(pos, R - 1)]
        l = logits_of(model, pass_rows(model, cache, [last] + d, pos - 1))
        t = [sampling.sample_row(l[i], temperature, top_k, top_p, seed, pos + i)[0] for i in range(R)]
        a, bonus = acc.accept(d, t)
        out.extend(t[: a + 1])
        lens.append(a)
        last, pos = bonus, pos + a + 1
    return out[:n_tokens], lens

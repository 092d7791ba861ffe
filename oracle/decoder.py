"""Attention-free synthetic decoder, serial and drafted (test infrastructure).

Stands in for the pages' 27B-class dense model (TensorFold README: decode
speed table for "Qwen3.8-27B + DFlash2"; 4-bit weights in groups of 64),
whose weights are not available.  It exists to exercise the verify pass end
to end: every W4 projection, the W4 LM head, keyed sampling and acceptance.
Its arithmetic is a plain restatement chosen for this purpose:

    x   = emb[token]                                  (bf16 -> fp64)
    per block:  n = bf16(rms_norm(x));  h = bf16(silu(n Wg) * (n Wu));  x = x + h Wd
    logits = fp32( bf16(rms_norm(x)) Wlm )

rms_norm has gain 1 and eps 1e-6.  No attention means a row's logits depend
only on its input token; the position enters only through the sampling key.

``serial_decode`` samples one token per step (the pages' ``"draft": false``
reference).  ``drafted_decode`` verifies R rows per step and accepts the
longest matching prefix (``accept.accept``).  The invariant the pages state
-- a drafted run emits exactly the serial run's tokens -- is checked by
comparing ``token_sha`` of the two.
"""

from __future__ import annotations

import hashlib
import numpy as np

from .linear import w4_linear, bf16_to_f64
from .numerics import bf16_round, bf16_bits_of, rms_norm, silu
from . import sampling, accept as acc

EPS = 1e-6


def block_forward(x, blk, group: int):
    """One residual SwiGLU block on fp64 rows x [R][H]; returns the new x."""
    n_bits = bf16_bits_of(bf16_round(rms_norm(x, EPS)))
    g = w4_linear(blk["gate_codes"], blk["gate_scales"], n_bits, group)
    u = w4_linear(blk["up_codes"], blk["up_scales"], n_bits, group)
    h_bits = bf16_bits_of(bf16_round(silu(g) * u))
    return x + w4_linear(blk["down_codes"], blk["down_scales"], h_bits, group)


def final_input(x):
    """bf16 bits of the LM head's input."""
    return bf16_bits_of(bf16_round(rms_norm(x, EPS)))


def logits(model, tokens):
    """fp32 logits [R][V] for input tokens [R]."""
    toks = np.asarray(tokens, dtype=np.int64)
    x = bf16_to_f64(model["emb"][toks])
    for blk in model["blocks"]:
        x = block_forward(x, blk, model["group"])
    y = w4_linear(model["lm_codes"], model["lm_scales"], final_input(x), model["group"])
    return y.astype(np.float32)


def token_sha(tokens) -> str:
    """SHA-256 of the committed token ids as little-endian int32 (prompt excluded)."""
    return hashlib.sha256(np.asarray(tokens, dtype="<i4").tobytes()).hexdigest()


def serial_decode(model, prompt_token: int, n_tokens: int, temperature, top_k, top_p, seed):
    """One token per step, positions 1..n_tokens (the prompt token sits at position 0)."""
    out = []
    last = int(prompt_token)
    for pos in range(1, n_tokens + 1):
        l = logits(model, [last])
        t, _ = sampling.sample_row(l[0], temperature, top_k, top_p, seed, pos)
        out.append(t)
        last = t
    return out


def drafted_decode(model, prompt_token: int, n_tokens: int, R: int, temperature, top_k, top_p,
                   seed, draft_fn):
    """Verify R rows per step.  ``draft_fn(pos0, n)`` returns n draft tokens for
    positions pos0 .. pos0+n-1.  Returns (tokens, accepted lengths per step)."""
    out, lens = [], []
    last = int(prompt_token)
    pos0 = 1
    while len(out) < n_tokens:
        d = [int(v) for v in draft_fn(pos0, R - 1)]
        rows = [last] + d
        l = logits(model, rows)
        t = [sampling.sample_row(l[i], temperature, top_k, top_p, seed, pos0 + i)[0] for i in range(R)]
        a, bonus = acc.accept(d, t)
        out.extend(t[: a + 1])
        lens.append(a)
        last = bonus
        pos0 += a + 1
    return out[:n_tokens], lens

"""Longest-prefix acceptance of drafts (test infrastructure).

TensorFold README, section on the two guarantees: a draft is kept only when
it matches the token one-row decoding samples at its position, which is why a
drafted run emits exactly the serial run's tokens.

Indexing (the pages give none; this reading is used everywhere): a verify
pass has R rows; row i samples position ``pos0 + i`` and yields ``t[i]``;
draft ``d[i]`` (i < R-1) proposes the token at position ``pos0 + i`` and is
also the input of row i+1.  ``a`` is the first i with ``d[i] != t[i]``, or
R-1 when every draft matches; the pass commits ``t[0..a]`` (a+1 tokens) and
``t[a]`` is the bonus token that feeds the next pass.
"""

from __future__ import annotations


def accept(drafts, sampled):
    """(a, bonus) for drafts d[R-1] and sampled t[R]."""
    t = [int(v) for v in sampled]
    d = [int(v) for v in drafts]
    R = len(t)
    if R < 1 or len(d) != R - 1:
        raise ValueError("need R >= 1 sampled tokens and R-1 drafts")
    a = R - 1
    for i in range(R - 1):
        if d[i] != t[i]:
            a = i
            break
    return a, t[a]


def committed(drafts, sampled):
    """Tokens committed by one verify pass: t[0..a]."""
    a, _ = accept(drafts, sampled)
    return [int(v) for v in sampled[: a + 1]]

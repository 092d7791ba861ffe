"""Keyed Gumbel-max sampling over the top-k / top-p candidates (test infrastructure).

Source: TensorFold README, section on the two guarantees (keyed sampling):
position p gets the top-k/top-p candidate that maximises
``logit / T + g(seed, p, token)``, where ``g`` is Gumbel noise computed from a
hash of seed, position and token id; the CLI options table makes temperature 0
plain greedy decoding.

Readings fixed here where the pages are silent:

* hash: SplitMix64 finaliser (Steele, Lea & Flood, OOPSLA 2014, constants
  0x9E3779B97F4A7C15, 0xBF58476D1CE4E5B9, 0x94D049BB133111EB), composed as
  ``h = sm(sm(sm(seed) ^ pos) ^ token)`` with ``pos`` taken as a 64-bit
  two's-complement word and ``token`` as a zero-extended 32-bit word;
* uniform: ``u = ((h >> 11) + 0.5) / 2^53`` evaluated in fp64: the sum
  rounds to nearest-even, so the one top value ``h >> 11 = 2^53 - 1`` gives
  u = 1 exactly and then g = +inf by IEEE rules (probability 2^-53);
* Gumbel: ``g = -ln(-ln u)`` in fp64;
* candidate set: tokens ordered by (logit desc, id asc); keep the first
  ``k' = V if top_k <= 0 or top_k >= V else top_k``; then, when
  ``top_p < 1``, the smallest prefix whose renormalised mass reaches
  ``top_p`` (the token that crosses it is kept), with
  ``q_i = exp((l_i - l_0) / T) / sum_{j<k'} exp((l_j - l_0) / T)``,
  sums taken left to right in rank order, in fp64;
* selection: argmax of ``(double)l / (double)T + g`` over the candidates,
  ties to the lower id; ``T == 0`` is argmax of the logits over all V,
  ties to the lower id.
"""

from __future__ import annotations

import math
import numpy as np

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB


def splitmix64(z: int) -> int:
    """One SplitMix64 output for state ``z`` (state advanced by the golden gamma first)."""
    z = (z + GOLDEN) & M64
    z = ((z ^ (z >> 30)) * MIX1) & M64
    z = ((z ^ (z >> 27)) * MIX2) & M64
    return z ^ (z >> 31)


def key_hash(seed: int, pos: int, token: int) -> int:
    """64-bit key of (seed, position, token id)."""
    s = splitmix64(int(seed) & M64)
    s = splitmix64(s ^ (int(pos) & M64))
    return splitmix64(s ^ (int(token) & 0xFFFFFFFF))


def uniform_of(h: int) -> float:
    return ((h >> 11) + 0.5) / 9007199254740992.0  # 2^53


def gumbel_of(h: int) -> float:
    u = uniform_of(h)
    inner = -math.log(u)
    if inner == 0.0:
        # u rounded to exactly 1.0: IEEE log(0) = -inf, so g = +inf
        # (Python's math.log raises there instead of returning -inf).
        return math.inf
    return -math.log(inner)


def gumbel(seed: int, pos: int, token: int) -> float:
    return gumbel_of(key_hash(seed, pos, token))


def rank_order(logits_row) -> np.ndarray:
    """Token ids ordered by (logit desc, id asc)."""
    l = np.asarray(logits_row, dtype=np.float32).astype(np.float64)
    if not np.all(np.isfinite(l)):
        raise ValueError("non-finite logit")
    ids = np.arange(l.size)
    return np.lexsort((ids, -l))


def candidate_set(logits_row, temperature: float, top_k: int, top_p: float):
    """Candidate ids in rank order for T > 0 (see module docstring)."""
    l32 = np.asarray(logits_row, dtype=np.float32)
    V = l32.size
    order = rank_order(l32)
    kk = V if (top_k <= 0 or top_k >= V) else int(top_k)
    order = order[:kk]
    if float(np.float32(top_p)) >= 1.0:
        return order
    T = float(np.float32(temperature))
    l0 = float(l32[order[0]])
    e = [math.exp((float(l32[i]) - l0) / T) for i in order]
    Z = 0.0
    for v in e:
        Z += v
    p = float(np.float32(top_p))
    S = 0.0
    for m, v in enumerate(e, start=1):
        S += v / Z
        if S >= p:
            return order[:m]
    return order  # rounding left the total just below p: keep all k'


def topp_margin(logits_row, temperature: float, top_k: int, top_p: float) -> float:
    """How close the top-p cut of ``candidate_set`` is to flipping: the smaller
    of |S_m - p| and |S_(m-1) - p| for the cut m (the running sums as
    ``candidate_set`` forms them), inf when no top-p cut applies."""
    l32 = np.asarray(logits_row, dtype=np.float32)
    if float(np.float32(top_p)) >= 1.0 or float(np.float32(temperature)) == 0.0:
        return math.inf
    V = l32.size
    order = rank_order(l32)
    kk = V if (top_k <= 0 or top_k >= V) else int(top_k)
    order = order[:kk]
    T = float(np.float32(temperature))
    l0 = float(l32[order[0]])
    e = [math.exp((float(l32[i]) - l0) / T) for i in order]
    Z = 0.0
    for v in e:
        Z += v
    p = float(np.float32(top_p))
    S_prev, S = 0.0, 0.0
    for v in e:
        S_prev, S = S, S + v / Z
        if S >= p:
            return min(abs(S - p), abs(S_prev - p))
    return abs(S - p)


def sample_row(logits_row, temperature: float, top_k: int, top_p: float, seed: int, pos: int):
    """(token, gap): the keyed sample and the margin between the best and runner-up score.

    ``gap`` is +inf when there is a single candidate.
    """
    l32 = np.asarray(logits_row, dtype=np.float32)
    T = float(np.float32(temperature))
    if T < 0 or math.isnan(T):
        raise ValueError("temperature must be >= 0")
    if T == 0.0:
        order = rank_order(l32)
        best = int(order[0])
        gap = float(l32[order[0]]) - float(l32[order[1]]) if l32.size > 1 else math.inf
        return best, gap
    cand = candidate_set(l32, T, top_k, top_p)
    best_id, best_s, second = -1, -math.inf, -math.inf
    for i in cand:  # rank order; ties keep the lower id explicitly
        s = float(l32[i]) / T + gumbel(seed, pos, int(i))
        if s > best_s or (s == best_s and int(i) < best_id):
            second = max(second, best_s)
            best_id, best_s = int(i), s
        else:
            second = max(second, s)
    return best_id, best_s - second


def sample(logits, temperature: float, top_k: int, top_p: float, seed: int, pos):
    """Tokens [R] and gaps [R] for logits [R][V] at positions pos[R]."""
    logits = np.asarray(logits, dtype=np.float32)
    toks, gaps = [], []
    for r in range(logits.shape[0]):
        t, g = sample_row(logits[r], temperature, top_k, top_p, seed, int(pos[r]))
        toks.append(t)
        gaps.append(g)
    return np.array(toks, dtype=np.int32), np.array(gaps, dtype=np.float64)

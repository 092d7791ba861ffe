"""Top-k routed W4 SwiGLU experts (test infrastructure).

TensorFold README, "What each checkpoint needs" / source layout: the MoE
model is served from 4-bit weights quantised in groups of 32.  The routing and
expert shapes are those of a 30B-A3B-class model (128 experts, top-8,
hidden 2048, expert FFN 768); the pages name the model class, not its
arithmetic, so these readings are used:

* ranking: experts ordered by (router logit desc, id asc).  softmax is
  strictly increasing in the logit, so this is the order of the routing
  probabilities, taken on the exact fp32 logits so rounding can't make ties;
* weights: the top-k probabilities renormalised to sum to 1, in fp64:
  ``w_j = exp(z_j - z_0) / sum_{i<k} exp(z_i - z_0)`` (left-to-right sum in
  rank order; the full softmax denominator cancels);
* expert: ``h = bf16(silu(x Wg) * (x Wu))``, ``y_e = h Wd``, all W4 layers
  evaluated by ``w4_linear`` (fp64), bf16 rounding of ``h`` in one step;
* combine: ``out = sum_{j=0..k-1} w_j * y_{e_j}`` in rank order, fp64.
"""

from __future__ import annotations

import math
import numpy as np

from .linear import w4_linear
from .numerics import bf16_round, bf16_bits_of, silu


def route(router_logits, top_k: int = 8):
    z = np.asarray(router_logits, dtype=np.float32)
    R, E = z.shape
    ids = np.empty((R, top_k), dtype=np.int64)
    w = np.empty((R, top_k), dtype=np.float64)
    for r in range(R):
        zr = z[r].astype(np.float64)
        if not np.all(np.isfinite(zr)):
            raise ValueError("non-finite router logit")
        order = np.lexsort((np.arange(E), -zr))[:top_k]
        ids[r] = order
        e = [math.exp(zr[i] - zr[order[0]]) for i in order]
        tot = 0.0
        for v in e:
            tot += v
        w[r] = [v / tot for v in e]
    return ids, w


def expert_forward(x_bits, W, e: int, group: int):
    """(h_bits [R][F], y [R][H]) of expert e for bf16 rows x_bits [R][H]."""
    g = w4_linear(W["gate_codes"][e], W["gate_scales"][e], x_bits, group)
    u = w4_linear(W["up_codes"][e], W["up_scales"][e], x_bits, group)
    h = bf16_round(silu(g) * u)
    h_bits = bf16_bits_of(h)
    y = w4_linear(W["down_codes"][e], W["down_scales"][e], h_bits, group)
    return h_bits, y


def moe(x_bits, router_logits, W, group: int = 32, top_k: int = 8):
    """(out [R][H] fp64, ids [R][k], w [R][k], y_sel [R][k][H] fp64)."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    ids, w = route(router_logits, top_k)
    R, H = x_bits.shape
    y_sel = np.zeros((R, top_k, H), dtype=np.float64)
    for e in np.unique(ids):
        rows = [r for r in range(R) if e in ids[r]]
        _, y = expert_forward(x_bits[rows], W, int(e), group)
        for i, r in enumerate(rows):
            j = int(np.nonzero(ids[r] == e)[0][0])
            y_sel[r, j] = y[i]
    out = np.zeros((R, H), dtype=np.float64)
    for j in range(top_k):
        out += w[:, j:j + 1] * y_sel[:, j, :]
    return out, ids, w, y_sel

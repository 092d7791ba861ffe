"""Host-side decode loop over ``tf_verify_step`` (serial and drafted).

The device does every step of a verify pass; the host only supplies draft
tokens and reads back, once per pass, the accepted length and the sampled
tokens (the pages' serial reference is ``R = 1``: one token a round).
"""

from __future__ import annotations

import hashlib

import numpy as np
import torch

from . import tf


def upload_model(weights: dict, rms_eps: float = 1e-6, device="cuda") -> tf.Model:
    """Pack numpy weights (canonical layout) into device matrices.

    ``weights``: emb (uint16 [V][H] bf16 bits), blocks: list of dicts with
    gate/up/down codes+scales, lm_codes, lm_scales, group.
    """
    G = weights["group"]

    def dev(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(device)

    emb = dev(weights["emb"], np.int16)
    V, H = weights["emb"].shape
    gu, dn = [], []
    F = None
    for blk in weights["blocks"]:
        F = blk["gate_codes"].shape[0]
        codes = np.concatenate([blk["gate_codes"], blk["up_codes"]], axis=0)
        scales = np.concatenate([blk["gate_scales"], blk["up_scales"]], axis=0)
        gu.append(tf.pack_w4(dev(codes, np.uint8), dev(scales, np.int16), G, gate_up=True))
        dn.append(tf.pack_w4(dev(blk["down_codes"], np.uint8), dev(blk["down_scales"], np.int16), G))
    lm = tf.pack_w4(dev(weights["lm_codes"], np.uint8), dev(weights["lm_scales"], np.int16), G)
    torch.cuda.synchronize()
    return tf.Model(emb, gu, dn, lm, V, H, F if F is not None else 64, G, rms_eps)


def token_sha(tokens) -> str:
    """SHA-256 of committed token ids as little-endian int32."""
    return hashlib.sha256(np.asarray(tokens, dtype="<i4").tobytes()).hexdigest()


class Decoder:
    """Device state for a decode loop: last token, position, drafts, outputs."""

    def __init__(self, model: tf.Model, max_rows: int = tf.MAX_ROWS, device="cuda", keep_logits: bool = False):
        self.model = model
        self.ws = tf.workspace(model.workspace_bytes(max_rows), device)
        self.last = torch.zeros(1, dtype=torch.int32, device=device)
        self.pos = torch.zeros(1, dtype=torch.int64, device=device)
        self.drafts = torch.zeros(max_rows, dtype=torch.int32, device=device)
        self.tokens = torch.zeros(max_rows, dtype=torch.int32, device=device)
        self.accepted = torch.zeros(1, dtype=torch.int32, device=device)
        self.logits = (torch.empty((max_rows, model.vocab), dtype=torch.float32, device=device)
                       if keep_logits else None)
        self.h_drafts = torch.zeros(max_rows, dtype=torch.int32).pin_memory()
        self.h_out = torch.zeros(1 + max_rows, dtype=torch.int32).pin_memory()
        self._out = torch.zeros(1 + max_rows, dtype=torch.int32, device=device)

    def reset(self, prompt_token: int, pos: int = 1):
        self.last.fill_(int(prompt_token))
        self.pos.fill_(int(pos))

    def step(self, R: int, drafts, temperature, top_k, top_p, seed):
        """One verify pass; returns (a, tokens t[0..R-1])."""
        if R > 1:
            self.h_drafts[: R - 1] = torch.as_tensor(np.asarray(drafts[: R - 1], dtype=np.int32))
            self.drafts[: R - 1].copy_(self.h_drafts[: R - 1], non_blocking=True)
        lg = self.logits[:R] if self.logits is not None else None
        self.model.verify_step(R, self.last, self.pos, self.drafts, temperature, top_k, top_p, seed,
                               self.tokens, self.accepted, self.ws, logits=lg)
        self._out[0:1].copy_(self.accepted)
        self._out[1:1 + R].copy_(self.tokens[:R])
        self.h_out[: 1 + R].copy_(self._out[: 1 + R], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        out = self.h_out[: 1 + R].tolist()
        return out[0], out[1:]


def serial_decode(dec: Decoder, prompt_token: int, n_tokens: int, temperature, top_k, top_p, seed):
    dec.reset(prompt_token, 1)
    out = []
    while len(out) < n_tokens:
        _, t = dec.step(1, [], temperature, top_k, top_p, seed)
        out.append(t[0])
    return out


def drafted_decode(dec: Decoder, prompt_token: int, n_tokens: int, R: int, temperature, top_k, top_p, seed,
                   draft_fn):
    """``draft_fn(pos0, n)`` gives the drafts for positions pos0 .. pos0+n-1."""
    dec.reset(prompt_token, 1)
    out, lens = [], []
    pos0 = 1
    while len(out) < n_tokens:
        d = list(draft_fn(pos0, R - 1))
        a, t = dec.step(R, d, temperature, top_k, top_p, seed)
        out.extend(t[: a + 1])
        lens.append(a)
        pos0 += a + 1
    return out[:n_tokens], lens


class GraphLoop:
    """Decoding with every verify pass chained on the device.

    Each pass takes its drafts from ``draft_table`` (device int32, index =
    position; unused when R = 1), runs ``tf_verify_step`` and writes its
    committed tokens into a device log; ``passes_per_graph`` passes are
    captured once as a CUDA graph (sampling settings and seed included) and
    replayed, and the host only checks the position between replays.
    """

    def __init__(self, dec: Decoder, n_tokens: int, R: int, temperature, top_k, top_p, seed,
                 draft_table: torch.Tensor = None, passes_per_graph: int = 8, prompt_token: int = 0):
        if R > 1 and draft_table is None:
            raise ValueError("a drafted run needs a draft table")
        self.dec, self.n_tokens, self.R, self.passes_per_graph = dec, n_tokens, R, passes_per_graph
        device = dec.last.device
        self.log = torch.zeros(n_tokens + (passes_per_graph + 1) * R, dtype=torch.int32, device=device)
        self.table = draft_table if draft_table is not None else torch.zeros(1, dtype=torch.int32, device=device)

        def one_pass():
            if R > 1:
                tf.gather_drafts(self.table, dec.pos, R, dec.drafts)
            dec.model.verify_step(R, dec.last, dec.pos, dec.drafts, temperature, top_k, top_p, seed, dec.tokens,
                                  dec.accepted, dec.ws)
            tf.commit_tokens(dec.tokens, dec.accepted, dec.pos, self.log)

        dec.reset(prompt_token, 1)
        one_pass()                      # first-call set-up happens outside the capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            for _ in range(passes_per_graph):
                one_pass()

    def run(self, prompt_token: int):
        """Returns (tokens, passes run); passes run counts whole replays."""
        self.dec.reset(prompt_token, 1)
        passes = 0
        while True:
            self.graph.replay()
            passes += self.passes_per_graph
            if int(self.dec.pos.item()) - 1 >= self.n_tokens:
                break
        return self.log[: self.n_tokens].tolist(), passes


def graph_decode(dec: Decoder, prompt_token: int, n_tokens: int, R: int, temperature, top_k, top_p, seed,
                 draft_table: torch.Tensor = None, passes_per_graph: int = 8):
    """One run of a freshly captured ``GraphLoop``: (tokens, passes run)."""
    loop = GraphLoop(dec, n_tokens, R, temperature, top_k, top_p, seed, draft_table, passes_per_graph,
                     prompt_token)
    return loop.run(prompt_token)

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


# ---------------------------------------------------------------- decoder with attention
class AttnModel:
    """The synthetic decoder with an attention sub-block before each MLP block.

    Block b: n = bf16(rms(x)); qkv = W_qkv n (queries n_q x 128, then keys and
    values n_kv x 128 each); the keys and values of the rows go into block b's
    KV cache at their positions; o = attention of the queries over the cache;
    x += W_o bf16(o); then the attention-free model's MLP block b.  Every
    projection is a W4 lane GEMM, so each row's bits do not depend on R.
    """

    def __init__(self, base: tf.Model, qkv, o, n_kv: int, group: int, max_len: int):
        if len(qkv) != len(base.gate_up) or len(o) != len(qkv):
            raise ValueError("one qkv and one output projection per block")
        self.base, self.qkv, self.o = base, list(qkv), list(o)
        self.n_kv, self.group, self.n_q = n_kv, group, n_kv * group
        self.max_len = max_len
        self.caches = [tf.KVCache(n_kv, max_len) for _ in self.qkv]


def upload_attn_model(weights: dict, n_kv: int, group: int, max_len: int, rms_eps: float = 1e-6,
                      device="cuda") -> AttnModel:
    """``weights`` as for upload_model plus ``attn``: per block qkv_codes/qkv_scales
    ([(n_q + 2 n_kv) * 128][hidden]) and o_codes/o_scales ([hidden][n_q * 128])."""
    base = upload_model(weights, rms_eps, device)
    G = weights["group"]

    def dev(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(device)

    qkv = [tf.pack_w4(dev(a["qkv_codes"], np.uint8), dev(a["qkv_scales"], np.int16), G) for a in weights["attn"]]
    o = [tf.pack_w4(dev(a["o_codes"], np.uint8), dev(a["o_scales"], np.int16), G) for a in weights["attn"]]
    torch.cuda.synchronize()
    return AttnModel(base, qkv, o, n_kv, group, max_len)


class AttnDecoder:
    """Decode loop state for an AttnModel; same interface as Decoder.

    A pass of R rows at position p (the next position to sample) feeds the last
    committed token and R - 1 drafts at cache positions p - 1 .. p + R - 2 and
    samples positions p .. p + R - 1.  Rejected rows leave stale cache entries
    behind; the next pass starts at the first of them and rewrites it before
    any row reads it.
    """

    def __init__(self, model: AttnModel, max_rows: int = tf.MAX_ROWS, device="cuda"):
        b = model.base
        H, V, F = b.hidden, b.vocab, b.ffn
        W = (model.n_q + 2 * model.n_kv) * tf.HEAD_DIM
        A = model.n_q * tf.HEAD_DIM
        self.model, self.max_rows = model, max_rows
        f32 = dict(dtype=torch.float32, device=device)
        i16 = dict(dtype=torch.int16, device=device)
        self.x = torch.zeros((max_rows, H), **f32)
        self.n = torch.zeros((max_rows, H), **i16)
        self.qkv = torch.zeros((max_rows, W), **f32)
        self.qkv_b = torch.zeros((max_rows, W), **i16)
        self.att = torch.zeros((max_rows, A), **f32)
        self.att_b = torch.zeros((max_rows, A), **i16)
        self.n_out = torch.zeros((max_rows, H), **i16)
        self.h_out = torch.zeros((max_rows, F), **i16)
        self.logits = torch.zeros((max_rows, V), **f32)
        gemm_ws = max(tf.lane_gemm_workspace_bytes(m.K, m.N, m.group) for m in model.qkv + model.o + [b.lm_head])
        self.ws_gemm = tf.workspace(gemm_ws, device)
        self.ws_block = tf.workspace(b.block_workspace_bytes(), device)
        self.ws_attn = tf.workspace(model.caches[0].workspace_bytes(model.group, max_rows), device)
        self.ws_status = tf.workspace(256, device)
        self.ws_sample = tf.workspace(tf.keyed_sample_workspace_bytes(max_rows, V), device)
        self.last = torch.zeros(1, dtype=torch.int32, device=device)
        self.drafts = torch.zeros(max_rows, dtype=torch.int32, device=device)
        self.kv_pos = torch.zeros(1, dtype=torch.int64, device=device)
        self.sample_pos = torch.zeros(max_rows, dtype=torch.int64, device=device)
        self.tokens = torch.zeros(max_rows, dtype=torch.int32, device=device)
        self.accepted = torch.zeros(1, dtype=torch.int32, device=device)
        self.h_pos = torch.zeros(1 + max_rows, dtype=torch.int64).pin_memory()
        self.h_drafts = torch.zeros(max_rows, dtype=torch.int32).pin_memory()
        self.h_result = torch.zeros(1 + max_rows, dtype=torch.int32).pin_memory()
        self._out = torch.zeros(1 + max_rows, dtype=torch.int32, device=device)
        self.pos = 1

    def reset(self, last_token: int, pos: int = 1):
        """Continue after a committed token ``last_token`` at position pos - 1."""
        self.last.fill_(int(last_token))
        self.pos = int(pos)

    def _rows(self, R: int, kv_pos0: int):
        """Embedding and every block for rows whose inputs are last, drafts[0..R-2]."""
        m, b = self.model, self.model.base
        qo, ko, vo = 0, m.n_q * tf.HEAD_DIM, (m.n_q + m.n_kv) * tf.HEAD_DIM
        x = self.x[:R]
        b.embed_rows(self.last, self.drafts, R, x, self.ws_status)
        for i in range(len(m.qkv)):
            tf.rmsnorm_bf16(x, b.rms_eps, out=self.n[:R])
            tf.lane_gemm_w4(m.qkv[i], self.n[:R], y=self.qkv[:R], ws=self.ws_gemm)
            tf.cast_bf16(self.qkv[:R], out=self.qkv_b[:R])
            m.caches[i].append(self.qkv_b[:R, ko:vo], self.qkv_b[:R, vo:], self.kv_pos, ws=self.ws_status)
            m.caches[i].attention(self.qkv_b[:R, qo:ko], m.group, self.kv_pos, out=self.att[:R], ws=self.ws_attn)
            tf.cast_bf16(self.att[:R], out=self.att_b[:R])
            tf.lane_gemm_w4_accumulate(m.o[i], self.att_b[:R], x, ws=self.ws_gemm)
            b.block(i, x, self.n_out[:R], self.h_out[:R], self.ws_block)

    def _set_positions(self, R: int, kv_pos0: int, sample_pos0: int):
        self.h_pos[0] = kv_pos0
        self.h_pos[1:1 + R] = torch.arange(sample_pos0, sample_pos0 + R, dtype=torch.int64)
        self.kv_pos.copy_(self.h_pos[0:1], non_blocking=True)
        self.sample_pos[:R].copy_(self.h_pos[1:1 + R], non_blocking=True)

    def prefill(self, tokens, block: int = tf.MAX_ROWS, first: int = 0):
        """Cache entries for tokens[first:] at their positions, ``block`` rows per
        pass, passes starting at multiples of ``block`` (a fixed grid of
        positions).  Every entry's bits are those of one-row decoding."""
        toks = [int(t) for t in tokens]
        p = first
        while p < len(toks):
            R = min(block - p % block, len(toks) - p)
            # the pinned staging buffers are reused: the previous pass's copies must have run
            torch.cuda.current_stream().synchronize()
            self.last.fill_(toks[p])
            if R > 1:
                self.h_drafts[: R - 1] = torch.as_tensor(toks[p + 1: p + R], dtype=torch.int32)
                self.drafts[: R - 1].copy_(self.h_drafts[: R - 1], non_blocking=True)
            self._set_positions(R, p, p + 1)
            self._rows(R, p)
            p += R
        torch.cuda.current_stream().synchronize()

    def step(self, R: int, drafts, temperature, top_k, top_p, seed):
        """One verify pass; returns (a, tokens t[0..R-1]) and advances the position."""
        b = self.model.base
        if R > 1:
            self.h_drafts[: R - 1] = torch.as_tensor(np.asarray(drafts[: R - 1], dtype=np.int32))
            self.drafts[: R - 1].copy_(self.h_drafts[: R - 1], non_blocking=True)
        self._set_positions(R, self.pos - 1, self.pos)
        self._rows(R, self.pos - 1)
        tf.rmsnorm_bf16(self.x[:R], b.rms_eps, out=self.n[:R])
        tf.lane_gemm_w4(b.lm_head, self.n[:R], y=self.logits[:R], ws=self.ws_gemm)
        tf.keyed_sample(self.logits[:R], temperature, top_k, top_p, seed, pos=self.sample_pos[:R],
                        tokens=self.tokens[:R], ws=self.ws_sample)
        tf.accept(self.drafts[: max(R - 1, 1)], self.tokens[:R], accepted=self.accepted, bonus=self.last)
        self._out[0:1].copy_(self.accepted)
        self._out[1:1 + R].copy_(self.tokens[:R])
        self.h_result[: 1 + R].copy_(self._out[: 1 + R], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        out = self.h_result[: 1 + R].tolist()
        self.pos += out[0] + 1
        return out[0], out[1:]


def attn_serial_decode(dec: AttnDecoder, last_token: int, pos: int, n_tokens: int, temperature, top_k, top_p,
                       seed):
    dec.reset(last_token, pos)
    out = []
    while len(out) < n_tokens:
        _, t = dec.step(1, [], temperature, top_k, top_p, seed)
        out.append(t[0])
    return out


def attn_drafted_decode(dec: AttnDecoder, last_token: int, pos: int, n_tokens: int, R: int, temperature, top_k,
                        top_p, seed, draft_fn):
    """``draft_fn(pos0, n)`` gives the drafts for positions pos0 .. pos0+n-1."""
    dec.reset(last_token, pos)
    out, lens = [], []
    while len(out) < n_tokens:
        pos0 = dec.pos
        a, t = dec.step(R, list(draft_fn(pos0, R - 1)), temperature, top_k, top_p, seed)
        out.extend(t[: a + 1])
        lens.append(a)
    return out[:n_tokens], lens

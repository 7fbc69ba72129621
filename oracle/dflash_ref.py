"""Float64 restatement of one DFlash drafting round (oracle; test infrastructure).

Only tests, the smoke entry and the bench's CPU-baseline leg may import this.
See the package docstring for the page titles behind the short citation tags.

Round structure ([Code walkthrough] §三 第1-3步; [Paper walkthrough] 设计):
  a1 fuse      c = RMSNorm(concat_5(features) @ W_fc^T)
  a2 inject    per draft layer: K = RoPE(k_norm(c @ W_k^T)), V = c @ W_v^T, appended
  a3 embed     block = [last verified token, 15 x mask]; h = E[block]
  a4/a5 layers pre-norm decoder layers; attention of the 16 block queries over
               [context K/V ; block K/V] with no mask
  a6 lm_head   tied embedding, argmax on block rows 1..15 -> 15 drafts
  a7 accept    longest matching prefix (cumulative product), bonus = target
               token at the first mismatch, context length += accepted count

Readings where the pages are silent:
  mask id = vocab-1; the 5 layers concatenate shallow->deep; fusion has no
  bias and its RMSNorm has a learned gain; c enters W_k/W_v without a norm;
  Qwen3-style layer (per-head q/k RMSNorm, SiLU-gated MLP, final norm);
  rotate-half RoPE with inv_freq_i = theta^(-2i/D); attention scale 1/sqrt(D);
  argmax ties go to the lowest id; the features appended after a round are the
  accepted count of rows, for the positions of the last verified token and the
  accepted drafts.
"""
from __future__ import annotations

import numpy as np

from workload.gen import bf16_bits_to_f32


# ----------------------------------------------------------------- helpers

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis.

    Used for the fusion norm ([Code walkthrough] §二.3, "线性投影 + RMSNorm";
    [Paper walkthrough] 设计 — Feature Fusion) and the drafter's layer norms.
    """
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half convention.

    x [..., n, heads, D], pos [n].  Dimension i (< D/2) pairs with i + D/2 and
    rotates by angle pos * theta^(-2i/D).  The pages name RoPE only through
    the drafter being a standard Qwen3/LLaMA-style layer; this is that
    family's convention.
    """
    D = x.shape[-1]
    half = D // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / D)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]  # [n, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softmax(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def argmax_first(x: np.ndarray) -> np.ndarray:
    """Index of the maximum along the last axis; ties go to the lowest index."""
    return np.argmax(x, axis=-1)


# ----------------------------------------------------------------- model

# matrices held as FP8 E4M3 with per-row scales in the low-precision variant
# (everything but the fusion projection and the norm gains)
FP8_WEIGHTS = ("embed", "wqkv", "wo", "w_gate_up", "w_down")

class OracleModel:
    """Drafter weights (bf16 bit patterns) with float64 views on demand.

    ``cache=True`` keeps float64 copies (small shapes); ``cache=False`` widens
    each matrix when used so full-size drafters fit in host memory.
    """

    def __init__(self, cfg, weights: dict, cache: bool = True, fp8: bool = False):
        self.cfg = cfg
        self.raw = weights
        self.cache = cache
        self.fp8 = fp8  # projections and the embedding as per-row-scaled E4M3 (oracle.fp8_ref)
        self._c = {}

    def _widen(self, name: str, src) -> np.ndarray:
        arr = bf16_to_f64(src)
        if self.fp8 and name in FP8_WEIGHTS:
            from .fp8_ref import dequantize_rows
            arr = dequantize_rows(arr)
        return arr

    def w(self, name: str, layer: int | None = None) -> np.ndarray:
        key = (name, layer)
        if key in self._c:
            return self._c[key]
        src = self.raw[name] if layer is None else self.raw["layers"][layer][name]
        arr = self._widen(name, src)
        if self.cache:
            self._c[key] = arr
        return arr

    def embed_rows(self, ids) -> np.ndarray:
        return self._widen("embed", self.raw["embed"][np.asarray(ids)])


# ----------------------------------------------------------------- a1, a2

def fuse_features(model: OracleModel, feats: np.ndarray) -> np.ndarray:
    """a1: target context feature from 5 target layers' hidden states.

    feats [n, 5, H] (bf16 bits or float64), layers ordered shallow -> deep
    ([Paper walkthrough] 设计 — Feature Fusion: 由浅到深 five layers,
    concatenated, one light projection; [Code walkthrough] §二.3: 一层线性投影
    + RMSNorm).  Returns c [n, H] float64.
    """
    cfg = model.cfg
    x = feats if feats.dtype == np.float64 else bf16_to_f64(feats)
    x = x.reshape(x.shape[0], cfg.n_fused * cfg.hidden)
    return rmsnorm(x @ model.w("fc").T, model.w("fc_norm"), cfg.rms_eps)


def inject_kv(model: OracleModel, layer: int, c: np.ndarray, pos: np.ndarray):
    """a2: project the fused feature into one draft layer's K/V.

    [Paper walkthrough] 设计 — KV Injection: the fused feature is projected
    directly by each draft layer's Key/Value projections and kept in the KV
    cache across drafting iterations; [News summary] "目标模型最懂": injected
    into every draft layer's K and V projections.  K gets the layer's per-head
    k-norm and RoPE at the context positions; V is the plain projection.
    Returns K, V [n, hkv, D].
    """
    cfg = model.cfg
    hq, hkv, D = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    wqkv = model.w("wqkv", layer)
    wk = wqkv[hq * D:(hq + hkv) * D]
    wv = wqkv[(hq + hkv) * D:]
    n = c.shape[0]
    k = (c @ wk.T).reshape(n, hkv, D)
    v = (c @ wv.T).reshape(n, hkv, D)
    k = rmsnorm(k, model.w("k_norm", layer), cfg.rms_eps)
    k = rope(k, pos, cfg.rope_theta)
    return k, v


# ----------------------------------------------------------------- a4, a5

def block_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """a5: softmax(q K^T / sqrt(D)) V with NO mask.

    q [S, hq, D]; K, V [L+S, hkv, D] = [context ; block].  Every block
    position sees the whole context and every other block position
    ([Code walkthrough] §二.2, is_causal=False).  Query head j reads KV head
    floor(j * hkv / hq) (grouped-query attention).
    """
    S, hq, D = q.shape
    hkv = K.shape[1]
    out = np.empty_like(q)
    scale = 1.0 / np.sqrt(D)
    for j in range(hq):
        kv = (j * hkv) // hq
        s = (q[:, j, :] @ K[:, kv, :].T) * scale
        out[:, j, :] = softmax(s) @ V[:, kv, :]
    return out


def decoder_layer(model: OracleModel, layer: int, h: np.ndarray, pos: np.ndarray,
                  ctx_k: np.ndarray, ctx_v: np.ndarray) -> np.ndarray:
    """a4: one pre-norm draft layer on the block's hidden states h [S, H].

    ([Paper walkthrough] 设计 — Parallel Drafting: one forward over the block,
    conditioned on the persistent target context in the KV cache.)  Layer
    type read as Qwen3-style: input RMSNorm, QKV projection, per-head q/k
    RMSNorm, RoPE at the block positions, attention (a5), output projection
    with residual, post-attention RMSNorm, SiLU-gated MLP with residual.
    """
    cfg = model.cfg
    hq, hkv, D, I = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate
    S = h.shape[0]
    eps = cfg.rms_eps
    x = rmsnorm(h, model.w("in_norm", layer), eps)
    qkv = x @ model.w("wqkv", layer).T
    q = qkv[:, :hq * D].reshape(S, hq, D)
    k = qkv[:, hq * D:(hq + hkv) * D].reshape(S, hkv, D)
    v = qkv[:, (hq + hkv) * D:].reshape(S, hkv, D)
    q = rope(rmsnorm(q, model.w("q_norm", layer), eps), pos, cfg.rope_theta)
    k = rope(rmsnorm(k, model.w("k_norm", layer), eps), pos, cfg.rope_theta)
    o = block_attention(q, np.concatenate([ctx_k, k], 0), np.concatenate([ctx_v, v], 0))
    h = h + o.reshape(S, hq * D) @ model.w("wo", layer).T
    y = rmsnorm(h, model.w("post_norm", layer), eps)
    gu = y @ model.w("w_gate_up", layer).T
    h = h + (silu(gu[:, :I]) * gu[:, I:]) @ model.w("w_down", layer).T
    return h


# ----------------------------------------------------------------- a6, a7

def lm_head_logits(model: OracleModel, h: np.ndarray, chunk: int = 1 << 14) -> np.ndarray:
    """a6 logits: RMSNorm(h, final gain) @ E^T with the tied embedding table.

    [Paper walkthrough] 设计 (reuses the target's embedding and LM head);
    [Code walkthrough] §二.3 (embed_tokens and lm_head bound to the target's).
    The vocabulary is walked in chunks only to bound host memory; every logit
    is the same single dot product either way.
    """
    cfg = model.cfg
    hn = rmsnorm(h, model.w("final_norm"), cfg.rms_eps)
    V = cfg.vocab
    out = np.empty((h.shape[0], V), dtype=np.float64)
    E = model.raw["embed"]
    for v0 in range(0, V, chunk):
        out[:, v0:v0 + chunk] = hn @ model._widen("embed", E[v0:v0 + chunk]).T
    return out


def accept_longest_prefix(draft: np.ndarray, target: np.ndarray):
    """a7: accept the longest matching prefix, then the bonus token.

    draft [S-1]: d_1..d_{S-1} (block positions 1..S-1); target [S]: t_0..t_{S-1},
    the target's own token after each block position.  d_{i+1} is accepted
    while it equals t_i, found with a cumulative product of the per-position
    matches ([Code walkthrough] §三 第3步); the first mismatch is replaced by
    the target's token (the bonus).  Worst case 1 token, best case S (16 at
    the trained block size; a smaller S at inference, [Paper walkthrough]
    Results: a large training block generalises to smaller inference blocks).
    Returns (tau, bonus) with tau = accepted drafts + 1.
    """
    nd = len(draft)
    match = (np.asarray(draft[:nd]) == np.asarray(target[:nd])).astype(np.int64)
    n = int(np.cumprod(match).sum())
    return n + 1, int(target[n])


def synthetic_target(draft: np.ndarray, m: np.ndarray, u: np.ndarray, vocab: int) -> np.ndarray:
    """Stand-in for the target model's verify step (benchmark harness, not the method).

    t_i = d_{i+1} if m_i else a uniform id different from d_{i+1} (u_i, bumped
    to (u_i+1) mod vocab on a collision), for i < S-1; t_{S-1} = u_{S-1}, with
    S-1 = len(draft).  The accepted length then depends only on m, never on
    the draft values.
    """
    nd = len(draft)
    t = np.empty(nd + 1, dtype=np.int64)
    for i in range(nd):
        d = int(draft[i])
        if m[i]:
            t[i] = d
        else:
            x = int(u[i])
            t[i] = (x + 1) % vocab if x == d else x
    t[nd] = int(u[nd])
    return t


# ----------------------------------------------------------------- state

class OracleRequest:
    """Per-request draft KV cache (float64) and context length."""

    def __init__(self, cfg, capacity: int):
        hkv, D = cfg.n_kv_heads, cfg.head_dim
        self.K = [np.zeros((capacity, hkv, D)) for _ in range(cfg.n_layers)]
        self.V = [np.zeros((capacity, hkv, D)) for _ in range(cfg.n_layers)]
        self.ctx_len = 0

    def ctx(self, layer):
        return self.K[layer][:self.ctx_len], self.V[layer][:self.ctx_len]


class OracleDrafter:
    """Round driver: fuse/inject, draft one block, accept/trim."""

    def __init__(self, model: OracleModel):
        self.model = model
        self.cfg = model.cfg

    def fuse_inject(self, req: OracleRequest, feats: np.ndarray):
        """a1 + a2 for n new rows at positions ctx_len .. ctx_len+n-1."""
        n = feats.shape[0]
        if n == 0:
            return
        c = fuse_features(self.model, feats)
        pos = np.arange(req.ctx_len, req.ctx_len + n)
        for l in range(self.cfg.n_layers):
            k, v = inject_kv(self.model, l, c, pos)
            req.K[l][pos] = k
            req.V[l][pos] = v
        req.ctx_len += n

    def draft(self, req: OracleRequest, last_tok: int, want_logits: bool = True):
        """a3-a6: one forward over [last_tok, mask x (S-1)]; returns a dict.

        Block = last verified token followed by S-1 mask ids ([Code walkthrough]
        §二.1, block size 16 = 1 known + 15 masks -> 15 candidates; S = cfg.block,
        smaller at inference per [Paper walkthrough] Results).
        """
        cfg = self.cfg
        S = cfg.block
        tokens = np.array([last_tok] + [cfg.mask_id] * (S - 1))
        h = self.model.embed_rows(tokens)
        pos = np.arange(req.ctx_len, req.ctx_len + S)
        for l in range(cfg.n_layers):
            ck, cv = req.ctx(l)
            h = decoder_layer(self.model, l, h, pos, ck, cv)
        logits = lm_head_logits(self.model, h[1:])
        draft = argmax_first(logits)
        top2 = np.partition(logits, -2, axis=-1)[:, -2:]
        margin = top2[:, 1] - top2[:, 0]
        out = {"draft": draft.astype(np.int64), "hidden": h, "margin": margin}
        if want_logits:
            out["logits"] = logits
        return out

    def accept_trim(self, req: OracleRequest, draft: np.ndarray, target: np.ndarray):
        """a7: tau, bonus and the confirmed length L + tau.

        The block's own K/V never enters the cache, so trimming the draft
        cache to the confirmed length leaves entries < L untouched; the tau
        new features arrive with the next fuse_inject.
        """
        tau, bonus = accept_longest_prefix(draft, target)
        return tau, bonus, req.ctx_len + tau

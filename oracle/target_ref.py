"""Float64 target model, verify step and speculative generation loop (oracle;
test infrastructure).

Only tests, the smoke entry and the bench's CPU-baseline leg may import this.

The verify step ([Code walkthrough] §三 第2步): the target runs one forward
over the block [b0, d_1..d_{S-1}] and gives, at every block position, its own
next token.  Acceptance keeps the longest matching prefix plus the target's
token at the first mismatch, and both caches are trimmed to the confirmed
length (§三 第3步); because a rejected position always falls back to the
target's own output, the generated text equals the target's own greedy
decoding (§三, "最终文本质量与目标模型直接生成完全一致").  The drafter's
features are hidden states of 5 target layers, shallow to deep ([Paper
walkthrough] 设计 — Feature Fusion), taken from the target's middle layers
with evenly spread layer ids ([Code walkthrough] §二.3), and the drafter
shares the target's embedding and LM head (§二.3).

Readings taken where the pages are silent:
  * the target is a stack of the same pre-norm Qwen3-style layers as the
    drafter (dflash_ref.decoder_layer) with CAUSAL attention: block row i
    sees the context and block rows 0..i;
  * the 5 taps are the residual stream after target layers
    tap_layers(L) = 1 + round(k (L-3) / 4), k = 0..4 (layers 1..L-2 evenly
    spread, first and last excluded), rounded to bf16 at the interface (the
    drafter's feature input is bf16);
  * generation starts from the target's greedy token at the last prompt
    position;
  * at temperature T > 0 the target samples its own token at every block
    position ([Code walkthrough] §三 第3步 compares the block with the
    target's sampled tokens; [Paper walkthrough] Results reports sampling at
    T = 1) by the Gumbel-max rule on a stream keyed by the position
    (sampling_ref.sample_target_rows), so a position's draw does not depend
    on which round or block it falls in -- the speculative loop then emits
    exactly the target's own sampled decoding.
"""
from __future__ import annotations

import numpy as np

from workload.gen import f64_to_bf16_bits

from .dflash_ref import (OracleModel, accept_longest_prefix, lm_head_logits, rmsnorm, rope, silu, softmax,
                         bf16_to_f64)


def tap_layers(n_layers: int, n_taps: int = 5) -> list[int]:
    """Target layers whose outputs are the drafter's features, shallow to deep."""
    assert n_layers >= n_taps + 2
    return [1 + (2 * k * (n_layers - 3) + (n_taps - 1)) // (2 * (n_taps - 1)) for k in range(n_taps)]


def causal_block_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, L: int) -> np.ndarray:
    """softmax(q K^T / sqrt(D)) V where block row i (position L+i) sees keys
    0..L+i: the context and block rows 0..i.  q [S, hq, D]; K, V [L+S, hkv, D];
    query head j reads KV head floor(j * hkv / hq)."""
    S, hq, D = q.shape
    hkv = K.shape[1]
    out = np.empty_like(q)
    scale = 1.0 / np.sqrt(D)
    mask = np.arange(L + S)[None, :] <= (L + np.arange(S))[:, None]
    for j in range(hq):
        kv = (j * hkv) // hq
        s = (q[:, j, :] @ K[:, kv, :].T) * scale
        s = np.where(mask, s, -np.inf)
        out[:, j, :] = softmax(s) @ V[:, kv, :]
    return out


def target_layer(model: OracleModel, layer: int, h: np.ndarray, L: int, ctx_k: np.ndarray, ctx_v: np.ndarray):
    """One causal target layer on block rows h [S, H] at positions L..L+S-1.
    Returns (h_out, k, v) with the block's own K/V [S, hkv, D]."""
    cfg = model.cfg
    hq, hkv, D, I = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate
    S = h.shape[0]
    eps = cfg.rms_eps
    pos = np.arange(L, L + S)
    x = rmsnorm(h, model.w("in_norm", layer), eps)
    qkv = x @ model.w("wqkv", layer).T
    q = qkv[:, :hq * D].reshape(S, hq, D)
    k = qkv[:, hq * D:(hq + hkv) * D].reshape(S, hkv, D)
    v = qkv[:, (hq + hkv) * D:].reshape(S, hkv, D)
    q = rope(rmsnorm(q, model.w("q_norm", layer), eps), pos, cfg.rope_theta)
    k = rope(rmsnorm(k, model.w("k_norm", layer), eps), pos, cfg.rope_theta)
    o = causal_block_attention(q, np.concatenate([ctx_k, k], 0), np.concatenate([ctx_v, v], 0), L)
    h = h + o.reshape(S, hq * D) @ model.w("wo", layer).T
    y = rmsnorm(h, model.w("post_norm", layer), eps)
    gu = y @ model.w("w_gate_up", layer).T
    h = h + (silu(gu[:, :I]) * gu[:, I:]) @ model.w("w_down", layer).T
    return h, k, v


class OracleTarget:
    """A target model over one request: its own float64 KV cache."""

    def __init__(self, model: OracleModel, n_layers: int, capacity: int):
        self.model = model
        self.cfg = model.cfg
        self.n_layers = n_layers
        self.taps = tap_layers(n_layers, self.cfg.n_fused)
        hkv, D = self.cfg.n_kv_heads, self.cfg.head_dim
        self.K = [np.zeros((capacity, hkv, D)) for _ in range(n_layers)]
        self.V = [np.zeros((capacity, hkv, D)) for _ in range(n_layers)]
        self.ctx_len = 0

    def forward(self, tokens, temperature: float = 0.0, seed: int = 0, slot: int = 0) -> dict:
        """The block's tokens at positions ctx_len.. (their K/V are written to
        the cache; ctx_len moves only with advance()).  Returns the logits of
        every row, its token -- the argmax, or at temperature > 0 the draw of
        sampling_ref.sample_target_rows -- with the top-2 margin of the
        (perturbed) scores, and the 5 tap features (float64 and bf16 bits)."""
        tokens = np.asarray(tokens)
        L = self.ctx_len
        S = len(tokens)
        h = self.model.embed_rows(tokens)
        feats = np.empty((S, len(self.taps), self.cfg.hidden))
        for l in range(self.n_layers):
            h, k, v = target_layer(self.model, l, h, L, self.K[l][:L], self.V[l][:L])
            self.K[l][L:L + S] = k
            self.V[l][L:L + S] = v
            if l in self.taps:
                feats[:, self.taps.index(l)] = h
        logits = lm_head_logits(self.model, h)
        if temperature > 0:
            from .sampling_ref import sample_target_rows
            tok, margin = sample_target_rows(logits, temperature, seed, slot, L)
        else:
            top2 = np.partition(logits, -2, axis=-1)[:, -2:]
            tok, margin = np.argmax(logits, -1).astype(np.int64), top2[:, 1] - top2[:, 0]
        return dict(logits=logits, tok=tok, margin=margin, feats=feats, feats_bf16=f64_to_bf16_bits(feats))

    def advance(self, n: int):
        self.ctx_len += int(n)

    def prefill(self, prompt, chunk: int = 16, temperature: float = 0.0, seed: int = 0, slot: int = 0) -> dict:
        """Run the prompt in chunks; returns the last chunk's outputs and the
        bf16 features of every prompt position."""
        prompt = np.asarray(prompt)
        feats = []
        out = None
        for p0 in range(0, len(prompt), chunk):
            out = self.forward(prompt[p0:p0 + chunk], temperature, seed, slot)
            self.advance(min(chunk, len(prompt) - p0))
            feats.append(out["feats_bf16"])
        return dict(last=out, feats_bf16=np.concatenate(feats, 0))


def greedy_generate(target: OracleTarget, prompt, n_new: int, temperature: float = 0.0, seed: int = 0,
                    slot: int = 0):
    """The target's own decoding: n_new tokens after the prompt, greedy, or
    at temperature > 0 each drawn as in sampling_ref.sample_target_rows;
    with each token's top-2 margin."""
    pf = target.prefill(prompt, temperature=temperature, seed=seed, slot=slot)
    g = int(pf["last"]["tok"][-1])
    out, margins = [g], [float(pf["last"]["margin"][-1])]
    while len(out) < n_new:
        o = target.forward([g], temperature, seed, slot)
        target.advance(1)
        g = int(o["tok"][0])
        out.append(g)
        margins.append(float(o["margin"][0]))
    return np.array(out, dtype=np.int64), np.array(margins)


def spec_generate(drafter, draft_req, target: OracleTarget, prompt, n_new: int, block: int, draft_fn=None,
                  temperature: float = 0.0, seed: int = 0, slot: int = 0):
    """Speculative generation: prefill both models, then rounds of draft ->
    verify -> accept -> trim until n_new tokens are out.  draft_fn(out, b0)
    may replace the drafter's tokens (tests that force long acceptances).
    At temperature > 0 the drafter draws each draft from its own softmax
    (sampling_ref.sample_drafts, request 0, round index of the generation)
    and the target samples its tokens by position; acceptance is unchanged."""
    from .sampling_ref import sample_drafts
    pf = target.prefill(prompt, temperature=temperature, seed=seed, slot=slot)
    drafter.fuse_inject(draft_req, pf["feats_bf16"])
    b0 = int(pf["last"]["tok"][-1])
    out = [b0]
    taus = []
    rnd = 0
    while len(out) < n_new:
        if draft_fn is not None:
            d = draft_fn(out, b0)
        elif temperature > 0:
            d, _ = sample_drafts(drafter.draft(draft_req, b0)["logits"], temperature, seed, 0, rnd)
        else:
            d = drafter.draft(draft_req, b0, want_logits=False)["draft"]
        rnd += 1
        d = np.asarray(d, dtype=np.int64)[:block - 1]
        v = target.forward(np.concatenate([[b0], d]), temperature, seed, slot)
        tau, bonus = accept_longest_prefix(d, v["tok"])
        target.advance(tau)
        drafter.fuse_inject(draft_req, v["feats_bf16"][:tau])
        out.extend(int(x) for x in d[:tau - 1])
        out.append(bonus)
        taus.append(tau)
        b0 = bonus
    return np.array(out[:n_new], dtype=np.int64), taus

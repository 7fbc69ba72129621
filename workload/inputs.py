"""Seeded synthetic inputs: weights, target features, stand-in verify streams.

Seeds (fixed): weights 0 (+config.seed), features 1, match/offset stream 2,
per-request context lengths and match probabilities 3.

* Weights: every projection matrix N(0, weight_std) in bf16, row-major
  [out_features, in_features]; RMSNorm gains 1 (or 1 + gain_std*N(0,1)).
* Features of request b at position p: row of 5*hidden N(0,1) bf16 values,
  addressed by (b, p) so the row does not depend on acceptance history.
* Stand-in verify stream of request b in round r: S = block match bits
  m_i ~ Bernoulli(p_b) and S uniform ids u_i in [0, vocab).
"""
from __future__ import annotations

import os

import numpy as np

from .gen import normal_bf16, stream_key, uniform

SEED_WEIGHTS = 0
SEED_FEATURES = 1
SEED_MATCH = 2
SEED_SCENARIO = 3

# stable ids of the weight tensors inside the weight stream
_GLOBAL_IDS = {"embed": 1, "fc": 2, "fc_norm": 3, "final_norm": 4}
_LAYER_IDS = {"wqkv": 1, "wo": 2, "w_gate_up": 3, "w_down": 4,
              "in_norm": 5, "post_norm": 6, "q_norm": 7, "k_norm": 8}
WEIGHT_NAMES = tuple(_GLOBAL_IDS) + tuple(_LAYER_IDS)


def _shape(cfg, name):
    H, I, V, D = cfg.hidden, cfg.intermediate, cfg.vocab, cfg.head_dim
    return {
        "embed": (V, H), "fc": (H, cfg.fused_dim), "fc_norm": (H,), "final_norm": (H,),
        "wqkv": (cfg.qkv_rows, H), "wo": (H, cfg.n_q_heads * D), "w_gate_up": (2 * I, H),
        "w_down": (H, I), "in_norm": (H,), "post_norm": (H,), "q_norm": (D,), "k_norm": (D,),
    }[name]


def _tensor(cfg, name, layer=None):
    shape = _shape(cfg, name)
    n = int(np.prod(shape))
    if layer is None:
        key = stream_key(SEED_WEIGHTS + cfg.seed, _GLOBAL_IDS[name])
    else:
        key = stream_key(SEED_WEIGHTS + cfg.seed, 1000 + layer, _LAYER_IDS[name])
    if len(shape) == 1:  # RMSNorm gain
        if cfg.gain_std == 0.0:
            return np.full(shape, 0x3F80, dtype=np.uint16)  # bf16 1.0
        return normal_bf16(key, 0, n, scale=cfg.gain_std, shift=1.0).reshape(shape)
    return normal_bf16(key, 0, n, scale=cfg.weight_std).reshape(shape)


def _arch_key(cfg) -> str:
    fields = (cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate,
              cfg.n_layers, cfg.vocab, cfg.n_fused, cfg.weight_std, cfg.gain_std, cfg.seed, "v1")
    return "w_" + "_".join(str(f) for f in fields)


def make_weights(cfg):
    """All drafter weights as bf16 bit patterns (numpy uint16), cached on disk
    under $DFLASH_WORKLOAD_CACHE when that variable is set.

    Returns {"embed", "fc", "fc_norm", "final_norm", "layers": [ {per-layer} ]}.
    Layer tensors: wqkv [(hq+2hkv)*D, H] (q rows, then k rows, then v rows),
    wo [H, hq*D], w_gate_up [2I, H] (gate rows then up rows), w_down [H, I],
    in_norm/post_norm [H], q_norm/k_norm [D].
    """
    cache = os.environ.get("DFLASH_WORKLOAD_CACHE")
    path = os.path.join(cache, _arch_key(cfg)) if cache else None

    def get(name, layer=None):
        if path is None:
            return _tensor(cfg, name, layer)
        f = os.path.join(path, name if layer is None else f"{name}.{layer}") + ".npy"
        if os.path.exists(f):
            return np.load(f, mmap_mode="r")
        a = _tensor(cfg, name, layer)
        os.makedirs(path, exist_ok=True)
        np.save(f + ".tmp.npy", a)
        os.replace(f + ".tmp.npy", f)
        return a

    w = {k: get(k) for k in _GLOBAL_IDS}
    w["layers"] = [{k: get(k, l) for k in _LAYER_IDS} for l in range(cfg.n_layers)]
    return w


SEED_TARGET = 4
SEED_PROMPT = 5


def make_target_weights(cfg, n_layers: int):
    """Weights of a random target model with the drafter's layer shape: its
    own n_layers layers and final norm (seed stream 4) and the drafter's
    embedding table, shared (the drafter reuses the target's embedding and
    LM head).  Same layout as make_weights; no fusion weights."""
    def tensor(name, layer=None):
        shape = _shape(cfg, name)
        n = int(np.prod(shape))
        ids = (_GLOBAL_IDS[name],) if layer is None else (1000 + layer, _LAYER_IDS[name])
        key = stream_key(SEED_TARGET + cfg.seed, *ids)
        if len(shape) == 1:
            if cfg.gain_std == 0.0:
                return np.full(shape, 0x3F80, dtype=np.uint16)
            return normal_bf16(key, 0, n, scale=cfg.gain_std, shift=1.0).reshape(shape)
        return normal_bf16(key, 0, n, scale=cfg.weight_std).reshape(shape)
    w = {"embed": make_weights(cfg)["embed"], "final_norm": tensor("final_norm")}
    w["layers"] = [{k: tensor(k, l) for k in _LAYER_IDS} for l in range(n_layers)]
    return w


def prompt_tokens(cfg, b: int, n: int) -> np.ndarray:
    """Prompt of request b: n ids uniform over the vocabulary minus the mask id."""
    u = uniform(stream_key(SEED_PROMPT + cfg.seed, b), np.arange(n))
    return np.minimum(np.floor(u * (cfg.vocab - 1)), cfg.vocab - 2).astype(np.int64)


def feature_rows(cfg, b: int, p0: int, n: int) -> np.ndarray:
    """Target features of request b at positions p0..p0+n-1: uint16 [n, 5, H]."""
    F = cfg.fused_dim
    key = stream_key(SEED_FEATURES + cfg.seed, b)
    return normal_bf16(key, p0 * F, n * F).reshape(n, cfg.n_fused, cfg.hidden)


def context_lengths(cfg) -> np.ndarray:
    """Prompt length of each request (int64 [B])."""
    if cfg.ctx0 is not None:
        return np.full(cfg.batch, cfg.ctx0, dtype=np.int64)
    lo, hi = cfg.ctx_range
    u = uniform(stream_key(SEED_SCENARIO + cfg.seed, 0), np.arange(cfg.batch))
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64)


def match_probs(cfg) -> np.ndarray:
    """Per-request probability that the stand-in target copies a draft token."""
    if cfg.match_p is not None:
        return np.full(cfg.batch, cfg.match_p, dtype=np.float64)
    lo, hi = cfg.p_range
    u = uniform(stream_key(SEED_SCENARIO + cfg.seed, 1), np.arange(cfg.batch))
    return lo + (hi - lo) * u


def match_stream(cfg, r: int, batch_ids=None):
    """Stand-in verify randomness for round r.

    Returns (m, u): m int32 [B, S] in {0,1}, u int32 [B, S] in [0, vocab), S = cfg.block.
    """
    ids = range(cfg.batch) if batch_ids is None else batch_ids
    probs = match_probs(cfg)
    S = cfg.block
    m = np.empty((len(ids), S), dtype=np.int32)
    u = np.empty((len(ids), S), dtype=np.int32)
    idx = np.arange(S)
    for j, b in enumerate(ids):
        m[j] = (uniform(stream_key(SEED_MATCH + cfg.seed, b, r, 0), idx) < probs[b]).astype(np.int32)
        u[j] = np.minimum(np.floor(uniform(stream_key(SEED_MATCH + cfg.seed, b, r, 1), idx)
                                   * cfg.vocab), cfg.vocab - 1).astype(np.int32)
    return m, u

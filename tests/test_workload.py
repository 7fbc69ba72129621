"""The seeded synthetic input recipe: shapes, distributions and addressing of
the weights, target features, prompts and stand-in verify streams that both
the CUDA path and the oracle consume.  CPU only."""
import numpy as np
import pytest

from workload import (bf16_bits_to_f32, context_lengths, feature_rows, get_config, make_target_weights, make_weights,
                      match_probs, match_stream, prompt_tokens)

TINY = get_config("tiny")


def _f(bits):
    return np.asarray(bf16_bits_to_f32(np.asarray(bits)), dtype=np.float64)


def test_weight_shapes_distributions_and_determinism():
    cfg = TINY
    w = make_weights(cfg)
    H, I, V, D = cfg.hidden, cfg.intermediate, cfg.vocab, cfg.head_dim
    assert w["embed"].shape == (V, H) and w["fc"].shape == (H, 5 * H)
    assert len(w["layers"]) == cfg.n_layers
    L0 = w["layers"][0]
    assert L0["wqkv"].shape == ((cfg.n_q_heads + 2 * cfg.n_kv_heads) * D, H)
    assert L0["wo"].shape == (H, cfg.n_q_heads * D)
    assert L0["w_gate_up"].shape == (2 * I, H) and L0["w_down"].shape == (H, I)
    for name in ("embed", "fc"):
        x = _f(w[name])
        assert abs(x.mean()) < 1e-3 and abs(x.std() - cfg.weight_std) < 0.02 * cfg.weight_std
    assert np.all(w["final_norm"] == 0x3F80) and np.all(L0["k_norm"] == 0x3F80)  # gains 1.0 (bf16)
    w2 = make_weights(cfg)
    assert np.array_equal(w["embed"], w2["embed"]) and np.array_equal(L0["w_down"], w2["layers"][0]["w_down"])
    assert not np.array_equal(w["layers"][0]["wo"], w["layers"][1]["wo"])


def test_test_gains_and_target_weights_share_the_embedding():
    cfg = get_config("tiny-gains")
    w = make_weights(cfg)
    g = _f(w["final_norm"])
    assert abs(g.mean() - 1.0) < 0.05 and 0.05 < g.std() < 0.15
    t = make_target_weights(cfg, 8)
    assert np.array_equal(t["embed"], w["embed"]) and len(t["layers"]) == 8
    assert not np.array_equal(t["layers"][0]["wqkv"], w["layers"][0]["wqkv"])


def test_features_are_addressed_by_request_and_position():
    cfg = TINY
    a = feature_rows(cfg, 2, 0, 40)
    assert a.shape == (40, 5, cfg.hidden)
    assert np.array_equal(feature_rows(cfg, 2, 13, 9), a[13:22])  # any chunking reads the same rows
    assert not np.array_equal(feature_rows(cfg, 3, 0, 40), a)
    x = _f(a)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02


def test_prompts_avoid_the_mask_id():
    cfg = TINY
    p = prompt_tokens(cfg, 0, 5000)
    assert p.min() >= 0 and p.max() <= cfg.vocab - 2
    assert len(np.unique(p)) > 0.6 * cfg.vocab
    assert np.array_equal(prompt_tokens(cfg, 0, 100), p[:100])


@pytest.mark.parametrize("name", ["qwen3-8b", "llama3.1-8b", "long-8layer", "batched-qwen3-8b"])
def test_scenario_lengths_and_match_probabilities(name):
    cfg = get_config(name)
    L = context_lengths(cfg)
    p = match_probs(cfg)
    assert L.shape == (cfg.batch,) and p.shape == (cfg.batch,)
    if cfg.ctx0 is not None:
        assert np.all(L == cfg.ctx0) and np.all(p == cfg.match_p)
    else:
        lo, hi = cfg.ctx_range
        assert L.min() >= lo and L.max() <= hi and len(np.unique(L)) > cfg.batch // 2
        plo, phi = cfg.p_range
        assert p.min() >= plo and p.max() <= phi


def test_match_stream_rates_and_ranges():
    cfg = get_config("qwen3-8b")
    ms = [match_stream(cfg, r) for r in range(400)]
    m = np.stack([a for a, _ in ms])
    u = np.stack([b for _, b in ms])
    assert m.shape == (400, cfg.batch, cfg.block) and set(np.unique(m)) <= {0, 1}
    assert abs(m.mean() - cfg.match_p) < 0.02
    assert u.min() >= 0 and u.max() < cfg.vocab
    m0, u0 = match_stream(cfg, 7)
    assert np.array_equal(m0, m[7]) and np.array_equal(u0, u[7])  # addressed by round, not drawn in sequence

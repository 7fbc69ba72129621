"""Pins for the float64 target model and speculative loop (oracle/target_ref.py).

What fixes them outside the oracle: causal attention written as plain loops
(brute force), the exactness of causal processing (a prompt run in 16-token
chunks or one token at a time gives the same logits), the tap definition
(the residual stream after the named layers), and losslessness: speculative
generation emits exactly the target's greedy tokens whatever the drafts are
([Code walkthrough] §三: a rejected position always falls back to the
target's own token).
"""
import numpy as np
import pytest

import oracle as O
import oracle.target_ref as T
from workload import get_config, make_target_weights, make_weights, prompt_tokens

CFG = get_config("tiny-gains")
NL = 8


@pytest.fixture(scope="module")
def models():
    tw = make_target_weights(CFG, NL)
    dw = make_weights(CFG)
    return O.OracleModel(CFG, tw), O.OracleModel(CFG, dw)


def test_causal_attention_brute_force():
    rng = np.random.default_rng(3)
    L, S, hq, hkv, D = 5, 4, 4, 2, 8
    q = rng.normal(size=(S, hq, D))
    K = rng.normal(size=(L + S, hkv, D))
    V = rng.normal(size=(L + S, hkv, D))
    got = T.causal_block_attention(q, K, V, L)
    for i in range(S):
        for j in range(hq):
            kv = j * hkv // hq
            n = L + i + 1
            s = np.array([q[i, j] @ K[t, kv] / np.sqrt(D) for t in range(n)])
            w = np.exp(s - s.max())
            w /= w.sum()
            ref = sum(w[t] * V[t, kv] for t in range(n))
            assert np.allclose(got[i, j], ref, atol=1e-12)


def test_tap_layers():
    assert T.tap_layers(8) == [1, 2, 4, 5, 6]
    for L in range(7, 40):
        t = T.tap_layers(L)
        assert t[0] == 1 and t[-1] == L - 2 and all(a < b for a, b in zip(t, t[1:]))


def test_chunked_prompt_equals_token_by_token(models):
    tm, _ = models
    prompt = prompt_tokens(CFG, 0, 37)
    a = T.OracleTarget(tm, NL, 64)
    b = T.OracleTarget(tm, NL, 64)
    pa = a.prefill(prompt, chunk=16)
    pb = b.prefill(prompt, chunk=1)
    assert np.allclose(pa["last"]["logits"][-1], pb["last"]["logits"][-1], rtol=0, atol=1e-10)
    assert np.allclose(bf16_f(pa["feats_bf16"]), bf16_f(pb["feats_bf16"]), atol=0.02)
    for l in range(NL):
        assert np.allclose(a.K[l][:37], b.K[l][:37], atol=1e-10)


def bf16_f(x):
    return O.bf16_to_f64(x)


def test_taps_are_the_residual_stream_after_the_tap_layers(models):
    tm, _ = models
    toks = prompt_tokens(CFG, 1, 6)
    t = T.OracleTarget(tm, NL, 16)
    out = t.forward(toks)
    h = tm.embed_rows(toks)
    z = np.zeros((0, CFG.n_kv_heads, CFG.head_dim))
    for l in range(NL):
        h, _, _ = T.target_layer(tm, l, h, 0, z, z)
        if l in t.taps:
            assert np.allclose(out["feats"][:, t.taps.index(l)], h, atol=1e-12)
    assert np.array_equal(out["tok"], np.argmax(O.lm_head_logits(tm, h), -1))


@pytest.mark.parametrize("mode", ["drafter", "perfect", "corrupt"])
def test_speculative_output_is_the_greedy_output(models, mode):
    tm, dm = models
    prompt = prompt_tokens(CFG, 2, 40)
    n_new = 48
    greedy, _ = T.greedy_generate(T.OracleTarget(tm, NL, 160), prompt, n_new)
    draft_fn = None
    if mode != "drafter":
        def draft_fn(out, b0, _g=greedy):
            # the greedy continuation after b0 (tau = S each round), or with one
            # wrong token at a position that moves from round to round
            k = len(out)
            d = np.array([_g[k + i] if k + i < len(_g) else 0 for i in range(CFG.block - 1)])
            if mode == "corrupt":
                j = (k * 7) % (CFG.block - 1)
                d[j] = (d[j] + 1) % (CFG.vocab - 1)
            return d
    drafter = O.OracleDrafter(dm)
    req = O.OracleRequest(CFG, 160)
    got, taus = T.spec_generate(drafter, req, T.OracleTarget(tm, NL, 160), prompt, n_new, CFG.block, draft_fn)
    assert np.array_equal(got, greedy)
    assert all(1 <= t <= CFG.block for t in taus)
    if mode == "perfect":
        assert all(t == CFG.block for t in taus[:-1])
    if mode == "corrupt":
        assert max(taus) > 1 and min(taus) < CFG.block


def test_planted_mistake_breaks_losslessness(models, monkeypatch):
    """A bonus taken from the next position (an off-by-one in the accept rule)
    makes the speculative output differ from the greedy one."""
    tm, dm = models

    def wrong_accept(draft, target):
        nd = len(draft)
        match = (np.asarray(draft) == np.asarray(target[:nd])).astype(np.int64)
        n = int(np.cumprod(match).sum())
        return n + 1, int(target[min(n + 1, nd)])
    monkeypatch.setattr(T, "accept_longest_prefix", wrong_accept)
    prompt = prompt_tokens(CFG, 3, 20)
    greedy, _ = T.greedy_generate(T.OracleTarget(tm, NL, 120), prompt, 20)
    got, _ = T.spec_generate(O.OracleDrafter(dm), O.OracleRequest(CFG, 120), T.OracleTarget(tm, NL, 120),
                             prompt, 20, CFG.block)
    assert not np.array_equal(got, greedy)


TEMP = 1.0


@pytest.mark.parametrize("mode", ["drafter", "perfect", "corrupt"])
def test_sampled_speculative_output_is_the_targets_sampled_output(models, mode):
    """At temperature 1 the verify step compares the block with the target's
    sampled tokens ([Code walkthrough] §三 第3步).  With the target's draws
    keyed by position, every emitted token is the target's own draw for its
    position given the same prefix, so speculative sampling emits exactly the
    target's own sampled decoding for the same seed, whatever the drafts."""
    tm, dm = models
    prompt = prompt_tokens(CFG, 4, 33)
    n_new, seed = 48, 77
    plain, _ = T.greedy_generate(T.OracleTarget(tm, NL, 160), prompt, n_new, TEMP, seed, slot=3)
    greedy, _ = T.greedy_generate(T.OracleTarget(tm, NL, 160), prompt, n_new)
    assert not np.array_equal(plain, greedy)  # the draws are not the argmax
    draft_fn = None
    if mode != "drafter":
        def draft_fn(out, b0, _g=plain):
            k = len(out)
            d = np.array([_g[k + i] if k + i < len(_g) else 0 for i in range(CFG.block - 1)])
            if mode == "corrupt":
                j = (k * 5) % (CFG.block - 1)
                d[j] = (d[j] + 1) % (CFG.vocab - 1)
            return d
    got, taus = T.spec_generate(O.OracleDrafter(dm), O.OracleRequest(CFG, 160), T.OracleTarget(tm, NL, 160), prompt,
                                n_new, CFG.block, draft_fn, temperature=TEMP, seed=seed, slot=3)
    assert np.array_equal(got, plain)
    if mode == "perfect":
        assert all(t == CFG.block for t in taus[:-1])
    if mode == "corrupt":
        assert max(taus) > 1 and min(taus) < CFG.block


def test_sampled_decoding_tends_to_greedy_as_temperature_vanishes(models):
    tm, _ = models
    prompt = prompt_tokens(CFG, 5, 20)
    cold, _ = T.greedy_generate(T.OracleTarget(tm, NL, 80), prompt, 24, 1e-9, 5)
    greedy, _ = T.greedy_generate(T.OracleTarget(tm, NL, 80), prompt, 24)
    assert np.array_equal(cold, greedy)


def test_target_draws_keyed_by_round_break_losslessness(models, monkeypatch):
    """Planted mistake: the target's stream keyed by the row within the block
    (as the drafter's is) instead of the position -- then a position's draw
    depends on where the block starts, and speculative sampling no longer
    reproduces the target's own sampled decoding."""
    import oracle.sampling_ref as SR
    tm, dm = models

    def by_row(z, temperature, seed, slot, pos0):
        d, mg = [], []
        for i in range(z.shape[0]):
            idx, m = SR.sample_row(z[i], temperature, SR.stream_key(seed, SR.TARGET, slot, i))
            d.append(idx)
            mg.append(m)
        return np.array(d, dtype=np.int64), np.array(mg)
    monkeypatch.setattr(SR, "sample_target_rows", by_row)
    prompt = prompt_tokens(CFG, 4, 33)
    plain, _ = T.greedy_generate(T.OracleTarget(tm, NL, 160), prompt, 40, TEMP, 77, slot=3)

    def draft_fn(out, b0):  # the plain sampled continuation, so blocks are accepted past row 0
        k = len(out)
        return np.array([plain[k + i] if k + i < len(plain) else 0 for i in range(CFG.block - 1)])
    got, _ = T.spec_generate(O.OracleDrafter(dm), O.OracleRequest(CFG, 160), T.OracleTarget(tm, NL, 160), prompt,
                             40, CFG.block, draft_fn, temperature=TEMP, seed=77, slot=3)
    assert not np.array_equal(got, plain)

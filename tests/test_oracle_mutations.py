"""Plant plausible mistakes in the CPU oracle and check that a pin catches each.

Every mutation replaces one oracle function (on the CPU, for the duration of
one test) with a subtly wrong variant -- a flipped sign, a dropped term, a
wrong index -- and runs the pins that cover it; at least one must fail.
"""
import numpy as np
import pytest

import oracle
import oracle.dflash_ref as R
import tests.test_oracle_pins as P


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(R, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _fails(*tests):
    for t in tests:
        try:
            t()
        except AssertionError:
            return True
    return False


def _rope_sign(x, pos, theta):
    D = x.shape[-1]
    h = D // 2
    inv = theta ** (-(2.0 * np.arange(h)) / D)
    a = np.asarray(pos, float)[:, None] * inv
    c, s = np.cos(a)[:, None], np.sin(a)[:, None]
    return np.concatenate([x[..., :h] * c + x[..., h:] * s, x[..., h:] * c - x[..., :h] * s], -1)


def _rope_interleaved(x, pos, theta):
    D = x.shape[-1]
    inv = theta ** (-(2.0 * np.arange(D // 2)) / D)
    a = np.asarray(pos, float)[:, None] * inv
    c, s = np.cos(a)[:, None], np.sin(a)[:, None]
    e, o = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = e * c - o * s
    out[..., 1::2] = o * c + e * s
    return out


def _attn_gqa_modulo(q, K, V):
    S, hq, D = q.shape
    hkv = K.shape[1]
    out = np.empty_like(q)
    for j in range(hq):
        kv = j % hkv
        s = q[:, j] @ K[:, kv].T / np.sqrt(D)
        out[:, j] = R.softmax(s) @ V[:, kv]
    return out


def _attn_scale_d(q, K, V):
    S, hq, D = q.shape
    hkv = K.shape[1]
    out = np.empty_like(q)
    for j in range(hq):
        kv = (j * hkv) // hq
        out[:, j] = R.softmax(q[:, j] @ K[:, kv].T / D) @ V[:, kv]
    return out


def _attn_causal_block(q, K, V):
    S, hq, D = q.shape
    hkv = K.shape[1]
    n = K.shape[0]
    out = np.empty_like(q)
    mask = np.arange(n)[None, :] > (n - S + np.arange(S))[:, None]
    for j in range(hq):
        kv = (j * hkv) // hq
        s = q[:, j] @ K[:, kv].T / np.sqrt(D)
        s = np.where(mask, -np.inf, s)
        out[:, j] = R.softmax(s) @ V[:, kv]
    return out


def _rms_no_mean(x, g, eps):
    return x / np.sqrt(np.sum(x * x, -1, keepdims=True) + eps) * g


def _rms_eps_outside(x, g, eps):
    return x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps) * g


def _accept_bonus_shift(draft, target):
    m = (np.asarray(draft[:15]) == np.asarray(target[:15])).astype(int)
    n = int(np.cumprod(m).sum())
    return n + 1, int(target[min(n + 1, 15)])


def _accept_count_all(draft, target):
    m = (np.asarray(draft[:15]) == np.asarray(target[:15])).astype(int)
    n = int(m.sum())
    return n + 1, int(target[n])


def _fuse_reversed(model, feats):
    cfg = model.cfg
    x = feats if feats.dtype == np.float64 else R.bf16_to_f64(feats)
    x = x[:, ::-1].reshape(x.shape[0], -1)
    return R.rmsnorm(x @ model.w("fc").T, model.w("fc_norm"), cfg.rms_eps)


def _fuse_no_gain(model, feats):
    cfg = model.cfg
    x = feats if feats.dtype == np.float64 else R.bf16_to_f64(feats)
    x = x.reshape(x.shape[0], -1)
    return R.rmsnorm(x @ model.w("fc").T, 1.0, cfg.rms_eps)


def _inject_normed_c(model, layer, c, pos):
    c2 = R.rmsnorm(c, model.w("in_norm", layer), model.cfg.rms_eps)
    return _ORIG_INJECT(model, layer, c2, pos)


def _inject_v_roped(model, layer, c, pos):
    k, v = _ORIG_INJECT(model, layer, c, pos)
    return k, R.rope(v, pos, model.cfg.rope_theta)


_ORIG_INJECT = R.inject_kv
_ORIG_LAYER = R.decoder_layer


def _layer_post_uses_in_gain(model, layer, h, pos, ck, cv):
    class W:
        def __init__(s, m):
            s.m, s.cfg, s.raw = m, m.cfg, m.raw

        def w(s, name, l=None):
            return s.m.w("in_norm" if name == "post_norm" else name, l)
    return _ORIG_LAYER(W(model), layer, h, pos, ck, cv)


def _layer_no_qnorm(model, layer, h, pos, ck, cv):
    class W:
        def __init__(s, m):
            s.m, s.cfg, s.raw = m, m.cfg, m.raw

        def w(s, name, l=None):
            if name == "q_norm":
                return np.full(s.cfg.head_dim, 1.0)
            return s.m.w(name, l)
    return _ORIG_LAYER(W(model), layer, h, pos, ck, cv)


_ORIG_LM = R.lm_head_logits


def _lm_no_final_norm(model, h, chunk=1 << 14):
    return h @ model.w("embed").T


def _lm_untied(model, h, chunk=1 << 14):
    """lm_head with a table other than the embedding (rows in reverse order)."""
    cfg = model.cfg
    hn = R.rmsnorm(h, model.w("final_norm"), cfg.rms_eps)
    return hn @ model.w("embed")[::-1].T


def _argmax_last(x):
    return x.shape[-1] - 1 - np.argmax(x[..., ::-1], axis=-1)


MUTATIONS = [
    ("rope", _rope_sign, [P.test_rope_complex_rotation_textbook]),
    ("rope", _rope_interleaved, [P.test_rope_complex_rotation_textbook]),
    ("block_attention", _attn_gqa_modulo,
     [lambda: P.test_attention_equals_library_sdpa_unmasked(37, 8, 2)]),
    ("block_attention", _attn_scale_d,
     [lambda: P.test_attention_equals_library_sdpa_unmasked(0, 4, 4)]),
    ("block_attention", _attn_causal_block,
     [P.test_attention_block_is_not_causal]),
    ("rmsnorm", _rms_no_mean, [P.test_rmsnorm_closed_form_and_library]),
    ("rmsnorm", _rms_eps_outside, [P.test_rmsnorm_closed_form_and_library]),
    ("accept_longest_prefix", _accept_bonus_shift,
     [lambda: [P.test_accept_golden(c) for c in P._load_accept_cases()]]),
    ("accept_longest_prefix", _accept_count_all,
     [lambda: [P.test_accept_golden(c) for c in P._load_accept_cases()]]),
    ("fuse_features", _fuse_reversed, [P.test_fusion_selects_layers_shallow_to_deep]),
    ("fuse_features", _fuse_no_gain, [P.test_fusion_selects_layers_shallow_to_deep]),
    ("inject_kv", _inject_normed_c, [P.test_inject_k_norm_and_rope_properties]),
    ("inject_kv", _inject_v_roped, [P.test_inject_k_norm_and_rope_properties]),
    ("decoder_layer", _layer_post_uses_in_gain, [P.test_decoder_layer_matches_library_assembly]),
    ("decoder_layer", _layer_no_qnorm, [P.test_decoder_layer_matches_library_assembly]),
    ("lm_head_logits", _lm_no_final_norm, [P.test_lm_head_equals_library_rms_norm_and_linear]),
    ("lm_head_logits", _lm_untied, [P.test_lm_head_is_tied_to_the_embedding]),
    ("argmax_first", _argmax_last, [P.test_argmax_ties_go_to_lowest_id]),
]


def _draft_variant(rows_from=1, b0_shift=0, fill=None):
    """OracleDrafter.draft with one planted slip: drafts from rows
    rows_from..rows_from+S-2, the block one position later, or the mask rows
    replaced by another token."""
    def draft(self, req, last_tok, want_logits=True):
        cfg = self.cfg
        S = cfg.block
        tokens = np.array([last_tok] + [cfg.mask_id if fill is None else fill] * (S - 1))
        h = self.model.embed_rows(tokens)
        pos = np.arange(req.ctx_len + b0_shift, req.ctx_len + b0_shift + S)
        for l in range(cfg.n_layers):
            ck, cv = req.ctx(l)
            h = R.decoder_layer(self.model, l, h, pos, ck, cv)
        logits = R.lm_head_logits(self.model, h[rows_from:rows_from + S - 1])
        top2 = np.partition(logits, -2, axis=-1)[:, -2:]
        out = {"draft": R.argmax_first(logits).astype(np.int64), "hidden": h, "margin": top2[:, 1] - top2[:, 0]}
        if want_logits:
            out["logits"] = logits
        return out
    return draft


DRAFT_PINS = [lambda: P.test_draft_block_rows_with_identity_layers(16), P.test_draft_block_positions_closed_form]
DRAFT_MUTATIONS = [
    ("rows 0..S-2", _draft_variant(rows_from=0)),
    ("b0 at L+1", _draft_variant(b0_shift=1)),
    ("b0 at L-1", _draft_variant(b0_shift=-1)),
    ("masks dropped", _draft_variant(fill=0)),
]


@pytest.mark.parametrize("label,fn", DRAFT_MUTATIONS, ids=[m[0] for m in DRAFT_MUTATIONS])
def test_planted_draft_block_mistake_is_caught(monkeypatch, label, fn):
    monkeypatch.setattr(R.OracleDrafter, "draft", fn)
    assert _fails(*DRAFT_PINS), f"no pin caught the planted mistake: {label}"


def test_unmutated_draft_block_passes_its_pins():
    for pin in DRAFT_PINS:
        pin()


@pytest.mark.parametrize("name,fn,pins", MUTATIONS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, fn, pins):
    _patch(monkeypatch, name, fn)
    assert _fails(*pins), f"no pin caught the planted mistake {fn.__name__} in {name}"

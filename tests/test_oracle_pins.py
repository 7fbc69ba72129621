"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks an oracle function against something other than itself:
the pages' stated acceptance semantics (golden cases), closed forms,
invariants, brute-force loops on tiny inputs, or a library routine that the
special case reduces to.  None of these tests needs a GPU.
"""
import itertools
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from workload import get_config, make_weights, feature_rows
from workload.gen import splitmix64_bits, f64_to_bf16_bits, bf16_bits_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ------------------------------------------------------------------ generator

def test_splitmix64_published_vector():
    # SplitMix64 reference outputs for initial state 1234567.
    got = splitmix64_bits(1234567, np.arange(5)).tolist()
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, 1.0 + 2 ** -9])
    b = f64_to_bf16_bits(x)
    back = bf16_bits_to_f32(b).astype(np.float64)
    # 1+2^-8 is a tie between 1 and 1+2^-7: even mantissa (1.0) wins;
    # 1+3*2^-8 ties between 1+2^-7 and 1+2^-6 -> 1+2^-6 (even).
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 0.0, 1.0]


# ------------------------------------------------------------------ a7 accept

def _brute_accept(draft, target):
    """Scan from the block head until the first mismatch (no cumprod)."""
    i = 0
    while i < len(draft) and draft[i] == target[i]:
        i += 1
    return i + 1, target[i]


def _load_accept_cases():
    cases = []
    with open(os.path.join(GOLDEN, "accept_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, d, t, tau, bonus = [s.strip() for s in line.split("|")]
            cases.append((name, [int(x) for x in d.split()], [int(x) for x in t.split()],
                          int(tau), int(bonus)))
    return cases


@pytest.mark.parametrize("case", _load_accept_cases(), ids=lambda c: c[0])
def test_accept_golden(case):
    _, d, t, tau, bonus = case
    assert O.accept_longest_prefix(np.array(d), np.array(t)) == (tau, bonus)


def test_accept_exhaustive_all_masks():
    """All 2^15 match patterns: cumprod form == first-mismatch scan, tau in [1,16]."""
    base = np.arange(100, 115)
    for bits in range(1 << 15):
        mism = np.array([(bits >> i) & 1 for i in range(15)], dtype=bool)
        target = np.concatenate([np.where(mism, base + 1000, base), [7]])
        tau, bonus = O.accept_longest_prefix(base, target)
        assert (tau, bonus) == _brute_accept(base, target)
        assert 1 <= tau <= 16


@pytest.mark.parametrize("S", [2, 8, 10])
def test_accept_exhaustive_smaller_blocks(S):
    """Inference at a smaller block S ([Paper walkthrough] Results): all 2^(S-1)
    match patterns against the first-mismatch scan, tau in [1, S], and the
    stand-in target has S tokens."""
    base = np.arange(100, 100 + S - 1)
    for bits in range(1 << (S - 1)):
        mism = np.array([(bits >> i) & 1 for i in range(S - 1)], dtype=bool)
        target = np.concatenate([np.where(mism, base + 1000, base), [7]])
        tau, bonus = O.accept_longest_prefix(base, target)
        assert (tau, bonus) == _brute_accept(base, target)
        assert 1 <= tau <= S
    t = O.synthetic_target(base, np.ones(S, bool), np.zeros(S, np.int64), 4096)
    assert t.shape == (S,) and O.accept_longest_prefix(base, t)[0] == S


def test_accept_mean_closed_form():
    """With i.i.d. matches of probability p, E[tau] = (1 - p^16) / (1 - p)."""
    p, R = 0.8, 40000
    r = np.random.default_rng(7)
    draft = np.arange(15)
    taus = []
    for _ in range(R):
        m = r.random(16) < p
        u = r.integers(0, 4096, 16)
        t = O.synthetic_target(draft, m, u, 4096)
        taus.append(O.accept_longest_prefix(draft, t)[0])
    expect = (1 - p ** 16) / (1 - p)
    se = np.std(taus) / np.sqrt(R)
    assert abs(np.mean(taus) - expect) < 5 * se


def test_synthetic_target_depends_only_on_matches():
    V = 50
    r = np.random.default_rng(3)
    for _ in range(500):
        m = r.random(16) < 0.7
        u = r.integers(0, V, 16)
        d1 = r.integers(0, V, 15)
        d2 = r.integers(0, V, 15)
        t1 = O.synthetic_target(d1, m, u, V)
        t2 = O.synthetic_target(d2, m, u, V)
        lead = 0
        while lead < 15 and m[lead]:
            lead += 1
        assert O.accept_longest_prefix(d1, t1)[0] == lead + 1
        assert O.accept_longest_prefix(d2, t2)[0] == lead + 1
        for i in range(15):
            assert (t1[i] == d1[i]) == bool(m[i])
            assert 0 <= t1[i] < V


# ------------------------------------------------------------------ norms, rope

def test_rmsnorm_closed_form_and_library():
    x = rng.standard_normal((7, 33)) * 3.0
    g = 1.0 + 0.1 * rng.standard_normal(33)
    y = O.rmsnorm(x, g, 0.0)
    # RMS of y/g is exactly 1 with eps = 0
    np.testing.assert_allclose(np.sqrt(np.mean((y / g) ** 2, -1)), 1.0, rtol=1e-12)
    # scale invariance
    np.testing.assert_allclose(O.rmsnorm(5.0 * x, g, 0.0), y, rtol=1e-12)
    # torch's RMSNorm routine
    ref = F.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rmsnorm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-14)


def test_rope_complex_rotation_textbook():
    """Rotate-half RoPE == complex multiply of (x_i + j x_{i+D/2}) by exp(j p theta^(-2i/D))."""
    D, theta = 16, 1e4
    x = rng.standard_normal((5, 3, D))
    pos = np.array([0, 1, 7, 100, 12345])
    got = O.rope(x, pos, theta)
    z = x[..., :D // 2] + 1j * x[..., D // 2:]
    w = np.exp(1j * pos[:, None, None] * theta ** (-np.arange(D // 2) * 2.0 / D))
    r = z * w
    np.testing.assert_allclose(got, np.concatenate([r.real, r.imag], -1), rtol=1e-12, atol=1e-12)


def test_rope_identity_norm_relative():
    D, theta = 64, 1e6
    x = rng.standard_normal((4, 2, D))
    np.testing.assert_array_equal(O.rope(x, np.zeros(4), theta), x)
    y = O.rope(x, np.array([3, 50, 999, 32000]), theta)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    dots = [np.sum(O.rope(q, np.array([m + s]), theta) * O.rope(k, np.array([n + s]), theta))
            for (m, n, s) in [(10, 3, 0), (10, 3, 500), (10, 3, 30000)]]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ------------------------------------------------------------------ a5 attention

def _brute_attention(q, K, V):
    S, hq, D = q.shape
    n, hkv, _ = K.shape
    out = np.zeros_like(q)
    for j in range(hq):
        kv = j // (hq // hkv)
        for i in range(S):
            s = [sum(q[i, j, d] * K[t, kv, d] for d in range(D)) / np.sqrt(D) for t in range(n)]
            mx = max(s)
            e = [np.exp(x - mx) for x in s]
            z = sum(e)
            for d in range(D):
                out[i, j, d] = sum(e[t] * V[t, kv, d] for t in range(n)) / z
    return out


def test_attention_bruteforce_tiny():
    q = rng.standard_normal((4, 4, 8))
    K = rng.standard_normal((9, 2, 8))
    V = rng.standard_normal((9, 2, 8))
    np.testing.assert_allclose(O.block_attention(q, K, V), _brute_attention(q, K, V), rtol=1e-11)


@pytest.mark.parametrize("L,hq,hkv", [(0, 4, 4), (0, 8, 2), (37, 8, 2), (130, 8, 1)])
def test_attention_equals_library_sdpa_unmasked(L, hq, hkv):
    S, D = 16, 32
    q = rng.standard_normal((S, hq, D))
    K = rng.standard_normal((L + S, hkv, D))
    V = rng.standard_normal((L + S, hkv, D))
    rep = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(rep, 0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(rep, 0)
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=False).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(O.block_attention(q, K, V), ref, rtol=1e-10, atol=1e-12)


def test_attention_context_permutation_invariant():
    q = rng.standard_normal((16, 4, 16))
    K = rng.standard_normal((50, 2, 16))
    V = rng.standard_normal((50, 2, 16))
    p = rng.permutation(50)
    np.testing.assert_allclose(O.block_attention(q, K[p], V[p]), O.block_attention(q, K, V),
                               rtol=1e-10)


def test_attention_block_is_not_causal():
    """The first block row must see the last block key (no causal mask)."""
    q = rng.standard_normal((16, 2, 8))
    K = rng.standard_normal((16, 2, 8))
    V = rng.standard_normal((16, 2, 8))
    V2 = V.copy()
    V2[15] += 10.0
    a = O.block_attention(q, K, V)
    b = O.block_attention(q, K, V2)
    assert np.abs(a[0] - b[0]).max() > 1e-3


def test_attention_rope_shift_invariance():
    """Shifting all positions (context and block) by a constant leaves attention unchanged."""
    D, theta = 32, 1e6
    q = rng.standard_normal((16, 4, D))
    k = rng.standard_normal((16 + 40, 2, D))
    v = rng.standard_normal((16 + 40, 2, D))
    pk = np.arange(56)
    pq = np.arange(40, 56)
    a = O.block_attention(O.rope(q, pq, theta), O.rope(k, pk, theta), v)
    b = O.block_attention(O.rope(q, pq + 777, theta), O.rope(k, pk + 777, theta), v)
    np.testing.assert_allclose(a, b, rtol=1e-8, atol=1e-10)


# ------------------------------------------------------------------ a1 fusion

def test_fusion_selects_layers_shallow_to_deep():
    cfg = get_config("tiny").with_(gain_std=0.1)
    w = make_weights(cfg)
    H = cfg.hidden
    feats = feature_rows(cfg, 0, 0, 6)
    ff = O.bf16_to_f64(feats)
    for layer in (0, 4):
        fc = np.zeros((H, 5 * H))
        fc[:, layer * H:(layer + 1) * H] = np.eye(H)
        w2 = dict(w)
        w2["fc"] = f64_to_bf16_bits(fc)
        m = O.OracleModel(cfg, w2)
        c = O.fuse_features(m, feats)
        ref = F.rms_norm(torch.from_numpy(ff[:, layer]), (H,),
                         torch.from_numpy(m.w("fc_norm")), eps=cfg.rms_eps).numpy()
        np.testing.assert_allclose(c, ref, rtol=1e-12, atol=1e-12)


def test_fusion_feature_scale_invariance():
    cfg = get_config("tiny")
    m = O.OracleModel(cfg, make_weights(cfg))
    f = O.bf16_to_f64(feature_rows(cfg, 0, 3, 4))
    # equal up to the eps term: relative change <= eps / (2 * mean square)
    np.testing.assert_allclose(O.fuse_features(m, 8.0 * f), O.fuse_features(m, f), rtol=1e-5)


# ------------------------------------------------------------------ a2 inject

def test_inject_k_norm_and_rope_properties():
    cfg = get_config("tiny-gains")
    m = O.OracleModel(cfg, make_weights(cfg))
    c = rng.standard_normal((5, cfg.hidden))
    k0, v0 = O.inject_kv(m, 1, c, np.zeros(5))
    # at position 0 RoPE is the identity: the k-normed vector divided by its
    # gain has RMS 1 (up to eps)
    g = m.w("k_norm", 1)
    rms = np.sqrt(np.mean((k0 / g) ** 2, -1))
    np.testing.assert_allclose(rms, 1.0, rtol=1e-4)
    k1, v1 = O.inject_kv(m, 1, c, np.arange(5) + 1000)
    np.testing.assert_allclose(np.linalg.norm(k1, axis=-1), np.linalg.norm(k0, axis=-1), rtol=1e-12)
    np.testing.assert_array_equal(v0, v1)
    # V is the plain projection by the layer's V rows
    D, hq, hkv = cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    wv = m.w("wqkv", 1)[(hq + hkv) * D:]
    np.testing.assert_allclose(v0.reshape(5, -1), c @ wv.T, rtol=1e-12)


# ------------------------------------------------------------------ a4 layer

def _torch_layer(m, l, h, pos, ck, cv):
    """The same pre-norm layer assembled from torch library routines (fp64)."""
    cfg = m.cfg
    hq, hkv, D, I = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.intermediate
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    h = T(h)
    x = F.rms_norm(h, (cfg.hidden,), T(m.w("in_norm", l)), eps=cfg.rms_eps)
    qkv = F.linear(x, T(m.w("wqkv", l)))
    S = h.shape[0]
    q = qkv[:, :hq * D].view(S, hq, D)
    k = qkv[:, hq * D:(hq + hkv) * D].view(S, hkv, D)
    v = qkv[:, (hq + hkv) * D:].view(S, hkv, D)
    q = F.rms_norm(q, (D,), T(m.w("q_norm", l)), eps=cfg.rms_eps)
    k = F.rms_norm(k, (D,), T(m.w("k_norm", l)), eps=cfg.rms_eps)

    def rot(t, p):  # complex-number form of RoPE
        z = torch.complex(t[..., :D // 2], t[..., D // 2:])
        ang = T(np.asarray(p, dtype=np.float64))[:, None, None] * \
            cfg.rope_theta ** (-torch.arange(D // 2, dtype=torch.float64) * 2.0 / D)
        r = z * torch.polar(torch.ones_like(ang), ang)
        return torch.cat([r.real, r.imag], -1)

    q, k = rot(q, pos), rot(k, pos)
    K = torch.cat([T(ck), k], 0).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    Vv = torch.cat([T(cv), v], 0).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2), K, Vv).permute(1, 0, 2).reshape(S, -1)
    h = h + F.linear(o, T(m.w("wo", l)))
    y = F.rms_norm(h, (cfg.hidden,), T(m.w("post_norm", l)), eps=cfg.rms_eps)
    gu = F.linear(y, T(m.w("w_gate_up", l)))
    h = h + F.linear(F.silu(gu[:, :I]) * gu[:, I:], T(m.w("w_down", l)))
    return h.numpy()


def test_decoder_layer_matches_library_assembly():
    cfg = get_config("tiny-gains")
    m = O.OracleModel(cfg, make_weights(cfg))
    h = rng.standard_normal((16, cfg.hidden))
    L = 21
    ck = rng.standard_normal((L, cfg.n_kv_heads, cfg.head_dim))
    cv = rng.standard_normal((L, cfg.n_kv_heads, cfg.head_dim))
    pos = np.arange(L, L + 16)
    np.testing.assert_allclose(O.decoder_layer(m, 1, h, pos, ck, cv),
                               _torch_layer(m, 1, h, pos, ck, cv), rtol=1e-9, atol=1e-11)


def test_decoder_layer_residual_structure():
    """With W_o = 0 and W_down = 0 the layer is the identity on h."""
    cfg = get_config("tiny")
    w = make_weights(cfg)
    w["layers"][0] = dict(w["layers"][0])
    w["layers"][0]["wo"] = np.zeros_like(w["layers"][0]["wo"])
    w["layers"][0]["w_down"] = np.zeros_like(w["layers"][0]["w_down"])
    m = O.OracleModel(cfg, w)
    h = rng.standard_normal((16, cfg.hidden))
    ck = np.zeros((0, cfg.n_kv_heads, cfg.head_dim))
    np.testing.assert_array_equal(O.decoder_layer(m, 0, h, np.arange(16), ck, ck), h)


# ------------------------------------------------------------------ a6 lm_head

def test_argmax_ties_go_to_lowest_id():
    x = np.array([[0.0, 3.0, 3.0, 1.0], [-1.0, -1.0, -2.0, -1.0], [0.0, -0.0, 0.0, -5.0]])
    assert O.argmax_first(x).tolist() == [1, 0, 0]


def test_lm_head_equals_library_rms_norm_and_linear():
    """a6 logits against torch's own RMSNorm and linear layer in float64, the
    table widened from the bf16 bits by torch (not by the oracle), with
    non-unit final gains and a chunk size that leaves a ragged last chunk."""
    cfg = get_config("tiny-gains")
    w = make_weights(cfg)
    m = O.OracleModel(cfg, w)
    h = rng.standard_normal((15, cfg.hidden)) * 3.0
    got = O.lm_head_logits(m, h, chunk=1000)
    bits = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).double()
    E, g = bits(w["embed"]), bits(w["final_norm"])
    want = F.linear(F.rms_norm(torch.from_numpy(h), (cfg.hidden,), weight=g, eps=cfg.rms_eps), E).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)


def test_lm_head_is_tied_to_the_embedding():
    """The lm_head is the embedding table itself ([Code walkthrough] 二.3,
    [Paper walkthrough] 设计: the drafter reuses the target's embedding and
    LM head): a hidden state equal to token v's embedding row scores v
    highest, because a random row's product with itself (|E_v|^2) dwarfs its
    products with the other rows (about |E_v| |E_u| / sqrt(H))."""
    cfg = get_config("tiny")
    w = make_weights(cfg)
    m = O.OracleModel(cfg, w)
    ids = np.array([0, 1, 17, 1000, 2048, cfg.vocab - 2, cfg.mask_id])
    logits = O.lm_head_logits(m, O.bf16_to_f64(w["embed"][ids]))
    assert O.argmax_first(logits).tolist() == ids.tolist()


# ------------------------------------------------------------------ a3-a6 draft block

def _identity_layers(cfg):
    """Weights whose every layer adds nothing to the residual stream (W_o = 0,
    W_down = 0), so the block's hidden states stay its embedding rows."""
    w = make_weights(cfg)
    w["layers"] = [dict(lw, wo=np.zeros_like(lw["wo"]), w_down=np.zeros_like(lw["w_down"])) for lw in w["layers"]]
    return w


@pytest.mark.parametrize("S", [16, 8])
def test_draft_block_rows_with_identity_layers(S):
    """Block = [last verified token, (S-1) x mask] ([Code walkthrough] 二.1:
    1 known token + 15 masks -> 15 candidates), drafts from rows 1..S-1.
    With identity layers the hidden state of row 0 is b0's embedding and of
    every other row the mask's; the drafts are then the lm_head's top id of
    the mask row (the mask id itself, the table being tied), never b0."""
    cfg = get_config("tiny").with_(block=S)
    w = _identity_layers(cfg)
    m = O.OracleModel(cfg, w)
    dr = O.OracleDrafter(m)
    req = O.OracleRequest(cfg, 64 + S)
    dr.fuse_inject(req, feature_rows(cfg, 0, 0, 64))
    b0 = 17
    out = dr.draft(req, b0)
    E = O.bf16_to_f64(w["embed"])
    np.testing.assert_array_equal(out["hidden"][0], E[b0])
    for i in range(1, S):
        np.testing.assert_array_equal(out["hidden"][i], E[cfg.mask_id])
    assert out["logits"].shape == (S - 1, cfg.vocab)
    assert out["draft"].tolist() == [cfg.mask_id] * (S - 1)


def _pos2d_model(S, eps):
    """A hand-built one-layer drafter in two dimensions: hidden 2, one head of
    dimension 2 (a single RoPE pair rotating by `position` radians), W_q, W_k,
    W_v, W_o and the fusion projection the identity, the MLP zero, all gains
    one.  Every weight is exact in bf16."""
    from workload.configs import DraftConfig
    cfg = DraftConfig(name="pos2d", hidden=2, n_q_heads=1, n_kv_heads=1, head_dim=2, intermediate=2, n_layers=1,
                      vocab=4, rope_theta=10000.0, batch=1, ctx0=3, rounds=1, match_p=0.5, n_fused=1, block=S,
                      rms_eps=eps)
    b = lambda a: f64_to_bf16_bits(np.asarray(a, dtype=np.float64))
    eye = np.eye(2)
    w = {"embed": b([[0.25, -1.0], [1.0, 0.5], [-2.0, 0.75], [-0.5, 1.0]]),
         "fc": b(eye), "fc_norm": b([1.0, 1.0]), "final_norm": b([1.0, 1.0]),
         "layers": [{"wqkv": b(np.vstack([eye, eye, eye])), "wo": b(eye), "w_gate_up": b(np.zeros((4, 2))),
                     "w_down": b(np.zeros((2, 2))), "in_norm": b([1.0, 1.0]), "post_norm": b([1.0, 1.0]),
                     "q_norm": b([1.0, 1.0]), "k_norm": b([1.0, 1.0])}]}
    return cfg, w


def test_draft_block_positions_closed_form():
    """Where the block sits: the context's keys at positions 0..L-1 and the
    block's rows at L..L+S-1, b0 at L (the reading that the block follows
    the confirmed context), all of them seen by every block row (no mask,
    [Code walkthrough] 二.2).  On the two-dimensional model every rotation is
    a plane rotation by the position in radians, so the layer's output is
    written out here with explicit rotation matrices and the softmax over
    scalar scores; drafts are the lm_head's choices for rows 1..S-1."""
    S, L, eps = 4, 3, 1e-6
    cfg, w = _pos2d_model(S, eps)
    dr = O.OracleDrafter(O.OracleModel(cfg, w))
    req = O.OracleRequest(cfg, L + S)
    x = np.array([[[0.5, 2.0]], [[-1.5, 0.25]], [[1.0, 1.0]]])  # three context features [L, 1, 2]
    dr.fuse_inject(req, x)
    b0 = 2
    out = dr.draft(req, b0)

    n = lambda v: v / np.sqrt(np.mean(v * v) + eps)
    rot = lambda a: np.array([[np.cos(a), -np.sin(a)], [np.sin(a), np.cos(a)]])
    E = O.bf16_to_f64(w["embed"])
    c = [n(x[j, 0]) for j in range(L)]                        # fused context features
    keys = [rot(j) @ n(c[j]) for j in range(L)]              # k-norm, then RoPE at position j
    vals = [c[j] for j in range(L)]
    toks = [b0] + [cfg.mask_id] * (S - 1)
    h = [E[t] for t in toks]
    xs = [n(v) for v in h]                                   # input norm
    keys += [rot(L + i) @ n(xs[i]) for i in range(S)]        # block keys at L..L+S-1
    vals += [xs[i] for i in range(S)]
    want = []
    for i in range(S):
        q = rot(L + i) @ n(xs[i])
        s = np.array([q @ k for k in keys]) / np.sqrt(2.0)
        p = np.exp(s - s.max())
        p /= p.sum()
        want.append(h[i] + sum(pj * vj for pj, vj in zip(p, vals)))
    want = np.array(want)
    np.testing.assert_allclose(out["hidden"], want, rtol=1e-12, atol=1e-12)
    drafts = [int(np.argmax(E @ n(want[i]))) for i in range(1, S)]
    assert out["draft"].tolist() == drafts


# ------------------------------------------------------------------ whole round

def _run_rounds(cfg, rounds, req_id=0, keep=None):
    from workload import match_stream, context_lengths
    w = make_weights(cfg)
    m = O.OracleModel(cfg, w)
    dr = O.OracleDrafter(m)
    L0 = int(context_lengths(cfg)[req_id])
    req = O.OracleRequest(cfg, L0 + 16 * (rounds + 1))
    dr.fuse_inject(req, feature_rows(cfg, req_id, 0, L0))
    last, hist = cfg.first_token, []
    pending = 0
    for r in range(rounds):
        if pending:
            dr.fuse_inject(req, feature_rows(cfg, req_id, req.ctx_len, pending))
        if keep is not None:
            keep.append([k[:req.ctx_len].copy() for k in req.K])
        out = dr.draft(req, last, want_logits=False)
        mm, uu = match_stream(cfg, r, [req_id])
        t = O.synthetic_target(out["draft"], mm[0], uu[0], cfg.vocab)
        tau, bonus, conf = dr.accept_trim(req, out["draft"], t)
        hist.append((tau, bonus, conf, out["draft"].copy()))
        last, pending = bonus, tau
    return req, hist


def test_round_invariants_and_persistence():
    cfg = get_config("tiny")
    snaps = []
    req, hist = _run_rounds(cfg, 5, keep=snaps)
    L = cfg.ctx0
    for (tau, bonus, conf, d) in hist:
        assert 1 <= tau <= 16
        assert conf == L + tau
        assert d.shape == (15,) and d.min() >= 0 and d.max() < cfg.vocab
        L = conf
    # context K written before a round is byte-identical after later rounds
    for i, snap in enumerate(snaps):
        for l in range(cfg.n_layers):
            np.testing.assert_array_equal(req.K[l][:snap[l].shape[0]], snap[l])


def test_round_tau_independent_of_drafts():
    """Under the stand-in verify, tau follows the match stream alone."""
    from workload import match_stream
    cfg = get_config("tiny")
    _, hist = _run_rounds(cfg, 6)
    for r, (tau, *_rest) in enumerate(hist):
        mm, _ = match_stream(cfg, r, [0])
        lead = 0
        while lead < 15 and mm[0][lead]:
            lead += 1
        assert tau == lead + 1


@pytest.mark.parametrize("name", ["tiny-gains", "small", "small-batch"])
def test_test_shapes_draft_diverse_ids(name):
    """The parity test shapes must draft varied ids (not one dominant token),
    otherwise the token comparisons would check little."""
    from tests.gpu_util import OracleRun
    cfg = get_config(name)
    o = OracleRun(cfg, 2)
    o.prefill()
    for _ in range(2):
        for od in o.round(want_logits=False):
            assert len(set(od["draft"].tolist())) >= 2

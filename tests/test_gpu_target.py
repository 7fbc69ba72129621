"""Target model (verify step) and speculative generation through the C ABI,
against the float64 oracle (oracle/target_ref.py)."""
import math

import numpy as np
import pytest

import oracle as O
import oracle.target_ref as T
from tests.gpu_util import MARGIN, TOL_REL_L2, rel_l2, to_np
from workload import get_config, make_target_weights, make_weights, prompt_tokens

pytestmark = pytest.mark.gpu

NL = 8  # target layers


def _handles(cfg, cap=256, attn_impl=0):
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    mpps = math.ceil(cap / 64) + 1
    tw, dw = make_target_weights(cfg, NL), make_weights(cfg)
    t = Drafter(cfg, weights_to_device(tw), max_batch=1, max_slots=2, max_pages=2 * mpps, max_pages_per_slot=mpps,
                max_rows=16, attn_impl=attn_impl, role=1)
    d = Drafter(cfg, weights_to_device(dw), max_batch=1, max_slots=2, max_pages=2 * mpps, max_pages_per_slot=mpps,
                max_rows=16, attn_impl=attn_impl)
    return t, d, O.OracleModel(cfg, tw), O.OracleModel(cfg, dw)


@pytest.mark.parametrize("attn_impl", [1, 2], ids=["attn-warp-mma", "attn-tcgen05"])
@pytest.mark.parametrize("name", ["tiny-gains", "small"])
def test_verify_block_matches_oracle(lib, name, attn_impl):
    """Every row's token, the tapped features and the cache, chunk by chunk
    over a 40-token prompt (causal within each chunk, the last chunk ragged)."""
    import torch
    cfg = get_config(name)
    t, _, tm, _ = _handles(cfg, attn_impl=attn_impl)
    ot = T.OracleTarget(tm, NL, 256)
    prompt = prompt_tokens(cfg, 0, 40)
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    slots = torch.tensor([1], **i32)
    tokens = torch.zeros(1, 16, **i32)
    out = torch.zeros(1, 16, **i32)
    nv = torch.zeros(1, **i32)
    feats = torch.zeros(1, 16, cfg.n_fused * cfg.hidden, dtype=torch.bfloat16, device=dev)
    for p0 in range(0, len(prompt), 16):
        chunk = prompt[p0:p0 + 16]
        n = len(chunk)
        tokens.zero_()
        tokens[0, :n] = torch.tensor(chunk, dtype=torch.int32)
        nv.fill_(n)
        t.verify_block(slots, tokens, out, nv, feats)
        t.advance(slots, nv)
        o = ot.forward(chunk)
        ot.advance(n)
        got = to_np(out)[0, :n]
        strong = o["margin"] > MARGIN
        assert np.array_equal(got[strong], o["tok"][strong]), (p0, got, o["tok"], o["margin"])
        f = to_np(feats)[0, :n].reshape(n, cfg.n_fused, cfg.hidden)
        assert rel_l2(f, o["feats"]) < TOL_REL_L2, p0
    L = len(prompt)
    assert int(to_np(t.slot_lengths(slots))[0]) == L
    for l in (0, NL - 1):
        k, v = t.read_kv(l, 1, 0, L)
        assert rel_l2(to_np(k), ot.K[l][:L]) < TOL_REL_L2 and rel_l2(to_np(v), ot.V[l][:L]) < TOL_REL_L2, l
    assert t.read_status() == 0


def _first_weak(margins, thr=MARGIN):
    weak = np.nonzero(np.asarray(margins) <= thr)[0]
    return int(weak[0]) if weak.size else len(margins)


@pytest.mark.parametrize("mode", ["drafter", "perfect", "corrupt"])
def test_speculative_generation_is_the_greedy_output(lib, mode):
    """The speculative output equals the target's own greedy decoding: on the
    GPU (same kernels, token by token) and against the oracle's greedy tokens
    up to its first near-tie."""
    from block_diffusion_speculative_hiddens_gb300.session import SpecDecoder, greedy_generate
    cfg = get_config("tiny-gains")
    t, d, tm, _ = _handles(cfg)
    prompt = prompt_tokens(cfg, 1, 40)
    n_new = 48
    og, om = T.greedy_generate(T.OracleTarget(tm, NL, 256), prompt, n_new)
    gg = greedy_generate(t, prompt, n_new, slot=0)
    k = _first_weak(om)
    assert gg[:k] == og[:k].tolist()
    override = None
    if mode != "drafter":
        def override(out, b0, _g=gg):
            kk = len(out)
            dd = [_g[kk + i] if kk + i < len(_g) else 0 for i in range(cfg.block - 1)]
            if mode == "corrupt":
                j = (kk * 7) % (cfg.block - 1)
                dd[j] = (dd[j] + 1) % (cfg.vocab - 1)
            return dd
    sd = SpecDecoder(d, t, slot=1)
    got = sd.generate(prompt, n_new, override)
    assert got == gg, (got, gg, sd.taus)
    if mode == "perfect":
        assert all(x == cfg.block for x in sd.taus[:-1])
    if mode == "corrupt":
        assert max(sd.taus) > 1
    assert t.read_status() == 0 and d.read_status() == 0


@pytest.mark.parametrize("mode", ["drafter", "perfect", "corrupt"])
def test_sampled_speculative_generation_is_the_targets_sampled_output(lib, mode):
    """At temperature 1 (drafts drawn from the drafter's softmax, the target's
    tokens sampled by position with dflash_verify_block_sample) the
    speculative output equals the target's own sampled decoding for the same
    seed and slot: on the GPU token by token, and against the oracle's
    sampled tokens up to its first near-tie of the perturbed scores."""
    from block_diffusion_speculative_hiddens_gb300.session import SpecDecoder, greedy_generate
    cfg = get_config("tiny-gains")
    t, d, tm, _ = _handles(cfg)
    prompt = prompt_tokens(cfg, 1, 40)
    n_new, temp, seed = 48, 1.0, 99
    gs = greedy_generate(t, prompt, n_new, slot=1, temperature=temp, seed=seed)
    t.reset_slot(1)
    gg = greedy_generate(t, prompt, n_new, slot=1)
    t.reset_slot(1)
    assert gs != gg  # the draws are not the argmax
    os_, om = T.greedy_generate(T.OracleTarget(tm, NL, 256), prompt, n_new, temp, seed, slot=1)
    k = _first_weak(om, MARGIN / temp)
    assert k > 0 and gs[:k] == os_[:k].tolist()
    override = None
    if mode != "drafter":
        def override(out, b0, _g=gs):
            kk = len(out)
            dd = [_g[kk + i] if kk + i < len(_g) else 0 for i in range(cfg.block - 1)]
            if mode == "corrupt":
                j = (kk * 5) % (cfg.block - 1)
                dd[j] = (dd[j] + 1) % (cfg.vocab - 1)
            return dd
    sd = SpecDecoder(d, t, slot=1, temperature=temp, seed=seed)
    got = sd.generate(prompt, n_new, override)
    assert got == gs, (got, gs, sd.taus)
    if mode == "perfect":
        assert all(x == cfg.block for x in sd.taus[:-1])
    if mode == "corrupt":
        assert max(sd.taus) > 1
    assert t.read_status() == 0 and d.read_status() == 0


def test_verify_sample_temperature_edges(lib):
    """T below 1e-6 is the argmax; a negative or NaN T is refused."""
    import torch
    from block_diffusion_speculative_hiddens_gb300.binding import DflashError
    cfg = get_config("tiny-gains")
    t, _, _, _ = _handles(cfg)
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    slots = torch.tensor([0], **i32)
    tokens = torch.tensor([prompt_tokens(cfg, 2, 16).tolist()], **i32)
    a, b = torch.zeros(1, 16, **i32), torch.zeros(1, 16, **i32)
    t.verify_block(slots, tokens, a)
    t.verify_block_sample(slots, tokens, b, 1e-9, 5)
    assert np.array_equal(to_np(a), to_np(b))
    for bad in (-1.0, float("nan")):
        with pytest.raises(DflashError):
            t.verify_block_sample(slots, tokens, b, bad, 5)
    assert t.read_status() == 0


def test_verify_block_batch_of_two_with_ragged_chunks(lib):
    """Two requests verified together, their last chunks of different lengths
    (37 and 33 prompt tokens): every request matches its own oracle."""
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    cfg = get_config("tiny-gains")
    tw = make_target_weights(cfg, NL)
    mpps = 8
    t = Drafter(cfg, weights_to_device(tw), max_batch=2, max_slots=2, max_pages=2 * mpps, max_pages_per_slot=mpps,
                max_rows=16, role=1)
    tm = O.OracleModel(cfg, tw)
    prompts = [prompt_tokens(cfg, 4, 37), prompt_tokens(cfg, 5, 33)]
    ots = [T.OracleTarget(tm, NL, 128) for _ in prompts]
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    slots = torch.tensor([0, 1], **i32)
    tokens = torch.zeros(2, 16, **i32)
    out = torch.zeros(2, 16, **i32)
    nv = torch.zeros(2, **i32)
    feats = torch.zeros(2, 16, cfg.n_fused * cfg.hidden, dtype=torch.bfloat16, device=dev)
    for p0 in range(0, 37, 16):
        chunks = [p[p0:p0 + 16] for p in prompts]
        tokens.zero_()
        for b, ch in enumerate(chunks):
            tokens[b, :len(ch)] = torch.tensor(ch, dtype=torch.int32)
            nv[b] = len(ch)
        t.verify_block(slots, tokens, out, nv, feats)
        t.advance(slots, nv)
        for b, ch in enumerate(chunks):
            o = ots[b].forward(ch)
            ots[b].advance(len(ch))
            n = len(ch)
            got = to_np(out)[b, :n]
            strong = o["margin"] > MARGIN
            assert np.array_equal(got[strong], o["tok"][strong]), (p0, b)
            f = to_np(feats)[b, :n].reshape(n, cfg.n_fused, cfg.hidden)
            assert rel_l2(f, o["feats"]) < TOL_REL_L2, (p0, b)
    lens = to_np(t.slot_lengths(slots))
    assert lens.tolist() == [37, 33]
    for b in range(2):
        k, v = t.read_kv(NL - 1, b, 0, int(lens[b]))
        assert rel_l2(to_np(k), ots[b].K[NL - 1][:lens[b]]) < TOL_REL_L2, b
    assert t.read_status() == 0


def test_drafter_calls_refused_on_a_target_handle(lib):
    """A target handle has no fusion weights: the injection and folded-round
    calls refuse it (DFLASH_ERR_INVALID_ARG) instead of reading an unpacked
    fusion block, and nothing is queued."""
    import torch
    from block_diffusion_speculative_hiddens_gb300.binding import DflashError
    cfg = get_config("tiny-gains")
    t, _, _, _ = _handles(cfg)
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    slots = torch.tensor([0], **i32)
    feats = torch.zeros(1, 16, cfg.n_fused * cfg.hidden, dtype=torch.bfloat16, device=dev)
    n_new = torch.tensor([4], **i32)
    for call in (lambda: t.fuse_inject(slots, feats, 16, n_new),
                 lambda: t.fuse_inject_noalloc(slots, feats, 16, n_new),
                 lambda: t.draft_round(slots, feats, 16, n_new, torch.ones(1, **i32), torch.zeros(1, 15, **i32))):
        with pytest.raises(DflashError) as e:
            call()
        assert e.value.code == 1
    assert to_np(t.slot_lengths(slots))[0] == 0
    assert t.read_status() == 0

"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import numpy as np
import pytest

import oracle as O
from tests.gpu_util import GpuRun, OracleRun, TOL_REL_L2, check_drafts, rel_l2, to_np
from workload import get_config, make_weights

pytestmark = pytest.mark.gpu

SMALL = ["tiny", "tiny-gains", "small", "small-batch"]


def _pair(name, rounds, attn_impl=0, **kw):
    cfg = get_config(name)
    w = make_weights(cfg)
    g = GpuRun(cfg, rounds, weights_np=w, attn_impl=attn_impl, **kw)
    o = OracleRun(cfg, rounds, weights_np=w, **kw)
    g.prefill()
    o.prefill()
    return cfg, g, o


@pytest.mark.parametrize("name", SMALL)
def test_inject_kv_matches_oracle(lib, name):
    cfg, g, o = _pair(name, 1)
    for j in range(len(g.ids)):
        L = int(g.ctx0[j])
        for l in range(cfg.n_layers):
            k, v = g.d.read_kv(l, j, 0, L)
            ok, ov = o.reqs[j].ctx(l)
            assert rel_l2(to_np(k), ok) < TOL_REL_L2, (name, j, l)
            assert rel_l2(to_np(v), ov) < TOL_REL_L2, (name, j, l)
            # every position, not just the aggregate
            kk = to_np(k).reshape(L, -1)
            err = np.linalg.norm(kk - ok.reshape(L, -1), axis=1) / np.linalg.norm(ok.reshape(L, -1), axis=1)
            assert err.max() < 3 * TOL_REL_L2
    assert g.d.read_status() == 0


# attention page loops: 1 warp MMAs, 2 tcgen05 (the default picks by capacity)
ATTN = [pytest.param(1, id="attn-warp-mma"), pytest.param(2, id="attn-tcgen05")]


@pytest.mark.parametrize("attn_impl", ATTN)
@pytest.mark.parametrize("name", SMALL)
def test_draft_round_matches_oracle(lib, name, attn_impl):
    cfg, g, o = _pair(name, 2, attn_impl=attn_impl)
    for r in range(2):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            # hidden states after the last layer (all 16 block rows)
            assert rel_l2(go["hidden"][j], od["hidden"]) < TOL_REL_L2
            # logits of rows 1..15
            assert rel_l2(go["logits"][j, 1:], od["logits"]) < TOL_REL_L2
            # fused argmax == argmax of the same kernel's materialised logits
            assert np.array_equal(go["draft"][j], np.argmax(go["logits"][j, 1:], -1))
            check_drafts(go["draft"][j], od)
            assert go["tau"][j] == od["tau"]
            assert go["ctx"][j] == od["ctx"]
            assert go["bonus"][j] == od["bonus"]
    assert g.d.read_status() == 0


@pytest.mark.parametrize("attn_impl", ATTN)
@pytest.mark.parametrize("folded", [False, True], ids=["separate", "folded"])
@pytest.mark.parametrize("name,rounds", [("tiny", 8), ("small-batch", 4)])
def test_rounds_accept_bit_exact(lib, name, rounds, folded, attn_impl):
    cfg, g, o = _pair(name, rounds, attn_impl=attn_impl)
    for r in range(rounds):
        go = g.round(folded=folded)
        oo = o.round(want_logits=False)
        for j, od in enumerate(oo):
            assert 1 <= go["tau"][j] <= 16
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
            check_drafts(go["draft"][j], od)
    lens = to_np(g.d.slot_lengths(g.state.slots))
    # the last round's accepted features are injected by the next round
    assert np.array_equal(lens + to_np(g.state.accept_len), [od["ctx"] for od in oo])


def test_batch16_round_matches_oracle(lib):
    """256 block tokens: every GEMM of the round (and the prefill's fusion and
    injection GEMMs, 128+ rows) shares its token tile across a cluster."""
    cfg, g, o = _pair("small-b16", 2)
    for j in range(len(g.ids)):
        L = int(g.ctx0[j])
        k, v = g.d.read_kv(1, j, 0, L)
        ok, ov = o.reqs[j].ctx(1)
        assert rel_l2(to_np(k), ok) < TOL_REL_L2 and rel_l2(to_np(v), ov) < TOL_REL_L2, j
    for r in range(2):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            assert rel_l2(go["hidden"][j], od["hidden"]) < TOL_REL_L2, (r, j)
            assert rel_l2(go["logits"][j, 1:], od["logits"]) < TOL_REL_L2, (r, j)
            assert np.array_equal(go["draft"][j], np.argmax(go["logits"][j, 1:], -1))
            check_drafts(go["draft"][j], od)
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
    assert g.d.read_status() == 0


@pytest.mark.parametrize("attn_impl", ATTN)
def test_global_merge_round_matches_oracle(lib, attn_impl):
    """More attention splits than clusters fit at once: the splits' partials
    are merged through global memory by a second kernel."""
    cfg, g, o = _pair("small-long", 2, attn_impl=attn_impl)
    plan = g.d.plan()
    if plan["attn_merge"] != "global" and attn_impl == 1:
        pytest.skip(f"the warp-MMA page loop's clusters all fit at once here: {plan}")
    assert plan["attn_merge"] == "global" and plan["attn_splits"] > 1, plan
    for r in range(2):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            assert rel_l2(go["hidden"][j], od["hidden"]) < TOL_REL_L2, (r, j)
            assert rel_l2(go["logits"][j, 1:], od["logits"]) < TOL_REL_L2, (r, j)
            check_drafts(go["draft"][j], od)
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
    assert g.d.read_status() == 0


@pytest.mark.parametrize("name", ["tiny-gains", "small-batch", "small-b16"])
def test_fp8_weights_round_matches_oracle(lib, name):
    """FP8 E4M3 weights with per-row scales (converted to f16 in the SM before
    each MMA) against the oracle computing with the same dequantised weights:
    injected K/V, hidden states, logits, drafts and acceptance."""
    cfg, g, o = _pair(name, 2, weight_fp8=1)
    for j in range(len(g.ids)):
        L = int(g.ctx0[j])
        k, v = g.d.read_kv(0, j, 0, L)
        ok, ov = o.reqs[j].ctx(0)
        assert rel_l2(to_np(k), ok) < TOL_REL_L2 and rel_l2(to_np(v), ov) < TOL_REL_L2, j
    for r in range(2):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            assert rel_l2(go["hidden"][j], od["hidden"]) < TOL_REL_L2, (r, j)
            assert rel_l2(go["logits"][j, 1:], od["logits"]) < TOL_REL_L2, (r, j)
            assert np.array_equal(go["draft"][j], np.argmax(go["logits"][j, 1:], -1))
            check_drafts(go["draft"][j], od)
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
    assert g.d.read_status() == 0


@pytest.mark.parametrize("T", [0.7, 1.5])
@pytest.mark.parametrize("name", ["tiny-gains", "small-batch"])
def test_sampled_drafts_match_oracle(lib, name, T):
    """Temperature > 0: each draft is the Gumbel-max draw from softmax(logits / T).

    The kernel's draw equals the host's Gumbel-max on the same kernel's logits
    with the oracle's generator (an independent implementation of the same
    published function) wherever the perturbed scores are not within float32
    rounding of a tie, and the oracle's own draw wherever its perturbed
    margin exceeds the logits' tolerance; acceptance stays bit-exact."""
    import oracle.sampling_ref as SR
    from tests.gpu_util import MARGIN
    cfg = get_config(name)
    w = make_weights(cfg)
    g = GpuRun(cfg, 3, weights_np=w, temperature=T, seed=4321)
    o = OracleRun(cfg, 3, weights_np=w, temperature=T, seed=4321)
    g.prefill()
    o.prefill()
    differs = 0
    for r in range(3):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            dh, mh = SR.sample_drafts(go["logits"][j, 1:].astype(np.float64), T, 4321, j, r)
            sure = mh > 1e-3
            assert np.array_equal(go["draft"][j][sure], dh[sure]), (r, j)
            check_drafts(go["draft"][j], od, margin=MARGIN / T)
            differs += int(np.sum(go["draft"][j] != np.argmax(go["logits"][j, 1:], -1)))
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
    assert differs > 0  # the draws are not the greedy argmax
    assert g.d.read_status() == 0


def test_sampling_temperature_edges(lib):
    """T below 1e-6 is the greedy argmax; a negative or NaN T is refused."""
    import torch
    from block_diffusion_speculative_hiddens_gb300.binding import DflashError
    cfg = get_config("tiny-gains")
    w = make_weights(cfg)
    a = GpuRun(cfg, 1, weights_np=w)
    b = GpuRun(cfg, 1, weights_np=w)
    a.prefill()
    b.prefill()
    da = a.round()["draft"]
    s = b.state
    rc = torch.zeros(1, dtype=torch.int32, device=b.dev)
    s.inject()
    b.d.draft_block_sample(s.slots, s.bonus, 1e-9, 7, rc, s.draft)
    assert np.array_equal(to_np(s.draft).astype(np.int64), da)
    for bad in (-0.5, float("nan")):
        with pytest.raises(DflashError):
            b.d.draft_block_sample(s.slots, s.bonus, bad, 7, rc, s.draft)
    assert b.d.read_status() == 0


# inference at blocks smaller than the trained 16: S-1 drafts, acceptance over S
SMALLER_BLOCKS = ["tiny-b8", "small-batch-b10"]


@pytest.mark.parametrize("attn_impl", ATTN)
@pytest.mark.parametrize("name", SMALLER_BLOCKS)
def test_smaller_block_round_matches_oracle(lib, name, attn_impl):
    cfg, g, o = _pair(name, 2, attn_impl=attn_impl)
    S = cfg.block
    assert S < 16
    for r in range(2):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            assert go["draft"][j].shape == (S - 1,)
            assert rel_l2(go["hidden"][j], od["hidden"]) < TOL_REL_L2
            assert rel_l2(go["logits"][j, 1:], od["logits"]) < TOL_REL_L2
            assert np.array_equal(go["draft"][j], np.argmax(go["logits"][j, 1:], -1))
            check_drafts(go["draft"][j], od)
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"])
    assert g.d.read_status() == 0


@pytest.mark.parametrize("folded", [False, True], ids=["separate", "folded"])
@pytest.mark.parametrize("name,rounds", [("tiny-b8", 8), ("small-batch-b10", 4)])
def test_smaller_block_rounds_and_cache(lib, name, rounds, folded):
    """Acceptance bit-exact over several rounds, and the cache afterwards holds
    exactly the oracle's context K/V: the padding rows of a smaller block are
    never written to it."""
    cfg, g, o = _pair(name, rounds)
    for r in range(rounds):
        go = g.round(folded=folded)
        oo = o.round(want_logits=False)
        for j, od in enumerate(oo):
            assert 1 <= go["tau"][j] <= cfg.block
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
            check_drafts(go["draft"][j], od)
    lens = to_np(g.d.slot_lengths(g.state.slots))
    for j in range(len(g.ids)):
        L = int(lens[j])
        for l in range(cfg.n_layers):
            k, v = g.d.read_kv(l, j, 0, L)
            ok, ov = o.reqs[j].ctx(l)
            assert rel_l2(to_np(k), ok[:L]) < TOL_REL_L2 and rel_l2(to_np(v), ov[:L]) < TOL_REL_L2, (j, l)
    assert g.d.read_status() == 0


@pytest.mark.parametrize("name", ["tiny-gains", "small-batch"])
def test_folded_round_equals_separate_calls(lib, name):
    """dflash_draft_round (K/V injection inside each layer's QKV GEMM) against
    dflash_fuse_inject + dflash_draft_block on the same inputs: the same
    acceptance every round, and the same injected K/V up to the fp32
    summation order of a differently split reduction."""
    cfg = get_config(name)
    w = make_weights(cfg)
    a = GpuRun(cfg, 4, weights_np=w)
    b = GpuRun(cfg, 4, weights_np=w)
    a.prefill()
    b.prefill()
    for r in range(4):
        ea = a.round(folded=True)
        eb = b.round(folded=False)
        for key in ("tau", "bonus", "ctx"):
            assert np.array_equal(ea[key], eb[key]), (r, key)
    for j in range(len(a.ids)):
        L = int(to_np(a.d.slot_lengths(a.state.slots))[j])
        for l in range(cfg.n_layers):
            ka, va = a.d.read_kv(l, j, 0, L)
            kb, vb = b.d.read_kv(l, j, 0, L)
            assert rel_l2(to_np(ka), to_np(kb)) < 1e-3 and rel_l2(to_np(va), to_np(vb)) < 1e-3, (j, l)
    assert a.d.read_status() == 0 and b.d.read_status() == 0


def test_context_kv_unchanged_by_later_rounds(lib):
    cfg, g, o = _pair("small", 4)
    L = int(g.ctx0[0])
    before = [tuple(to_np(t).copy() for t in g.d.read_kv(l, 0, 0, L)) for l in range(cfg.n_layers)]
    for _ in range(4):
        g.round()
    for l in range(cfg.n_layers):
        k, v = g.d.read_kv(l, 0, 0, L)
        assert np.array_equal(to_np(k), before[l][0]) and np.array_equal(to_np(v), before[l][1])


def test_graph_replay_equals_eager(lib):
    import torch
    from block_diffusion_speculative_hiddens_gb300.session import run_round
    cfg = get_config("small-batch")
    w = make_weights(cfg)
    a = GpuRun(cfg, 4, weights_np=w)
    b = GpuRun(cfg, 4, weights_np=w)
    a.prefill()
    b.prefill()
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        b.d.graph_begin(st)
        run_round(b.state, b.verify, st)
        nk = b.d.graph_end(st)
    assert nk >= 5
    for _ in range(4):
        ea = a.round()
        with torch.cuda.stream(st):
            b.d.graph_launch(st)
        st.synchronize()
        s = b.state
        for key, t in (("draft", s.draft), ("tau", s.accept_len), ("bonus", s.bonus), ("ctx", s.ctx_len)):
            assert np.array_equal(ea[key], to_np(t).astype(np.int64)), key


def test_batch_invariance(lib):
    """Each request of a batch behaves as the same request run alone.

    Accept lengths and lengths are bit-exact; drafts follow the margin rule
    against the oracle (the split-KV count depends on the batch size, so the
    attention's summation order may differ between the two runs)."""
    cfg = get_config("small-batch")
    w = make_weights(cfg)
    full = GpuRun(cfg, 3, weights_np=w)
    full.prefill()
    orc = OracleRun(cfg, 3, weights_np=w)
    orc.prefill()
    res_full = [full.round() for _ in range(3)]
    res_orc = [orc.round(want_logits=False) for _ in range(3)]
    for b in range(cfg.batch):
        one = GpuRun(cfg, 3, weights_np=w, batch_ids=[b])
        one.prefill()
        for r in range(3):
            ro = one.round()
            assert ro["tau"][0] == res_full[r]["tau"][b] == res_orc[r][b]["tau"]
            assert ro["ctx"][0] == res_full[r]["ctx"][b] == res_orc[r][b]["ctx"]
            check_drafts(ro["draft"][0], res_orc[r][b])
            check_drafts(res_full[r]["draft"][b], res_orc[r][b])


@pytest.mark.parametrize("S", [16, 10, 8, 2])
def test_accept_trim_exhaustive_patterns(lib, S):
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    cfg = get_config("tiny").with_(block=S)
    d = Drafter(cfg, weights_to_device(make_weights(cfg)), max_batch=64, max_slots=64, max_pages=64,
                max_pages_per_slot=1, max_rows=64)
    rng = np.random.default_rng(5)
    for rep in range(40):
        B = 64 if rep % 2 else int(rng.integers(1, 65))
        draft = rng.integers(0, 7, (B, S - 1)).astype(np.int32)
        target = rng.integers(0, 7, (B, S)).astype(np.int32)
        # force structured patterns: all right, all wrong, single mismatch at k
        for b in range(B):
            kind = (rep * 64 + b) % (S + 2)
            if kind == 0:
                target[b, :S - 1] = draft[b]
            elif kind == 1:
                target[b, :S - 1] = draft[b] + 1
            elif kind < S + 1:
                target[b, :S - 1] = draft[b]
                if kind - 2 < S - 1:
                    target[b, kind - 2] = draft[b, kind - 2] + 1
        dev = torch.device("cuda:0")
        T = lambda a: torch.from_numpy(a).to(dev)
        slots = torch.arange(B, dtype=torch.int32, device=dev)
        acc = torch.zeros(B, dtype=torch.int32, device=dev)
        bon = torch.zeros_like(acc)
        ctx = torch.zeros_like(acc)
        d.accept_trim(slots, T(draft), T(target), acc, bon, ctx)
        acc, bon, ctx = to_np(acc), to_np(bon), to_np(ctx)
        for b in range(B):
            tau, bonus = O.accept_longest_prefix(draft[b], target[b])
            assert (acc[b], bon[b], ctx[b]) == (tau, bonus, tau)
    assert d.read_status() == 0


def test_edge_cases_and_errors(lib):
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    from block_diffusion_speculative_hiddens_gb300.binding import DflashError, DEV_ARG
    cfg = get_config("tiny")
    d = Drafter(cfg, weights_to_device(make_weights(cfg)), max_batch=2, max_slots=2, max_pages=8,
                max_pages_per_slot=4, max_rows=64)
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    empty = torch.zeros(0, **i32)
    d.draft_block(empty, empty, torch.zeros(0, 15, **i32))       # batch 0: no-op
    d.fuse_inject(empty, None, 0, empty)
    with pytest.raises(DflashError) as e:                         # batch > max_batch
        s3 = torch.arange(3, **i32)
        d.draft_block(s3, s3, torch.zeros(3, 15, **i32))
    assert e.value.code == 1
    with pytest.raises(DflashError) as e:                         # rows > max_rows
        d.fuse_inject(torch.arange(2, **i32), torch.zeros(2, 40, cfg.fused_dim, dtype=torch.bfloat16,
                                                          device=dev), 40, torch.zeros(2, **i32))
    assert e.value.code == 3
    # n_new beyond rows_per_req and an out-of-range slot are device-side errors, not faults
    feats = torch.zeros(1, 8, cfg.fused_dim, dtype=torch.bfloat16, device=dev)
    d.fuse_inject(torch.tensor([0], **i32), feats, 8, torch.tensor([9], **i32))
    assert d.read_status() & DEV_ARG
    d.fuse_inject(torch.tensor([5], **i32), feats, 8, torch.tensor([1], **i32))
    assert d.read_status() & DEV_ARG
    assert d.read_status() == 0                                   # cleared by the read
    # page capacity: 4 pages of 64 positions per slot
    big = torch.zeros(1, 64, cfg.fused_dim, dtype=torch.bfloat16, device=dev)
    for _ in range(4):
        d.fuse_inject(torch.tensor([1], **i32), big, 64, torch.tensor([64], **i32))
    st = d.read_status()
    assert st & 0x08  # DEV_CAPACITY: 256 positions + a 16-token block do not fit in 4 pages
    lens = to_np(d.slot_lengths(torch.tensor([0, 1], **i32)))
    assert lens[1] == 192  # the 4th chunk was refused, earlier ones kept
    d.reset_slot(1)
    assert to_np(d.slot_lengths(torch.tensor([1], **i32)))[0] == 0
    assert d.read_status() == 0
    # an out-of-range slot in a draft call is a device-side error too: the
    # request is computed from slot 0's lengths and written nowhere
    before = [to_np(t).copy() for t in d.read_kv(0, 0, 0, 64)]
    d.draft_block(torch.tensor([7], **i32), torch.tensor([1], **i32), torch.zeros(1, 15, **i32))
    assert d.read_status() & DEV_ARG
    after = [to_np(t) for t in d.read_kv(0, 0, 0, 64)]
    assert all(np.array_equal(x, y, equal_nan=True) for x, y in zip(before, after))


# attention shapes beyond the workloads': one query head per KV head, head_dim 64 with G = 4 and 8
ATTN_SHAPES = ["small-g1", "small-d64-g4", "small-d64-g8"]


@pytest.mark.parametrize("attn_impl", ATTN)
@pytest.mark.parametrize("name", ATTN_SHAPES)
def test_attention_shapes_round_matches_oracle(lib, name, attn_impl):
    cfg, g, o = _pair(name, 2, attn_impl=attn_impl)
    for j in range(len(g.ids)):
        L = int(g.ctx0[j])
        k, v = g.d.read_kv(1, j, 0, L)
        ok, ov = o.reqs[j].ctx(1)
        assert rel_l2(to_np(k), ok) < TOL_REL_L2 and rel_l2(to_np(v), ov) < TOL_REL_L2, j
    for r in range(2):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            assert rel_l2(go["hidden"][j], od["hidden"]) < TOL_REL_L2, (r, j)
            assert rel_l2(go["logits"][j, 1:], od["logits"]) < TOL_REL_L2, (r, j)
            assert np.array_equal(go["draft"][j], np.argmax(go["logits"][j, 1:], -1))
            strong, _ = check_drafts(go["draft"][j], od)
            assert strong >= 5, (r, j, strong)
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
    assert g.d.read_status() == 0


def test_misaligned_features_refused_before_anything_is_queued(lib):
    """Feature rows the TMA descriptor cannot address (not 16-byte aligned)
    are refused by the host-side check before the page allocation is queued:
    the slot's length and pages stay as they were."""
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    cfg = get_config("tiny")
    d = Drafter(cfg, weights_to_device(make_weights(cfg)), max_batch=1, max_slots=1, max_pages=8,
                max_pages_per_slot=8, max_rows=64)
    dev = torch.device("cuda:0")
    i32 = dict(dtype=torch.int32, device=dev)
    slot = torch.tensor([0], **i32)
    buf = torch.zeros(1, 9, cfg.fused_dim, dtype=torch.bfloat16, device=dev)
    d.fuse_inject(slot, buf[:, :8].contiguous(), 8, torch.tensor([8], **i32))
    torch.cuda.synchronize()
    before = to_np(d.slot_lengths(slot))[0]
    n_new = torch.tensor([4], **i32)
    rc = d.lib.dflash_fuse_inject(d.h, slot.data_ptr(), 1, buf.data_ptr() + 2, 4, n_new.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == 1  # DFLASH_ERR_INVALID_ARG
    rc = d.lib.dflash_fuse_inject_noalloc(d.h, slot.data_ptr(), 1, buf.data_ptr() + 2, 4, n_new.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == 1
    torch.cuda.synchronize()
    assert to_np(d.slot_lengths(slot))[0] == before == 8
    with pytest.raises(ValueError):  # the binding refuses it before the library sees it
        d.fuse_inject(slot, buf.view(-1)[1:1 + 4 * cfg.fused_dim].view(1, 4, cfg.fused_dim), 4, n_new)
    assert d.read_status() == 0


def test_bounded_wait_gives_up_and_reports(lib):
    """A bounded in-kernel wait on a barrier nothing arrives at gives up after
    its limit, sets DFLASH_DEV_TIMEOUT and returns; the context stays usable
    and a round afterwards matches the oracle."""
    import time
    from block_diffusion_speculative_hiddens_gb300.binding import DEV_TIMEOUT
    cfg, g, o = _pair("tiny-gains", 1)
    t0 = time.perf_counter()
    g.d.check_wait_timeout(2000)  # 2 ms
    st = g.d.read_status()
    dt = time.perf_counter() - t0
    assert st & DEV_TIMEOUT and dt < 5.0
    assert g.d.read_status() == 0  # cleared by the read
    go = g.round()
    od = o.round(want_logits=False)[0]
    assert (go["tau"][0], go["bonus"][0], go["ctx"][0]) == (od["tau"], od["bonus"], od["ctx"])
    check_drafts(go["draft"][0], od)
    assert g.d.read_status() == 0


def test_create_refuses_weights_beyond_f16(lib):
    """A weight the f16 copies cannot hold makes dflash_create fail with
    DFLASH_ERR_RANGE instead of silently holding inf; FP8 weights (per-row
    scales) take the same matrix."""
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    from block_diffusion_speculative_hiddens_gb300.binding import DflashError
    cfg = get_config("tiny")
    w = weights_to_device(make_weights(cfg))
    w["layers"][1]["wo"][3, 7] = 1.0e5
    kw = dict(max_batch=1, max_slots=1, max_pages=4, max_pages_per_slot=4, max_rows=16)
    with pytest.raises(DflashError) as e:
        Drafter(cfg, w, **kw)
    assert e.value.code == 7
    d = Drafter(cfg, w, weight_fp8=1, **kw)
    assert d.read_status() == 0


def test_batch32_rounds_inject_only_the_appended_rows(lib):
    """Batch 32: a round's injection covers 512 feature rows, more than one
    token tile, so the library gathers the appended rows (each request's
    accept_len first rows) and the fusion and injection GEMMs compute those
    alone.  Acceptance bit-exact over three rounds, hidden states and logits
    against the oracle, and afterwards every request's cache equal to the
    oracle's context K/V."""
    cfg, g, o = _pair("small-b32", 3)
    for r in range(3):
        go = g.round(debug=True)
        oo = o.round(want_logits=True)
        for j, od in enumerate(oo):
            assert rel_l2(go["hidden"][j], od["hidden"]) < TOL_REL_L2, (r, j)
            assert rel_l2(go["logits"][j, 1:], od["logits"]) < TOL_REL_L2, (r, j)
            check_drafts(go["draft"][j], od)
            assert (go["tau"][j], go["bonus"][j], go["ctx"][j]) == (od["tau"], od["bonus"], od["ctx"]), (r, j)
    assert len(set(int(t) for t in go["tau"])) > 3  # ragged acceptance: the gather matters
    lens = to_np(g.d.slot_lengths(g.state.slots))
    for j in range(len(g.ids)):
        L = int(lens[j])
        for l in range(cfg.n_layers):
            k, v = g.d.read_kv(l, j, 0, L)
            ok, ov = o.reqs[j].ctx(l)
            assert rel_l2(to_np(k), ok[:L]) < TOL_REL_L2 and rel_l2(to_np(v), ov[:L]) < TOL_REL_L2, (j, l)
    assert g.d.read_status() == 0

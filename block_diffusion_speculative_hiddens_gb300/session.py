"""Round driver over the C ABI: device-resident state for a batch of requests.

A round is fuse_inject(previous round's accepted features) -> draft_block ->
verify (the caller's target model, or the benchmark's stand-in) ->
accept_trim.  Every buffer that links one round to the next (accept_len,
bonus, confirmed length, block features) stays on the device, so a round --
or many -- can be captured once as a CUDA graph and replayed.
"""
from __future__ import annotations

import torch

from .binding import Drafter


class RoundState:
    def __init__(self, drafter: Drafter, batch: int, slots=None, first_token: int = 1):
        cfg = drafter.cfg
        dev = torch.device(f"cuda:{drafter.device}")
        i32 = dict(dtype=torch.int32, device=dev)
        self.d = drafter
        self.batch = batch
        self.slots = (torch.arange(batch, **i32) if slots is None
                      else torch.as_tensor(slots, dtype=torch.int32).to(dev))
        self.bonus = torch.full((batch,), first_token, **i32)    # next round's last verified token
        self.accept_len = torch.zeros(batch, **i32)              # next round's n_new
        self.ctx_len = torch.zeros(batch, **i32)                 # confirmed length after accept
        self.draft = torch.zeros(batch, cfg.block - 1, **i32)
        self.target = torch.zeros(batch, cfg.block, **i32)
        self.feats = torch.zeros(batch, cfg.block, cfg.n_fused * cfg.hidden, dtype=torch.bfloat16,
                                 device=dev)
        self.temperature = 0.0     # 0: greedy drafts
        self.seed = 0
        self.round_ctr = None      # device int32 round index read by the sampling draft

    def set_sampling(self, temperature: float, seed: int, round_ctr):
        """Draw drafts from softmax(logits / temperature); round_ctr is a device
        int32 the caller advances once per round (the stand-in verify does)."""
        self.temperature = float(temperature)
        self.seed = int(seed)
        self.round_ctr = round_ctr

    def prefill(self, feats, n_new, stream=None):
        """Inject prompt features: feats [batch, rows, n_fused*H] bf16, n_new [batch] int32 (device)."""
        self.d.fuse_inject(self.slots, feats, feats.shape[1], n_new, stream)

    def inject(self, stream=None):
        self.d.fuse_inject(self.slots, self.feats, self.d.cfg.block, self.accept_len, stream)

    def draft_block(self, stream=None):
        if self.temperature > 0:
            self.d.draft_block_sample(self.slots, self.bonus, self.temperature, self.seed, self.round_ctr,
                                      self.draft, None, stream)
        else:
            self.d.draft_block(self.slots, self.bonus, self.draft, stream)

    def draft_round(self, stream=None):
        """inject + draft_block as one call (injection folded into each layer's QKV GEMM)."""
        self.d.draft_round(self.slots, self.feats, self.d.cfg.block, self.accept_len, self.bonus, self.draft,
                           stream)

    def accept(self, stream=None):
        self.d.accept_trim(self.slots, self.draft, self.target, self.accept_len, self.bonus,
                           self.ctx_len, stream)


class SyntheticVerify:
    """Benchmark stand-in for the target's verify step (see dflash_harness_verify).

    match/offs: int32 [rounds, batch, block] device tensors drawn by the workload
    generator; feat_stream: [batch, rows, n_fused*H] bf16 device tensor of the
    target features of every position (or None to leave state.feats alone).
    """

    def __init__(self, state: RoundState, match, offs, feat_stream=None):
        self.s = state
        self.match = match.contiguous()
        self.offs = offs.contiguous()
        self.rounds_cap = match.shape[0]
        self.feat_stream = feat_stream
        self.round_ctr = torch.zeros(1, dtype=torch.int32, device=state.slots.device)

    def __call__(self, stream=None):
        s = self.s
        fs = self.feat_stream
        s.d.harness_verify(s.slots, s.draft, self.match, self.offs, self.rounds_cap, self.round_ctr,
                           s.target, fs, 0 if fs is None else fs.shape[1],
                           None if fs is None else s.feats, stream)


def run_round(state: RoundState, verify, stream=None, folded: bool = False):
    """One drafting-plus-acceptance round on the given stream.

    folded=False issues dflash_fuse_inject and dflash_draft_block (the faster
    order at batch 1 on GB300); True uses dflash_draft_round, which computes
    the injection inside the layers' QKV projections.
    """
    if folded:
        state.draft_round(stream)
    else:
        state.inject(stream)
        state.draft_block(stream)
    verify(stream)
    state.accept(stream)


class SpecDecoder:
    """Speculative generation for one request with a drafter handle and a
    target handle (role 1) of the same shape family: prefill both models in
    16-token chunks, then rounds of draft -> verify -> accept -> trim
    (dflash_draft_block, dflash_verify_block, dflash_accept_trim,
    dflash_advance, dflash_fuse_inject).  The output equals the target's own
    greedy decoding, or at temperature > 0 (drafts drawn from the drafter's
    softmax, the target's tokens sampled by position with
    dflash_verify_block_sample) the target's own sampled decoding for the same
    seed.  `draft_override(out, b0)` may supply the drafts instead of the
    drafter (tests that force long acceptances)."""

    def __init__(self, drafter: Drafter, target: Drafter, slot: int = 0, stream=None, temperature: float = 0.0,
                 seed: int = 0):
        cfg = drafter.cfg
        dev = torch.device(f"cuda:{drafter.device}")
        i32 = dict(dtype=torch.int32, device=dev)
        self.d, self.t, self.stream = drafter, target, stream
        self.S = cfg.block
        self.slots = torch.tensor([slot], **i32)
        self.tokens = torch.zeros(1, 16, **i32)
        self.out_tok = torch.zeros(1, 16, **i32)
        self.n_valid = torch.zeros(1, **i32)
        self.feats = torch.zeros(1, 16, cfg.n_fused * cfg.hidden, dtype=torch.bfloat16, device=dev)
        self.draft = torch.zeros(1, self.S - 1, **i32)
        self.accept_len = torch.zeros(1, **i32)
        self.bonus = torch.zeros(1, **i32)
        self.ctx = torch.zeros(1, **i32)
        self.rnd = torch.zeros(1, **i32)  # the drafter's round index (its draws' stream)
        self.temperature, self.seed = float(temperature), int(seed)
        self.taus = []

    def _verify(self, n_valid=None):
        if self.temperature > 0:
            self.t.verify_block_sample(self.slots, self.tokens, self.out_tok, self.temperature, self.seed, n_valid,
                                       self.feats, self.stream)
        else:
            self.t.verify_block(self.slots, self.tokens, self.out_tok, n_valid, self.feats, self.stream)

    def prefill(self, prompt) -> int:
        """Both models over the prompt; returns the target's greedy token after it."""
        prompt = [int(x) for x in prompt]
        s = self.stream
        n = 0
        for p0 in range(0, len(prompt), 16):
            chunk = prompt[p0:p0 + 16]
            n = len(chunk)
            self.tokens.zero_()
            self.tokens[0, :n] = torch.tensor(chunk, dtype=torch.int32)
            self.n_valid.fill_(n)
            self._verify(self.n_valid)
            self.d.fuse_inject(self.slots, self.feats, 16, self.n_valid, s)
            self.t.advance(self.slots, self.n_valid, s)
        return int(self.out_tok[0, n - 1].item())

    def generate(self, prompt, n_new: int, draft_override=None):
        s = self.stream
        b0 = self.prefill(prompt)
        out = [b0]
        self.bonus.fill_(b0)
        while len(out) < n_new:
            if draft_override is not None:
                self.draft.copy_(torch.as_tensor(draft_override(out, b0), dtype=torch.int32).view(1, -1))
            elif self.temperature > 0:
                self.rnd.fill_(len(self.taus))
                self.d.draft_block_sample(self.slots, self.bonus, self.temperature, self.seed, self.rnd, self.draft,
                                          None, s)
            else:
                self.d.draft_block(self.slots, self.bonus, self.draft, s)
            self.tokens[:, 0] = self.bonus
            self.tokens[:, 1:self.S] = self.draft
            self._verify()
            self.d.accept_trim(self.slots, self.draft, self.out_tok[:, :self.S].contiguous(), self.accept_len,
                               self.bonus, self.ctx, s)
            self.t.advance(self.slots, self.accept_len, s)
            self.d.fuse_inject(self.slots, self.feats, 16, self.accept_len, s)
            tau = int(self.accept_len.item())
            d = self.draft[0].tolist()
            b0 = int(self.bonus.item())
            out.extend(d[:tau - 1])
            out.append(b0)
            self.taus.append(tau)
        return out[:n_new]


def greedy_generate(target: Drafter, prompt, n_new: int, slot: int = 0, stream=None, temperature: float = 0.0,
                    seed: int = 0):
    """The target's own decoding through dflash_verify_block with one live
    row per step (what speculative generation must equal): greedy, or at
    temperature > 0 sampled by position (dflash_verify_block_sample)."""
    dev = torch.device(f"cuda:{target.device}")
    i32 = dict(dtype=torch.int32, device=dev)
    slots = torch.tensor([slot], **i32)
    tokens = torch.zeros(1, 16, **i32)
    out_tok = torch.zeros(1, 16, **i32)
    n_valid = torch.zeros(1, **i32)
    prompt = [int(x) for x in prompt]

    def verify(sl, tk, ot, nv):
        if temperature > 0:
            target.verify_block_sample(sl, tk, ot, temperature, seed, nv, None, stream)
        else:
            target.verify_block(sl, tk, ot, nv, None, stream)
    n = 0
    for p0 in range(0, len(prompt), 16):
        chunk = prompt[p0:p0 + 16]
        n = len(chunk)
        tokens.zero_()
        tokens[0, :n] = torch.tensor(chunk, dtype=torch.int32)
        n_valid.fill_(n)
        verify(slots, tokens, out_tok, n_valid)
        target.advance(slots, n_valid, stream)
    g = int(out_tok[0, n - 1].item())
    out = [g]
    n_valid.fill_(1)
    while len(out) < n_new:
        tokens[0, 0] = g
        verify(slots, tokens, out_tok, n_valid)
        target.advance(slots, n_valid, stream)
        g = int(out_tok[0, 0].item())
        out.append(g)
    return out

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

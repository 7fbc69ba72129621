"""Helpers for the GPU parity tests: drive the CUDA path and the CPU oracle
over the same seeded inputs.  The oracle never sees a value produced by the
CUDA path; both sides read only the workload generators."""
from __future__ import annotations

import math

import numpy as np

import oracle as O
import oracle.sampling_ref as SR
from workload import (context_lengths, feature_rows, make_weights, match_stream)

TOL_REL_L2 = 1e-2      # hidden states, logits, K/V
MARGIN = 0.05          # draft tokens must match where the oracle's top-1 margin exceeds this


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def to_np(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


# ---------------------------------------------------------------- GPU side

class GpuRun:
    """CUDA-path driver: prefill every request, then rounds with the stand-in verify."""

    def __init__(self, cfg, rounds: int, weights_np=None, batch_ids=None, prefill_chunk=4096,
                 ctx=None, attn_impl: int = 0, temperature: float = 0.0, seed: int = 0, weight_fp8: int = 0):
        import torch
        from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
        from block_diffusion_speculative_hiddens_gb300.session import RoundState, SyntheticVerify
        self.cfg = cfg
        self.ids = list(range(cfg.batch)) if batch_ids is None else list(batch_ids)
        B = len(self.ids)
        self.ctx0 = (context_lengths(cfg)[self.ids] if ctx is None else np.asarray(ctx)).astype(int)
        self.rounds = rounds
        w = make_weights(cfg) if weights_np is None else weights_np
        self.w_dev = weights_to_device(w)
        cap = int(self.ctx0.max()) + cfg.block * (rounds + 2) + 64
        mpps = math.ceil(cap / 64) + 1
        self.stream_rows = cap
        self.chunk = min(prefill_chunk, int(self.ctx0.max()))
        self.d = Drafter(cfg, self.w_dev, max_batch=B, max_slots=B, max_pages=mpps * B,
                         max_pages_per_slot=mpps, max_rows=max(self.chunk, B * cfg.block),
                         attn_impl=attn_impl, weight_fp8=weight_fp8)
        dev = torch.device("cuda:0")
        self.dev = dev
        # feature stream: every position a request can reach
        F = cfg.fused_dim
        fs = np.zeros((B, cap, F), dtype=np.uint16)
        for j, b in enumerate(self.ids):
            n = min(cap, int(self.ctx0[j]) + cfg.block * (rounds + 2))
            fs[j, :n] = feature_rows(cfg, b, 0, n).reshape(n, F)
        self.feat_stream = torch.from_numpy(fs.view(np.int16)).view(torch.bfloat16).to(dev)
        m = np.empty((max(rounds, 1), B, cfg.block), dtype=np.int32)
        u = np.empty_like(m)
        for r in range(rounds):
            m[r], u[r] = match_stream(cfg, r, self.ids)
        self.match = torch.from_numpy(m).to(dev)
        self.offs = torch.from_numpy(u).to(dev)
        self.state = RoundState(self.d, B, first_token=cfg.first_token)
        self.verify = SyntheticVerify(self.state, self.match, self.offs, self.feat_stream)
        if temperature > 0:
            self.state.set_sampling(temperature, seed, self.verify.round_ctr)

    def prefill(self):
        import torch
        cfg = self.cfg
        for j in range(len(self.ids)):
            slot = torch.tensor([j], dtype=torch.int32, device=self.dev)
            L = int(self.ctx0[j])
            for p0 in range(0, L, self.chunk):
                n = min(self.chunk, L - p0)
                feats = self.feat_stream[j:j + 1, p0:p0 + n]
                self.d.fuse_inject(slot, feats, n, torch.tensor([n], dtype=torch.int32, device=self.dev))

    def round(self, debug=False, folded=False):
        """One round; returns dict of host arrays (draft, target, tau, bonus, ctx) and debug tensors."""
        import torch
        from block_diffusion_speculative_hiddens_gb300.session import run_round
        s = self.state
        out = {}
        if debug:
            cfg = self.cfg
            B = s.batch
            s.inject()
            # the debug outputs always hold 16 rows per request (rows S..15 pad a smaller block)
            hidden = torch.empty(B * 16, cfg.hidden, dtype=torch.float32, device=self.dev)
            logits = torch.empty(B * 16, cfg.vocab, dtype=torch.float32, device=self.dev)
            if s.temperature > 0:
                self.d.draft_block_sample(s.slots, s.bonus, s.temperature, s.seed, s.round_ctr, s.draft, logits)
            else:
                self.d.draft_block_debug(s.slots, s.bonus, s.draft, hidden, logits)
            self.verify()
            s.accept()
            out["hidden"] = to_np(hidden).reshape(B, 16, cfg.hidden)[:, :cfg.block]
            out["logits"] = to_np(logits).reshape(B, 16, cfg.vocab)[:, :cfg.block]
        else:
            run_round(s, self.verify, folded=folded)
        torch.cuda.synchronize()
        out.update(draft=to_np(s.draft).astype(np.int64), target=to_np(s.target).astype(np.int64),
                   tau=to_np(s.accept_len).astype(np.int64), bonus=to_np(s.bonus).astype(np.int64),
                   ctx=to_np(s.ctx_len).astype(np.int64))
        return out


# ---------------------------------------------------------------- oracle side

class OracleRun:
    def __init__(self, cfg, rounds: int, weights_np=None, batch_ids=None, ctx=None, cache=True,
                 temperature: float = 0.0, seed: int = 0, weight_fp8: int = 0):
        self.temperature = temperature
        self.seed = seed
        self.cfg = cfg
        self.ids = list(range(cfg.batch)) if batch_ids is None else list(batch_ids)
        self.ctx0 = (context_lengths(cfg)[self.ids] if ctx is None else np.asarray(ctx)).astype(int)
        w = make_weights(cfg) if weights_np is None else weights_np
        self.model = O.OracleModel(cfg, w, cache=cache, fp8=bool(weight_fp8))
        self.dr = O.OracleDrafter(self.model)
        self.reqs = [O.OracleRequest(cfg, int(L) + cfg.block * (rounds + 2)) for L in self.ctx0]
        self.last = [cfg.first_token] * len(self.ids)
        self.pending = [0] * len(self.ids)
        self.r = 0

    def prefill(self):
        for j, b in enumerate(self.ids):
            self.dr.fuse_inject(self.reqs[j], feature_rows(self.cfg, b, 0, int(self.ctx0[j])))

    def round(self, want_logits=True):
        cfg = self.cfg
        mm, uu = match_stream(cfg, self.r, self.ids)
        res = []
        for j, b in enumerate(self.ids):
            req = self.reqs[j]
            if self.pending[j]:
                self.dr.fuse_inject(req, feature_rows(cfg, b, req.ctx_len, self.pending[j]))
            o = self.dr.draft(req, self.last[j], want_logits=want_logits or self.temperature > 0)
            if self.temperature > 0:  # drafts drawn from softmax(logits / T); margins of the perturbed scores
                o["draft"], o["margin"] = SR.sample_drafts(o["logits"], self.temperature, self.seed, j, self.r)
                o["sampled"] = True
            t = O.synthetic_target(o["draft"], mm[j], uu[j], cfg.vocab)
            tau, bonus, conf = self.dr.accept_trim(req, o["draft"], t)
            o.update(target=t, tau=tau, bonus=bonus, ctx=conf)
            res.append(o)
            self.last[j], self.pending[j] = bonus, tau
        self.r += 1
        return res


def check_drafts(gpu_draft, o, margin=MARGIN):
    """Tokens equal wherever the oracle margin exceeds `margin`; elsewhere the
    GPU's token must be a near-maximum of the oracle's logits."""
    d = np.asarray(gpu_draft)
    strong = o["margin"] > margin
    assert np.array_equal(d[strong], o["draft"][strong]), (d, o["draft"], o["margin"])
    if "logits" in o and not o.get("sampled"):
        lg = o["logits"]
        top = lg.max(-1)
        got = lg[np.arange(len(d)), d]
        assert np.all(got >= top - margin), (got, top)
    return int(strong.sum()), len(d)

#!/usr/bin/env python
"""Benchmark: one DFlash drafting-plus-acceptance round per step on GB300.

Workload (default): the Qwen3-8B-shaped drafter at batch 1 -- hidden 4096,
32/8 heads x 128, SwiGLU 12288, 5 layers, vocabulary 151936, fusion
20480 -> 4096 -- with a 2048-token prompt, block 16 and a stand-in verify
that copies each draft with probability 0.9.  One step = fuse+inject the
previous round's accepted features, draft one block, stand-in verify,
accept/trim, all captured in one CUDA graph.  Synthetic seeded data and
random-init weights of that architecture.

Every scenario pass is the workload's round count from its prompts; timed
steps cycle through identically prefilled groups of request slots, one pass
per group, so K steps always run rounds of the stated scenario.  Other
workloads (`--config llama3.1-8b | batched-qwen3-8b | long-8layer`) run the
same way at their own batch; large feature streams are drawn on the GPU.

Prints one JSON line (rank 0).  `--impl reference` times the float64 CPU
oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "drafted tok/s & draft-round latency (µs), Qwen3-8B-shape b16; % HBM roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed rounds (default 512 at batch 1, one scenario pass of the workload otherwise)")
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3-8b")
    ap.add_argument("--rounds-per-slot", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=25.0)
    ap.add_argument("--block", type=int, default=None,
                    help="inference block size S in [2, 16] (default: the workload's, 16): S-1 drafts per round")
    ap.add_argument("--attn-impl", type=int, default=0, choices=[0, 1, 2],
                    help="attention page loop: 0 chosen by the library, 1 warp MMAs, 2 tcgen05")
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="draft at this temperature (> 0: each draft drawn from softmax(logits / T))")
    ap.add_argument("--seed", type=int, default=1234, help="seed of the drafts' random streams (temperature > 0)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp8"],
                    help="drafter weights as given (bf16, held as f16) or FP8 E4M3 with per-row scales")
    ap.add_argument("--spec-generate", type=int, default=0,
                    help="instead of the drafting rounds: greedy speculative generation of this many tokens "
                         "with a random-weight target model (--target-layers) of the workload's layer shape")
    ap.add_argument("--target-layers", type=int, default=8)
    ap.add_argument("--fold-inject", action="store_true",
                    help="issue dflash_draft_round instead of dflash_fuse_inject + dflash_draft_block")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def tensor_peaks():
    """Dense bf16 tensor peaks (TFLOP/s): burst and sustained, measured else fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"]))
    except Exception:
        return 1900.0, 1700.0


def gemm_source_hash():
    """sha256 over the GEMM kernel's sources: gemm.cu, common.cuh and the
    GemmParams block of internal.h (the rest of that header is other kernels')."""
    import hashlib
    csrc = os.path.join(ROOT, "block_diffusion_speculative_hiddens_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("gemm.cu", "common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(csrc, "internal.h")) as f:
        text = f.read()
    m = re.search(r"struct GemmParams \{.*?\n\};", text, re.S)
    h.update(m.group(0).encode() if m else b"")
    return h.hexdigest()


def lm_head_traffic(cfg):
    """DRAM bytes per lm_head launch from the committed ncu summary, or None
    when the GEMM sources changed since the counters were taken (or for a
    workload the summary does not cover)."""
    try:
        with open(os.path.join(ROOT, "profiles", "lm_head_traffic_mid.md")) as f:
            text = f.read()
        want = re.search(r"^source_sha256: ([0-9a-f]{64})$", text, re.M).group(1)
        traffic = int(re.search(r"^traffic_bytes_per_launch: (\d+)$", text, re.M).group(1))
    except Exception:
        return None
    if gemm_source_hash() != want or cfg.name != "qwen3-8b":
        return None
    return traffic


# ------------------------------------------------------------------ clocks

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="dflash_clocks_", suffix=".csv")
        self.f = open(self.path, "w")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                       "-i", str(gpu_index), "-lms", "20"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self, t0: float, t1: float):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                        float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
                except Exception:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside if inside else rows
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed region" if inside else "whole run (no sample fell inside the timed region)"}


# ------------------------------------------------------------------ oracle timing

def oracle_round_seconds(cfg, budget_s: float, max_rounds: int):
    """Time the float64 CPU oracle on rounds of `cfg` (request 0) after an untimed prefill."""
    import numpy as np
    import oracle as O
    from workload import feature_rows, make_weights, match_stream
    w = make_weights(cfg)
    model = O.OracleModel(cfg, w, cache=False)
    dr = O.OracleDrafter(model)
    L0 = int(cfg.ctx0 or cfg.ctx_range[0])
    req = O.OracleRequest(cfg, L0 + cfg.block * (max_rounds + 2))
    dr.fuse_inject(req, feature_rows(cfg, 0, 0, L0))
    last, pending = cfg.first_token, 0
    times, taus = [], []
    start = time.perf_counter()
    for r in range(max_rounds):
        t0 = time.perf_counter()
        if pending:
            dr.fuse_inject(req, feature_rows(cfg, 0, req.ctx_len, pending))
        o = dr.draft(req, last, want_logits=False)
        mm, uu = match_stream(cfg, r, [0])
        t = O.synthetic_target(o["draft"], mm[0], uu[0], cfg.vocab)
        tau, bonus, _ = dr.accept_trim(req, o["draft"], t)
        times.append(time.perf_counter() - t0)
        taus.append(tau)
        last, pending = bonus, tau
        if time.perf_counter() - start > budget_s:
            break
    return times, taus


# ------------------------------------------------------------------ GPU arm

def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the job's time is its slowest replica's)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput of `world` replicas: all ranks' units over the slowest time."""
    return units_per_rank * world / seconds


def roofline_bound(flops: float, nbytes: float, hbm_gbs: float, tflops: float) -> str:
    """"hbm" when a kernel's arithmetic intensity (flops per algorithmic byte)
    is below the ridge point of the two peaks, else "tensor"."""
    return "hbm" if flops / nbytes < tflops * 1e12 / (hbm_gbs * 1e9) else "tensor"


def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, binding, weights_to_device
    from block_diffusion_speculative_hiddens_gb300.session import RoundState, SyntheticVerify, run_round
    from workload import context_lengths, feature_rows, get_config, make_weights, match_stream

    torch.cuda.set_device(local_rank)
    dev = torch.device(f"cuda:{local_rank}")
    cfg = get_config(args.config)
    if args.block:
        cfg = cfg.with_(block=args.block)
    S = cfg.block                                        # S-1 drafts per request per round
    B = cfg.batch
    ctx = context_lengths(cfg).astype(int)               # prompt length per request
    R = args.rounds_per_slot or cfg.rounds
    K = args.steps if args.steps is not None else (512 if B == 1 else R)
    W = args.warmup
    n_groups = math.ceil(K / R) + 1                      # + one group of B slots for warm-up
    n_slots = n_groups * B
    cap = int(ctx.max()) + cfg.block * (max(R, W) + 2) + 64
    mpps = math.ceil(cap / 64) + 1
    F = cfg.fused_dim

    w_dev = weights_to_device(make_weights(cfg), local_rank)
    # target features of every position a request reaches: the workload's
    # position-keyed stream when it is small, else N(0,1) drawn on the device
    # from a per-request seeded generator (same distribution, same shapes)
    if B * cap * F <= 4e8:
        fs = np.stack([feature_rows(cfg, b, 0, cap).reshape(cap, F) for b in range(B)])
        feat_stream = binding.bf16_host(fs).to(dev)
        feat_src = "workload generator"
    else:
        fs = None
        feat_stream = torch.empty(B, cap, F, dtype=torch.bfloat16, device=dev)
        for b in range(B):
            g = torch.Generator(device=dev)
            g.manual_seed(1_000_003 * (cfg.seed + 1) + b)
            feat_stream[b].normal_(generator=g)
        feat_src = "device generator (torch.normal_, seeded per request)"
    m = np.empty((max(R, W), B, S), dtype=np.int32)
    u = np.empty_like(m)
    for r in range(max(R, W)):
        m[r], u[r] = match_stream(cfg, r, list(range(B)))
    match, offs = torch.from_numpy(m).to(dev), torch.from_numpy(u).to(dev)

    chunk = 2048
    d = Drafter(cfg, w_dev, max_batch=B, max_slots=n_slots, max_pages=mpps * n_slots,
                max_pages_per_slot=mpps, max_rows=max(chunk, S * B), device=local_rank, attn_impl=args.attn_impl,
                weight_fp8=1 if args.weights == "fp8" else 0)
    stream = torch.cuda.Stream(device=dev)

    def prefill(g, timed=False):
        """Inject every prompt of slot group g in chunks; with timed, returns
        the device time (ms) of the fuse_inject calls alone."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)] if timed else None
        with torch.cuda.stream(stream):
            calls = []
            for b in range(B):
                slot = torch.tensor([g * B + b], dtype=torch.int32, device=dev)
                for p0 in range(0, int(ctx[b]), chunk):
                    n = min(chunk, int(ctx[b]) - p0)
                    calls.append((slot, b, p0, n, torch.tensor([n], dtype=torch.int32, device=dev)))
            if timed:
                stream.synchronize()
                ev[0].record(stream)
            for slot, b, p0, n, n_dev in calls:
                d.fuse_inject(slot, feat_stream[b:b + 1, p0:p0 + n], n, n_dev, stream)
            if timed:
                ev[1].record(stream)
        if timed:
            ev[1].synchronize()
            return ev[0].elapsed_time(ev[1])
        return None

    states, verifies = [], []
    for g in range(n_groups):
        prefill(g)
        st = RoundState(d, B, slots=[g * B + b for b in range(B)], first_token=cfg.first_token)
        states.append(st)
        verifies.append(SyntheticVerify(st, match, offs, feat_stream))
        if args.temperature > 0:
            st.set_sampling(args.temperature, args.seed, verifies[-1].round_ctr)
    stream.synchronize()

    # warm-up: W rounds on the spare group, as one graph
    wst, wv = states[-1], verifies[-1]
    d.graph_begin(stream)
    for _ in range(W):
        run_round(wst, wv, stream, folded=args.fold_inject)
    d.graph_end(stream)
    d.graph_launch(stream)
    stream.synchronize()

    # timed: K rounds, R per group, one graph; lm_head bracketed by event probes
    d.probe_arm(binding.KID_LM_HEAD, K)
    n0 = d.launch_count()
    d.graph_begin(stream)
    for i in range(K):
        run_round(states[i // R], verifies[i // R], stream, folded=args.fold_inject)
    n_kernels = d.graph_end(stream)
    launches_captured = d.launch_count() - n0
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    d.graph_launch(stream)
    e1.record(stream)
    e1.synchronize()
    t_wall1 = time.time()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    ms = e0.elapsed_time(e1)
    lm_ms = d.probe_read(K)
    status = d.read_status()
    accepted = 0
    for g in range(n_groups - 1):
        if min(R, K - g * R) > 0:
            accepted += int((states[g].ctx_len.cpu().numpy() - ctx).sum())
    ms = max_over_ranks(ms, world, dev)

    # ---- the stand-in verify on its own, and the per-round distribution: one
    # more graph of up to R rounds on a fresh copy of the prompts, with
    # timeline marks at every round start and around the verify (the marks'
    # event nodes cost a little overlap, so the headline mean stays the
    # unmarked graph's, minus the verify's mean)
    Ki = min(R, K)
    gi = n_groups - 1
    for b in range(B):
        d.reset_slot(gi * B + b, stream)
    prefill_ms = prefill(gi, timed=True)
    st_i = RoundState(d, B, slots=[gi * B + b for b in range(B)], first_token=cfg.first_token)
    ver_i = SyntheticVerify(st_i, match, offs, feat_stream)
    if args.temperature > 0:
        st_i.set_sampling(args.temperature, args.seed, ver_i.round_ctr)

    def marked_verify(s_=None):
        d.mark(s_)
        ver_i(s_)
        d.mark(s_)

    d.marks_arm(3 * Ki + 1)
    d.graph_begin(stream)
    for _ in range(Ki):
        d.mark(stream)
        run_round(st_i, marked_verify, stream, folded=args.fold_inject)
    d.mark(stream)
    d.graph_end(stream)
    d.graph_launch(stream)
    stream.synchronize()
    iv = d.marks_read(3 * Ki)
    verify_ms = statistics.mean(iv[1::3])
    per_round_ms = sorted(a + c for a, c in zip(iv[0::3], iv[2::3]))
    pct = lambda q: per_round_ms[min(len(per_round_ms) - 1, int(q * len(per_round_ms)))]

    # ---- end to end through the C ABI with host buffers: per step H2D of the
    # block's target features and verify streams, one round, D2H of the result
    e2e = None
    E = min(args.e2e_steps, R)
    if E > 0:
        for b in range(B):
            d.reset_slot(gi * B + b, stream)
        prefill(gi)
        st = RoundState(d, B, slots=[gi * B + b for b in range(B)], first_token=cfg.first_token)
        m_dev = torch.zeros(1, B, S, dtype=torch.int32, device=dev)
        u_dev = torch.zeros_like(m_dev)
        ver = SyntheticVerify(st, m_dev, u_dev, None)
        if args.temperature > 0:
            st.set_sampling(args.temperature, args.seed, ver.round_ctr)
        d.graph_begin(stream)
        run_round(st, ver, stream, folded=args.fold_inject)
        d.graph_end(stream)
        feats_h = torch.empty(B, S, F, dtype=torch.bfloat16).pin_memory()
        mu_h = torch.empty(2, B, S, dtype=torch.int32).pin_memory()
        out_h = torch.empty(B, S - 1 + 3, dtype=torch.int32).pin_memory()
        if fs is not None:
            fs_host = binding.bf16_host(fs)
        else:  # the device-drawn stream's first rows stand in on the host
            fs_host = feat_stream[:, :S].cpu()
        stream.synchronize()
        # the round's inject consumes the previous round's block features
        # (positions prev_L .. prev_L+S-1 of each request, the first accept_len)
        prev_L = ctx.copy()
        cur_L = ctx.copy()
        t0 = time.perf_counter()
        for r in range(E):
            for b in range(B):
                if fs is not None:
                    feats_h[b].copy_(fs_host[b, prev_L[b]:prev_L[b] + S])
                else:
                    feats_h[b].copy_(fs_host[b])
            mu_h[0].copy_(torch.from_numpy(m[r % len(m)]))
            mu_h[1].copy_(torch.from_numpy(u[r % len(u)]))
            with torch.cuda.stream(stream):
                st.feats.copy_(feats_h, non_blocking=True)
                m_dev[0].copy_(mu_h[0], non_blocking=True)
                u_dev[0].copy_(mu_h[1], non_blocking=True)
                d.graph_launch(stream)
                out_h[:, :S - 1].copy_(st.draft, non_blocking=True)
                out_h[:, S - 1].copy_(st.accept_len, non_blocking=True)
                out_h[:, S].copy_(st.bonus, non_blocking=True)
                out_h[:, S + 1].copy_(st.ctx_len, non_blocking=True)
            stream.synchronize()
            prev_L, cur_L = cur_L, out_h[:, S + 1].numpy().astype(int)
        h2d = feats_h.numel() * 2 + mu_h.numel() * 4
        d2h = out_h.numel() * 4
        t_e2e = time.perf_counter() - t0
        t_e2e = max_over_ranks(t_e2e, world, dev)
        e2e = {"value": round(replica_rate((S - 1) * B * E, world, t_e2e), 1), "unit": "tok/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": E,
               "round_us": round(t_e2e / E * 1e6, 1),
               "note": "includes the stand-in verify kernel"}

    # ---- rooflines: the dominant kernel (lm_head + argmax) and the round
    hbm, _, peak_src = peaks()
    tf_burst, tf_sust = tensor_peaks()
    H, V, D = cfg.hidden, cfg.vocab, cfg.head_dim
    M = S * B                                            # block rows the method computes
    fp8 = args.weights == "fp8"
    wb = 1 if fp8 else 2                                 # bytes per projection / embedding weight
    lm_bytes = V * H * wb + (V * 4 if fp8 else 0) + M * H * 2
    lm_flops = 2.0 * M * V * H
    lm_avg_ms = statistics.mean(lm_ms) if lm_ms else float("nan")
    round_ms_incl = ms / K
    round_ms = round_ms_incl - verify_ms  # the stand-in verify is not part of the round
    tau = accepted / (K * B)
    avg_ctx = float(ctx.mean()) + tau * (R / 2)
    kv_bytes = B * cfg.n_layers * (avg_ctx + S) * cfg.n_kv_heads * D * 2 * 2
    if fp8:  # FP8 projections and embedding (+ a float scale per row); the fusion projection stays 2 bytes
        fc_bytes = 2 * H * F
        rows = V + cfg.n_layers * (cfg.qkv_rows + H + 2 * cfg.intermediate + H)
        w_bytes = (cfg.weight_bytes() - fc_bytes) // 2 + fc_bytes + 4 * rows
    else:
        w_bytes = cfg.weight_bytes()
    round_bytes = w_bytes + kv_bytes + B * tau * F * 2
    layer_params = cfg.qkv_rows * H + H * cfg.n_q_heads * D + 3 * cfg.intermediate * H
    inj_params = H * F + cfg.n_layers * 2 * cfg.n_kv_heads * D * H
    round_flops = 2.0 * M * (cfg.n_layers * layer_params + V * H) + 2.0 * B * tau * inj_params
    prefill_flops = 2.0 * float(ctx.sum()) * inj_params
    if roofline_bound(lm_flops, lm_bytes, hbm, tf_sust) == "hbm":
        lm_roof = {"bound": "hbm", "achieved": round(lm_bytes / (lm_avg_ms * 1e-3) / 1e9, 1), "peak": hbm,
                   "unit": "GB/s", "frac": round(lm_bytes / (lm_avg_ms * 1e-3) / 1e9 / hbm, 4),
                   "traffic": None if fp8 else lm_head_traffic(cfg), "peak_source": f"{peak_src} copy bandwidth"}
    else:
        ach = lm_flops / (lm_avg_ms * 1e-3) / 1e12
        lm_roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": tf_sust, "unit": "TFLOP/s",
                   "frac": round(ach / tf_sust, 4), "traffic": None,
                   "peak_source": "measured bf16 sustained (f16 dense rate equals bf16 on this part)"}
    lm_roof.update({"kernel": "lm_head+argmax (tcgen05 GEMM)", "bytes_per_launch": lm_bytes,
                    "flops_per_launch": lm_flops, "avg_launch_us": round(lm_avg_ms * 1e3, 2)})
    ctx_desc = f"prompt {int(ctx[0])}" if cfg.ctx0 else f"prompts U[{cfg.ctx_range[0]}, {cfg.ctx_range[1]}]"
    p_desc = f"match p {cfg.match_p}" if cfg.match_p is not None else f"match p U[{cfg.p_range[0]}, {cfg.p_range[1]}]"
    res = {
        "metric": METRIC,
        "value": round(replica_rate((S - 1) * B, world, round_ms * 1e-3), 1),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(round_ms, 4),
        "round_us": round(round_ms * 1e3, 1),
        "round_us_p10_p50_p90": [round(pct(0.1) * 1e3, 1), round(pct(0.5) * 1e3, 1), round(pct(0.9) * 1e3, 1)],
        "round_us_with_stand_in_verify": round(round_ms_incl * 1e3, 1),
        "stand_in_verify_us": round(verify_ms * 1e3, 1),
        "accepted_tok_s": round(accepted * world / (round_ms * K * 1e-3), 1),
        "mean_tau": round(tau, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 activations, fp8 e4m3 weights" if fp8 else "f16",
        "data": f"synthetic (seeded N(0,1) target features from the {feat_src}, N(0,0.02) random-init weights, "
                "stand-in verify)",
        "config": {"workload": f"{cfg.name} drafter batch {B}: H{H}, {cfg.n_q_heads}q/{cfg.n_kv_heads}kv x"
                               f"{D}, I{cfg.intermediate}, {cfg.n_layers} layers, V{V}, fusion "
                               f"{F}->{H}, {ctx_desc}, block {S}, {p_desc}",
                   "batch": B, "prompt_mean": float(ctx.mean()), "rounds_per_slot": R,
                   "attn_impl": ["library choice", "warp MMAs", "tcgen05"][args.attn_impl],
                   "weights": "fp8 e4m3, per-row scales" if args.weights == "fp8" else "bf16 (held as f16)",
                   "drafting": (f"sampled at temperature {args.temperature} (Gumbel-max, seed {args.seed})"
                                if args.temperature > 0 else "greedy argmax"),
                   "round_call": "dflash_draft_round" if args.fold_inject
                   else "dflash_fuse_inject+dflash_draft_block", "slot_groups": n_groups - 1,
                   "l2": "inputs larger than L2 (the drafter's weights stream every round)",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": launches_captured,
        "plan": d.plan(),
        "graph_kernel_nodes": n_kernels,
        "roofline": lm_roof,
        "round_roofline": {"bytes_per_round": int(round_bytes), "achieved_gbs": round(
            round_bytes / (round_ms * 1e-3) / 1e9, 1), "frac": round(round_bytes / (round_ms * 1e-3) / 1e9 / hbm, 4)},
        "round_tensor": {"flops_per_round": round_flops, "achieved_tflops": round(
            round_flops / (round_ms * 1e-3) / 1e12, 1), "peak": tf_sust,
            "frac": round(round_flops / (round_ms * 1e-3) / 1e12 / tf_sust, 4)},
        "prefill": {"tokens": int(ctx.sum()), "us": round(prefill_ms * 1e3, 1),
                    "tok_s": round(float(ctx.sum()) / (prefill_ms * 1e-3), 1),
                    "flops": prefill_flops, "tensor_frac": round(prefill_flops / (prefill_ms * 1e-3) / 1e12 / tf_burst, 4),
                    "call": f"dflash_fuse_inject per request in {chunk}-token chunks (device time, not in the round)"},
        "clocks": clk,
        "status_word": status,
        "e2e": e2e,
    }
    return res, cfg


def run_spec_generate(args):
    """Greedy speculative generation (draft -> verify -> accept -> trim per
    round, host loop) with a random-weight target of the drafter's layer
    shape; times the whole generation and the verify calls."""
    import numpy as np
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, weights_to_device
    from block_diffusion_speculative_hiddens_gb300.session import SpecDecoder
    from workload import get_config, make_target_weights, make_weights, prompt_tokens
    cfg = get_config(args.config)
    P = int(cfg.ctx0 or cfg.ctx_range[0])
    n_new = args.spec_generate
    cap = P + 16 * (n_new + 2) + 64
    mpps = math.ceil(cap / 64) + 1
    kw = dict(max_batch=1, max_slots=1, max_pages=mpps, max_pages_per_slot=mpps, max_rows=16,
              attn_impl=args.attn_impl)
    t = Drafter(cfg, weights_to_device(make_target_weights(cfg, args.target_layers)), role=1, **kw)
    d = Drafter(cfg, weights_to_device(make_weights(cfg)), **kw)
    prompt = prompt_tokens(cfg, 0, P)
    times = []
    ev = []
    orig = t.verify_block

    def timed_verify(*a, **k):  # CUDA events around every verify call
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        orig(*a, **k)
        e1.record()
        ev.append((e0, e1))
    t.verify_block = timed_verify
    for rep_ in range(2):  # the first pass warms up; its slot is reset before the timed one
        for x in (t, d):
            x.reset_slot(0)
        ev.clear()
        sd = SpecDecoder(d, t, slot=0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        out = sd.generate(prompt, n_new)
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    n_prefill = math.ceil(P / 16)
    verify_us = [a.elapsed_time(b) * 1e3 for a, b in ev[n_prefill:]]
    rounds = len(sd.taus)
    return {"metric": "greedy speculative generation, random-weight target", "value": round(n_new / times[-1], 1),
            "unit": "tok/s", "higher_is_better": True, "generated": len(out), "rounds": rounds,
            "mean_tau": round(float(np.mean(sd.taus)), 3), "wall_s": round(times[-1], 4),
            "verify_us_median": round(float(np.median(verify_us)), 1) if verify_us else None,
            "note": "host loop with one host read per round; prefill included; the random drafter rarely matches "
                    "the random target, so tau is near 1",
            "config": {"workload": f"{cfg.name} drafter + {args.target_layers}-layer target of the same layer "
                                   f"shape, prompt {P}, block 16", "target_layers": args.target_layers}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the CPU oracle on the host cores; rank 0 alone, other ranks exit
        if rank != 0:
            return
        from workload import get_config
        cfg = get_config(args.config)
        if args.block:
            cfg = cfg.with_(block=args.block)
        budget = 150.0
        K, W = max(1, args.steps or 8), max(0, args.warmup)
        times, taus = oracle_round_seconds(cfg, budget, W + K)
        warm = min(W, len(times) - 1)  # the budget may stop early: keep at least one timed round
        used = times[warm:]
        rs = statistics.mean(used)
        val = (cfg.block - 1) / rs
        stopped = len(times) < W + K
        line = {"impl": "reference", "metric": METRIC, "value": round(val, 3), "unit": "tok/s",
                "n_gpus": args.gpus, "steps": len(used), "warmup": warm,
                "ms_per_step": round(rs * 1e3, 1), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": f"{cfg.name} drafter, one request of batch {cfg.batch} at a time, "
                                       f"prompt {cfg.ctx0 or cfg.ctx_range[0]}, block {cfg.block}"},
                "cpu_baseline": {"value": round(val, 3), "unit": "tok/s", "cores": os.cpu_count(),
                                 "kind": "oracle",
                                 "sample": f"{len(used)} timed rounds after {warm} warm-up rounds of request 0, "
                                           f"after an untimed {cfg.ctx0 or cfg.ctx_range[0]}-token prefill"
                                           + (f"; stopped by the {budget:.0f} s budget" if stopped else "")},
                "e2e": {"value": round(val, 3), "unit": "tok/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    if args.spec_generate:
        if rank == 0:
            print(json.dumps(run_spec_generate(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    res, cfg = run_gpu(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times, taus = oracle_round_seconds(cfg, args.cpu_budget_s, 4)
        rs = statistics.mean(times)
        res["cpu_baseline"] = {"value": round((cfg.block - 1) / rs, 3), "unit": "tok/s", "cores": os.cpu_count(),
                               "kind": "oracle",
                               "sample": f"{len(times)} round(s) of the same workload (request 0) after an "
                                         f"untimed {cfg.ctx0 or cfg.ctx_range[0]}-token prefill, float64 NumPy"}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark: one DFlash drafting-plus-acceptance round per step on one GB300.

Headline workload (default): the Qwen3-8B-shaped drafter at batch 1 -- hidden
4096, 32/8 heads x 128, SwiGLU 12288, 5 layers, vocabulary 151936, fusion
20480 -> 4096 -- with a 2048-token prompt, block 16 and a stand-in verify that
copies each draft with probability 0.9.  One step = accept/trim the previous
round, fuse+inject its accepted features, draft one block; the stand-in
verify runs between rounds and is timed apart, in the same CUDA graph.
Synthetic seeded data and random-init weights of that architecture.

Every scenario pass is the workload's round count from its prompts; timed
steps cycle through identically prefilled groups of request slots, one pass
per group, so K steps always run rounds of the stated scenario.  After the
headline, the default run measures the other drafting workloads (tiny,
Llama-3.1-8B shape, batched Qwen3-8B shape, long-context 8-layer) with a
short run each and reports them under "workloads" (`--workloads none` skips
them; `--config NAME` makes another workload the headline).

The library drives one GPU; `--gpus N` with N > 1 prints a one-line record
saying so and exits (replicas are independent processes, one per GPU, each
running this benchmark on its own).

Prints one JSON line.  `--impl reference` times the float64 CPU oracle on the
host cores instead.
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
    ap.add_argument("--rounds-per-slot", type=int, default=None,
                    help="rounds of the scenario per slot group (default: the workload's round count)")
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
    ap.add_argument("--workloads", default="all",
                    help="after the headline, also measure: all (tiny, llama3.1-8b, batched-qwen3-8b, "
                         "long-8layer), none, or a comma-separated list")
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

def oracle_round_seconds(cfg, budget_s: float, max_rounds: int, weights=None):
    """Time the float64 CPU oracle on rounds of `cfg` (request 0) after an untimed prefill."""
    import numpy as np
    import oracle as O
    from workload import feature_rows, make_weights, match_stream
    w = make_weights(cfg) if weights is None else weights
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

def roofline_bound(flops: float, nbytes: float, hbm_gbs: float, tflops: float) -> str:
    """"hbm" when a kernel's arithmetic intensity (flops per algorithmic byte)
    is below the ridge point of the two peaks, else "tensor"."""
    return "hbm" if flops / nbytes < tflops * 1e12 / (hbm_gbs * 1e9) else "tensor"


# The workloads every default run measures after the headline one, each with
# a short run of timed rounds (the batched round is ~6 ms, the others < 2 ms).
EXTRA_WORKLOADS = ("tiny", "llama3.1-8b", "batched-qwen3-8b", "long-8layer")
EXTRA_STEPS = {"tiny": 64, "llama3.1-8b": 32, "batched-qwen3-8b": 16, "long-8layer": 32}
FEATS_ON_HOST_MAX = 4e8  # feature-stream elements drawn by the workload generator; larger: on the device


def device_weights(cfg, dev, seed: int) -> dict:
    """Random-init weights of cfg's architecture drawn on the device: every
    projection N(0, weight_std) in bf16, RMSNorm gains 1 -- the distribution
    and layout of workload.make_weights, from a seeded torch generator."""
    import torch
    from workload.inputs import WEIGHT_NAMES, _shape
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def t(name):
        shape = _shape(cfg, name)
        if len(shape) == 1:
            return torch.ones(shape, dtype=torch.bfloat16, device=dev)
        x = torch.empty(shape, dtype=torch.float32, device=dev)
        x.normal_(0.0, cfg.weight_std, generator=g)
        return x.to(torch.bfloat16)

    glob = [n for n in WEIGHT_NAMES if n in ("embed", "fc", "fc_norm", "final_norm")]
    out = {n: t(n) for n in glob}
    out["layers"] = [{n: t(n) for n in WEIGHT_NAMES if n not in glob} for _ in range(cfg.n_layers)]
    return out


def feature_stream(cfg, B, cap, dev):
    """Target features of every position [B, cap, F] bf16 on the device: the
    workload's position-keyed stream when small, else N(0,1) drawn on the
    device from a per-request seeded generator (same distribution and shape).
    Returns (tensor, host numpy bits or None, description)."""
    import numpy as np
    import torch
    from block_diffusion_speculative_hiddens_gb300 import binding
    from workload import feature_rows
    F = cfg.fused_dim
    if B * cap * F <= FEATS_ON_HOST_MAX:
        fs = np.stack([feature_rows(cfg, b, 0, cap).reshape(cap, F) for b in range(B)])
        return binding.bf16_host(fs).to(dev), fs, "workload generator"
    out = torch.empty(B, cap, F, dtype=torch.bfloat16, device=dev)
    for b in range(B):
        g = torch.Generator(device=dev)
        g.manual_seed(1_000_003 * (cfg.seed + 1) + b)
        out[b].normal_(generator=g)
    return out, None, "device generator (torch.normal_, seeded per request)"


def measure(cfg, w_dev, dev, K, W, *, attn_impl=0, weight_fp8=0, temperature=0.0, seed=0, fold=False,
            e2e_steps=0, weights_desc="workload generator", rounds_per_slot=None):
    """Run K timed drafting rounds of `cfg` (after W warm-up rounds) as one
    CUDA graph and return the measurements.

    Timed graph: per round fuse_inject + draft_block, the stand-in verify,
    accept_trim.  The graph is timed with CUDA events on its stream; the
    stand-in verify writes device timestamps (%globaltimer) when it may
    start (the drafter's kernels before it complete) and when its last block
    is done, so the drafter's time -- the graph's time outside the verify
    windows -- and its per-round intervals (accept of the previous round +
    inject + draft of this one) come from the same replay, with no extra
    node in the graph; the lm_head launches carry CUDA-event probes in the
    same graph."""
    import numpy as np
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, binding
    from block_diffusion_speculative_hiddens_gb300.session import RoundState, SyntheticVerify, run_round
    from workload import context_lengths, match_stream

    S, B = cfg.block, cfg.batch
    ctx = context_lengths(cfg).astype(int)
    R = rounds_per_slot or cfg.rounds
    n_groups = math.ceil(K / R) + 1                      # + one group of B slots for warm-up
    n_slots = n_groups * B
    cap = int(ctx.max()) + S * (max(R, W) + 2 + TRACED_ROUNDS) + 64
    mpps = math.ceil(cap / 64) + 1
    F = cfg.fused_dim
    feat_stream, fs, feat_src = feature_stream(cfg, B, cap, dev)
    m = np.empty((max(R, W), B, S), dtype=np.int32)
    u = np.empty_like(m)
    for r in range(max(R, W)):
        m[r], u[r] = match_stream(cfg, r, list(range(B)))
    match, offs = torch.from_numpy(m).to(dev), torch.from_numpy(u).to(dev)

    chunk = 2048
    d = Drafter(cfg, w_dev, max_batch=B, max_slots=n_slots, max_pages=mpps * n_slots, max_pages_per_slot=mpps,
                max_rows=max(chunk, S * B), device=dev.index, attn_impl=attn_impl, weight_fp8=weight_fp8)
    stream = torch.cuda.Stream(device=dev)

    def prefill(g, timed=False):
        """Inject every prompt of slot group g in chunks; with timed, the
        device time (ms) of the fuse_inject calls alone."""
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

    def new_state(g, verify_feats=True):
        st = RoundState(d, B, slots=[g * B + b for b in range(B)], first_token=cfg.first_token)
        ver = SyntheticVerify(st, match, offs, feat_stream if verify_feats else None)
        if temperature > 0:
            st.set_sampling(temperature, seed, ver.round_ctr)
        return st, ver

    states, verifies = [], []
    for g in range(n_groups - 1):
        prefill(g)
        st, ver = new_state(g)
        states.append(st)
        verifies.append(ver)
    gw = n_groups - 1
    prefill_ms = prefill(gw, timed=True)                 # the warm-up group's prefill, timed on its own
    wst, wv = new_state(gw)
    stream.synchronize()

    # warm-up: W rounds on the spare group, as one graph
    d.graph_begin(stream)
    for _ in range(W):
        run_round(wst, wv, stream, folded=fold)
    d.graph_end(stream)
    d.graph_launch(stream)
    stream.synchronize()

    # timed: K rounds, R per slot group, one graph; the verify windows stamped on the device
    stamps = torch.zeros(K, 2, dtype=torch.int64, device=dev)
    d.stamps_arm(stamps, K)
    d.probe_arm(binding.KID_LM_HEAD, K)
    n0 = d.launch_count()
    d.graph_begin(stream)
    for i in range(K):
        run_round(states[i // R], verifies[i // R], stream, folded=fold)
    n_kernels = d.graph_end(stream)
    d.stamps_arm(None, 0)
    launches = d.launch_count() - n0
    stream.synchronize()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
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
    clk = clocks.stop(t_wall0, t_wall1)
    total_ms = e0.elapsed_time(e1)
    st_ns = stamps.cpu().numpy().astype(np.int64)
    lm_ms = d.probe_read(K)
    status = d.read_status()
    accepted = 0
    for g in range(n_groups - 1):
        if min(R, K - g * R) > 0:
            accepted += int((states[g].ctx_len.cpu().numpy() - ctx).sum())

    verify_ms = [(int(e) - int(s)) * 1e-6 for s, e in st_ns]         # the stand-in verify windows
    round_ms = (total_ms - sum(verify_ms)) / K           # every kernel of the K rounds but the verify
    full = sorted((int(st_ns[r][0]) - int(st_ns[r - 1][1])) * 1e-6 for r in range(1, K))  # accept + inject + draft
    pct = (lambda q: full[min(len(full) - 1, int(q * len(full)))]) if full else (lambda q: round_ms)

    # ---- rooflines: the dominant kernel (lm_head + argmax) and the round
    hbm, _, peak_src = peaks()
    tf_burst, tf_sust = tensor_peaks()
    H, V, D = cfg.hidden, cfg.vocab, cfg.head_dim
    M = S * B                                            # block rows the method computes
    fp8 = bool(weight_fp8)
    wb = 1 if fp8 else 2                                 # bytes per projection / embedding weight
    lm_bytes = V * H * wb + (V * 4 if fp8 else 0) + M * H * 2
    lm_flops = 2.0 * M * V * H
    lm_avg_ms = statistics.mean(lm_ms) if lm_ms else float("nan")
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
        ach = lm_bytes / (lm_avg_ms * 1e-3) / 1e9
        lm_roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                   "frac": round(ach / hbm, 4), "frac_of_8000": round(ach / 8000.0, 4),
                   "traffic": None if fp8 else lm_head_traffic(cfg),
                   "peak_source": f"{peak_src} copy bandwidth"}
        if lm_roof["traffic"] is not None:
            lm_roof["traffic_source"] = ("ncu capture on the mid shape, scaled to this launch by the weight "
                                         "bytes it streams (profiles/lm_head_traffic_mid.md)")
    else:
        ach = lm_flops / (lm_avg_ms * 1e-3) / 1e12
        lm_roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": tf_sust, "unit": "TFLOP/s",
                   "frac": round(ach / tf_sust, 4), "traffic": None,
                   "peak_source": "measured bf16 sustained (f16 dense rate equals bf16 on this part)"}
    lm_roof.update({"kernel": "lm_head+argmax (tcgen05 GEMM)", "bytes_per_launch": lm_bytes,
                    "flops_per_launch": lm_flops, "avg_launch_us": round(lm_avg_ms * 1e3, 2)})
    gbs = round_bytes / (round_ms * 1e-3) / 1e9
    res = {
        "value": round((S - 1) * B / (round_ms * 1e-3), 1),
        "round_us": round(round_ms * 1e3, 1),
        "round_us_p10_p50_p90": [round(pct(0.1) * 1e3, 1), round(pct(0.5) * 1e3, 1), round(pct(0.9) * 1e3, 1)],
        "round_samples": len(full),
        "stand_in_verify_us": round(statistics.mean(verify_ms) * 1e3, 1),
        "round_us_with_stand_in_verify": round(total_ms / K * 1e3, 1),
        "accepted_tok_s": round(accepted / (round_ms * K * 1e-3), 1),
        "mean_tau": round(tau, 3),
        "roofline": lm_roof,
        "round_roofline": {"bytes_per_round": int(round_bytes), "achieved_gbs": round(gbs, 1),
                           "frac": round(gbs / hbm, 4), "frac_of_8000": round(gbs / 8000.0, 4)},
        "round_tensor": {"flops_per_round": round_flops, "achieved_tflops": round(
            round_flops / (round_ms * 1e-3) / 1e12, 1), "peak": tf_sust,
            "frac": round(round_flops / (round_ms * 1e-3) / 1e12 / tf_sust, 4)},
        "prefill": {"tokens": int(ctx.sum()), "us": round(prefill_ms * 1e3, 1),
                    "tok_s": round(float(ctx.sum()) / (prefill_ms * 1e-3), 1),
                    "flops": prefill_flops,
                    "tensor_frac": round(prefill_flops / (prefill_ms * 1e-3) / 1e12 / tf_burst, 4),
                    "call": f"dflash_fuse_inject per request in {chunk}-token chunks (device time, not in the round)"},
        "clocks": clk,
        "status_word": status,
        "gpu_launches": launches,
        "graph_kernel_nodes": n_kernels,
        "plan": d.plan(),
        "steps": K,
        "warmup": W,
        "rounds_per_slot": R,
        "slot_groups": n_groups - 1,
        "feature_source": feat_src,
        "weights_source": weights_desc,
    }

    # ---- where the round's time goes: one more round of the warm-up group,
    # captured with every GEMM and attention launch writing per-CTA
    # %globaltimer stamps, replayed TRACED_ROUNDS - 1 times; each launch's
    # time runs from the previous traced launch's end to its own (the small
    # kernels between them count with the launch after them)
    if not fold:
        kt = kernel_times(d, binding, run_round, wst, wv, stream, cfg)
        if kt is not None:
            status |= d.read_status()
            res["status_word"] = status
            g_us, a_us = kt["gemm_us"], kt["attention_us"]
            res["kernel_time"] = kt
            res["gemm_tensor"] = {"flops_per_round": round_flops, "us_per_round": round(g_us, 1),
                                  "achieved_tflops": round(round_flops / (g_us * 1e-6) / 1e12, 1), "peak": tf_sust,
                                  "frac": round(round_flops / (g_us * 1e-6) / 1e12 / tf_sust, 4)}
            res["attention_hbm"] = {"kv_bytes_per_round": int(kv_bytes), "us_per_round": round(a_us, 1),
                                    "achieved_gbs": round(kv_bytes / (a_us * 1e-6) / 1e9, 1),
                                    "frac": round(kv_bytes / (a_us * 1e-6) / 1e9 / hbm, 4)}

    # ---- end to end through the C ABI with host buffers: per round the
    # block's target features and verify streams go host -> device from
    # pinned memory and the round's result comes back; the host prepares
    # round r+1's inputs while round r runs (double-buffered staging)
    if e2e_steps > 0:
        E = min(e2e_steps, R)
        for b in range(B):
            d.reset_slot(gw * B + b, stream)
        prefill(gw)
        st = RoundState(d, B, slots=[gw * B + b for b in range(B)], first_token=cfg.first_token)
        m_dev = torch.zeros(1, B, S, dtype=torch.int32, device=dev)
        u_dev = torch.zeros_like(m_dev)
        ver = SyntheticVerify(st, m_dev, u_dev, None)
        if temperature > 0:
            st.set_sampling(temperature, seed, ver.round_ctr)
        d.graph_begin(stream)
        run_round(st, ver, stream, folded=fold)
        d.graph_end(stream)
        feats_h = [torch.empty(B, S, F, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        mu_h = [torch.empty(2, B, S, dtype=torch.int32).pin_memory() for _ in range(2)]
        out_h = [torch.empty(B, S + 2, dtype=torch.int32).pin_memory() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        fs_host = binding.bf16_host(fs) if fs is not None else feat_stream[:, :S].cpu()
        m_t, u_t = torch.from_numpy(m), torch.from_numpy(u)
        stream.synchronize()

        def prepare(buf, r, pos):
            """Inputs of round r: the features of the block positions of round
            r-1 (pos = that round's first position), the verify streams."""
            for b in range(B):
                if fs is not None:
                    feats_h[buf][b].copy_(fs_host[b, pos[b]:pos[b] + S])
                else:  # the device-drawn stream's first rows stand in on the host
                    feats_h[buf][b].copy_(fs_host[b])
            mu_h[buf][0].copy_(m_t[r % len(m_t)])
            mu_h[buf][1].copy_(u_t[r % len(u_t)])

        t0 = time.perf_counter()
        prepare(0, 0, ctx)
        for r in range(E):
            buf = r & 1
            with torch.cuda.stream(stream):
                st.feats.copy_(feats_h[buf], non_blocking=True)
                m_dev[0].copy_(mu_h[buf][0], non_blocking=True)
                u_dev[0].copy_(mu_h[buf][1], non_blocking=True)
                d.graph_launch(stream)
                out_h[buf][:, :S - 1].copy_(st.draft, non_blocking=True)
                out_h[buf][:, S - 1].copy_(st.accept_len, non_blocking=True)
                out_h[buf][:, S].copy_(st.ctx_len, non_blocking=True)
                done[buf].record(stream)
            if r + 1 < E:
                if r >= 1:  # round r+1 injects round r's block features: round r starts at r-1's confirmed length
                    done[buf ^ 1].synchronize()
                    pos = out_h[buf ^ 1][:, S].numpy().astype(int)
                else:
                    pos = ctx
                prepare(buf ^ 1, r + 1, pos)
        done[(E - 1) & 1].synchronize()
        t_e2e = time.perf_counter() - t0
        h2d = feats_h[0].numel() * 2 + mu_h[0].numel() * 4
        d2h = out_h[0].numel() * 4
        res["e2e"] = {"value": round((S - 1) * B * E / t_e2e, 1), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "steps": E, "round_us": round(t_e2e / E * 1e6, 1),
                      "note": "dflash_graph_launch of one round per step with pinned host staging, double-buffered; "
                              "includes the stand-in verify kernel"}
    d.close()
    del d, states, verifies, feat_stream, match, offs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


TRACED_ROUNDS = 4  # rounds the kernel-time pass adds to the warm-up group (capture + replays)


def kernel_times(d, binding, run_round, st, ver, stream, cfg):
    """GEMM and attention time of one live round (us), from a traced replay;
    None when the launches cannot be attributed."""
    import numpy as np
    import torch
    cap = 16384
    buf = torch.zeros(cap, 8, dtype=torch.int64, device=stream.device)
    d.trace_arm(binding.KID_ALL, buf, cap)
    d.graph_begin(stream)
    run_round(st, ver, stream)
    d.graph_end(stream)
    d.trace_arm(0)
    for _ in range(TRACED_ROUNDS - 1):
        d.graph_launch(stream)
    stream.synchronize()
    rows = buf.cpu().numpy().astype(np.int64)
    names = ["fc", "inject"] + ["qkv", "attention", "wo", "gate_up", "down"] * cfg.n_layers + ["lm_head"]
    segs, pos = [], 0
    while pos < cap and rows[pos, 0] > 0 and len(segs) < len(names):
        grid = int(rows[pos, 6]) >> 32
        if grid <= 0 or pos + grid > cap:
            return None
        seg = rows[pos:pos + grid]
        segs.append((int(seg[:, 0][seg[:, 0] > 0].min()), int(seg[:, 5].max())))
        pos += grid
    if len(segs) != len(names):
        return None
    own = {}
    prev_end = segs[0][0]
    for (start, end), nm in zip(segs, names):
        own[nm] = own.get(nm, 0.0) + (end - prev_end) * 1e-3
        prev_end = end
    gemm = sum(v for k, v in own.items() if k != "attention")
    return {"gemm_us": round(gemm, 1), "attention_us": round(own["attention"], 1),
            "per_kind_us": {k: round(v, 1) for k, v in own.items()},
            "traced_us": round((segs[-1][1] - segs[0][0]) * 1e-3, 1),
            "source": "one traced replay of a round (per-CTA %globaltimer stamps); a launch's time runs from the "
                      "previous traced launch's end to its own, the small kernels between counting with the next"}


def workload_desc(cfg, ctx_mean):
    B, H, D, F = cfg.batch, cfg.hidden, cfg.head_dim, cfg.fused_dim
    ctx_desc = f"prompt {cfg.ctx0}" if cfg.ctx0 else f"prompts U[{cfg.ctx_range[0]}, {cfg.ctx_range[1]}]"
    p_desc = f"match p {cfg.match_p}" if cfg.match_p is not None else f"match p U[{cfg.p_range[0]}, {cfg.p_range[1]}]"
    return (f"{cfg.name} drafter batch {B}: H{H}, {cfg.n_q_heads}q/{cfg.n_kv_heads}kv x{D}, I{cfg.intermediate}, "
            f"{cfg.n_layers} layers, V{cfg.vocab}, fusion {F}->{H}, {ctx_desc}, block {cfg.block}, {p_desc}")


SUMMARY_KEYS = ("value", "round_us", "round_us_p10_p50_p90", "round_samples", "stand_in_verify_us", "mean_tau",
                "accepted_tok_s", "roofline", "round_roofline", "round_tensor", "prefill", "clocks", "steps",
                "warmup", "gpu_launches", "plan", "status_word", "weights_source", "feature_source", "gemm_tensor",
                "attention_hbm", "kernel_time")


def run_gpu(args):
    import torch
    from block_diffusion_speculative_hiddens_gb300 import weights_to_device
    from workload import context_lengths, get_config, make_weights

    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    cfg = get_config(args.config)
    if args.block:
        cfg = cfg.with_(block=args.block)
    B = cfg.batch
    K = args.steps if args.steps is not None else (512 if B == 1 else (args.rounds_per_slot or cfg.rounds))
    W = args.warmup
    w_np = make_weights(cfg)
    w_dev = weights_to_device(w_np, 0)
    head = measure(cfg, w_dev, dev, K, W, attn_impl=args.attn_impl, weight_fp8=1 if args.weights == "fp8" else 0,
                   temperature=args.temperature, seed=args.seed, fold=args.fold_inject, e2e_steps=args.e2e_steps,
                   rounds_per_slot=args.rounds_per_slot)
    ctx = context_lengths(cfg)
    res = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "tok/s",
        "n_gpus": 1,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(head["round_us"] * 1e-3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 activations, fp8 e4m3 weights" if args.weights == "fp8" else "f16",
        "data": f"synthetic (seeded N(0,1) target features from the {head['feature_source']}, N(0,0.02) "
                "random-init weights from the workload generator, stand-in verify)",
        "config": {"workload": workload_desc(cfg, float(ctx.mean())), "batch": B, "prompt_mean": float(ctx.mean()),
                   "rounds_per_slot": head["rounds_per_slot"], "slot_groups": head["slot_groups"],
                   "attn_impl": ["library choice", "warp MMAs", "tcgen05"][args.attn_impl],
                   "weights": "fp8 e4m3, per-row scales" if args.weights == "fp8" else "bf16 (held as f16)",
                   "drafting": (f"sampled at temperature {args.temperature} (Gumbel-max, seed {args.seed})"
                                if args.temperature > 0 else "greedy argmax"),
                   "round_call": "dflash_draft_round" if args.fold_inject
                   else "dflash_fuse_inject+dflash_draft_block",
                   "l2": "inputs larger than L2 (the drafter's weights stream every round)",
                   "parallelism": "single GPU"},
        "timing": "one CUDA graph of the K timed rounds, timed with CUDA events on its stream; the stand-in verify "
                  "stamps its window on the device (%globaltimer): ms_per_step is the graph's time outside the "
                  "verify windows / K, the percentiles are the same replay's per-round intervals between verify "
                  "windows (each an accept, a fuse_inject and a draft_block)",
    }
    res.update({k: head[k] for k in ("round_us", "round_us_p10_p50_p90", "round_samples", "stand_in_verify_us",
                                     "round_us_with_stand_in_verify", "accepted_tok_s", "mean_tau", "gpu_launches",
                                     "plan", "graph_kernel_nodes", "roofline", "round_roofline", "round_tensor",
                                     "prefill", "clocks", "status_word")})
    res.update({k: head[k] for k in ("gemm_tensor", "attention_hbm", "kernel_time") if k in head})
    if "e2e" in head:
        res["e2e"] = head["e2e"]

    names = [] if args.workloads == "none" else (
        list(EXTRA_WORKLOADS) if args.workloads == "all" else [n for n in args.workloads.split(",") if n])
    workloads = {cfg.name: {k: head[k] for k in SUMMARY_KEYS if k in head}} if names else {}
    for name in names:
        if name == cfg.name:
            continue
        wc = get_config(name)
        if name == "tiny":
            wd, src = weights_to_device(make_weights(wc), 0), "workload generator"
        elif (wc.hidden, wc.n_q_heads, wc.n_kv_heads, wc.intermediate, wc.n_layers, wc.vocab, wc.seed) == \
                (cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.intermediate, cfg.n_layers, cfg.vocab, cfg.seed) \
                and args.weights == "bf16":
            wd, src = w_dev, "workload generator (the headline drafter's weights)"
        else:
            wd, src = device_weights(wc, dev, 7919 + len(workloads)), \
                "device generator (torch.normal_ N(0,0.02), seeded; gains 1)"
        r = measure(wc, wd, dev, EXTRA_STEPS.get(name, 16), min(W, 3), attn_impl=args.attn_impl, weights_desc=src)
        if wd is not w_dev:
            del wd
        s = {k: r[k] for k in SUMMARY_KEYS if k in r}
        s["workload"] = workload_desc(wc, 0.0)
        workloads[name] = s
    if workloads:
        res["workloads"] = workloads
    return res, cfg, w_np


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


ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def oracle_one_thread(name: str, rounds: int, budget_s: float):
    """The oracle's round time on one host thread (a child process whose BLAS
    runs single-threaded), or None if it could not run."""
    env = dict(os.environ, **{k: "1" for k in ONE_THREAD_ENV})
    code = ("import json, statistics, sys; sys.path.insert(0, %r); import bench; from workload import get_config; "
            "t, _ = bench.oracle_round_seconds(get_config(%r), %r, %d); print(json.dumps(t))"
            % (ROOT, name, budget_s, rounds))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=budget_s * 4 + 60)
        times = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception:
        return None
    return times


def cpu_baseline_line(cfg, weights, budget_s):
    times, _ = oracle_round_seconds(cfg, budget_s, 4, weights=weights)
    rs = statistics.mean(times)
    out = {"value": round((cfg.block - 1) / rs, 3), "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"{len(times)} round(s) of the same workload (request 0) after an untimed "
                     f"{cfg.ctx0 or cfg.ctx_range[0]}-token prefill, float64 NumPy, BLAS on every host core"}
    one = oracle_one_thread("tiny", 8, 20.0)
    if one:
        rs1 = statistics.mean(one)
        out["tiny_one_thread"] = {"value": round(15 / rs1, 3), "unit": "tok/s", "cores": 1,
                                  "ms_per_round": round(rs1 * 1e3, 2),
                                  "sample": f"{len(one)} rounds of the tiny workload after its 128-token prefill, "
                                            "one host thread"}
    return out


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

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

    if args.gpus > 1 or world > 1:
        # one GPU per process: there is no multi-GPU path to run or time
        if rank == 0:
            print(json.dumps({"metric": METRIC, "n_gpus": max(args.gpus, world), "value": None,
                              "unavailable": "single-GPU library: a replica per GPU is an independent process "
                                             "running this benchmark with --gpus 1; nothing is shared or "
                                             "exchanged between GPUs, so no multi-GPU run is made"}), flush=True)
        return

    import torch
    if args.spec_generate:
        print(json.dumps(run_spec_generate(args)), flush=True)
        return
    res, cfg, w_np = run_gpu(args)
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_line(cfg, w_np, args.cpu_budget_s)
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

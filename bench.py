#!/usr/bin/env python
"""Benchmark: one DFlash drafting-plus-acceptance round per step on GB300.

Workload (default): the Qwen3-8B-shaped drafter at batch 1 -- hidden 4096,
32/8 heads x 128, SwiGLU 12288, 5 layers, vocabulary 151936, fusion
20480 -> 4096 -- with a 2048-token prompt, block 16 and a stand-in verify
that copies each draft with probability 0.9.  One step = fuse+inject the
previous round's accepted features, draft one block, stand-in verify,
accept/trim, all captured in one CUDA graph.  Synthetic seeded data and
random-init weights of that architecture.

Every scenario pass is 64 rounds from the 2048-token prompt; timed steps
cycle through identically prefilled request slots, 64 rounds per slot, so K
steps always run rounds of the stated scenario.

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
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3-8b")
    ap.add_argument("--rounds-per-slot", type=int, default=None)
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=25.0)
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
    req = O.OracleRequest(cfg, L0 + 16 * (max_rounds + 2))
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

def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch
    from block_diffusion_speculative_hiddens_gb300 import Drafter, binding, weights_to_device
    from block_diffusion_speculative_hiddens_gb300.session import RoundState, SyntheticVerify, run_round
    from workload import feature_rows, get_config, make_weights, match_stream

    torch.cuda.set_device(local_rank)
    dev = torch.device(f"cuda:{local_rank}")
    cfg = get_config(args.config)
    assert cfg.batch == 1 and cfg.ctx0, "bench workload is a batch-1 scenario"
    B = 1
    R = args.rounds_per_slot or cfg.rounds
    K, W = args.steps, args.warmup
    n_slots = math.ceil(K / R) + 1                       # + one slot for warm-up
    L0 = cfg.ctx0
    cap = L0 + cfg.block * (max(R, W) + 2) + 64
    mpps = math.ceil(cap / 64) + 1

    w_dev = weights_to_device(make_weights(cfg), local_rank)
    F = cfg.fused_dim
    fs = feature_rows(cfg, 0, 0, cap).reshape(1, cap, F)
    feat_stream = binding.bf16_host(fs).to(dev)
    m = np.empty((max(R, W), 1, 16), dtype=np.int32)
    u = np.empty_like(m)
    for r in range(max(R, W)):
        m[r], u[r] = match_stream(cfg, r, [0])
    match, offs = torch.from_numpy(m).to(dev), torch.from_numpy(u).to(dev)

    chunk = 2048
    d = Drafter(cfg, w_dev, max_batch=B, max_slots=n_slots, max_pages=mpps * n_slots,
                max_pages_per_slot=mpps, max_rows=max(chunk, 16 * B), device=local_rank)
    stream = torch.cuda.Stream(device=dev)
    states, verifies = [], []
    with torch.cuda.stream(stream):
        for j in range(n_slots):
            st = RoundState(d, B, slots=[j], first_token=cfg.first_token)
            for p0 in range(0, L0, chunk):
                n = min(chunk, L0 - p0)
                d.fuse_inject(st.slots, feat_stream[:, p0:p0 + n], n,
                              torch.tensor([n], dtype=torch.int32, device=dev), stream)
            states.append(st)
            verifies.append(SyntheticVerify(st, match, offs, feat_stream))
    stream.synchronize()

    # warm-up: W rounds on the spare slot, as one graph
    wst, wv = states[-1], verifies[-1]
    d.graph_begin(stream)
    for _ in range(W):
        run_round(wst, wv, stream, folded=args.fold_inject)
    d.graph_end(stream)
    d.graph_launch(stream)
    stream.synchronize()

    # timed: K rounds, R per slot, one graph; lm_head bracketed by event probes
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
    for j in range(n_slots - 1):
        rounds_j = min(R, K - j * R)
        if rounds_j > 0:
            accepted += int(states[j].ctx_len.item()) - L0
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # ---- the stand-in verify on its own, and the per-round distribution: one
    # more graph of up to R rounds on a fresh copy of the prompt, with
    # timeline marks at every round start and around the verify (the marks'
    # event nodes cost a little overlap, so the headline mean stays the
    # unmarked graph's, minus the verify's mean)
    Ki = min(R, K)
    st_i = RoundState(d, B, slots=[n_slots - 1], first_token=cfg.first_token)
    d.reset_slot(n_slots - 1, stream)
    with torch.cuda.stream(stream):
        for p0 in range(0, L0, chunk):
            n = min(chunk, L0 - p0)
            d.fuse_inject(st_i.slots, feat_stream[:, p0:p0 + n], n,
                          torch.tensor([n], dtype=torch.int32, device=dev), stream)
    ver_i = SyntheticVerify(st_i, match, offs, feat_stream)

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
        st = RoundState(d, B, slots=[n_slots - 1], first_token=cfg.first_token)
        d.reset_slot(n_slots - 1, stream)
        for p0 in range(0, L0, chunk):
            n = min(chunk, L0 - p0)
            d.fuse_inject(st.slots, feat_stream[:, p0:p0 + n], n,
                          torch.tensor([n], dtype=torch.int32, device=dev), stream)
        m_dev = torch.zeros(1, 1, 16, dtype=torch.int32, device=dev)
        u_dev = torch.zeros_like(m_dev)
        ver = SyntheticVerify(st, m_dev, u_dev, None)
        d.graph_begin(stream)
        run_round(st, ver, stream, folded=args.fold_inject)
        d.graph_end(stream)
        feats_h = torch.empty(1, 16, F, dtype=torch.bfloat16).pin_memory()
        mu_h = torch.empty(2, 16, dtype=torch.int32).pin_memory()
        out_h = torch.empty(15 + 3, dtype=torch.int32).pin_memory()
        fs_host = binding.bf16_host(fs[0])
        stream.synchronize()
        # the round's inject consumes the previous round's block features
        # (positions prev_L .. prev_L+15, the first accept_len of them)
        prev_L = cur_L = L0
        h2d = d2h = 0
        t0 = time.perf_counter()
        for r in range(E):
            feats_h.copy_(fs_host[prev_L:prev_L + 16].unsqueeze(0))
            mu_h[0].copy_(torch.from_numpy(m[r % len(m), 0]))
            mu_h[1].copy_(torch.from_numpy(u[r % len(u), 0]))
            with torch.cuda.stream(stream):
                st.feats.copy_(feats_h, non_blocking=True)
                m_dev[0, 0].copy_(mu_h[0], non_blocking=True)
                u_dev[0, 0].copy_(mu_h[1], non_blocking=True)
                d.graph_launch(stream)
                out_h[:15].copy_(st.draft[0], non_blocking=True)
                out_h[15:16].copy_(st.accept_len, non_blocking=True)
                out_h[16:17].copy_(st.bonus, non_blocking=True)
                out_h[17:18].copy_(st.ctx_len, non_blocking=True)
            stream.synchronize()
            prev_L, cur_L = cur_L, int(out_h[17])
            h2d = feats_h.numel() * 2 + mu_h.numel() * 4
            d2h = out_h.numel() * 4
        t_e2e = time.perf_counter() - t0
        if world > 1:
            t = torch.tensor([t_e2e], dtype=torch.float64, device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            t_e2e = float(t.item())
        e2e = {"value": round(15 * B * E * world / t_e2e, 1), "unit": "tok/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": E,
               "round_us": round(t_e2e / E * 1e6, 1)}

    # ---- roofline of the dominant kernel (lm_head + argmax) and of the round
    hbm, bf16_tf, peak_src = peaks()
    H, V = cfg.hidden, cfg.vocab
    lm_bytes = V * H * 2 + 16 * B * H * 2
    lm_avg_ms = statistics.mean(lm_ms) if lm_ms else float("nan")
    lm_gbs = lm_bytes / (lm_avg_ms * 1e-3) / 1e9
    round_ms_incl = ms / K
    round_ms = round_ms_incl - verify_ms  # the stand-in verify is not part of the round
    wb = cfg.weight_bytes()
    avg_ctx = L0 + accepted / max(1, (n_slots - 1)) / 2
    kv_bytes = cfg.n_layers * (avg_ctx + 16) * cfg.n_kv_heads * cfg.head_dim * 2 * 2
    round_bytes = wb + kv_bytes + 8 * F * 2
    res = {
        "metric": METRIC,
        "value": round(15 * B * world / (round_ms * 1e-3), 1),
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
        "mean_tau": round(accepted / K, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded N(0,1) target features, N(0,0.02) random-init weights, stand-in verify)",
        "config": {"workload": f"{cfg.name} drafter batch 1: H{H}, {cfg.n_q_heads}q/{cfg.n_kv_heads}kv x"
                               f"{cfg.head_dim}, I{cfg.intermediate}, {cfg.n_layers} layers, V{V}, fusion "
                               f"{F}->{H}, prompt {L0}, block 16, match p {cfg.match_p}",
                   "batch": B, "prompt": L0, "rounds_per_slot": R,
                   "round_call": "dflash_draft_round" if args.fold_inject
                   else "dflash_fuse_inject+dflash_draft_block", "slots": n_slots - 1,
                   "l2": "inputs larger than L2 (3.3 GB of weights stream every round)",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": launches_captured,
        "graph_kernel_nodes": n_kernels,
        "roofline": {"bound": "hbm", "kernel": "lm_head+argmax (tcgen05 GEMM)",
                     "achieved": round(lm_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(lm_gbs / hbm, 4), "traffic": lm_head_traffic(cfg), "peak_source": peak_src,
                     "bytes_per_launch": lm_bytes, "avg_launch_us": round(lm_avg_ms * 1e3, 2)},
        "round_roofline": {"bytes_per_round": int(round_bytes), "achieved_gbs": round(
            round_bytes / (round_ms * 1e-3) / 1e9, 1), "frac": round(round_bytes / (round_ms * 1e-3) / 1e9 / hbm, 4)},
        "clocks": clk,
        "status_word": status,
        "e2e": e2e,
    }
    return res, cfg


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
        budget = 150.0
        times, taus = oracle_round_seconds(cfg, budget, max(1, args.steps))
        used = times[1:] if len(times) > 1 else times
        rs = statistics.mean(used)
        val = 15 / rs
        line = {"impl": "reference", "metric": METRIC, "value": round(val, 3), "unit": "tok/s",
                "n_gpus": args.gpus, "steps": len(used), "warmup": len(times) - len(used),
                "ms_per_step": round(rs * 1e3, 1), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": f"{cfg.name} drafter batch 1, prompt {cfg.ctx0}, block 16"},
                "cpu_baseline": {"value": round(val, 3), "unit": "tok/s", "cores": os.cpu_count(),
                                 "kind": "oracle",
                                 "sample": f"{len(times)} rounds of request 0 after an untimed {cfg.ctx0}-token "
                                           f"prefill, stopped after {budget:.0f} s"},
                "e2e": {"value": round(val, 3), "unit": "tok/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    res, cfg = run_gpu(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times, taus = oracle_round_seconds(cfg, args.cpu_budget_s, 4)
        rs = statistics.mean(times)
        res["cpu_baseline"] = {"value": round(15 / rs, 3), "unit": "tok/s", "cores": os.cpu_count(),
                               "kind": "oracle",
                               "sample": f"{len(times)} round(s) of the same workload (request 0) after an "
                                         f"untimed {cfg.ctx0}-token prefill, float64 NumPy"}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

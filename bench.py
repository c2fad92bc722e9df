#!/usr/bin/env python
"""Benchmark of the hybrid attention step (Hybrid Forcing) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hf|reference]

One step = the whole hot path over one chunk of the 832x480 streaming
workload ("realistic": batch 1, 12 heads, head_dim 128, 1560 tokens per
latent frame, 3-frame chunk, 9-frame window, block 64, top-K 25 % = 57 of
225 key blocks, 30 frames already in the linear state):
  hf_absorb_evicted_strided  (the 3 frames the chunk evicts, from the ring)
  hf_hybrid_forward          (pool -> score/top-K -> state prep -> sparse
                              attention with fused linear read + sum)
Inputs are synthetic (seeded Philox, see workloads.py) and resident in HBM;
L2 is flushed (256 MB write) before every timed step; each step is timed
with CUDA events on the launching stream.  value = algorithmic FLOPs of the
step / device time (effective TFLOP/s); us_per_latent_frame = time / 3.

--impl reference times the CPU oracle (plain C, fp64) on the host cores on
a bounded sample of the same step.  Multi-GPU (torchrun): every rank runs
an independent replica (the layer shards over heads with no exchange);
value = all ranks' FLOPs / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hybrid-attn layer µs per latent frame & effective TFLOP/s (% bf16 TC peak), 1 B300"
WORKLOAD = "realistic"
L2_FLUSH_BYTES = 256 << 20


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def step_flops(w, idx: np.ndarray, n_ev_tokens: int) -> dict:
    """Algorithmic FLOPs of one step (only what the method must compute).
    idx: int32 [BH, nQB, K] selected key blocks."""
    d, nf, beta, bpf = w.head_dim, w.tokens_per_frame, w.block_size, w.blocks_per_frame
    BH = w.heads_total
    blk_rows = np.array([min(beta, nf - j * beta) for j in range(bpf)], np.int64)
    nk_sel = blk_rows[idx % bpf].sum(axis=2)                  # [BH, nQB] selected key tokens
    nq = np.tile(blk_rows, w.chunk_frames)[None, :]           # [1, nQB] query tokens per block
    attn = 4.0 * d * float((nq * nk_sel).sum())
    Nq = w.chunk_frames * nf
    lin = (2.0 * d * d + 2.0 * d) * Nq * BH
    absorb = (2.0 * d * d + d) * n_ev_tokens * BH
    score = 2.0 * w.n_qb() * (w.n_win(0) * bpf) * d * BH
    return {"attn": attn, "lin": lin, "absorb": absorb, "score": score,
            "total": attn + lin + absorb + score}


def step_bytes(w, n_ev_tokens: int) -> dict:
    BH, d, nf = w.heads_total, w.head_dim, w.tokens_per_frame
    Nq = w.chunk_frames * nf
    Nk = w.n_win(0) * nf
    q = BH * Nq * d * 2
    kv = 2 * BH * Nk * d * 2
    o = q
    ev = 2 * BH * n_ev_tokens * d * 2
    state = 2 * BH * (d * d + d) * 4
    pool = q + BH * Nk * d * 2           # pooling reads Q and K of the window
    return {"compulsory": q + kv + o + ev + state, "pool": pool, "absorb": ev + state}


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# --------------------------------------------------------------------------
def oracle_sample(w, rows_per_head: int, inputs, seed: int = 0):
    """Runs the oracle on a row sample of the step (all heads: pooling,
    scores and top-K in full, attention + linear read for the sampled rows)
    plus the absorb of the evicted frames of two heads.  Returns
    (seconds, algorithmic FLOPs of the sample)."""
    import oracle
    Q, Kw, Vw, Kev3, Vev3, S, z = inputs
    nq = w.chunk_frames * w.tokens_per_frame
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(nq, size=rows_per_head, replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    out = oracle.hybrid_forward(Q, Kw, Vw, S, z, C=w.chunk_frames, n_win=w.n_win(0), nf=w.tokens_per_frame,
                                beta=w.block_size, k=w.k_for(0), rows=rows)
    oracle.state_from_frames(Kev3[:2], Vev3[:2], S[:2], z[:2])
    dt = time.perf_counter() - t0
    idx = out["idx"]
    d, nf, beta, bpf = w.head_dim, w.tokens_per_frame, w.block_size, w.blocks_per_frame
    blk_rows = np.array([min(beta, nf - j * beta) for j in range(bpf)], np.int64)
    qb = (rows // nf) * bpf + (rows % nf) // beta
    nk = blk_rows[idx[:, qb, :] % bpf].sum(axis=2)           # [BH, R]
    flops = 4.0 * d * float(nk.sum()) + (2.0 * d * d + 2.0 * d) * len(rows) * w.heads_total
    flops += (2.0 * d * d + d) * Kev3.shape[1] * 2
    flops += 2.0 * w.n_qb() * w.n_kb(0) * d * w.heads_total
    return dt, flops


def oracle_inputs(w):
    """CPU copies of the step's inputs for the oracle (generated on the CPU)."""
    import oracle
    from hybrid_sparse_linear_scores_b300 import synth
    from hybrid_sparse_linear_scores_b300.workloads import frames_tensor
    flat = lambda x: x.reshape(x.shape[0], -1, x.shape[-1])
    Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(0)))
    Kw = flat(frames_tensor(w, synth.STREAM_K, w.window(0)))
    Vw = flat(frames_tensor(w, synth.STREAM_V, w.window(0)))
    ev = w.window(0)[:w.chunk_frames]
    Kev3 = flat(frames_tensor(w, synth.STREAM_K, ev))
    Vev3 = flat(frames_tensor(w, synth.STREAM_V, ev))
    # the state content does not change the oracle's work: a small absorbed history
    S, z = oracle.state_from_frames(Kev3, Vev3)
    return Q, Kw, Vw, Kev3, Vev3, S, z


def cpu_baseline(w, target_s: float):
    import oracle
    inputs = oracle_inputs(w)
    dt, fl = oracle_sample(w, 8, inputs)
    per_row = max(dt / 8, 1e-4)
    rows = int(max(8, min(w.chunk_frames * w.tokens_per_frame, target_s / per_row)))
    dt, fl = oracle_sample(w, rows, inputs, seed=1)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{rows} query rows of each of {w.heads_total} heads (pooling, scores and top-K of all "
                      f"blocks) + absorb of {w.chunk_frames} frames for 2 heads; {dt:.1f} s wall",
            "seconds": dt}


def run_reference(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.barrier()
            dist.destroy_process_group()
            return
    import oracle
    from hybrid_sparse_linear_scores_b300.workloads import CONFIGS
    w = CONFIGS[args.workload]
    inputs = oracle_inputs(w)
    dt, _ = oracle_sample(w, 8, inputs)
    budget = 150.0 / max(1, args.steps + args.warmup)         # whole run within a few minutes
    rows = int(max(4, min(w.chunk_frames * w.tokens_per_frame, budget / max(dt / 8, 1e-4))))
    for i in range(args.warmup):
        oracle_sample(w, rows, inputs, seed=100 + i)
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = oracle_sample(w, rows, inputs, seed=i)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_desc(w), "sample_rows_per_head": rows},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"{rows} query rows per head of {w.heads_total} heads + absorb of "
                                       f"{w.chunk_frames} frames for 2 heads, per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def workload_desc(w):
    return (f"{w.name}: b{w.batch} H{w.heads} d{w.head_dim} N_f{w.tokens_per_frame} C{w.chunk_frames} "
            f"W{w.window_frames} beta{w.block_size} K{w.k_for(0)}/{w.n_kb(0)} state {w.absorbed_frames} frames")


# --------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------
def run_hf(args):
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from hybrid_sparse_linear_scores_b300 import binding as hb
    from hybrid_sparse_linear_scores_b300 import synth
    from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer
    from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, frames_tensor

    w = CONFIGS[args.workload]
    cfg = hb.make_config(w.batch, w.heads, w.head_dim, w.tokens_per_frame, w.window_frames, w.chunk_frames,
                         w.block_size, w.k_for(0))
    L = HybridAttentionLayer(cfg, dev)
    flat = lambda x: x.reshape(x.shape[0], -1, x.shape[-1])
    # state: the absorbed history, built on the device
    for f0 in range(0, w.absorbed_before(0), 6):
        fr = list(range(f0, min(f0 + 6, w.absorbed_before(0))))
        K = frames_tensor(w, synth.STREAM_K, fr, dev)
        V = frames_tensor(w, synth.STREAM_V, fr, dev)
        hb.hf_absorb_evicted(cfg, L.S, L.z, flat(K), flat(V), len(fr) * w.tokens_per_frame, L.ws)
    win = w.window(0)
    Kw = frames_tensor(w, synth.STREAM_K, win, dev)
    Vw = frames_tensor(w, synth.STREAM_V, win, dev)
    for i, f in enumerate(win):
        L.Kc[:, f % w.window_frames] = Kw[:, i]
        L.Vc[:, f % w.window_frames] = Vw[:, i]
    L.frames = w.frames_so_far(0)
    Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(0), dev))
    O = torch.empty_like(Q)
    idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(0)), dtype=torch.int32, device=dev)
    evict_slot = win[0] % w.window_frames                    # the oldest chunk's slots (contiguous)
    n_ev = w.chunk_frames * w.tokens_per_frame
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    E = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in E:
        e.record(stream)

    def one_step(events=None):
        if events is not None:
            events[0].record(stream)
        L.absorb_slots(evict_slot, w.chunk_frames, stream)
        if events is not None:
            hb.hf_hybrid_forward_profiled(cfg, Q, L.Kc, L.Vc, L.ss, L.slot_map(), L.n_win(), L.S, L.z, O, idx, L.ws,
                                          events[1:6], stream)
        else:
            L.forward(Q, O, idx, stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        one_step(E)
    torch.cuda.synchronize()
    L.check_device_status()
    fl = step_flops(w, idx.cpu().numpy(), n_ev)
    by = step_bytes(w, n_ev)

    # ---- timed region: K steps, L2 flushed before each, events per kernel ----
    names = ["absorb", "pool", "score_topk", "state_prep", "attention"]
    times = {n: [] for n in names}
    step_ms = []
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        evs = []
        for _ in range(args.steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            flush.zero_()
            one_step(ev)
            evs.append(ev)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    if ws > 1:
        dist.barrier()
    for ev in evs:
        for i, n in enumerate(names):
            times[n].append(ev[i].elapsed_time(ev[i + 1]))
        step_ms.append(ev[0].elapsed_time(ev[5]))
    L.check_device_status()
    clocks = clk.summary()
    ms = statistics.mean(step_ms)
    if ws > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # warm-L2 timing, for context
    for _ in range(3):
        one_step()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(args.steps):
        one_step()
    s1.record(stream)
    torch.cuda.synchronize()
    warm_ms = s0.elapsed_time(s1) / args.steps

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.skip_e2e:
        Qh = Q.cpu().pin_memory()
        Kn = Kw[:, -w.chunk_frames:].contiguous().cpu().pin_memory()
        Vn = Vw[:, -w.chunk_frames:].contiguous().cpu().pin_memory()
        Oh = torch.empty(Q.shape, dtype=Q.dtype).pin_memory()
        Qd, Knd, Vnd = torch.empty_like(Q), torch.empty_like(Kw[:, :w.chunk_frames]), torch.empty_like(
            Kw[:, :w.chunk_frames])
        chunk_slot = w.chunk(0)[0] % w.window_frames

        def e2e_step():
            Qd.copy_(Qh, non_blocking=True)
            Knd.copy_(Kn, non_blocking=True)
            Vnd.copy_(Vn, non_blocking=True)
            L.absorb_slots(evict_slot, w.chunk_frames, stream)
            L.Kc[:, chunk_slot:chunk_slot + w.chunk_frames].copy_(Knd)
            L.Vc[:, chunk_slot:chunk_slot + w.chunk_frames].copy_(Vnd)
            L.forward(Qd, O, idx, stream)
            Oh.copy_(O, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        h2d = Qh.numel() * 2 + Kn.numel() * 2 + Vn.numel() * 2
        d2h = Oh.numel() * 2
        e2e = {"value": fl["total"] * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    pk = peaks()
    attn_ms = statistics.mean(times["attention"])
    attn_tf = (fl["attn"] + fl["lin"]) / (attn_ms * 1e-3) / 1e12
    value = fl["total"] * ws / (ms * 1e-3) / 1e12
    per_kernel = {n: {"ms": statistics.mean(times[n]), "share": statistics.mean(times[n]) / ms} for n in names}
    per_kernel["absorb"]["GB_s"] = by["absorb"] / (per_kernel["absorb"]["ms"] * 1e-3) / 1e9
    per_kernel["pool"]["GB_s"] = by["pool"] / (per_kernel["pool"]["ms"] * 1e-3) / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if os.path.exists(tp):
        traffic = json.load(open(tp)).get("dram_bytes_per_launch")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "l2": "flushed (256 MB write) before every step; "
                   "step time = CUDA events around the step's kernels", "parallelism": f"replicas x{ws}"},
        "us_per_latent_frame": 1000 * ms / w.chunk_frames,
        "pct_bf16_peak": 100 * value / pk["bf16_tflops"],
        "warm_l2_ms_per_step": warm_ms,
        "flops_per_step": fl, "bytes_per_step": by,
        "kernels": per_kernel,
        "roofline": {"bound": "tensor", "kernel": "attention (sparse softmax + fused linear read)",
                     "achieved": attn_tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": attn_tf / pk["bf16_tflops"], "traffic": traffic,
                     "peak_source": pk["source"] + " burst", "peak_sustained": pk["bf16_tflops_sustained"]},
        "gpu_launches": 5 * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if e2e:
        line["e2e"] = e2e
    if rank == 0 and ws == 1 and not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_baseline_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("hf", "reference"), default="hf")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_hf(args)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the hybrid attention step (Hybrid Forcing) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hf|reference]

One step = the whole hot path over one chunk of the 832x480 streaming
workload ("realistic": batch 1, 12 heads, head_dim 128, 1560 tokens per
latent frame, 3-frame chunk, 9-frame window, block 64, top-K 25 % = 57 of
225 key blocks, 30 frames already in the linear state):
  hf_absorb_evicted_strided  (the 3 frames the chunk evicts, from the ring;
                              it also writes the state's tensor-core operand)
  hf_pool_keys               (key blocks of the chunk's 3 new frames, into
                              the pooled-key cache)
  hf_hybrid_forward_ex       (prologue: query pooling, scores against the
                              cached key pools, top-K; then sparse attention
                              with the linear read and the sum fused in)
The absorb runs on a second stream beside the key pooling and the prologue,
which do not read the state; the attention waits for it (an event).
Inputs are synthetic (seeded Philox, see workloads.py) and resident in HBM.
The step is captured once as a CUDA graph (its 4 kernels on two streams, no
host work in between) and replayed; L2 is flushed (256 MB write) before every timed
replay, and each replay is timed with CUDA events on the launching stream.
value = algorithmic FLOPs of the step / device time (effective TFLOP/s);
us_per_latent_frame = time / 3.  A second graph of the same step records
events between its kernels (external event nodes) for the per-kernel
breakdown and the attention kernel's roofline figure.  e2e streams chunks from pinned host memory through
stream.HostStreamer (copies overlapped with compute).

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
DENOISE_STEPS = 4          # "few-step" denoising per chunk (the pages give no number)
ROPE_BASE = 10000.0        # rotary base frequency of the RoPE pre-step (the pages give none)


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    """The slowest rank's value (every rank gets it); x itself when ws == 1."""
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, ws: int, ms_slowest: float) -> float:
    """Whole-job TFLOP/s: the work of all ws ranks over the slowest rank's time."""
    return flops_per_rank_step * ws / (ms_slowest * 1e-3) / 1e12


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
    # the prologue reads the chunk's queries (pooled keys and indices are small and
    # stay in L2); the absorb reads the evicted K/V and the state and writes the
    # state and its bf16 hi/lo tensor-core operand
    prologue = q
    pool_k = BH * w.chunk_frames * nf * d * 2   # pooling the new chunk's keys (the cache holds the rest)
    smma = BH * d * d * 2 * 2
    return {"compulsory": q + kv + o + ev + state, "prologue": prologue, "pool_k": pool_k,
            "absorb": ev + state + smma}


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
    # the state's content does not change the oracle's work: a small absorbed history
    S, z = oracle.state_from_frames(Kev3, Vev3)
    return Q, Kw, Vw, Kev3, Vev3, S, z


def oracle_step(w, inputs, heads, rows, seed: int = 0):
    """The oracle on (a sample of) one step: for the given heads, the absorb
    of the chunk's evicted frames, pooling, scores and top-K of every block,
    and attention + linear read for `rows` query rows (None = all rows).
    Returns (seconds, algorithmic FLOPs done)."""
    import oracle
    Q, Kw, Vw, Kev3, Vev3, S, z = inputs
    nq = w.chunk_frames * w.tokens_per_frame
    r = None
    if rows is not None and rows < nq:
        rng = np.random.default_rng(seed)
        r = np.sort(rng.choice(nq, size=rows, replace=False)).astype(np.int32)
    hs = list(heads)
    t0 = time.perf_counter()
    oracle.state_from_frames(Kev3[hs], Vev3[hs], S[hs], z[hs])
    out = oracle.hybrid_forward(Q[hs], Kw[hs], Vw[hs], S[hs], z[hs], C=w.chunk_frames, n_win=w.n_win(0),
                                nf=w.tokens_per_frame, beta=w.block_size, k=w.k_for(0), rows=r)
    dt = time.perf_counter() - t0
    idx = out["idx"]
    d, nf, beta, bpf = w.head_dim, w.tokens_per_frame, w.block_size, w.blocks_per_frame
    blk_rows = np.array([min(beta, nf - j * beta) for j in range(bpf)], np.int64)
    rr = np.arange(nq) if r is None else r
    qb = (rr // nf) * bpf + (rr % nf) // beta
    nk = blk_rows[idx[:, qb, :] % bpf].sum(axis=2)           # [heads, R]
    H = len(hs)
    flops = 4.0 * d * float(nk.sum()) + (2.0 * d * d + 2.0 * d) * len(rr) * H
    flops += (2.0 * d * d + d) * Kev3.shape[1] * H
    flops += 2.0 * w.n_qb() * w.n_kb(0) * d * H
    return dt, flops


def sample_plan(w, inputs, budget_s: float):
    """(heads, rows) of a sample that takes about budget_s on this host."""
    nq = w.chunk_frames * w.tokens_per_frame
    H = w.heads_total
    t_small, _ = oracle_step(w, inputs, [0], 4)
    t_big, _ = oracle_step(w, inputs, [0], 68)
    per_row = max((t_big - t_small) / 64, 1e-6)               # one head
    fixed = max(t_small - 4 * per_row, 1e-4)                  # one head: absorb, pooling, scores, top-K
    full_head = fixed + nq * per_row
    if budget_s >= H * full_head:
        return list(range(H)), None
    heads = max(1, min(H, int(budget_s // full_head)))
    if heads > 1:
        return list(range(heads)), None
    rows = int(max(4, min(nq, (budget_s - fixed) / per_row)))
    return [0], rows


def describe_sample(w, heads, rows):
    nq = w.chunk_frames * w.tokens_per_frame
    hs = f"{len(heads)} of {w.heads_total} heads"
    rs = f"all {nq} query rows" if rows is None else f"{rows} of {nq} query rows"
    return (f"{hs}, {rs}: absorb of the {w.chunk_frames} evicted frames, pooling, scores and top-K of all "
            f"blocks, sparse attention + linear read of the rows")


def cpu_baseline(w, target_s: float):
    """The oracle as it stands, on the whole step if it fits in target_s,
    repeated until at least target_s of CPU work."""
    import oracle
    inputs = oracle_inputs(w)
    heads, rows = sample_plan(w, inputs, target_s)
    tot_t, tot_f, n = 0.0, 0.0, 0
    while tot_t < target_s and n < 50:
        dt, fl = oracle_step(w, inputs, heads, rows, seed=n)
        tot_t += dt
        tot_f += fl
        n += 1
    return {"value": tot_f / tot_t / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{describe_sample(w, heads, rows)}; {n} repetition(s), {tot_t:.1f} s wall",
            "seconds": tot_t}


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
    budget = min(30.0, 150.0 / max(1, args.steps + args.warmup))   # whole run within a few minutes
    heads, rows = sample_plan(w, inputs, budget)
    for i in range(args.warmup):
        oracle_step(w, inputs, heads, rows, seed=100 + i)
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = oracle_step(w, inputs, heads, rows, seed=i)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = describe_sample(w, heads, rows) + " per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload_desc(w), "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def workload_desc(w):
    return (f"{w.name}: b{w.batch} H{w.heads} d{w.head_dim} N_f{w.tokens_per_frame} C{w.chunk_frames} "
            f"W{w.window_frames} beta{w.block_size} K{w.k_for(0)}/{w.n_kb(0)} state {w.absorbed_frames} frames")


def attention_traffic():
    """DRAM bytes per launch of the attention kernel from the committed ncu
    capture, or None when the kernel's sources changed since it was taken."""
    import hashlib
    tp = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if not os.path.exists(tp):
        return None
    rec = json.load(open(tp))
    h = hashlib.sha256()
    for f in rec.get("sources", []):
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if h.hexdigest() != rec.get("sources_sha256"):
        return None
    return rec.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# the CUDA path
# --------------------------------------------------------------------------
def build_layer(w, cfg, dev, spare_slots: int = 0):
    """A layer holding the workload's step-0 window and absorbed history."""
    from hybrid_sparse_linear_scores_b300 import binding as hb
    from hybrid_sparse_linear_scores_b300 import synth
    from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer
    from hybrid_sparse_linear_scores_b300.workloads import frames_tensor
    L = HybridAttentionLayer(cfg, dev, spare_slots=spare_slots)
    flat = lambda x: x.reshape(x.shape[0], -1, x.shape[-1])
    for f0 in range(0, w.absorbed_before(0), 6):
        fr = list(range(f0, min(f0 + 6, w.absorbed_before(0))))
        K = frames_tensor(w, synth.STREAM_K, fr, dev)
        V = frames_tensor(w, synth.STREAM_V, fr, dev)
        hb.hf_absorb_evicted(L.cfg, L.S, L.z, flat(K), flat(V), len(fr) * w.tokens_per_frame, L.ws)
    win = w.window(0)
    Kw = frames_tensor(w, synth.STREAM_K, win, dev)
    Vw = frames_tensor(w, synth.STREAM_V, win, dev)
    for i, f in enumerate(win):
        L.Kc[:, f % L.R] = Kw[:, i]
        L.Vc[:, f % L.R] = Vw[:, i]
    L.frames = w.frames_so_far(0)
    return L, Kw, Vw


def time_graph(fn, dev, flush, n):
    """Mean ms of `fn(stream)` captured as one CUDA graph, L2 flushed before each replay."""
    cap = torch.cuda.Stream(dev)
    with torch.cuda.stream(cap):
        fn(cap)                                                   # untimed first launch on this stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fn(torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        flush.zero_()
        g.replay()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)


def extra_measurements(w, cfg, dev, L, Q, O, idx, evict_slot, chunk_slots, flush, step_ms, args):
    """More figures on the same box, beside the step:
    - denoise_reuse: a chunk denoised in DENOISE_STEPS steps.  The window's
      K/V and the state do not change between the steps of one chunk, so
      absorb and key pooling run once and the forward once per step.
    - dense_swa_w21: the plain sliding-window attention the method replaces
      (W = 21 frames, every key block selected, empty state: the method's own
      dense special case), same chunk, same kernels.
    - rope_prestep: the relative temporal RoPE pre-step on the chunk's
      queries and the window's keys (HBM-bound).
    - long_horizon: the 240-frame stream through the layer, step times in
      buckets of 10 steps (flat when the state's cost does not grow)."""
    from hybrid_sparse_linear_scores_b300 import binding as hb
    from hybrid_sparse_linear_scores_b300 import synth
    from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, frames_tensor
    n = min(args.steps, 100)
    out = {}

    def chunk(stream):
        L.absorb_slots(evict_slot, w.chunk_frames, stream)
        L.pool_slots(chunk_slots, stream)
        for _ in range(DENOISE_STEPS):
            L.forward(Q, O, idx, stream)
    ms_chunk = time_graph(chunk, dev, flush, n)
    L.check_device_status()
    out["denoise_reuse"] = {"denoise_steps": DENOISE_STEPS, "ms_per_chunk": ms_chunk,
                            "us_per_latent_frame": 1000 * ms_chunk / w.chunk_frames,
                            "reading": "'few-step' denoising taken as 4 steps per chunk",
                            "how": "one CUDA graph per chunk: absorb + key pooling once, then 4 forwards"}

    # relative temporal RoPE pre-step: the chunk's queries (offsets W-C..W-1) in
    # place, the window's keys from the unrotated ring into a rotated copy
    Wn = w.n_win(0)
    Qr = Q.clone()
    Kr = torch.empty_like(L.Kc)
    nfd = w.tokens_per_frame * w.head_dim
    q_off = list(range(Wn - w.chunk_frames, Wn))

    def rope(stream):
        hb.hf_rope_relative(L.cfg, Qr, Qr, w.chunk_frames * nfd, nfd, list(range(w.chunk_frames)), q_off, Wn - 1,
                            w.head_dim, ROPE_BASE, stream)
        hb.hf_rope_relative(L.cfg, L.Kc, Kr, L.R * L.ss * w.head_dim, L.ss * w.head_dim, L.slot_map(),
                            list(range(Wn)), Wn - 1, w.head_dim, ROPE_BASE, stream)
    ms_rope = time_graph(rope, dev, flush, n)
    rope_bytes = 2 * (w.chunk_frames + Wn) * w.heads_total * nfd * 2
    hbm = peaks()["hbm_gbs"]
    out["rope_prestep"] = {"ms_per_step": ms_rope, "bytes": rope_bytes,
                           "GB_s": rope_bytes / (ms_rope * 1e-3) / 1e9,
                           "hbm_frac": rope_bytes / (ms_rope * 1e-3) / 1e9 / hbm,
                           "how": "hf_rope_relative on the chunk's Q (in place) and the window's K (ring -> rotated "
                                  "copy), offsets relative to the window, bound W-1, all channels, base 10000; "
                                  "2 launches in one CUDA graph, L2 flushed before each replay"}
    del Qr, Kr

    # the whole step with the relative RoPE on (EN section 2.C): absorb, rotation
    # of the window's keys (ring -> rotated copy) and of the chunk's queries by
    # their window-relative offsets, pooling of the rotated window's key blocks
    # (every frame's offset moves with the window), prologue, attention
    from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer, RelativeRope
    Lr = HybridAttentionLayer(cfg, dev, rope=RelativeRope(rot_dims=w.head_dim, base=ROPE_BASE))
    Lr.Kc.copy_(L.Kc)
    Lr.Vc.copy_(L.Vc)
    Lr.S.copy_(L.S)
    Lr.z.copy_(L.z)
    Lr.state_changed()
    Lr.frames = L.frames

    def rope_step(stream):
        Lr.absorb_slots(evict_slot, w.chunk_frames, stream)
        Lr.forward(Q, O, idx, stream)
    ms_rstep = time_graph(rope_step, dev, flush, n)
    Lr.check_device_status()
    out["step_with_rope"] = {"ms_per_step": ms_rstep, "us_per_latent_frame": 1000 * ms_rstep / w.chunk_frames,
                             "vs_step": ms_rstep / step_ms,
                             "how": "layer.step's forward with RelativeRope(rot_dims=d, base 10000, bound W-1): absorb, "
                                    "RoPE of the window keys and chunk queries, key pooling of the 9 rotated frames, "
                                    "prologue, attention; one CUDA graph, L2 flushed before each replay"}
    del Lr

    wd = CONFIGS["dense_w21"]
    cfg_d = hb.make_config(wd.batch, wd.heads, wd.head_dim, wd.tokens_per_frame, wd.window_frames,
                           wd.chunk_frames, wd.block_size, wd.k_for(0))
    Ld, _, _ = build_layer(wd, cfg_d, dev)
    Ld.pool_slots(Ld.slot_map())
    Qd = frames_tensor(wd, synth.STREAM_Q, wd.chunk(0), dev).reshape(wd.heads_total, -1, wd.head_dim)
    Od = torch.empty_like(Qd)
    idx_d = torch.empty((wd.heads_total, wd.n_qb(), wd.k_for(0)), dtype=torch.int32, device=dev)
    ms_d = time_graph(lambda st: Ld.forward(Qd, Od, idx_d, st), dev, flush, n)
    Ld.check_device_status()
    nq, nk = wd.chunk_frames * wd.tokens_per_frame, wd.window_frames * wd.tokens_per_frame
    fl_d = 4.0 * wd.head_dim * nq * nk * wd.heads_total
    out["dense_swa_w21"] = {"workload": workload_desc(wd), "ms_per_chunk": ms_d,
                            "us_per_latent_frame": 1000 * ms_d / wd.chunk_frames,
                            "attention_tflops": fl_d / (ms_d * 1e-3) / 1e12,
                            "hybrid_step_speedup": ms_d / step_ms,
                            "how": "hf_hybrid_forward_ex (cached key pools) with topk = all blocks and S = z = 0, "
                                   "one CUDA graph, L2 flushed before each replay"}
    del Ld

    # long horizon: the 240-frame stream (80 chunks) through the layer's own
    # step (absorb of the evicted frames, ring write + key pooling, forward);
    # every step timed, medians per 10-step bucket should be flat
    from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer
    w3 = CONFIGS["stream"]
    cfg3 = hb.make_config(w3.batch, w3.heads, w3.head_dim, w3.tokens_per_frame, w3.window_frames,
                          w3.chunk_frames, w3.block_size, w3.k_for(w3.steps - 1))
    L3 = HybridAttentionLayer(cfg3, dev)
    state_bytes = {L3.S.numel() * 4 + L3.z.numel() * 4}
    per_step = []
    for st in range(w3.steps):
        L3.cfg.topk = w3.k_for(st)
        Kn = frames_tensor(w3, synth.STREAM_K, w3.chunk(st), dev)
        Vn = frames_tensor(w3, synth.STREAM_V, w3.chunk(st), dev)
        Q3 = frames_tensor(w3, synth.STREAM_Q, w3.chunk(st), dev).reshape(w3.heads_total, -1, w3.head_dim)
        O3 = torch.empty_like(Q3)
        idx3 = torch.empty((w3.heads_total, w3.n_qb(), w3.k_for(st)), dtype=torch.int32, device=dev)
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        L3.step(Q3, Kn, Vn, O3, idx3)
        e1.record()
        torch.cuda.synchronize()
        per_step.append(e0.elapsed_time(e1))
        state_bytes.add(L3.S.numel() * 4 + L3.z.numel() * 4)
    L3.check_device_status()
    buckets = [statistics.median(per_step[i:i + 10]) for i in range(0, len(per_step), 10)]
    out["long_horizon"] = {"workload": f"{w3.name}: {w3.steps} chunks of {w3.chunk_frames} frames "
                                       f"(b{w3.batch} H{w3.heads} d{w3.head_dim} N_f{w3.tokens_per_frame} "
                                       f"W{w3.window_frames} beta{w3.block_size}, K = 25 % of the window)",
                           "bucket_median_ms_per_step": buckets,
                           "state_bytes": sorted(state_bytes),
                           "how": "layer.step per chunk (absorb, ring write + key pooling, forward), eager "
                                  "launches, CUDA events around each step, L2 flushed before each"}
    del L3
    return out


def forward_breakdown(L, Q, O, idx, dev, flush, n):
    """Mean ms of the layer's forward (cached key pools) as one CUDA graph, and
    of its prologue and attention kernels (external event records between
    them), L2 flushed before each replay."""
    cap = torch.cuda.Stream(dev)
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    stream = torch.cuda.current_stream(dev)
    for e in ev:
        e.record(stream)
    with torch.cuda.stream(cap):
        L.forward(Q, O, idx, cap)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        L.forward(Q, O, idx, torch.cuda.current_stream(dev), ev)
    torch.cuda.synchronize()
    pro, att = [], []
    for i in range(n + 3):
        flush.zero_()
        g.replay()
        torch.cuda.synchronize()
        if i >= 3:
            pro.append(ev[1].elapsed_time(ev[2]))
            att.append(ev[2].elapsed_time(ev[3]))
    total = time_graph(lambda st: L.forward(Q, O, idx, st), dev, flush, n)
    return total, statistics.mean(pro), statistics.mean(att)


def workload_figures(dev, flush, n):
    """Secondary figures on the other workloads of the same layer shape: the
    sparsity/block sweep (top-K 10/25/50/100 % of the window's key blocks,
    blocks of 64 and 128 tokens, clustered keys) and the 40-head layer.  Per
    workload: the forward with cached key pools (prologue + attention) per
    latent frame, and the attention kernel's effective TFLOP/s and fraction of
    the measured bf16 peak; for the 40-head layer also the whole step."""
    from hybrid_sparse_linear_scores_b300 import binding as hb
    from hybrid_sparse_linear_scores_b300 import synth
    from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, SWEEP, frames_tensor
    pk = peaks()
    out = {"sweep": [], "wide": None}
    flat = lambda x: x.reshape(x.shape[0], -1, x.shape[-1])
    for w in list(SWEEP) + [CONFIGS["wide"]]:
        cfg = hb.make_config(w.batch, w.heads, w.head_dim, w.tokens_per_frame, w.window_frames, w.chunk_frames,
                             w.block_size, w.k_for(0))
        L, _, _ = build_layer(w, cfg, dev)
        Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(0), dev))
        O = torch.empty_like(Q)
        idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(0)), dtype=torch.int32, device=dev)
        L.forward(Q, O, idx)                      # pools the window into the cache
        torch.cuda.synchronize()
        fwd_ms, pro_ms, att_ms = forward_breakdown(L, Q, O, idx, dev, flush, n)
        L.check_device_status()
        n_ev = w.chunk_frames * w.tokens_per_frame
        fl = step_flops(w, idx.cpu().numpy(), n_ev)
        att_tf = (fl["attn"] + fl["lin"]) / (att_ms * 1e-3) / 1e12
        rec = {"workload": workload_desc(w), "forward_ms": fwd_ms,
               "forward_us_per_latent_frame": 1000 * fwd_ms / w.chunk_frames,
               "prologue_ms": pro_ms, "attention_ms": att_ms, "attention_tflops": att_tf,
               "attention_frac": att_tf / pk["bf16_tflops"], "attention_gflop": (fl["attn"] + fl["lin"]) / 1e9}
        if w.name == "wide":
            first = w.window(0)[0] % L.R
            slots = [f % L.R for f in w.chunk(0)]

            def step(stream):
                L.absorb_slots(first, w.chunk_frames, stream)
                L.pool_slots(slots, stream)
                L.forward(Q, O, idx, stream)
            ms = time_graph(step, dev, flush, n)
            L.check_device_status()
            rec.update({"step_ms": ms, "step_us_per_latent_frame": 1000 * ms / w.chunk_frames,
                        "step_tflops": fl["total"] / (ms * 1e-3) / 1e12})
            out["wide"] = rec
        else:
            out["sweep"].append(rec)
        del L
        torch.cuda.synchronize()
    return out


def pinned_h2d_rate(dev, nbytes: int = 43130880, n: int = 10, trials: int = 3):
    """GB/s of one plain copy of nbytes from pinned host memory to the device
    (the size of a chunk's Q, K and V), CUDA events on the copying stream; the
    best of a few trials of n copies (the host link is shared with the rest of
    the machine)."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(dev)
    best = 0.0
    with torch.cuda.stream(st):
        for _ in range(3):
            d.copy_(h, non_blocking=True)
        for _ in range(trials):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(n):
                d.copy_(h, non_blocking=True)
            e1.record(st)
            e1.synchronize()
            best = max(best, nbytes * n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    return best


def streamer_copies_alone(streamer, Qh, Kh, Vh, Oh, n: int):
    """ms per chunk of the host streamer's own copies with no compute between
    them: the same pinned buffers, the same calls (Q by one copy, K/V by the
    ring write's pitched per-frame copies, O back on the device-to-host
    stream once its chunk's copy-in has landed) on the same two copy streams.
    Host wall clock over n chunks, as for the end-to-end figure; if the two
    agree, the end-to-end step runs at the host link's rate."""
    from hybrid_sparse_linear_scores_b300 import binding as hb
    L = streamer.L
    slots = L.chunk_slots()

    def one(i):
        b = i % 2
        with torch.cuda.stream(streamer.h2d):
            streamer.h2d.wait_event(streamer.ev_d2h[b])   # Qd[b] / Od[b] reuse, as the forward would
            streamer.Qd[b].copy_(Qh, non_blocking=True)
            hb.hf_ring_write(L.cfg, Kh, Vh, L.Kc, L.Vc, L.ss, slots, streamer.h2d)
            streamer.ev_h2d[b].record(streamer.h2d)
        with torch.cuda.stream(streamer.d2h):
            streamer.d2h.wait_event(streamer.ev_h2d[b])
            Oh[b].copy_(streamer.Od[b], non_blocking=True)
            streamer.ev_d2h[b].record(streamer.d2h)

    for i in range(4):
        one(i)
    streamer.synchronize()
    t0 = time.perf_counter()
    for i in range(n):
        one(i)
    streamer.synchronize()
    return 1000 * (time.perf_counter() - t0) / n


def run_hf(args):
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from hybrid_sparse_linear_scores_b300 import binding as hb
    from hybrid_sparse_linear_scores_b300 import synth
    from hybrid_sparse_linear_scores_b300.stream import HostStreamer
    from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, frames_tensor

    w = CONFIGS[args.workload]
    cfg = hb.make_config(w.batch, w.heads, w.head_dim, w.tokens_per_frame, w.window_frames, w.chunk_frames,
                         w.block_size, w.k_for(0))
    L, Kw, Vw = build_layer(w, cfg, dev)
    flat = lambda x: x.reshape(x.shape[0], -1, x.shape[-1])
    Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(0), dev))
    O = torch.empty_like(Q)
    idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(0)), dtype=torch.int32, device=dev)
    evict_slot = w.window(0)[0] % L.R                     # the oldest chunk's slots (contiguous)
    chunk_slots = [f % L.R for f in w.chunk(0)]           # the slots the chunk's frames were written to
    n_ev = w.chunk_frames * w.tokens_per_frame
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    side = torch.cuda.Stream(dev)
    ev_fork, ev_state = torch.cuda.Event(), torch.cuda.Event()

    def one_step(stream, events=None):
        """absorb the evicted frames (on a side stream: it writes the state and
        its tensor-core operand) beside the key pooling of the new chunk and the
        forward's prologue (selection), which do not read the state; then the
        attention, which waits for the absorb (as HybridAttentionLayer.step does
        when the chunk's slots are not the evicted ones)."""
        ev_fork.record(stream)
        side.wait_event(ev_fork)
        if events is not None:
            events[0].record(side)
        L.absorb_slots(evict_slot, w.chunk_frames, side, share_sms=True)
        if events is not None:
            events[1].record(side)
        ev_state.record(side)
        if events is not None:
            events[2].record(stream)
        L.pool_slots(chunk_slots, stream)
        L.forward(Q, O, idx, stream, events[3:] if events is not None else None, state_ready=ev_state,
                  after_pool_keys=True)

    stream = torch.cuda.current_stream(dev)
    L.forward(Q, O, idx, stream)                          # fills the key-pool cache for the window
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        one_step(stream)
    torch.cuda.synchronize()
    L.check_device_status()
    fl = step_flops(w, idx.cpu().numpy(), n_ev)
    by = step_bytes(w, n_ev)

    # ---- the step as one CUDA graph (4 kernels, no host work between them) ----
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.stream(cap):
        one_step(cap)                                      # untimed: first launch on this stream
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=cap):
        one_step(torch.cuda.current_stream(dev))
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K graph replays, L2 flushed before each ----
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    if ws > 1:
        dist.barrier()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    L.check_device_status()
    clocks = clk.summary()
    ms = max_over_ranks(statistics.mean(step_ms), ws, dev)

    # ---- per-kernel breakdown: the same step captured with event records between
    #      its kernels (external event nodes, so they time every replay) ----
    # events: [0] absorb [1] (side stream); [2] hf_pool_keys [3] (the forward's window
    # key pooling: none with cached pools) [4] prologue [5] attention (after its wait
    # for the absorb) [6]
    names = ["absorb", "pool_keys", "prologue", "attention"]
    spans = {"absorb": (0, 1), "pool_keys": (2, 3), "prologue": (4, 5), "attention": (5, 6)}
    times = {n: [] for n in names}
    n_prof = min(args.steps, 200)
    pev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(7)]
    for e in pev:                                         # create the CUDA events before the capture
        e.record(stream)
    torch.cuda.synchronize()
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=cap):
        one_step(torch.cuda.current_stream(dev), pev)
    torch.cuda.synchronize()
    for _ in range(n_prof):
        flush.zero_()
        graph_ev.replay()
        torch.cuda.synchronize()
        for n in names:
            a, b = spans[n]
            times[n].append(pev[a].elapsed_time(pev[b]))

    # warm-L2 timing of the graphed step, for context
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(n_prof):
        graph.replay()
    s1.record(stream)
    torch.cuda.synchronize()
    warm_ms = s0.elapsed_time(s1) / n_prof
    L.check_device_status()

    # ---- end to end: chunks streamed from pinned host memory ----
    e2e = None
    if not args.skip_e2e:
        L2, _, _ = build_layer(w, cfg, dev, spare_slots=w.chunk_frames)
        streamer = HostStreamer(L2)
        Qh = Q.cpu().pin_memory()
        Kh = Kw[:, -w.chunk_frames:].contiguous().cpu().pin_memory()
        Vh = Vw[:, -w.chunk_frames:].contiguous().cpu().pin_memory()
        Oh = [torch.empty(Q.shape, dtype=Q.dtype).pin_memory() for _ in range(2)]
        for i in range(4):
            streamer.push(Qh, Kh, Vh, Oh[i % 2])
        streamer.synchronize()
        n_e2e = min(args.steps, 500)
        b0, d0 = streamer.h2d_bytes, streamer.d2h_bytes
        t0 = time.perf_counter()
        for i in range(n_e2e):
            streamer.push(Qh, Kh, Vh, Oh[i % 2])
        streamer.synchronize()
        e2e_ms = max_over_ranks(1000 * (time.perf_counter() - t0) / n_e2e, ws, dev)
        L2.check_device_status()
        h2d_step = (streamer.h2d_bytes - b0) // n_e2e
        copies_ms = streamer_copies_alone(streamer, Qh, Kh, Vh, Oh, n_e2e)
        e2e = {"value": job_throughput(fl["total"], ws, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d_step,
               "d2h_bytes_per_step": (streamer.d2h_bytes - d0) // n_e2e, "ms_per_step": e2e_ms,
               "h2d_GB_s_implied": h2d_step / (e2e_ms * 1e-3) / 1e9,
               "copies_alone_ms_per_step": copies_ms,
               "h2d_GB_s_copies_alone": h2d_step / (copies_ms * 1e-3) / 1e9,
               "h2d_GB_s_plain_pinned_copy": pinned_h2d_rate(dev, int(h2d_step)),
               "how": "HostStreamer: per chunk, Q and the chunk's K/V copied from pinned host memory and O "
                      "copied back, on copy streams overlapped with the neighbouring chunks' compute; "
                      f"host wall clock over {n_e2e} chunks"}

    extra = {}
    if not args.skip_extras:
        # secondary figures: a failure there is reported in the line, not allowed to
        # take the step's own measurement with it
        try:
            extra = extra_measurements(w, cfg, dev, L, Q, O, idx, evict_slot, chunk_slots, flush, ms, args)
        except Exception as exc:   # noqa: BLE001 - reported, not swallowed
            print(f"bench: extra measurements failed: {exc!r}", file=sys.stderr, flush=True)
            extra = {"extras_error": repr(exc)}
        try:
            extra["workloads"] = workload_figures(dev, flush, min(args.steps, 50))
        except Exception as exc:   # noqa: BLE001 - reported, not swallowed
            print(f"bench: workload figures failed: {exc!r}", file=sys.stderr, flush=True)
            extra["workloads_error"] = repr(exc)
        torch.cuda.synchronize()
        L.check_device_status()

    pk = peaks()
    attn_ms = statistics.mean(times["attention"])
    attn_tf = (fl["attn"] + fl["lin"]) / (attn_ms * 1e-3) / 1e12
    value = job_throughput(fl["total"], ws, ms)
    per_kernel = {n: {"ms": statistics.mean(times[n])} for n in names}
    tot_k = sum(v["ms"] for v in per_kernel.values())
    for n in names:
        per_kernel[n]["share"] = per_kernel[n]["ms"] / tot_k
    for n, key in (("absorb", "absorb"), ("prologue", "prologue"), ("pool_keys", "pool_k")):
        per_kernel[n]["GB_s"] = by[key] / (per_kernel[n]["ms"] * 1e-3) / 1e9
        per_kernel[n]["hbm_frac"] = per_kernel[n]["GB_s"] / pk["hbm_gbs"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "l2": "flushed (256 MB write) before every step",
                   "timing": "CUDA events around each replay of the step's CUDA graph (absorb on a second "
                             "stream beside the key pooling of the new chunk and the forward's prologue; then the "
                             "attention, which waits for the absorb: 4 kernels)",
                   "parallelism": f"replicas x{ws}"},
        "us_per_latent_frame": 1000 * ms / w.chunk_frames,
        "median_ms_per_step": statistics.median(step_ms),
        "p10_ms_per_step": statistics.quantiles(step_ms, n=10)[0] if len(step_ms) > 1 else step_ms[0],
        "p90_ms_per_step": statistics.quantiles(step_ms, n=10)[8] if len(step_ms) > 1 else step_ms[0],
        "median_us_per_latent_frame": 1000 * statistics.median(step_ms) / w.chunk_frames,
        "pct_bf16_peak": 100 * value / pk["bf16_tflops"],
        "warm_l2_ms_per_step": warm_ms,
        "flops_per_step": fl, "bytes_per_step": by,
        "kernels": per_kernel,
        "roofline": {"bound": "tensor", "kernel": "attention (sparse softmax + fused linear read)",
                     "achieved": attn_tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": attn_tf / pk["bf16_tflops"], "traffic": attention_traffic(),
                     "peak_source": pk["source"] + " burst", "peak_sustained": pk["bf16_tflops_sustained"]},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    line.update(extra)
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
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("hf", "reference"), default="hf")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-extras", action="store_true", help="skip the denoise-reuse and dense-baseline figures")
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

"""The five synthetic workloads of the hybrid attention step, and their inputs.

A workload fixes the attention shapes of one layer of a streaming video
transformer at 832x480 (1560 tokens per latent frame, 30x52 after 2x2
patchify), the window/chunk/block geometry, the top-K budget and a value
recipe.  Inputs are drawn with :mod:`synth` and are pure functions of
(seed, tensor, frame, head, token, channel).

Streaming schedule (Hybrid Forcing, "Hybrid Attention": frames that leave
the sliding window are folded into the linear state): step s appends the
chunk frames [C*s, C*s + C); the window then holds the last
n_win = min(W, frames so far) frames, chunk included; every older frame has
been absorbed into the state.  Ring slot of frame f is f mod W.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

from . import synth

RECIPES = ("normal", "frame_mean", "drift", "clustered")


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    head_dim: int
    tokens_per_frame: int
    chunk_frames: int
    window_frames: int
    block_size: int
    seed: int
    recipe: str
    topk: int = 0              # fixed K (0: use topk_frac)
    topk_frac: float = 0.0     # K = ceil(frac * nKB), clamped to [1, nKB]
    absorbed_frames: int = 0   # single-step workloads: frames already in the state
    steps: int = 1             # streaming workloads: number of chunks

    # ---- geometry of the step (shapes only) ----
    @property
    def blocks_per_frame(self) -> int:
        return -(-self.tokens_per_frame // self.block_size)

    def frames_so_far(self, step: int) -> int:
        """Frames generated once step `step` has appended its chunk."""
        if self.steps == 1:
            return self.absorbed_frames + self.window_frames
        return self.chunk_frames * (step + 1)

    def n_win(self, step: int) -> int:
        return min(self.window_frames, self.frames_so_far(step))

    def window(self, step: int) -> list[int]:
        f = self.frames_so_far(step)
        return list(range(f - self.n_win(step), f))

    def chunk(self, step: int) -> list[int]:
        return self.window(step)[-self.chunk_frames:]

    def absorbed_before(self, step: int) -> int:
        """Frames [0, absorbed_before) are in the state during step `step`."""
        return self.frames_so_far(step) - self.n_win(step)

    def newly_absorbed(self, step: int) -> list[int]:
        """Frames this step absorbs (evicted by the arrival of its chunk)."""
        lo = 0 if step == 0 else self.absorbed_before(step - 1)
        if self.steps == 1:
            lo = 0
        return list(range(lo, self.absorbed_before(step)))

    def n_kb(self, step: int) -> int:
        return self.n_win(step) * self.blocks_per_frame

    def n_qb(self) -> int:
        return self.chunk_frames * self.blocks_per_frame

    def k_for(self, step: int) -> int:
        nkb = self.n_kb(step)
        if self.topk > 0:
            k = self.topk
        else:
            k = math.ceil(self.topk_frac * nkb - 1e-9)
        return max(1, min(k, nkb))

    def slot_map(self, step: int) -> list[int]:
        return [f % self.window_frames for f in self.window(step)]

    @property
    def heads_total(self) -> int:
        return self.batch * self.heads


def _frame_means(w: Workload, stream: int, frames, device) -> torch.Tensor:
    """Per-(head, frame) mean vector, [BH, F, 1, d] float64."""
    heads = range(w.heads_total)
    d = w.head_dim
    if w.recipe == "frame_mean":
        return 0.5 * synth.normal_field(w.seed, synth.STREAM_MEAN[stream], frames, heads, 1, d, device)
    # drift: mu_0 ~ N(0, 0.5^2), mu_f = mu_{f-1} + N(0, 0.05^2); summed on the CPU in frame order
    fmax = max(frames)
    mu0 = 0.5 * synth.normal_field(w.seed, synth.STREAM_MEAN[stream], [0], heads, 1, d, "cpu")
    if fmax > 0:
        inc = 0.05 * synth.normal_field(w.seed, synth.STREAM_DRIFT[stream], range(1, fmax + 1), heads, 1, d, "cpu")
        mus = torch.cat((mu0, mu0 + torch.cumsum(inc, dim=1)), dim=1)
    else:
        mus = mu0
    idx = torch.as_tensor(list(frames), dtype=torch.int64)
    return mus[:, idx].to(device)


def frames_tensor(w: Workload, stream: int, frames, device="cpu") -> torch.Tensor:
    """bf16 [BH, len(frames), N_f, d] for tensor `stream` (synth.STREAM_Q/K/V)."""
    frames = list(frames)
    heads = range(w.heads_total)
    nf, d = w.tokens_per_frame, w.head_dim
    if len(frames) == 0:
        return torch.zeros((w.heads_total, 0, nf, d), dtype=torch.bfloat16, device=device)
    x = synth.normal_field(w.seed, stream, frames, heads, nf, d, device)
    if w.recipe in ("frame_mean", "drift"):
        x = x + _frame_means(w, stream, frames, device)
    elif w.recipe == "clustered" and stream == synth.STREAM_K:
        centres = synth.normal_field(w.seed, synth.STREAM_CENTRES, [0], heads, 16, d, device)[:, 0]
        ids = synth.uniform_u32(w.seed, synth.STREAM_CLUSTER_ID, frames, heads, nf, device) >> 28
        bh = torch.arange(w.heads_total, device=device).view(-1, 1, 1).expand_as(ids)
        x = centres[bh, ids] + 0.3 * x
    return synth.to_bf16(x)


def to_ring(win: torch.Tensor, w: Workload, step: int, slot_stride: int | None = None) -> torch.Tensor:
    """Lay logical window frames [BH, n_win, N_f, d] into ring slots
    [BH, W, slot_stride, d] (slot of frame f = f mod W; unused rows zero)."""
    bh, n, nf, d = win.shape
    ss = slot_stride or nf
    ring = torch.zeros((bh, w.window_frames, ss, d), dtype=win.dtype, device=win.device)
    for i, f in enumerate(w.window(step)):
        ring[:, f % w.window_frames, :nf] = win[:, i]
    return ring


CONFIGS: dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 2, 64, 128, 1, 2, 32, seed=0, recipe="normal", topk=4, steps=6),
    "realistic": Workload("realistic", 1, 12, 128, 1560, 3, 9, 64, seed=1, recipe="frame_mean",
                          topk_frac=0.25, absorbed_frames=30),
    "stream": Workload("stream", 1, 12, 128, 1560, 3, 9, 64, seed=2, recipe="drift",
                       topk_frac=0.25, steps=80),
    "wide": Workload("wide", 1, 40, 128, 1560, 3, 9, 64, seed=4, recipe="frame_mean",
                     topk_frac=0.25, absorbed_frames=60),
    # the dense sliding-window baseline that the method replaces: W = 21 frames,
    # every key block selected, nothing in the state
    "dense_w21": Workload("dense_w21", 1, 12, 128, 1560, 3, 21, 64, seed=5, recipe="frame_mean",
                          topk_frac=1.0),
}


def sweep_point(frac: float, block: int) -> Workload:
    """Sparsity/block sweep on the realistic shapes with clustered keys.
    At 100 % the state is empty (the dense sliding-window check)."""
    absorbed = 0 if frac >= 1.0 else 30
    return Workload(f"sweep_k{int(round(frac * 100))}_b{block}", 1, 12, 128, 1560, 3, 9, block,
                    seed=3, recipe="clustered", topk_frac=frac, absorbed_frames=absorbed)


SWEEP = [sweep_point(f, b) for b in (64, 128) for f in (0.10, 0.25, 0.50, 1.00)]


def scaled(w: Workload, **kw) -> Workload:
    """Same recipe and geometry rules with some sizes changed (parity cases)."""
    return replace(w, **kw)

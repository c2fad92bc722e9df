"""Shared helpers of the GPU parity tests: build one streaming step of a
workload on the device (through the C ABI) and the same step in the oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from hybrid_sparse_linear_scores_b300 import binding as hb
from hybrid_sparse_linear_scores_b300 import synth
from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer
from hybrid_sparse_linear_scores_b300.workloads import Workload, frames_tensor

MAX_ABS = 2e-2     # output tolerance vs the fp64 oracle: max |delta|
REL_L2 = 5e-3      #                                     relative L2
# The absorbed state S: bf16 hi+lo products (exact to ~2^-17 relative) summed
# by the tensor core for at most 2 x 8 K-steps of one 128-token tile (its
# internal adds may truncate: <= 32 * 2^-23 = 3.8e-6 relative per tile), then
# tiles, CTAs and calls summed in fp32 round-to-nearest.  2e-5 relative L2
# leaves a 5x margin; z is a plain fp32 sum (1e-5).
STATE_REL_L2 = 2e-5
Z_REL_L2 = 1e-5


def config_of(w: Workload, step: int, eps: float = 1e-6) -> hb.HFConfig:
    return hb.make_config(w.batch, w.heads, w.head_dim, w.tokens_per_frame, w.window_frames, w.chunk_frames,
                          w.block_size, w.k_for(step), 0.0, eps)


def flat(x: torch.Tensor) -> torch.Tensor:
    """[BH, F, N_f, d] -> [BH, F*N_f, d]"""
    return x.reshape(x.shape[0], -1, x.shape[-1])


class Step:
    """Inputs of one step (device copies) and the device layer holding them."""

    def __init__(self, w: Workload, step: int, device, absorb_on_gpu: bool = True):
        self.w, self.step = w, step
        self.cfg = config_of(w, step)
        self.layer = HybridAttentionLayer(self.cfg, device)
        self.ev = list(range(w.absorbed_before(step)))
        self.win = w.window(step)
        self.Kev = frames_tensor(w, synth.STREAM_K, self.ev, device)
        self.Vev = frames_tensor(w, synth.STREAM_V, self.ev, device)
        if self.ev and absorb_on_gpu:
            n = len(self.ev) * w.tokens_per_frame
            hb.hf_absorb_evicted(self.cfg, self.layer.S, self.layer.z, flat(self.Kev), flat(self.Vev), n,
                                 self.layer.ws)
        self.Kwin = frames_tensor(w, synth.STREAM_K, self.win, device)
        self.Vwin = frames_tensor(w, synth.STREAM_V, self.win, device)
        for i, f in enumerate(self.win):
            self.layer.Kc[:, f % w.window_frames, :w.tokens_per_frame] = self.Kwin[:, i]
            self.layer.Vc[:, f % w.window_frames, :w.tokens_per_frame] = self.Vwin[:, i]
        self.layer.frames = w.frames_so_far(step)
        self.Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(step), device))

    def run_forward(self):
        w = self.w
        O = torch.empty_like(self.Q)
        idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(self.step)), dtype=torch.int32, device=self.Q.device)
        self.layer.forward(self.Q, O, idx)
        torch.cuda.synchronize()
        self.layer.check_device_status()
        return O, idx

    def oracle_state(self):
        if not self.ev:
            return None, None
        return oracle.state_from_frames(flat(self.Kev).cpu(), flat(self.Vev).cpu())

    def oracle_forward(self, rows=None, split=False, S=None, z=None):
        w = self.w
        if S is None and self.ev:
            S, z = self.oracle_state()
        return oracle.hybrid_forward(self.Q.cpu(), flat(self.Kwin).cpu(), flat(self.Vwin).cpu(), S, z,
                                     C=w.chunk_frames, n_win=w.n_win(self.step), nf=w.tokens_per_frame,
                                     beta=w.block_size, k=w.k_for(self.step), rows=rows, split=split)


def compare(got: torch.Tensor, ref: np.ndarray, max_abs=MAX_ABS, rel_l2=REL_L2, what="output"):
    g = got.detach().double().cpu().numpy()
    diff = g - ref
    ma = float(np.abs(diff).max()) if diff.size else 0.0
    rl = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    assert ma <= max_abs and rl <= rel_l2, f"{what}: max|d| = {ma:.3e} (<= {max_abs}), rel L2 = {rl:.3e} (<= {rel_l2})"
    return ma, rl


def compare_state(S, z, S_ref, z_ref):
    """The device state against the oracle's fp64 state."""
    s_max = float(np.abs(S_ref).max())
    compare(S, S_ref, max_abs=8 * STATE_REL_L2 * s_max, rel_l2=STATE_REL_L2, what="S")
    compare(z, z_ref, max_abs=8 * Z_REL_L2 * float(np.abs(z_ref).max()), rel_l2=Z_REL_L2, what="z")


def sample_rows(w: Workload, per_head: int, seed: int = 0) -> np.ndarray:
    """Query rows spread over every tile of the chunk, including each frame's
    ragged last block and its last row."""
    nq = w.chunk_frames * w.tokens_per_frame
    rng = np.random.default_rng(seed)
    must = []
    for c in range(w.chunk_frames):
        base = c * w.tokens_per_frame
        must += [base, base + w.tokens_per_frame - 1, base + (w.blocks_per_frame - 1) * w.block_size]
    extra = rng.choice(nq, size=max(0, per_head - len(must)), replace=False)
    return np.unique(np.concatenate([np.array(must), extra])).astype(np.int32)

"""Device state of one streaming hybrid attention layer, driven through the C ABI.

The layer owns (in device memory, allocated by torch):
  - the key/value ring of W frame slots, [BH, W, slot_stride, d] bf16,
  - the linear state S [BH, d, d] and z [BH, d] (fp32),
  - the library workspace.
A chunk of C frames is processed as in Hybrid Forcing's streaming loop
(English technical summary, section 2.A.1: frames that leave the sliding
window are absorbed into the compact state): first the frames this chunk
evicts are absorbed into (S, z) straight from their ring slots, then the
chunk's keys/values take those slots, then the hybrid forward runs over the
window.  Logical window order (oldest first) is passed as the slot map, so
no frame is ever moved.
"""

from __future__ import annotations

import torch

from . import binding as hb


class HybridAttentionLayer:
    def __init__(self, cfg: hb.HFConfig, device="cuda", slot_stride: int | None = None):
        self.cfg = cfg
        self.device = torch.device(device)
        self.BH = cfg.batch * cfg.heads
        self.W = cfg.window_frames
        self.C = cfg.chunk_frames
        self.nf = cfg.tokens_per_frame
        self.d = cfg.head_dim
        self.ss = slot_stride or self.nf
        self.Kc = torch.zeros((self.BH, self.W, self.ss, self.d), dtype=torch.bfloat16, device=self.device)
        self.Vc = torch.zeros_like(self.Kc)
        self.S = torch.zeros((self.BH, self.d, self.d), dtype=torch.float32, device=self.device)
        self.z = torch.zeros((self.BH, self.d), dtype=torch.float32, device=self.device)
        self.ws = torch.zeros(hb.hf_workspace_size(cfg), dtype=torch.uint8, device=self.device)
        self.frames = 0

    # ---- window bookkeeping (host) ----
    def n_win(self) -> int:
        return min(self.W, self.frames)

    def slot_map(self) -> list[int]:
        first = self.frames - self.n_win()
        return [(first + w) % self.W for w in range(self.n_win())]

    def frames_to_evict(self) -> list[int]:
        """Frames the next chunk pushes out of the window (oldest first)."""
        first = self.frames - self.n_win()               # oldest frame in the window now
        keep_from = max(0, self.frames + self.C - self.W)  # oldest frame after the chunk arrives
        return list(range(first, max(first, keep_from)))

    # ---- the three phases of a step ----
    def absorb_evicted(self, stream=None) -> int:
        """Absorb the frames the next chunk evicts, from their ring slots."""
        frames = self.frames_to_evict()
        runs: list[list[int]] = []
        for f in frames:   # group into runs of consecutive slots (one call each)
            s = f % self.W
            if runs and self.ss == self.nf and runs[-1][-1] + 1 == s:
                runs[-1].append(s)
            else:
                runs.append([s])
        for run in runs:
            self.absorb_slots(run[0], len(run), stream)
        return len(frames)

    def absorb_slots(self, first_slot: int, n_slots: int, stream=None):
        hb.hf_absorb_evicted_strided(self.cfg, self.S, self.z, self.Kc[:, first_slot], self.Vc[:, first_slot],
                                     n_slots * self.nf, self.W * self.ss, self.ws,
                                     stream)

    def write_chunk(self, K_new: torch.Tensor, V_new: torch.Tensor):
        """K_new, V_new: [BH, C, N_f, d] bf16 for the next C frames."""
        for c in range(self.C):
            slot = (self.frames + c) % self.W
            self.Kc[:, slot, :self.nf].copy_(K_new[:, c])
            self.Vc[:, slot, :self.nf].copy_(V_new[:, c])
        self.frames += self.C

    def forward(self, Q: torch.Tensor, O: torch.Tensor, idx_out: torch.Tensor | None = None, stream=None):
        """Q, O: [BH, C*N_f, d] bf16.  idx_out: optional int32 [BH, nQB, K_eff]."""
        hb.hf_hybrid_forward(self.cfg, Q, self.Kc, self.Vc, self.ss, self.slot_map(), self.n_win(), self.S, self.z,
                             O, idx_out, self.ws, stream)

    def step(self, Q, K_new, V_new, O, idx_out=None, stream=None):
        self.absorb_evicted(stream)
        self.write_chunk(K_new, V_new)
        self.forward(Q, O, idx_out, stream)

    def check_device_status(self, stream=None):
        rc, site = hb.hf_get_device_status(self.ws, stream)
        if rc != hb.HF_OK:
            raise hb.HFError(rc, "device status", f"site {site}: {hb.lib().hf_last_error().decode()}")

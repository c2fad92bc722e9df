"""Device state of one streaming hybrid attention layer, driven through the C ABI.

The layer owns (in device memory, allocated by torch):
  - the key/value ring of frame slots, [BH, R, slot_stride, d] bf16, with
    R = W + spare_slots (W = window frames, the chunk included),
  - the linear state S [BH, d, d] and z [BH, d] (fp32),
  - the library workspace.
A chunk of C frames is processed as in Hybrid Forcing's streaming loop
(English technical summary, section 2.A.1: frames that leave the sliding
window are absorbed into the compact state): first the frames this chunk
evicts are absorbed into (S, z) straight from their ring slots, then the
chunk's keys/values take those slots, then the hybrid forward runs over the
window.  Logical window order (oldest first) is passed as the slot map, so
no frame is ever moved.  Frame f lives in slot f mod R.

With spare_slots = C the next chunk's keys/values can be copied in while the
current chunk's forward still reads the window (HostStreamer below).  With a
RelativeRope the forward first rotates the window's keys into a copy and the
chunk's queries by their window-relative offsets (the ring keeps the
unrotated keys for the absorb).  The C
ABI sees a ring of R slots (its config's window_frames = R) and a window of
n_win <= W frames; the top-K count is the config's fixed topk.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as hb


@dataclass(frozen=True)
class RelativeRope:
    """The relative temporal RoPE of the layer (English technical summary,
    section 2.C: temporal RoPE indices are window-relative and held under one
    fixed bound).  Each forward rotates the chunk's queries and the window's
    keys by their frame's offset inside the current window (oldest frame 0),
    clamped to max_offset (None: the window's largest offset, W - 1); values
    and the linear state are not rotated."""
    rot_dims: int
    base: float = 10000.0
    max_offset: int | None = None


class HybridAttentionLayer:
    def __init__(self, cfg: hb.HFConfig, device="cuda", slot_stride: int | None = None, spare_slots: int = 0,
                 rope: RelativeRope | None = None):
        self.window = cfg.window_frames                  # W: frames attended (chunk included)
        self.R = cfg.window_frames + spare_slots         # ring slots
        self.cfg = hb.HFConfig.from_buffer_copy(cfg)     # the ABI's view: window_frames = ring slots
        self.cfg.window_frames = self.R
        self.device = torch.device(device)
        self.BH = cfg.batch * cfg.heads
        self.W = self.R
        self.C = cfg.chunk_frames
        self.nf = cfg.tokens_per_frame
        self.d = cfg.head_dim
        self.ss = slot_stride or self.nf
        self.Kc = torch.zeros((self.BH, self.R, self.ss, self.d), dtype=torch.bfloat16, device=self.device)
        self.Vc = torch.zeros_like(self.Kc)
        self.S = torch.zeros((self.BH, self.d, self.d), dtype=torch.float32, device=self.device)
        self.z = torch.zeros((self.BH, self.d), dtype=torch.float32, device=self.device)
        self.ws = torch.zeros(hb.hf_workspace_size(self.cfg), dtype=torch.uint8, device=self.device)
        self.frames = 0
        # ring slots whose pooled key blocks are in the workspace's cache (host bookkeeping)
        self.pooled: set[int] = set()
        # with RoPE: the window's keys rotated for the current step (the ring keeps
        # the unrotated keys, which the absorb reads), and the chunk's rotated queries
        self.rope = rope
        self.Kr = torch.zeros_like(self.Kc) if rope is not None else None
        self.Qr: torch.Tensor | None = None
        # whether the workspace holds S as the linear read's tensor-core operand:
        # every absorb and every forward leave it so (the zeroed workspace holds
        # the operand of S = 0); writing S directly needs state_changed()
        self.state_prepared = True
        self._side: torch.cuda.Stream | None = None
        self._ev_fork = self._ev_state = None

    # ---- window bookkeeping (host) ----
    def n_win(self) -> int:
        return min(self.window, self.frames)

    def slot_map(self) -> list[int]:
        first = self.frames - self.n_win()
        return [(first + w) % self.R for w in range(self.n_win())]

    def frames_to_evict(self) -> list[int]:
        """Frames the next chunk pushes out of the window (oldest first)."""
        first = self.frames - self.n_win()                      # oldest frame in the window now
        keep_from = max(0, self.frames + self.C - self.window)  # oldest frame after the chunk arrives
        return list(range(first, max(first, keep_from)))

    def _slot_runs(self, frames) -> list[list[int]]:
        """Frames grouped into runs of consecutive ring slots."""
        runs: list[list[int]] = []
        for f in frames:
            s = f % self.R
            if runs and self.ss == self.nf and runs[-1][-1] + 1 == s:
                runs[-1].append(s)
            else:
                runs.append([s])
        return runs

    # ---- the three phases of a step ----
    def absorb_evicted(self, stream=None, share_sms: bool = False) -> int:
        """Absorb the frames the next chunk evicts, from their ring slots."""
        frames = self.frames_to_evict()
        for run in self._slot_runs(frames):
            self.absorb_slots(run[0], len(run), stream, share_sms)
        return len(frames)

    def absorb_slots(self, first_slot: int, n_slots: int, stream=None, share_sms: bool = False):
        """share_sms: the absorb runs beside other kernels (on about half of the
        SMs, fewer tiles in flight; the state differs from the unshared absorb
        only in the order of one fp32 reduction)."""
        hb.hf_absorb_evicted_strided(self.cfg, self.S, self.z, self.Kc[:, first_slot], self.Vc[:, first_slot],
                                     n_slots * self.nf, self.R * self.ss, self.ws, stream,
                                     hb.HF_ABSORB_SHARE_SMS if share_sms else 0)
        self.state_prepared = True

    def state_changed(self):
        """Call after writing S or z directly: the next forward converts S again."""
        self.state_prepared = False

    def chunk_slots(self) -> list[int]:
        """Ring slots of the next chunk's frames."""
        return [(self.frames + c) % self.R for c in range(self.C)]

    def write_chunk(self, K_new: torch.Tensor, V_new: torch.Tensor, stream=None):
        """K_new, V_new: contiguous [BH, C, N_f, d] bf16 for the next C frames.
        The chunk's key blocks are pooled into the cache right after the copy
        (with RoPE the forward pools the rotated window instead)."""
        slots = self.chunk_slots()
        hb.hf_ring_write(self.cfg, K_new, V_new, self.Kc, self.Vc, self.ss, slots, stream)
        if self.rope is None:
            self.pool_slots(slots, stream)
        else:
            self.invalidate_key_cache(slots)
        self.frames += self.C

    def pool_slots(self, slots, stream=None):
        """Pool the key blocks of freshly written ring slots into the cache."""
        hb.hf_pool_keys(self.cfg, self.Kc, self.ss, list(slots), self.ws, stream)
        self.pooled.update(slots)

    def invalidate_key_cache(self, slots=None):
        """Forget cached key pools (all, or of `slots`) after writing Kc directly."""
        if slots is None:
            self.pooled.clear()
        else:
            self.pooled.difference_update(slots)

    def _state_flags(self) -> int:
        return hb.HF_FWD_STATE_PREPARED if self.state_prepared else 0

    def forward(self, Q: torch.Tensor, O: torch.Tensor, idx_out: torch.Tensor | None = None, stream=None,
                events=None, state_ready=None, after_pool_keys: bool = False):
        """Q, O: [BH, C*N_f, d] bf16.  idx_out: optional int32 [BH, nQB, K_eff].
        Uses the cached key pools when every window slot is in the cache;
        otherwise pools the whole window (which fills the cache).
        state_ready: optional torch.cuda.Event (recorded after the absorb that
        produced the state, on another stream) that the attention waits for.
        after_pool_keys: the last kernel on `stream` is this layer's key pooling
        (pool_slots), launched after Q and the state were written: the forward
        may then start while it runs (HF_FWD_AFTER_POOL_KEYS)."""
        sm = self.slot_map()
        if self.rope is not None:
            self._forward_rope(Q, O, idx_out, stream, events, state_ready)
            return
        cached = all(sl in self.pooled for sl in sm)
        flags = (hb.HF_FWD_CACHED_KEYS if cached else 0) | self._state_flags()
        if after_pool_keys:
            flags |= hb.HF_FWD_AFTER_POOL_KEYS
        hb.hf_hybrid_forward_ex(self.cfg, Q, self.Kc, self.Vc, self.ss, sm, self.n_win(), self.S, self.z, O, idx_out,
                                self.ws, flags, events, stream, state_ready)
        self.pooled.update(sm)
        self.state_prepared = True

    def rope_offsets(self) -> tuple[list[int], list[int], int]:
        """(key offsets of the window's frames in logical order, query offsets
        of the chunk's frames, the bound) for the current window."""
        n = self.n_win()
        bound = self.rope.max_offset if self.rope.max_offset is not None else self.window - 1
        return list(range(n)), list(range(n - self.C, n)), bound

    def _forward_rope(self, Q, O, idx_out, stream, events, state_ready=None):
        """Rotate the window's keys (ring -> rotated copy) and the chunk's
        queries by their window-relative offsets, pool the rotated window's key
        blocks (every frame's offset moved with the window), then the forward
        on the rotated keys and queries and the unrotated values."""
        r = self.rope
        sm = self.slot_map()
        k_off, q_off, bound = self.rope_offsets()
        if self.Qr is None or self.Qr.shape != Q.shape:
            self.Qr = torch.empty_like(Q)
        nfd = self.nf * self.d
        hb.hf_rope_relative(self.cfg, self.Kc, self.Kr, self.R * self.ss * self.d, self.ss * self.d, sm, k_off, bound,
                            r.rot_dims, r.base, stream)
        hb.hf_rope_relative(self.cfg, Q, self.Qr, self.C * nfd, nfd, list(range(self.C)), q_off, bound, r.rot_dims,
                            r.base, stream)
        hb.hf_pool_keys(self.cfg, self.Kr, self.ss, sm, self.ws, stream)
        hb.hf_hybrid_forward_ex(self.cfg, self.Qr, self.Kr, self.Vc, self.ss, sm, self.n_win(), self.S, self.z, O,
                                idx_out, self.ws, hb.HF_FWD_CACHED_KEYS | hb.HF_FWD_AFTER_POOL_KEYS | self._state_flags(),
                                events, stream, state_ready)
        self.pooled.clear()   # the cache holds this step's rotated pools
        self.state_prepared = True

    def can_overlap_absorb(self) -> bool:
        """The absorb of the evicted frames may run beside the next chunk's ring
        write, key pooling and selection when the chunk's slots are not the
        evicted ones (spare slots) and no RoPE rewrites the window's keys."""
        return self.rope is None and self.R >= self.window + self.C

    def step(self, Q, K_new, V_new, O, idx_out=None, stream=None):
        if not self.can_overlap_absorb():
            self.absorb_evicted(stream)
            self.write_chunk(K_new, V_new, stream)
            self.forward(Q, O, idx_out, stream, after_pool_keys=True)
            return
        # the absorb on a side stream; ring write, key pooling and the prologue
        # on `stream`; the attention (the only reader of the state) waits for it
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        if self._side is None:
            self._side = torch.cuda.Stream(self.device)
            self._ev_fork, self._ev_state = torch.cuda.Event(), torch.cuda.Event()
        self._ev_fork.record(main)
        self._side.wait_event(self._ev_fork)
        self.absorb_evicted(self._side, share_sms=True)
        self._ev_state.record(self._side)
        self.write_chunk(K_new, V_new, main)
        self.forward(Q, O, idx_out, main, state_ready=self._ev_state, after_pool_keys=True)

    # ---- checkpoint / resume ----
    def state_dict(self) -> dict:
        """Everything the stream needs to continue: ring, state, frame count."""
        return {"Kc": self.Kc.clone(), "Vc": self.Vc.clone(), "S": self.S.clone(), "z": self.z.clone(),
                "frames": self.frames}

    def load_state_dict(self, sd: dict):
        self.Kc.copy_(sd["Kc"])
        self.Vc.copy_(sd["Vc"])
        self.S.copy_(sd["S"])
        self.z.copy_(sd["z"])
        self.frames = int(sd["frames"])
        self.state_changed()
        self.invalidate_key_cache()   # the next forward re-pools the window

    def check_device_status(self, stream=None):
        rc, site = hb.hf_get_device_status(self.ws, stream)
        if rc != hb.HF_OK:
            raise hb.HFError(rc, "device status", f"site {site}: {hb.lib().hf_last_error().decode()}")


class HostStreamer:
    """Streams chunks from pinned host memory through a layer, overlapping the
    host<->device copies with compute.

    The layer needs spare_slots >= chunk_frames.  Frame f lives in slot
    f mod R (R = W + spare), so the slots the next chunk takes held frames
    that the current step absorbs; once that absorb is done, the next chunk's
    copy-in runs while the current forward still reads the window.  Q and O
    are double-buffered on the device.  Three streams (compute,
    host->device, device->host) ordered by events.

    push(Qh, Kh, Vh, Oh): Qh, Oh [BH, C*N_f, d] and Kh, Vh [BH, C, N_f, d],
    bf16 pinned host tensors.  Per chunk, on the compute stream: absorb the
    frames the chunk's arrival evicted (still in their slots), then, once the
    chunk's copies have landed, the hybrid forward; then O is copied back.
    Oh is valid after synchronize().
    """

    def __init__(self, layer: HybridAttentionLayer):
        assert layer.R >= layer.window + layer.C, "HostStreamer needs spare_slots >= chunk_frames"
        self.L = layer
        dev = layer.device
        shape = (layer.BH, layer.C * layer.nf, layer.d)
        self.Qd = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.Od = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.cs = torch.cuda.Stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.n = 0
        self.ev_h2d = [torch.cuda.Event() for _ in range(2)]
        self.ev_fwd = [torch.cuda.Event() for _ in range(2)]
        self.ev_d2h = [torch.cuda.Event() for _ in range(2)]
        self.ev_absorb = torch.cuda.Event()
        self.h2d_bytes = 0
        self.d2h_bytes = 0

    def push(self, Qh, Kh, Vh, Oh):
        L, b = self.L, self.n % 2
        # 1. copy-in: the chunk's slots were absorbed by the previous step;
        #    Qd[b] was last read by the forward two chunks back.
        slots = L.chunk_slots()
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.ev_absorb)
            self.h2d.wait_event(self.ev_fwd[b])
            self.Qd[b].copy_(Qh, non_blocking=True)
            # one pitched copy per frame and tensor straight from the pinned buffers
            hb.hf_ring_write(L.cfg, Kh, Vh, L.Kc, L.Vc, L.ss, slots, self.h2d)
            self.ev_h2d[b].record(self.h2d)
        self.h2d_bytes += (Qh.numel() + Kh.numel() + Vh.numel()) * 2
        # 2. compute: absorb the frames this chunk's arrival evicts (they are
        #    still in their slots), then the forward once the copies landed.
        evicted = L.frames_to_evict()
        L.frames += L.C
        for run in L._slot_runs(evicted):
            L.absorb_slots(run[0], len(run), self.cs)
        self.ev_absorb.record(self.cs)
        self.cs.wait_event(self.ev_h2d[b])
        L.pool_slots(slots, self.cs)                  # the chunk's key blocks, once they landed
        self.cs.wait_event(self.ev_d2h[b])            # Od[b] has been read back
        L.forward(self.Qd[b], self.Od[b], None, self.cs)
        self.ev_fwd[b].record(self.cs)
        # 3. copy-out
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.ev_fwd[b])
            Oh.copy_(self.Od[b], non_blocking=True)
            self.ev_d2h[b].record(self.d2h)
        self.d2h_bytes += Oh.numel() * 2
        self.n += 1

    def synchronize(self):
        self.d2h.synchronize()
        self.cs.synchronize()
        self.h2d.synchronize()

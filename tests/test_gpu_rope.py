"""The relative temporal RoPE pre-step on the GPU against the oracle
(Hybrid Forcing, English technical summary, section 2.C: temporal RoPE
indices under a fixed upper bound, positions as relative offsets)."""

import numpy as np
import pytest
import torch

import oracle
from hybrid_sparse_linear_scores_b300 import binding as hb

from gpu_harness import compare

pytestmark = pytest.mark.gpu


def _cfg(BH, d, nf, W, C):
    return hb.make_config(1, BH, d, nf, W, C, 64, 4)


def test_rope_matches_oracle(cuda_device):
    """Compact [BH, F, N_f, d] frames, a ragged token count (two CTAs per
    frame, the second partial), offsets above the bound (clamped) and
    rot_dims < d (the other channels pass bit for bit)."""
    BH, F, nf, d = 3, 5, 100, 128
    offsets, max_off, rot = [0, 2, 4, 11, 7], 8, 96
    gen = torch.Generator().manual_seed(21)
    x = torch.randn(BH, F, nf, d, generator=gen).to(torch.bfloat16)
    xd = x.to(cuda_device)
    y = torch.empty_like(xd)
    cfg = _cfg(BH, d, nf, 9, 3)
    hb.hf_rope_relative(cfg, xd, y, F * nf * d, nf * d, list(range(F)), offsets, max_off, rot, 10000.0,
                        torch.cuda.current_stream(cuda_device))
    torch.cuda.synchronize()
    ref = oracle.rope_relative(x, offsets, max_off, rot, 10000.0)
    compare(y, ref, what="rope")
    assert torch.equal(y[..., rot:].cpu().view(torch.int16), x[..., rot:].view(torch.int16))
    # in place gives the same bits
    z = xd.clone()
    hb.hf_rope_relative(cfg, z, z, F * nf * d, nf * d, list(range(F)), offsets, max_off, rot, 10000.0,
                        torch.cuda.current_stream(cuda_device))
    torch.cuda.synchronize()
    assert torch.equal(z.view(torch.int16), y.view(torch.int16))
    # frame 3 (offset 11) is rotated exactly as an offset of 8
    w = torch.empty_like(xd[:, 3:4])
    hb.hf_rope_relative(cfg, xd[:, 3:4].contiguous(), w, nf * d, nf * d, [0], [8], max_off, rot, 10000.0,
                        torch.cuda.current_stream(cuda_device))
    torch.cuda.synchronize()
    assert torch.equal(w[:, 0].view(torch.int16), y[:, 3].view(torch.int16))


def test_rope_ring_layout(cuda_device):
    """Window frames read from ring slots with a padded slot stride into a
    rotated copy of the ring: the listed slots get their frame's rotation,
    every other slot and the padding rows keep the copy's old contents."""
    BH, R, ss, nf, d = 4, 7, 80, 70, 64
    slots, offsets, max_off = [5, 0, 3], [0, 1, 2], 2
    gen = torch.Generator().manual_seed(22)
    ring = torch.randn(BH, R, ss, d, generator=gen).to(torch.bfloat16)
    src = ring.to(cuda_device)
    dst = torch.full((BH, R, ss, d), 3.0, dtype=torch.bfloat16, device=cuda_device)
    cfg = _cfg(BH, d, nf, R, 3)
    hb.hf_rope_relative(cfg, src, dst, R * ss * d, ss * d, slots, offsets, max_off, d, 500.0,
                        torch.cuda.current_stream(cuda_device))
    torch.cuda.synchronize()
    frames = torch.stack([ring[:, s, :nf] for s in slots], dim=1)      # [BH, F, nf, d]
    ref = oracle.rope_relative(frames, offsets, max_off, d, 500.0)
    out = dst.cpu()
    for f, s in enumerate(slots):
        compare(out[:, s, :nf], ref[:, f], what=f"rope slot {s}")
    untouched = torch.ones(R, dtype=torch.bool)
    untouched[slots] = False
    assert torch.all(out[:, untouched] == 3.0)
    assert torch.all(out[:, :, nf:] == 3.0)

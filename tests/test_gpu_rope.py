"""The relative temporal RoPE pre-step on the GPU against the oracle
(Hybrid Forcing, English technical summary, section 2.C: temporal RoPE
indices under a fixed upper bound, positions as relative offsets)."""

import numpy as np
import pytest
import torch

import oracle
from hybrid_sparse_linear_scores_b300 import binding as hb
from hybrid_sparse_linear_scores_b300 import synth
from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer, RelativeRope
from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, Workload, frames_tensor

from gpu_harness import compare, config_of, flat

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


ROPE_STREAMS = {
    "tiny": CONFIGS["tiny"],
    "d128_b64_ragged": Workload("rope_s", 1, 2, 128, 200, 3, 9, 64, seed=31, recipe="drift", topk_frac=0.25, steps=5),
}


@pytest.mark.parametrize("name", list(ROPE_STREAMS))
def test_layer_step_with_relative_rope(name, cuda_device):
    """layer.step with the relative RoPE on, streamed until frames are
    evicted: every step's rotated window keys and chunk queries against the
    oracle's rope_relative (window-relative offsets, bound W - 1), and the
    step's selection (bit-exact) and output against the oracle's forward on
    those rotated tensors, with the state built from the unrotated evicted
    keys (the linear state is not rotated)."""
    w = ROPE_STREAMS[name]
    rot = w.head_dim - 16 if w.head_dim > 64 else w.head_dim
    cfg = config_of(w, w.steps - 1)
    layer = HybridAttentionLayer(cfg, cuda_device, rope=RelativeRope(rot_dims=rot))
    BH, nf, d, C = w.heads_total, w.tokens_per_frame, w.head_dim, w.chunk_frames
    for s in range(w.steps):
        layer.cfg.topk = w.k_for(s)
        Kn = frames_tensor(w, synth.STREAM_K, w.chunk(s), cuda_device)
        Vn = frames_tensor(w, synth.STREAM_V, w.chunk(s), cuda_device)
        Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(s), cuda_device))
        O = torch.empty_like(Q)
        idx = torch.empty((BH, w.n_qb(), w.k_for(s)), dtype=torch.int32, device=cuda_device)
        layer.step(Q, Kn, Vn, O, idx)
        torch.cuda.synchronize()
        layer.check_device_status()
        k_off, q_off, bound = layer.rope_offsets()
        assert bound == w.window_frames - 1 and k_off == list(range(w.n_win(s)))
        win = w.window(s)
        K_unrot = frames_tensor(w, synth.STREAM_K, win)
        Kr = layer.Kr[:, layer.slot_map(), :nf]                      # [BH, n_win, N_f, d], logical order
        compare(Kr, oracle.rope_relative(K_unrot, k_off, bound, rot), what=f"{name} step {s} keys")
        Qr = layer.Qr.reshape(BH, C, nf, d)
        compare(Qr, oracle.rope_relative(Q.reshape(BH, C, nf, d).cpu(), q_off, bound, rot),
                what=f"{name} step {s} queries")
        ev = list(range(w.absorbed_before(s)))
        S = z = None
        if ev:
            S, z = oracle.state_from_frames(flat(frames_tensor(w, synth.STREAM_K, ev)),
                                            flat(frames_tensor(w, synth.STREAM_V, ev)))
        ref = oracle.hybrid_forward(layer.Qr.cpu(), flat(Kr).cpu(), flat(frames_tensor(w, synth.STREAM_V, win)), S,
                                    z, C=C, n_win=w.n_win(s), nf=nf, beta=w.block_size, k=w.k_for(s))
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"], err_msg=f"{name} step {s}")
        compare(O, ref["O"], what=f"{name} step {s}")

"""Streaming on the GPU: the long-horizon stream (80 chunks of 3 frames, 240
frames) against the oracle at sampled steps, checkpoint/resume, and the
host streamer (copies overlapped with compute) against the plain layer.

Hybrid Forcing, English technical summary, section 2.A.1: the state absorbs
every frame evicted from the window, at constant size whatever the length
of the video."""

import numpy as np
import pytest
import torch

import oracle
from hybrid_sparse_linear_scores_b300 import synth
from hybrid_sparse_linear_scores_b300.stream import HostStreamer, HybridAttentionLayer
from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, Workload, frames_tensor

from gpu_harness import compare, compare_state, config_of, flat, sample_rows

pytestmark = pytest.mark.gpu


def chunk_inputs(w: Workload, s: int, dev):
    Kn = frames_tensor(w, synth.STREAM_K, w.chunk(s), dev)
    Vn = frames_tensor(w, synth.STREAM_V, w.chunk(s), dev)
    Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(s), dev))
    return Q, Kn, Vn


def test_long_horizon_stream(cuda_device):
    """240 frames through the layer's ring: at steps {0, 1, 2, 3, 40, 79} all
    selected indices are exact and sampled rows of three heads match the
    oracle, whose state is absorbed frame by frame in fp64 alongside; the
    device state matches it at the end; the state never changes size."""
    w = CONFIGS["stream"]
    check = {0, 1, 2, 3, 40, 79}
    heads = [0, 5, 11]
    cfg = config_of(w, w.steps - 1)
    L = HybridAttentionLayer(cfg, cuda_device)
    state_bytes = L.S.numel() * 4 + L.z.numel() * 4
    S_ref = np.zeros((len(heads), w.head_dim, w.head_dim))
    z_ref = np.zeros((len(heads), w.head_dim))
    for s in range(w.steps):
        cfg.topk = w.k_for(s)
        L.cfg.topk = w.k_for(s)
        Q, Kn, Vn = chunk_inputs(w, s, cuda_device)
        O = torch.empty_like(Q)
        idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(s)), dtype=torch.int32, device=cuda_device)
        L.step(Q, Kn, Vn, O, idx)
        new = w.newly_absorbed(s)
        if new:
            Ke = flat(frames_tensor(w, synth.STREAM_K, new, cuda_device)[heads]).cpu()
            Ve = flat(frames_tensor(w, synth.STREAM_V, new, cuda_device)[heads]).cpu()
            S_ref, z_ref = oracle.state_from_frames(Ke, Ve, S_ref, z_ref)
        assert L.S.numel() * 4 + L.z.numel() * 4 == state_bytes
        if s not in check:
            continue
        torch.cuda.synchronize()
        L.check_device_status()
        win = w.window(s)
        Kw = flat(frames_tensor(w, synth.STREAM_K, win, cuda_device)).cpu()
        Vw = flat(frames_tensor(w, synth.STREAM_V, win, cuda_device)).cpu()
        geo = dict(C=w.chunk_frames, n_win=w.n_win(s), nf=w.tokens_per_frame, beta=w.block_size, k=w.k_for(s))
        ref_idx = oracle.hybrid_forward(Q.cpu(), Kw, Vw, None, None, rows=np.array([0], np.int32), **geo)["idx"]
        np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx, err_msg=f"step {s}")
        rows = sample_rows(w, 48, seed=s)
        have_state = w.absorbed_before(s) > 0
        ref = oracle.hybrid_forward(Q[heads].cpu(), Kw[heads], Vw[heads], S_ref if have_state else None,
                                    z_ref if have_state else None, rows=rows, **geo)
        compare(O[heads][:, rows], ref["O"], what=f"stream step {s}")
    compare_state(L.S[heads], L.z[heads], S_ref, z_ref)


def test_checkpoint_resume_is_bit_identical(cuda_device):
    """Save the streaming state after 3 chunks, restore it into a fresh layer
    and continue: every later output and index is bit-identical to the
    uninterrupted run (all kernels are deterministic)."""
    w = Workload("ckpt", 1, 2, 128, 200, 2, 6, 64, seed=31, recipe="drift", topk_frac=0.3, steps=8)
    cfg = config_of(w, w.steps - 1)
    A = HybridAttentionLayer(cfg, cuda_device)
    outs_a, saved = [], None
    for s in range(w.steps):
        A.cfg.topk = w.k_for(s)
        Q, Kn, Vn = chunk_inputs(w, s, cuda_device)
        O = torch.empty_like(Q)
        idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(s)), dtype=torch.int32, device=cuda_device)
        A.step(Q, Kn, Vn, O, idx)
        outs_a.append((O, idx))
        if s == 2:
            torch.cuda.synchronize()
            saved = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in A.state_dict().items()}
    B = HybridAttentionLayer(cfg, cuda_device)
    B.load_state_dict(saved)
    for s in range(3, w.steps):
        B.cfg.topk = w.k_for(s)
        Q, Kn, Vn = chunk_inputs(w, s, cuda_device)
        O = torch.empty_like(Q)
        idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(s)), dtype=torch.int32, device=cuda_device)
        B.step(Q, Kn, Vn, O, idx)
        torch.cuda.synchronize()
        assert torch.equal(idx, outs_a[s][1]), f"step {s}"
        assert torch.equal(O.view(torch.int16), outs_a[s][0].view(torch.int16)), f"step {s}"


def test_host_streamer_matches_layer_steps(cuda_device):
    """Chunks pushed from pinned host memory through HostStreamer (ring with
    spare slots, copies on their own streams) give bit-identical outputs to
    the plain layer stepping the same chunks."""
    w = Workload("hs", 1, 3, 128, 300, 3, 9, 64, seed=41, recipe="drift", topk=20, steps=7)
    cfg = config_of(w, w.steps - 1)
    ref = HybridAttentionLayer(cfg, cuda_device)
    L = HybridAttentionLayer(cfg, cuda_device, spare_slots=w.chunk_frames)
    hs = HostStreamer(L)
    outs_ref, outs_host, keep = [], [], []
    for s in range(w.steps):
        Q, Kn, Vn = chunk_inputs(w, s, cuda_device)
        O = torch.empty_like(Q)
        ref.step(Q, Kn, Vn, O)
        outs_ref.append(O)
        Oh = torch.empty(Q.shape, dtype=Q.dtype).pin_memory()
        host = (Q.cpu().pin_memory(), Kn.cpu().pin_memory(), Vn.cpu().pin_memory())
        keep.append(host)                   # host buffers live until the copies are done
        hs.push(*host, Oh)
        outs_host.append(Oh)
    hs.synchronize()
    torch.cuda.synchronize()
    ref.check_device_status()
    L.check_device_status()
    for s in range(w.steps):
        assert torch.equal(outs_host[s].view(torch.int16), outs_ref[s].cpu().view(torch.int16)), f"chunk {s}"
    assert torch.equal(L.S, ref.S) and torch.equal(L.z, ref.z)


@pytest.mark.parametrize("where", ["pinned_host", "device"])
def test_ring_write_places_frames(where, cuda_device):
    """hf_ring_write puts frame f of every head into rows [0, N_f) of ring
    slot slots[f], bit for bit, from pinned host memory or from device
    memory, and leaves the other slots and the padding rows of the written
    slots (slot_stride > N_f) untouched."""
    from hybrid_sparse_linear_scores_b300 import binding as hb
    BH, nf, d, R, ss, C = 6, 100, 64, 7, 112, 3
    cfg = hb.make_config(1, BH, d, nf, R, C, 64, 4)
    gen = torch.Generator().manual_seed(5)
    K = torch.randn(BH, C, nf, d, generator=gen).to(torch.bfloat16)
    V = torch.randn(BH, C, nf, d, generator=gen).to(torch.bfloat16)
    Ks, Vs = (K.pin_memory(), V.pin_memory()) if where == "pinned_host" else (K.to(cuda_device), V.to(cuda_device))
    slots = [5, 0, 3]
    fill = torch.full((BH, R, ss, d), 7.0, dtype=torch.bfloat16)
    Kc, Vc = fill.to(cuda_device), fill.to(cuda_device)
    hb.hf_ring_write(cfg, Ks, Vs, Kc, Vc, ss, slots, torch.cuda.current_stream(cuda_device))
    torch.cuda.synchronize()
    for src, ring in ((K, Kc), (V, Vc)):
        ref = fill.clone()
        for f, sl in enumerate(slots):
            ref[:, sl, :nf] = src[:, f]
        assert torch.equal(ring.cpu().view(torch.int16), ref.view(torch.int16))


def test_overlapped_step_matches_sequential_step(cuda_device):
    """With spare ring slots the layer's step runs the absorb on a side stream
    beside the ring write, key pooling and prologue (the attention waits for
    it), on fewer SMs; indices are identical and outputs and state agree with
    the sequential step of a layer without spare slots up to the order of the
    absorb's cluster reduction (a few fp32 ulps of the state)."""
    w = Workload("ovl", 1, 3, 128, 300, 3, 9, 64, seed=43, recipe="drift", topk=20, steps=7)
    cfg = config_of(w, w.steps - 1)
    seq = HybridAttentionLayer(cfg, cuda_device)
    ovl = HybridAttentionLayer(cfg, cuda_device, spare_slots=w.chunk_frames)
    assert ovl.can_overlap_absorb() and not seq.can_overlap_absorb()
    for s in range(w.steps):
        Q, Kn, Vn = chunk_inputs(w, s, cuda_device)
        outs = []
        for L in (seq, ovl):
            O = torch.empty_like(Q)
            idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(s)), dtype=torch.int32, device=cuda_device)
            L.step(Q, Kn, Vn, O, idx)
            outs.append((O, idx))
        torch.cuda.synchronize()
        assert torch.equal(outs[0][1], outs[1][1]), f"step {s}"
        a, b = outs[0][0].float(), outs[1][0].float()
        assert float((a - b).abs().max()) <= 2.0 ** -7 * float(a.abs().max()), f"step {s}"
        assert float((a - b).norm() / a.norm()) <= 1e-4, f"step {s}"
    seq.check_device_status()
    ovl.check_device_status()
    for x, y in ((seq.S, ovl.S), (seq.z, ovl.z)):
        assert float((x - y).norm() / x.norm()) <= 1e-6


def test_state_operand_from_absorb_matches_prologue(cuda_device):
    """The absorb writes the state's tensor-core operand; a forward that uses it
    (HF_FWD_STATE_PREPARED, S not read) is bit-identical to one whose prologue
    converts S itself."""
    from hybrid_sparse_linear_scores_b300 import binding as hb
    w = Workload("prep", 1, 2, 128, 300, 3, 9, 64, seed=47, recipe="drift", topk=25, steps=5)
    cfg = config_of(w, w.steps - 1)
    L = HybridAttentionLayer(cfg, cuda_device)
    for s in range(w.steps - 1):
        Q, Kn, Vn = chunk_inputs(w, s, cuda_device)
        L.step(Q, Kn, Vn, torch.empty_like(Q))
    s = w.steps - 1
    Q, Kn, Vn = chunk_inputs(w, s, cuda_device)
    L.absorb_evicted()
    L.write_chunk(Kn, Vn)
    outs = []
    for flags in (hb.HF_FWD_CACHED_KEYS | hb.HF_FWD_STATE_PREPARED, hb.HF_FWD_CACHED_KEYS):
        O = torch.empty_like(Q)
        idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(s)), dtype=torch.int32, device=cuda_device)
        S = None if flags & hb.HF_FWD_STATE_PREPARED else L.S
        hb.hf_hybrid_forward_ex(L.cfg, Q, L.Kc, L.Vc, L.ss, L.slot_map(), L.n_win(), S, L.z, O, idx, L.ws, flags)
        outs.append((O, idx))
    torch.cuda.synchronize()
    L.check_device_status()
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))

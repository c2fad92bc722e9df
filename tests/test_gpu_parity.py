"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs.  Indices bit-exact; outputs within max|d| <= 2e-2 and
relative L2 <= 5e-3 of the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from hybrid_sparse_linear_scores_b300 import binding as hb
from hybrid_sparse_linear_scores_b300 import synth
from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer
from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, SWEEP, Workload, frames_tensor, scaled

from gpu_harness import STATE_REL_L2, Step, compare, compare_state, config_of, flat, sample_rows

pytestmark = pytest.mark.gpu

# Small shapes that still span several tiles and a ragged tail, one per
# (head_dim, block size) path of the kernels.
SMALL = {
    "d128_b64_ragged8": Workload("s1", 1, 2, 128, 200, 3, 9, 64, seed=11, recipe="frame_mean", topk_frac=0.25,
                                 absorbed_frames=4),
    "d128_b128_ragged44": Workload("s2", 1, 2, 128, 300, 3, 9, 128, seed=12, recipe="clustered", topk_frac=0.25,
                                   absorbed_frames=3),
    "d128_b32_ragged4": Workload("s3", 1, 2, 128, 100, 2, 5, 32, seed=13, recipe="normal", topk_frac=0.3,
                                 absorbed_frames=2),
    "d64_b64": Workload("s4", 2, 2, 64, 130, 1, 4, 64, seed=14, recipe="normal", topk_frac=0.5, absorbed_frames=5),
    "d64_b128_dense_empty": Workload("s5", 1, 1, 64, 200, 2, 3, 128, seed=15, recipe="normal", topk_frac=1.0),
    "d128_b64_k1": Workload("s6", 1, 3, 128, 192, 1, 3, 64, seed=16, recipe="frame_mean", topk=1,
                            absorbed_frames=1),
    "d128_b64_one_frame_window": Workload("s7", 1, 2, 128, 96, 1, 1, 64, seed=17, recipe="normal", topk=2),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_hybrid_forward_small(name, cuda_device):
    w = SMALL[name]
    st = Step(w, 0, cuda_device)
    O, idx = st.run_forward()
    ref = st.oracle_forward()
    np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
    compare(O, ref["O"], what=name)


def test_tiny_stream_every_step(cuda_device):
    """The tiny workload streamed for 6 frames through the layer's own ring:
    absorb of the evicted frame from its slot, then the forward."""
    w = CONFIGS["tiny"]
    cfg = config_of(w, w.steps - 1)
    layer = HybridAttentionLayer(cfg, cuda_device)
    for s in range(w.steps):
        cfg.topk = w.k_for(s)
        Kn = frames_tensor(w, synth.STREAM_K, w.chunk(s), cuda_device)
        Vn = frames_tensor(w, synth.STREAM_V, w.chunk(s), cuda_device)
        Q = flat(frames_tensor(w, synth.STREAM_Q, w.chunk(s), cuda_device))
        O = torch.empty_like(Q)
        idx = torch.empty((w.heads_total, w.n_qb(), w.k_for(s)), dtype=torch.int32, device=cuda_device)
        layer.step(Q, Kn, Vn, O, idx)
        torch.cuda.synchronize()
        layer.check_device_status()
        ref = Step(w, s, "cpu", absorb_on_gpu=False).oracle_forward()
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"], err_msg=f"step {s}")
        compare(O, ref["O"], what=f"tiny step {s}")


def all_head_indices(st: Step, w: Workload, margin: bool = False):
    """The oracle's selection for every head (pooling, scores and top-K run on
    all heads; one query row of attention is enough for that)."""
    return oracle.hybrid_forward(st.Q.cpu(), flat(st.Kwin).cpu(), flat(st.Vwin).cpu(), None, None,
                                 C=w.chunk_frames, n_win=w.n_win(0), nf=w.tokens_per_frame, beta=w.block_size,
                                 k=w.k_for(0), rows=[0], margin=margin)


@pytest.mark.parametrize("name", ["realistic", "wide", "dense_w21"])
def test_full_config_sampled_rows(name, cuda_device):
    """Full size: the indices of every head exact; outputs on rows sampled
    over every tile, on every head (every fifth head of the 40-head layer).
    dense_w21 is the dense sliding-window baseline (W = 21, every block
    selected, empty state)."""
    w = CONFIGS[name]
    st = Step(w, 0, cuda_device)
    O, idx = st.run_forward()
    np.testing.assert_array_equal(idx.cpu().numpy(), all_head_indices(st, w)["idx"])
    rows = sample_rows(w, 160)
    heads = list(range(w.heads_total)) if w.heads_total <= 12 else list(range(0, w.heads_total, 5))
    S, z = st.oracle_state()
    ref = oracle.hybrid_forward(st.Q[heads].cpu(), flat(st.Kwin[heads]).cpu(), flat(st.Vwin[heads]).cpu(),
                                None if S is None else S[heads], None if z is None else z[heads],
                                C=w.chunk_frames, n_win=w.n_win(0), nf=w.tokens_per_frame,
                                beta=w.block_size, k=w.k_for(0), rows=rows)
    compare(O[heads][:, rows], ref["O"], what=name)


@pytest.mark.parametrize("w", SWEEP, ids=[w.name for w in SWEEP])
def test_sweep_sampled_rows(w, cuda_device):
    """The sparsity/block sweep (clustered keys: the near-tie stress): the
    indices of all 12 heads exact, with the smallest float64 margin between
    the K-th and (K+1)-th score printed; outputs on sampled rows of 3 heads."""
    st = Step(w, 0, cuda_device)
    O, idx = st.run_forward()
    sel = all_head_indices(st, w, margin=True)
    np.testing.assert_array_equal(idx.cpu().numpy(), sel["idx"])
    if w.k_for(0) < w.n_kb(0):
        print(f"{w.name}: smallest float64 score margin between ranks K and K+1 over all heads: "
              f"{float(sel['margin'].min()):.3e}")
    heads = [0, 5, 11]
    rows = sample_rows(w, 96, seed=1)
    S, z = st.oracle_state()
    ref = oracle.hybrid_forward(st.Q[heads].cpu(), flat(st.Kwin[heads]).cpu(), flat(st.Vwin[heads]).cpu(),
                                None if S is None else S[heads], None if z is None else z[heads],
                                C=w.chunk_frames, n_win=w.n_win(0), nf=w.tokens_per_frame, beta=w.block_size,
                                k=w.k_for(0), rows=rows)
    compare(O[heads][:, rows], ref["O"], what=w.name)


@pytest.mark.parametrize("name", ["d128_b64_ragged8", "d128_b128_ragged44", "d128_b32_ragged4", "d64_b64"])
def test_cached_key_pools_bit_identical(name, cuda_device):
    """hf_pool_keys + hf_hybrid_forward_ex(HF_FWD_CACHED_KEYS) gives the same
    indices and output bits as pooling the whole window in the forward, with
    the ring slots pooled in an order different from the window's."""
    w = SMALL[name]
    st = Step(w, 0, cuda_device)
    L = st.layer
    O_ref, idx_ref = st.run_forward()                       # pools every window frame
    # wipe the cache, then pool the window's slots one call per slot, newest first
    L.ws[1024:].zero_()
    L.invalidate_key_cache()
    for sl in reversed(L.slot_map()):
        L.pool_slots([sl])
    O = torch.empty_like(st.Q)
    idx = torch.empty_like(idx_ref)
    hb.hf_hybrid_forward_ex(L.cfg, st.Q, L.Kc, L.Vc, L.ss, L.slot_map(), L.n_win(), L.S, L.z, O, idx, L.ws,
                            hb.HF_FWD_CACHED_KEYS)
    torch.cuda.synchronize()
    L.check_device_status()
    assert torch.equal(idx, idx_ref)
    assert torch.equal(O.view(torch.int16), O_ref.view(torch.int16))


def test_pool_keys_rejects_bad_slots(cuda_device):
    w = SMALL["d128_b64_ragged8"]
    L = HybridAttentionLayer(config_of(w, 0), cuda_device)
    for slots in ([w.window_frames], [-1], [0, 0]):
        with pytest.raises(hb.HFError) as e:
            hb.hf_pool_keys(L.cfg, L.Kc, L.ss, slots, L.ws)
        assert e.value.code == 1


def test_standalone_entry_points(cuda_device):
    """hf_block_scores, hf_topk_blocks, hf_sparse_swa_attn, hf_linear_read,
    hf_absorb_evicted each against the matching oracle step."""
    w = SMALL["d128_b64_ragged8"]
    st = Step(w, 0, cuda_device)
    cfg, L = st.cfg, st.layer
    BH, nqb, nkb, k = w.heads_total, w.n_qb(), w.n_kb(0), w.k_for(0)
    # scores: bit-exact float32
    scores = torch.empty((BH, nqb, nkb), dtype=torch.float32, device=cuda_device)
    hb.hf_block_scores(cfg, st.Q, L.Kc, L.ss, L.slot_map(), L.n_win(), scores, L.ws)
    idx = torch.empty((BH, nqb, k), dtype=torch.int32, device=cuda_device)
    hb.hf_topk_blocks(cfg, scores, nqb, nkb, idx)
    torch.cuda.synchronize()
    for h in range(BH):
        qp = oracle.pool(st.Q[h].cpu().reshape(w.chunk_frames, w.tokens_per_frame, -1), w.block_size)
        kp = oracle.pool(st.Kwin[h].cpu(), w.block_size)
        s_ref = oracle.scores(qp, kp)
        np.testing.assert_array_equal(scores[h].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
        np.testing.assert_array_equal(idx[h].cpu().numpy(), oracle.topk(s_ref, k))
    # sparse attention alone (fp32 output) and the linear read alone
    O_swa = torch.empty(st.Q.shape, dtype=torch.float32, device=cuda_device)
    hb.hf_sparse_swa_attn(cfg, st.Q, L.Kc, L.Vc, L.ss, L.slot_map(), L.n_win(), idx, O_swa, L.ws)
    O_lin = torch.empty_like(O_swa)
    hb.hf_linear_read(cfg, st.Q, L.S, L.z, O_lin)
    torch.cuda.synchronize()
    L.check_device_status()
    ref = st.oracle_forward(split=True)
    compare(O_swa, ref["O_swa"], max_abs=1e-2, rel_l2=3e-3, what="O_swa")
    compare(O_lin, ref["O_lin"], max_abs=1e-4, rel_l2=1e-5, what="O_lin")
    # accumulate: O_swa + o_lin in fp32 equals the oracle's sum
    hb.hf_linear_read(cfg, st.Q, L.S, L.z, O_swa, accumulate=True)
    torch.cuda.synchronize()
    compare(O_swa, ref["O"], max_abs=1e-2, rel_l2=3e-3, what="O_swa + O_lin")
    # the state itself
    S_ref, z_ref = st.oracle_state()
    compare_state(L.S, L.z, S_ref, z_ref)


@pytest.mark.parametrize("name", ["realistic", "wide"])
def test_absorb_full_config(name, cuda_device):
    w = CONFIGS[name]
    st = Step(w, 0, cuda_device)
    torch.cuda.synchronize()
    st.layer.check_device_status()
    heads = [0, w.heads_total - 1]
    S_ref, z_ref = oracle.state_from_frames(flat(st.Kev[heads]).cpu(), flat(st.Vev[heads]).cpu())
    compare_state(st.layer.S[heads], st.layer.z[heads], S_ref, z_ref)


def test_incremental_absorb_matches_one_shot(cuda_device):
    """Absorbing frame by frame equals absorbing all frames at once (fp32 sums
    in different orders: close, not bit-equal)."""
    w = CONFIGS["realistic"]
    cfg = config_of(w, 0)
    L1 = HybridAttentionLayer(cfg, cuda_device)
    L2 = HybridAttentionLayer(cfg, cuda_device)
    K = frames_tensor(w, synth.STREAM_K, range(6), cuda_device)
    V = frames_tensor(w, synth.STREAM_V, range(6), cuda_device)
    hb.hf_absorb_evicted(cfg, L1.S, L1.z, flat(K), flat(V), 6 * w.tokens_per_frame, L1.ws)
    for f in range(6):
        hb.hf_absorb_evicted(cfg, L2.S, L2.z, flat(K[:, f:f + 1].contiguous()), flat(V[:, f:f + 1].contiguous()),
                             w.tokens_per_frame, L2.ws)
    torch.cuda.synchronize()
    d = (L1.S - L2.S).norm() / L1.S.norm()
    assert float(d) < STATE_REL_L2


def test_deterministic_repeat(cuda_device):
    w = CONFIGS["realistic"]
    st = Step(w, 0, cuda_device)
    O1, i1 = st.run_forward()
    O2, i2 = st.run_forward()
    assert torch.equal(i1, i2)
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))


def test_ring_slot_map_is_honoured(cuda_device):
    """The same logical window laid into the ring at a rotated position gives
    bit-identical results."""
    w = SMALL["d128_b64_ragged8"]
    st = Step(w, 0, cuda_device)
    O1, i1 = st.run_forward()
    L = st.layer
    rot = 4
    Kc2 = torch.roll(L.Kc, rot, dims=1).contiguous()
    Vc2 = torch.roll(L.Vc, rot, dims=1).contiguous()
    sm = [(s + rot) % w.window_frames for s in L.slot_map()]
    O2 = torch.empty_like(O1)
    i2 = torch.empty_like(i1)
    hb.hf_hybrid_forward(st.cfg, st.Q, Kc2, Vc2, L.ss, sm, L.n_win(), L.S, L.z, O2, i2, L.ws)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(O1.view(torch.int16), O2.view(torch.int16))


def test_padded_slot_stride(cuda_device):
    """slot_stride > N_f: rows past N_f in a slot are never read."""
    w = SMALL["d128_b64_ragged8"]
    st = Step(w, 0, cuda_device)
    O1, i1 = st.run_forward()
    L = st.layer
    pad = 56
    Kc2 = torch.full((L.BH, L.W, L.ss + pad, L.d), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    Vc2 = torch.full_like(Kc2, float("nan"))
    Kc2[:, :, :L.ss] = L.Kc
    Vc2[:, :, :L.ss] = L.Vc
    O2 = torch.empty_like(O1)
    i2 = torch.empty_like(i1)
    hb.hf_hybrid_forward(st.cfg, st.Q, Kc2, Vc2, L.ss + pad, L.slot_map(), L.n_win(), L.S, L.z, O2, i2, L.ws)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(O1.view(torch.int16), O2.view(torch.int16))


def test_bounded_wait_reports_timeout(cuda_device):
    """A wait on a barrier nothing releases ends after its limit with
    HF_ERR_TIMEOUT in the status word; the context stays usable."""
    ws = torch.zeros(1024, dtype=torch.uint8, device=cuda_device)
    hb.hf_selftest_wait_timeout(ws, 2000)
    rc, site = hb.hf_get_device_status(ws)
    assert rc == 4 and site == 301
    rc, site = hb.hf_get_device_status(ws)
    assert rc == 0
    x = torch.ones(4, device=cuda_device)
    assert float(x.sum()) == 4.0


def test_bad_index_is_reported(cuda_device):
    """An out-of-range block index given to the attention entry point is
    caught on the device (HF_ERR_DEVICE_CHECK), nothing is read out of bounds."""
    w = SMALL["d128_b64_ragged8"]
    st = Step(w, 0, cuda_device)
    L = st.layer
    idx = torch.zeros((w.heads_total, w.n_qb(), w.k_for(0)), dtype=torch.int32, device=cuda_device)
    idx[0, 0, 0] = 10_000
    O = torch.empty(st.Q.shape, dtype=torch.float32, device=cuda_device)
    hb.hf_sparse_swa_attn(st.cfg, st.Q, L.Kc, L.Vc, L.ss, L.slot_map(), L.n_win(), idx, O, L.ws)
    rc, site = hb.hf_get_device_status(L.ws)
    assert rc == 5 and site == 110


def test_stale_split_counters_do_not_change_a_forward(cuda_device):
    """A launch that gives up part-way (a bounded wait that ran out) can leave
    the arrival counters of split tile pairs non-zero in the workspace.  Plant
    such leftovers (the bytes a stuck count would leave, written from the
    host: no wait is made to run out on the GPU) and check that the next
    forward on the same workspace is bit-identical to a clean one: the
    forward resets the counters before its attention kernel runs."""
    w = CONFIGS["realistic"]
    st = Step(w, 0, cuda_device)
    O1, i1 = st.run_forward()
    G = 128 // w.block_size
    pairs = w.heads_total * ((-(-w.n_qb() // G) + 1) // 2)
    counters = st.layer.ws[1024:1024 + 8 * pairs]          # uint32 [pairs][2] at offset 1024
    for fill in (1, 0xFF):
        counters.fill_(fill)
        O2, i2 = st.run_forward()
        assert torch.equal(i1, i2)
        assert torch.equal(O1.view(torch.int16), O2.view(torch.int16)), f"counter bytes 0x{fill:02x}"

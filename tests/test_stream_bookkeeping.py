"""Host-side bookkeeping of the streaming layer (no kernels run): which
frames each chunk evicts into the state, where the chunk's frames go in the
K/V ring, and the window's slot map (Hybrid Forcing, English technical
summary, section 2.A.1: frames leaving the sliding window are absorbed into
the linear state; section 2.A.2: attention over the last W frames)."""

import pytest

from hybrid_sparse_linear_scores_b300 import binding as hb
from hybrid_sparse_linear_scores_b300.stream import HybridAttentionLayer


def _layer(W, C, spare, nf=64, slot_stride=None):
    cfg = hb.make_config(1, 1, 64, nf, W, C, 64, 1)
    return HybridAttentionLayer(cfg, device="cpu", slot_stride=slot_stride, spare_slots=spare)


@pytest.mark.parametrize("W,C,spare", [(9, 3, 0), (9, 3, 3), (5, 2, 0), (4, 1, 1), (7, 7, 0)])
def test_every_frame_is_absorbed_once_and_in_order(W, C, spare):
    """Over a long stream the evicted frames are exactly the frames that leave
    the window, each once, oldest first; the window's slot map lists the last
    min(W, frames) frames in order, frame f in slot f mod R."""
    L = _layer(W, C, spare)
    absorbed = []
    for step in range(100):
        ev = L.frames_to_evict()
        after = L.frames + C
        assert ev == list(range(max(0, L.frames - W), max(0, after - W)))
        absorbed += ev
        L.frames = after
        win = list(range(max(0, L.frames - W), L.frames))
        assert L.n_win() == len(win)
        assert L.slot_map() == [f % L.R for f in win]
    assert absorbed == list(range(100 * C - W))


@pytest.mark.parametrize("W,C,spare", [(9, 3, 0), (9, 3, 3), (4, 1, 1)])
def test_chunk_slots(W, C, spare):
    """The next chunk's frames take consecutive ring positions f mod R.  With
    no spare slots they are the slots of the frames the chunk evicts (once the
    window is full); with C spare slots they hold no frame of the current
    window, so the chunk can be copied in while the window is still read."""
    L = _layer(W, C, spare)
    for step in range(40):
        slots = L.chunk_slots()
        assert slots == [(L.frames + c) % L.R for c in range(C)]
        window_slots = set(L.slot_map())
        if spare >= C:
            assert not window_slots & set(slots)
        elif L.frames >= W:
            assert set(slots) == {f % L.R for f in L.frames_to_evict()}
        L.frames += C


def test_slot_runs_group_consecutive_slots():
    """Evicted frames are absorbed in runs of consecutive ring slots (one
    strided absorb per run); a run never wraps around the ring, and padded
    slots (slot stride > N_f) are never merged into one run."""
    L = _layer(9, 3, 0)
    assert L._slot_runs([6, 7, 8]) == [[6, 7, 8]]
    assert L._slot_runs([7, 8, 9, 10]) == [[7, 8], [0, 1]]      # slots 7, 8, 0, 1
    P = _layer(9, 3, 0, slot_stride=80)
    assert P._slot_runs([3, 4, 5]) == [[3], [4], [5]]

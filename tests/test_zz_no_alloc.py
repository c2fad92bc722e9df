"""hf_hybrid_forward_noalloc: the hybrid forward for callers that cannot
allocate device memory (a custom-operator interface that passes only inputs,
outputs and a stream; code running under CUDA graph capture, where cudaMalloc
is not allowed; an engine that keeps all device memory in its own pool).  It
runs the same kernels as hf_hybrid_forward with the workspace in the
library's static device array instead of a caller buffer, so its indices and
output must match hf_hybrid_forward's.

This file is named to be collected last: a run that stops at the first
failure has then already run every other test."""

import numpy as np
import pytest
import torch

from hybrid_sparse_linear_scores_b300 import binding as hb
from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, Workload

from gpu_harness import MAX_ABS, REL_L2, Step, config_of


def _compare_to_workspace_path(st: Step):
    """One call of each entry point on the same inputs; returns the status
    word address the no-alloc call reported."""
    w, L = st.w, st.layer
    dev = st.Q.device
    shape_idx = (w.heads_total, w.n_qb(), w.k_for(st.step))
    O_ref = torch.empty_like(st.Q)
    idx_ref = torch.empty(shape_idx, dtype=torch.int32, device=dev)
    hb.hf_hybrid_forward(st.cfg, st.Q, L.Kc, L.Vc, L.ss, L.slot_map(), L.n_win(), L.S, L.z, O_ref, idx_ref, L.ws)
    O = torch.full_like(st.Q, float("nan"))
    idx = torch.full(shape_idx, -1, dtype=torch.int32, device=dev)
    status_word = hb.hf_hybrid_forward_noalloc(st.cfg, st.Q, L.Kc, L.Vc, L.ss, L.slot_map(), L.n_win(), L.S, L.z,
                                               O, idx)
    torch.cuda.synchronize()
    L.check_device_status()
    rc, site = hb.hf_get_device_status(status_word)
    assert rc == hb.HF_OK, f"no-alloc forward reported device status {rc} at site {site}"
    np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy())
    a, b = O.double().cpu().numpy(), O_ref.double().cpu().numpy()
    assert np.isfinite(a).all()
    diff = a - b
    assert float(np.abs(diff).max()) <= MAX_ABS
    assert float(np.linalg.norm(diff) / np.linalg.norm(b)) <= REL_L2
    return status_word


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward_twice(cuda_device):
    """Two calls in a row, on two different layers (the second smaller than
    the first, so it runs over what the first left in the scratch)."""
    big = Step(CONFIGS["realistic"], 0, cuda_device)
    small = Workload("na", 1, 2, 128, 200, 3, 9, 64, seed=21, recipe="frame_mean", topk_frac=0.25,
                     absorbed_frames=4)
    s1 = _compare_to_workspace_path(big)
    s2 = _compare_to_workspace_path(Step(small, 0, cuda_device))
    assert s1 == s2 and s1 != 0   # one array per device, same address every call


def test_noalloc_rejects_configs_beyond_the_scratch():
    """Checked on the host before any CUDA call, so this runs without a GPU."""
    w = CONFIGS["wide"]
    cfg = config_of(w, 0)
    split_part = 160 * 2 * 2 * 128 * (128 + 4) * 4     # HF_SPLIT_PARTIAL_BYTES(128)
    assert hb.hf_workspace_size(cfg) - split_part <= (16 << 20)   # the 40-head layer fits
    big = hb.make_config(4, 40, 128, 1560, 9, 3, 64, 57)
    assert hb.hf_workspace_size(big) - split_part > (16 << 20)
    with pytest.raises(hb.HFError) as e:
        hb.hf_hybrid_forward_noalloc(big, 16, 16, 16, 1560, None, 9, 16, 16, 16, None, stream=0)
    assert e.value.code == 2 and "static scratch" in str(e.value)

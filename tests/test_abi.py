"""The C-ABI library loads without a GPU, exports every entry point that
include/hf.h declares, and rejects bad arguments synchronously (before any
CUDA call), so these run on a CPU-only host."""

import ctypes
import re

import pytest

from hybrid_sparse_linear_scores_b300 import binding as hb
from hybrid_sparse_linear_scores_b300.workloads import CONFIGS, SWEEP


def test_library_exports_every_declared_function():
    declared = hb.declared_functions()
    assert len(declared) >= 14
    L = hb.lib()
    for name in declared:
        assert hasattr(L, name), name
    for required in ("hf_absorb_evicted", "hf_block_scores", "hf_topk_blocks", "hf_sparse_swa_attn",
                     "hf_linear_read", "hf_hybrid_forward"):
        assert required in declared


def test_abi_version_and_status_strings():
    L = hb.lib()
    assert L.hf_abi_version() == 3
    for code, name in hb.STATUS.items():
        assert L.hf_status_string(code).decode() == name


def cfg_of(w, **over):
    c = dict(batch=w.batch, heads=w.heads, head_dim=w.head_dim, tokens_per_frame=w.tokens_per_frame,
             window_frames=w.window_frames, chunk_frames=w.chunk_frames, block_size=w.block_size,
             topk=w.k_for(w.steps - 1))
    c.update(over)
    return hb.make_config(**c)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_workspace_size_covers_buffers(name):
    w = CONFIGS[name]
    cfg = cfg_of(w)
    n = hb.hf_workspace_size(cfg)
    BH, d = w.heads_total, w.head_dim
    nkb = w.window_frames * w.blocks_per_frame
    floor = 256 + BH * (w.n_qb() + nkb) * d * 4 + BH * 2 * d * d * 2
    assert n >= floor and n % 1024 == 0


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=96), 2), (dict(head_dim=0), 2), (dict(block_size=48), 2), (dict(topk=0), 1),
    (dict(chunk_frames=10), 1), (dict(window_frames=0), 2), (dict(window_frames=65), 2),
    (dict(batch=0), 1), (dict(tokens_per_frame=0), 1), (dict(lin_eps=-1.0), 1),
    (dict(tokens_per_frame=100000, block_size=32), 2),
])
def test_config_validation(bad, code):
    cfg = cfg_of(CONFIGS["realistic"], **bad)
    with pytest.raises(hb.HFError) as ei:
        hb.hf_workspace_size(cfg)
    assert ei.value.code == code


FAKE = 1 << 20   # an aligned, never-dereferenced address: calls must fail before using it


def _fwd(cfg, **kw):
    a = dict(Q=FAKE, Kc=FAKE, Vc=FAKE, slot_stride=cfg.tokens_per_frame, slot_map=None, n_win=cfg.window_frames,
             S=FAKE, z=FAKE, O=FAKE, idx_out=None, ws=FAKE)
    a.update(kw)
    return hb.hf_hybrid_forward(cfg, a["Q"], a["Kc"], a["Vc"], a["slot_stride"], a["slot_map"], a["n_win"], a["S"],
                                a["z"], a["O"], a["idx_out"], a["ws"], stream=0)


@pytest.mark.parametrize("kw,msg", [
    (dict(Q=0), "Q is NULL"), (dict(S=FAKE + 4), "not 16-byte aligned"), (dict(n_win=2), "n_win"),
    (dict(n_win=10), "n_win"), (dict(slot_stride=100), "slot_stride"),
    (dict(slot_map=[0, 1, 2, 3, 4, 5, 6, 7, 7]), "used twice"), (dict(slot_map=[0, 1, 2, 3, 4, 5, 6, 7, 9]), "outside"),
    (dict(idx_out=FAKE + 8), "idx_out"),
])
def test_forward_argument_errors_are_synchronous(kw, msg):
    cfg = cfg_of(CONFIGS["realistic"])
    with pytest.raises(hb.HFError) as ei:
        _fwd(cfg, **kw)
    assert ei.value.code == 1
    assert msg in str(ei.value)


def test_absorb_and_topk_argument_errors():
    cfg = cfg_of(CONFIGS["realistic"])
    with pytest.raises(hb.HFError):
        hb.hf_absorb_evicted(cfg, FAKE, FAKE, FAKE, FAKE, -1, FAKE, stream=0)
    with pytest.raises(hb.HFError):
        hb.hf_absorb_evicted_strided(cfg, FAKE, FAKE, FAKE, FAKE, 100, 50, FAKE, stream=0)
    with pytest.raises(hb.HFError) as ei:
        hb.hf_topk_blocks(cfg, FAKE, 75, 2000, FAKE, stream=0)
    assert ei.value.code == 2
    with pytest.raises(hb.HFError):
        hb.hf_selftest_wait_timeout(FAKE, 0, stream=0)
    # n_ev_tokens = 0 is a no-op that never touches the device
    hb.hf_absorb_evicted(cfg, FAKE, FAKE, None, None, 0, FAKE, stream=0)


@pytest.mark.parametrize("kw,msg", [
    (dict(K_src=0), "K_src is NULL"), (dict(Vc=0), "Vc is NULL"), (dict(slots=[]), "n_frames"),
    (dict(slots=[0, 0]), "given twice"), (dict(slots=[9]), "outside"), (dict(slots=[-1]), "outside"),
    (dict(slot_stride=100), "slot_stride"),
])
def test_ring_write_argument_errors_are_synchronous(kw, msg):
    cfg = cfg_of(CONFIGS["realistic"])
    a = dict(K_src=FAKE, V_src=FAKE, Kc=FAKE, Vc=FAKE, slot_stride=cfg.tokens_per_frame, slots=[0, 1, 2])
    a.update(kw)
    with pytest.raises(hb.HFError) as ei:
        hb.hf_ring_write(cfg, a["K_src"], a["V_src"], a["Kc"], a["Vc"], a["slot_stride"], a["slots"], stream=0)
    assert ei.value.code == 1
    assert msg in str(ei.value)


def test_header_documents_every_entry_point():
    """Every declared function carries a comment block in the header."""
    text = open(hb.HEADER).read()
    for name in hb.declared_functions():
        m = re.search(r"/\*(?:(?!\*/).)*\*/\s*HF_API[^;]*\b" + name + r"\s*\(", text, re.S)
        assert m, name


@pytest.mark.parametrize("kw,msg", [
    (dict(src=0), "src is NULL"), (dict(rot_dims=12), "rot_dims"), (dict(rot_dims=136), "rot_dims"),
    (dict(max_offset=-1), "max_offset"), (dict(theta_base=1.0), "theta_base"), (dict(frame_stride=1560 * 128 + 4), "multiples of 8"),
    (dict(frame_stride=64), "frame_stride"), (dict(slots=[0, 0], offsets=[0, 1]), "given twice"),
    (dict(slots=[64], offsets=[0]), "outside"), (dict(head_stride=1560 * 128), "head_stride"),
    (dict(slots=[], offsets=[]), "n_frames"),
])
def test_rope_argument_errors_are_synchronous(kw, msg):
    cfg = cfg_of(CONFIGS["realistic"])
    a = dict(src=FAKE, dst=FAKE, head_stride=9 * 1560 * 128, frame_stride=1560 * 128, slots=[0, 1, 2],
             offsets=[6, 7, 8], max_offset=8, rot_dims=128, theta_base=10000.0)
    a.update(kw)
    with pytest.raises(hb.HFError) as ei:
        hb.hf_rope_relative(cfg, a["src"], a["dst"], a["head_stride"], a["frame_stride"], a["slots"], a["offsets"],
                            a["max_offset"], a["rot_dims"], a["theta_base"], stream=0)
    assert ei.value.code == 1
    assert msg in str(ei.value)


@pytest.mark.parametrize("kw,msg", [
    (dict(Kc=0), "Kc is NULL"), (dict(ws=FAKE + 8), "ws is not 16-byte aligned"),
    (dict(slots=[0, 0]), "given twice"), (dict(slots=[9]), "outside"), (dict(slots=[-1]), "outside"),
    (dict(slot_stride=100), "slot_stride"), (dict(slots=list(range(10))), "n_slots"),
])
def test_pool_keys_argument_errors_are_synchronous(kw, msg):
    cfg = cfg_of(CONFIGS["realistic"])
    a = dict(Kc=FAKE, slot_stride=cfg.tokens_per_frame, slots=[0, 1, 2], ws=FAKE)
    a.update(kw)
    with pytest.raises(hb.HFError) as ei:
        hb.hf_pool_keys(cfg, a["Kc"], a["slot_stride"], a["slots"], a["ws"], stream=0)
    assert ei.value.code == 1
    assert msg in str(ei.value)


def test_pool_keys_of_no_slot_is_a_no_op():
    cfg = cfg_of(CONFIGS["realistic"])
    hb.hf_pool_keys(cfg, FAKE, cfg.tokens_per_frame, [], FAKE, stream=0)

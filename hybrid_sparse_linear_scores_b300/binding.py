"""ctypes binding of libhf.so (include/hf.h), same names as the C entry points.

Argument marshalling only: tensors are passed as raw device pointers, every
step runs in the library's CUDA kernels.  There is no fallback: if libhf.so
is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libhf.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "hf.h")

HF_OK = 0
STATUS = {0: "HF_OK", 1: "HF_ERR_INVALID_ARG", 2: "HF_ERR_UNSUPPORTED", 3: "HF_ERR_CUDA",
          4: "HF_ERR_TIMEOUT", 5: "HF_ERR_DEVICE_CHECK"}


class HFError(RuntimeError):
    def __init__(self, code: int, func: str, detail: str):
        self.code = code
        super().__init__(f"{func}: {STATUS.get(code, code)}: {detail}")


class HFConfig(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("tokens_per_frame", ctypes.c_int32), ("window_frames", ctypes.c_int32),
                ("chunk_frames", ctypes.c_int32), ("block_size", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("lin_eps", ctypes.c_float)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} not found: build it with "
                               "`python -m hybrid_sparse_linear_scores_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        cfgp = ctypes.POINTER(HFConfig)
        sig = {
            "hf_abi_version": ([], _I),
            "hf_status_string": ([_I], ctypes.c_char_p),
            "hf_last_error": ([], ctypes.c_char_p),
            "hf_workspace_size": ([cfgp, ctypes.POINTER(ctypes.c_size_t)], _I),
            "hf_state_reset": ([cfgp, _P, _P, _P], _I),
            "hf_absorb_evicted": ([cfgp, _P, _P, _P, _P, _I, _P, _P], _I),
            "hf_absorb_evicted_strided": ([cfgp, _P, _P, _P, _P, _I, ctypes.c_int64, _P, _P, ctypes.c_uint32], _I),
            "hf_block_scores": ([cfgp, _P, _P, _I, _P, _I, _P, _P, _P], _I),
            "hf_topk_blocks": ([cfgp, _P, _I, _I, _P, _P], _I),
            "hf_sparse_swa_attn": ([cfgp, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P], _I),
            "hf_linear_read": ([cfgp, _P, _P, _P, _P, _I, _P], _I),
            "hf_hybrid_forward": ([cfgp, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _P, _P], _I),
            "hf_hybrid_forward_profiled": ([cfgp, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _P, _P,
                                            ctypes.POINTER(ctypes.c_void_p)], _I),
            "hf_hybrid_forward_noalloc": ([cfgp, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P,
                                           ctypes.POINTER(ctypes.c_void_p), _P], _I),
            "hf_hybrid_forward_ex": ([cfgp, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _P, _P, ctypes.c_uint32,
                                      ctypes.POINTER(ctypes.c_void_p), _P], _I),
            "hf_pool_keys": ([cfgp, _P, _I, _P, _I, _P, _P], _I),
            "hf_ring_write": ([cfgp, _P, _P, _P, _P, _I, _P, _I, _P], _I),
            "hf_rope_relative": ([cfgp, _P, _P, ctypes.c_int64, ctypes.c_int64, _P, _P, _I, _I, _I,
                                  ctypes.c_float, _P], _I),
            "hf_get_device_status": ([_P, _P, ctypes.POINTER(_I)], _I),
            "hf_selftest_wait_timeout": ([_P, _I, _P], _I),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/hf.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^HF_API\s+(?:const\s+)?[a-z_0-9]+\s*\*?\s*(hf_[a-z_0-9]+)\s*\(", text, re.M)))


def make_config(batch, heads, head_dim, tokens_per_frame, window_frames, chunk_frames, block_size, topk,
                softmax_scale=0.0, lin_eps=1e-6) -> HFConfig:
    return HFConfig(batch, heads, head_dim, tokens_per_frame, window_frames, chunk_frames, block_size, topk,
                    softmax_scale, lin_eps)


def _check(rc: int, name: str):
    if rc != HF_OK:
        raise HFError(rc, name, lib().hf_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _slots(slot_map):
    if slot_map is None:
        return None
    arr = (ctypes.c_int32 * len(slot_map))(*[int(s) for s in slot_map])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def hf_workspace_size(cfg: HFConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().hf_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "hf_workspace_size")
    return n.value


def hf_state_reset(cfg, S, z, stream=None):
    _check(lib().hf_state_reset(ctypes.byref(cfg), _ptr(S), _ptr(z), _stream(stream)), "hf_state_reset")


def hf_absorb_evicted(cfg, S, z, K_ev, V_ev, n_ev_tokens, ws, stream=None):
    _check(lib().hf_absorb_evicted(ctypes.byref(cfg), _ptr(S), _ptr(z), _ptr(K_ev), _ptr(V_ev), int(n_ev_tokens),
                                   _ptr(ws), _stream(stream)), "hf_absorb_evicted")


def hf_absorb_evicted_strided(cfg, S, z, K_ev, V_ev, n_ev_tokens, head_stride_tokens, ws, stream=None, flags=0):
    _check(lib().hf_absorb_evicted_strided(ctypes.byref(cfg), _ptr(S), _ptr(z), _ptr(K_ev), _ptr(V_ev),
                                           int(n_ev_tokens), int(head_stride_tokens), _ptr(ws), _stream(stream),
                                           ctypes.c_uint32(int(flags))),
           "hf_absorb_evicted_strided")


def hf_block_scores(cfg, Q, Kc, slot_stride, slot_map, n_win, scores, ws, stream=None):
    sm = _slots(slot_map)
    _check(lib().hf_block_scores(ctypes.byref(cfg), _ptr(Q), _ptr(Kc), int(slot_stride), sm and sm[0], int(n_win),
                                 _ptr(scores), _ptr(ws), _stream(stream)), "hf_block_scores")


def hf_topk_blocks(cfg, scores, nQB, nKB, idx, stream=None):
    _check(lib().hf_topk_blocks(ctypes.byref(cfg), _ptr(scores), int(nQB), int(nKB), _ptr(idx), _stream(stream)),
           "hf_topk_blocks")


def hf_sparse_swa_attn(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, idx, O_swa, ws, stream=None):
    sm = _slots(slot_map)
    _check(lib().hf_sparse_swa_attn(ctypes.byref(cfg), _ptr(Q), _ptr(Kc), _ptr(Vc), int(slot_stride), sm and sm[0],
                                    int(n_win), _ptr(idx), _ptr(O_swa), _ptr(ws), _stream(stream)),
           "hf_sparse_swa_attn")


def hf_linear_read(cfg, Q, S, z, O, accumulate=False, stream=None):
    _check(lib().hf_linear_read(ctypes.byref(cfg), _ptr(Q), _ptr(S), _ptr(z), _ptr(O), int(bool(accumulate)),
                                _stream(stream)), "hf_linear_read")


def hf_hybrid_forward(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, ws, stream=None):
    sm = _slots(slot_map)
    _check(lib().hf_hybrid_forward(ctypes.byref(cfg), _ptr(Q), _ptr(Kc), _ptr(Vc), int(slot_stride), sm and sm[0],
                                   int(n_win), _ptr(S), _ptr(z), _ptr(O), _ptr(idx_out), _ptr(ws), _stream(stream)),
           "hf_hybrid_forward")


def hf_hybrid_forward_profiled(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, ws, events,
                               stream=None):
    """events: HF_FWD_EVENTS (4) torch.cuda.Event objects (before the key
    pooling, before the prologue, before the attention kernel, after it).
    torch creates an event's CUDA handle on its first record and only
    reports times for events it has recorded, so each event is recorded by
    torch first; the library then records it again at its own point."""
    st = _stream(stream)
    import torch
    ts = torch.cuda.ExternalStream(st.value) if st.value else torch.cuda.current_stream()
    for e in events:
        if e is not None:
            e.record(ts)
    sm = _slots(slot_map)
    ev = (ctypes.c_void_p * HF_FWD_EVENTS)(*[ctypes.c_void_p(e.cuda_event) if e is not None else None for e in events])
    _check(lib().hf_hybrid_forward_profiled(ctypes.byref(cfg), _ptr(Q), _ptr(Kc), _ptr(Vc), int(slot_stride),
                                            sm and sm[0], int(n_win), _ptr(S), _ptr(z), _ptr(O), _ptr(idx_out),
                                            _ptr(ws), st, ev), "hf_hybrid_forward_profiled")


HF_FWD_CACHED_KEYS = 1
HF_FWD_STATE_PREPARED = 2
HF_FWD_AFTER_POOL_KEYS = 4
HF_ABSORB_SHARE_SMS = 1
HF_FWD_EVENTS = 4


def hf_pool_keys(cfg, Kc, slot_stride, slots, ws, stream=None):
    """Pool the key blocks of the given ring slots into the workspace's cache."""
    sl = _slots(list(slots))
    _check(lib().hf_pool_keys(ctypes.byref(cfg), _ptr(Kc), int(slot_stride), sl and sl[0], len(list(slots)),
                              _ptr(ws), _stream(stream)), "hf_pool_keys")


def hf_ring_write(cfg, K_src, V_src, Kc, Vc, slot_stride, slots, stream=None):
    """Copy a chunk's K, V ([BH, n, N_f, d], device or pinned host) into ring slots."""
    slots = list(slots)
    for t in (K_src, V_src):
        if hasattr(t, "is_contiguous") and not t.is_contiguous():
            raise ValueError("hf_ring_write: sources must be contiguous")
    sl = _slots(slots)
    _check(lib().hf_ring_write(ctypes.byref(cfg), _ptr(K_src), _ptr(V_src), _ptr(Kc), _ptr(Vc), int(slot_stride),
                               sl[0], len(slots), _stream(stream)), "hf_ring_write")


def hf_rope_relative(cfg, src, dst, head_stride, frame_stride, slots, offsets, max_offset, rot_dims,
                     theta_base=10000.0, stream=None):
    """Relative temporal RoPE of frames slots[f] (offset offsets[f], clamped to
    [0, max_offset]); strides in elements; dst may be src."""
    slots, offsets = list(slots), list(offsets)
    if len(slots) != len(offsets):
        raise ValueError("hf_rope_relative: one offset per frame")
    sl, of = _slots(slots), _slots(offsets)
    _check(lib().hf_rope_relative(ctypes.byref(cfg), _ptr(src), _ptr(dst), int(head_stride), int(frame_stride),
                                  sl and sl[0], of and of[0], len(slots), int(max_offset), int(rot_dims),
                                  float(theta_base), _stream(stream)), "hf_rope_relative")


def hf_hybrid_forward_ex(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, ws, flags=0, events=None,
                         stream=None, state_ready=None):
    """hf_hybrid_forward with flags (HF_FWD_CACHED_KEYS, HF_FWD_STATE_PREPARED),
    optional per-kernel events (HF_FWD_EVENTS torch.cuda.Event objects, handled
    as in hf_hybrid_forward_profiled) and an optional torch.cuda.Event, already
    recorded, that the attention kernel waits for (the state's producer)."""
    st = _stream(stream)
    ev = None
    if events is not None:
        import torch
        ts = torch.cuda.ExternalStream(st.value) if st.value else torch.cuda.current_stream()
        for e in events:
            if e is not None and not e.cuda_event:   # torch creates the CUDA event on its first record
                e.record(ts)
        ev = (ctypes.c_void_p * HF_FWD_EVENTS)(*[ctypes.c_void_p(e.cuda_event) if e is not None else None for e in events])
    sm = _slots(slot_map)
    ready = ctypes.c_void_p(state_ready.cuda_event) if state_ready is not None else None
    _check(lib().hf_hybrid_forward_ex(ctypes.byref(cfg), _ptr(Q), _ptr(Kc), _ptr(Vc), int(slot_stride), sm and sm[0],
                                      int(n_win), _ptr(S), _ptr(z), _ptr(O), _ptr(idx_out), _ptr(ws), st,
                                      ctypes.c_uint32(int(flags)), ev, ready), "hf_hybrid_forward_ex")


def hf_hybrid_forward_noalloc(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, stream=None):
    """hf_hybrid_forward without a workspace argument (the library's static
    device scratch stands in for it).  Returns the device address of the
    scratch's status word, to pass as ``ws`` to :func:`hf_get_device_status`."""
    sm = _slots(slot_map)
    status_word = ctypes.c_void_p(0)
    _check(lib().hf_hybrid_forward_noalloc(ctypes.byref(cfg), _ptr(Q), _ptr(Kc), _ptr(Vc), int(slot_stride),
                                           sm and sm[0], int(n_win), _ptr(S), _ptr(z), _ptr(O), _ptr(idx_out),
                                           ctypes.byref(status_word), _stream(stream)),
           "hf_hybrid_forward_noalloc")
    return status_word.value


def hf_get_device_status(ws, stream=None) -> tuple[int, int]:
    """(status code, site) of the first device-side error since the last call."""
    site = ctypes.c_int32(0)
    rc = lib().hf_get_device_status(_ptr(ws), _stream(stream), ctypes.byref(site))
    return rc, site.value


def hf_selftest_wait_timeout(ws, limit_us, stream=None):
    _check(lib().hf_selftest_wait_timeout(_ptr(ws), int(limit_us), _stream(stream)), "hf_selftest_wait_timeout")

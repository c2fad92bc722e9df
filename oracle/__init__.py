"""CPU oracle for the hybrid attention step (fp64; float32 only where the
block selection is defined in float32).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (``hybrid_sparse_linear_scores_b300``) and never imports it;
the two see the same seeded input bytes and nothing else.

The arithmetic lives in ``hf_oracle.c`` (see its header for the step-by-step
definition and the passages each step follows); this module only marshals
numpy/torch arrays into it.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        lib.hfo_pool.argtypes = [_P, _I, _I, _I, _I, _P]
        lib.hfo_scores.argtypes = [_P, _I, _P, _I, _I, _P]
        lib.hfo_topk.argtypes = [_P, _I, _I, _I, _P]
        lib.hfo_topk.restype = _I
        lib.hfo_score_margin.argtypes = [_P, _I, _P, _I, _I, _I, _P]
        lib.hfo_absorb.argtypes = [_P, _P, _P, _P, _I, _I]
        lib.hfo_absorb_heads.argtypes = [_I, _P, _P, _P, _P, _I, _I]
        lib.hfo_linear_read.argtypes = [_P, _I, _P, _P, _I, _D, _P]
        lib.hfo_sparse_attn.argtypes = [_P, _P, _P, _I, _I, _I, _I, _P, _I, _D, _P, _I, _P]
        lib.hfo_hybrid_forward.argtypes = [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _D, _D,
                                           _P, _I, _P, _P, _P, _P, _P]
        lib.hfo_hybrid_forward.restype = _I
        lib.hfo_max_threads.restype = _I
        lib.hfo_rope_relative.argtypes = [_P, _I, _I, _I, _I, _P, _I, _I, _D, _P]
        _lib = lib
    return _lib


def _bf16_bits(x) -> np.ndarray:
    """bf16 torch tensor (or uint16 ndarray) -> contiguous uint16 ndarray."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    """OpenMP threads the oracle runs on."""
    return _load().hfo_max_threads()


def pool(x, beta: int) -> np.ndarray:
    """Mean-pooled blocks (float32).  x: bf16 [n_frames, N_f, d] of one head."""
    xb = _bf16_bits(x)
    nfr, nf, d = xb.shape
    bpf = -(-nf // beta)
    out = np.empty((nfr * bpf, d), np.float32)
    _load().hfo_pool(_ptr(xb), nfr, nf, d, beta, _ptr(out))
    return out


def scores(qp: np.ndarray, kp: np.ndarray) -> np.ndarray:
    qp = np.ascontiguousarray(qp, np.float32)
    kp = np.ascontiguousarray(kp, np.float32)
    s = np.empty((qp.shape[0], kp.shape[0]), np.float32)
    _load().hfo_scores(_ptr(qp), qp.shape[0], _ptr(kp), kp.shape[0], qp.shape[1], _ptr(s))
    return s


def topk(s: np.ndarray, k: int) -> np.ndarray:
    s = np.ascontiguousarray(s, np.float32)
    idx = np.empty((s.shape[0], k), np.int32)
    rc = _load().hfo_topk(_ptr(s), s.shape[0], s.shape[1], k, _ptr(idx))
    if rc != 0:
        raise ValueError("oracle top-K: k out of range or non-finite score")
    return idx


def score_margin(qp: np.ndarray, kp: np.ndarray, k: int) -> np.ndarray:
    qp = np.ascontiguousarray(qp, np.float32)
    kp = np.ascontiguousarray(kp, np.float32)
    m = np.empty(qp.shape[0], np.float64)
    _load().hfo_score_margin(_ptr(qp), qp.shape[0], _ptr(kp), kp.shape[0], qp.shape[1], k, _ptr(m))
    return m


def absorb(S: np.ndarray, z: np.ndarray, k, v) -> None:
    """In place: S [d,d] += sum phi(k) v^T, z [d] += sum phi(k).  k, v: bf16 [n, d]."""
    kb, vb = _bf16_bits(k), _bf16_bits(v)
    assert S.dtype == np.float64 and S.flags.c_contiguous and z.dtype == np.float64
    n, d = kb.shape
    _load().hfo_absorb(_ptr(S), _ptr(z), _ptr(kb), _ptr(vb), n, d)


def linear_read(q, S: np.ndarray, z: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    qb = _bf16_bits(q)
    nq, d = qb.shape
    S = np.ascontiguousarray(S, np.float64)
    z = np.ascontiguousarray(z, np.float64)
    o = np.empty((nq, d), np.float64)
    _load().hfo_linear_read(_ptr(qb), nq, _ptr(S), _ptr(z), d, eps, _ptr(o))
    return o


def sparse_attn(q, k, v, C: int, nf: int, beta: int, idx: np.ndarray, scale: float = 0.0,
                rows=None) -> np.ndarray:
    """One head.  q bf16 [C*N_f, d]; k, v bf16 [n_win*N_f, d] logical order;
    idx int32 [C*bpf, K].  Returns float64 [len(rows) or C*N_f, d]."""
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    d = qb.shape[-1]
    idx = np.ascontiguousarray(idx, np.int32)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    n = C * nf if r is None else len(r)
    o = np.empty((n, d), np.float64)
    _load().hfo_sparse_attn(_ptr(qb), _ptr(kb), _ptr(vb), C, nf, d, beta, _ptr(idx), idx.shape[1],
                            scale, None if r is None else _ptr(r), 0 if r is None else len(r), _ptr(o))
    return o


def hybrid_forward(Q, K, V, S, z, *, C: int, n_win: int, nf: int, beta: int, k: int,
                   scale: float = 0.0, eps: float = 1e-6, rows=None, split: bool = False,
                   margin: bool = False):
    """The whole step for all heads.

    Q bf16 [BH, C*N_f, d]; K, V bf16 [BH, n_win*N_f, d] (logical window order,
    oldest frame first); S float64 [BH, d, d] and z [BH, d], or None for the
    empty state.  Returns dict(idx=int32 [BH, nQB, K], O=float64 [BH, R, d],
    and O_swa/O_lin if split, margin if margin)."""
    Qb, Kb, Vb = _bf16_bits(Q), _bf16_bits(K), _bf16_bits(V)
    BH, nq, d = Qb.shape
    assert nq == C * nf and Kb.shape == (BH, n_win * nf, d) and Vb.shape == Kb.shape
    bpf = -(-nf // beta)
    if S is not None:
        S = np.ascontiguousarray(S, np.float64)
        z = np.ascontiguousarray(z, np.float64)
        assert S.shape == (BH, d, d) and z.shape == (BH, d)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    R = nq if r is None else len(r)
    idx = np.empty((BH, C * bpf, k), np.int32)
    O = np.empty((BH, R, d), np.float64)
    Os = np.empty_like(O) if split else None
    Ol = np.empty_like(O) if split else None
    mg = np.empty((BH, C * bpf), np.float64) if margin else None
    rc = _load().hfo_hybrid_forward(
        BH, _ptr(Qb), _ptr(Kb), _ptr(Vb), None if S is None else _ptr(S),
        None if S is None else _ptr(z), C, n_win, nf, d, beta, k, scale, eps,
        None if r is None else _ptr(r), 0 if r is None else R, _ptr(idx), _ptr(O),
        None if Os is None else _ptr(Os), None if Ol is None else _ptr(Ol),
        None if mg is None else _ptr(mg))
    if rc != 0:
        raise ValueError("oracle hybrid_forward: bad argument or non-finite score")
    out = {"idx": idx, "O": O}
    if split:
        out["O_swa"], out["O_lin"] = Os, Ol
    if margin:
        out["margin"] = mg
    return out


def rope_relative(x, offsets, max_offset: int, rot_dims: int, base: float = 10000.0) -> np.ndarray:
    """Relative temporal RoPE (step 8 of hf_oracle.c).  x: bf16 [BH, F, N_f, d];
    offsets: frame offsets inside the window (length F).  Returns fp64."""
    xb = _bf16_bits(x)
    BH, F, nf, d = xb.shape
    off = np.ascontiguousarray(offsets, np.int32)
    assert off.shape == (F,)
    y = np.empty((BH, F, nf, d), np.float64)
    _load().hfo_rope_relative(_ptr(xb), BH, F, nf, d, _ptr(off), int(max_offset), int(rot_dims), float(base), _ptr(y))
    return y


def state_from_frames(Kev, Vev, S=None, z=None) -> tuple[np.ndarray, np.ndarray]:
    """S, z (float64) of all heads after absorbing tokens Kev, Vev bf16
    [BH, n, d], starting from (S, z) or from the empty state."""
    Kb, Vb = _bf16_bits(Kev), _bf16_bits(Vev)
    BH, n, d = Kb.shape
    S = np.zeros((BH, d, d), np.float64) if S is None else np.array(S, np.float64, order="C")
    z = np.zeros((BH, d), np.float64) if z is None else np.array(z, np.float64, order="C")
    _load().hfo_absorb_heads(BH, _ptr(S), _ptr(z), _ptr(Kb), _ptr(Vb), n, d)
    return S, z

"""Seeded synthetic inputs for the hybrid attention step.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests.  It holds none of the method's arithmetic: it only turns
(seed, stream, frame, head, token, channel) into bf16 values with the
distributions the workloads call for.

Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11), written here from its published
definition, evaluated with int64 torch ops so that it runs identically on
the CPU and on a GPU.  Every 32-bit product is split into 16-bit halves so
no intermediate exceeds 2^49 (no reliance on signed-overflow wrap-around).
Two uniforms -> Box-Muller (float64) -> float32 -> bf16 (round to nearest
even).  One Philox call yields four normals, used for channels 4i..4i+3.

Because every value is a pure function of its coordinates, any frame can be
generated on its own; a frame that is in the window at one step and evicted
at a later one has the same bytes both times.
"""

from __future__ import annotations

import math

import torch

_M32 = 0xFFFFFFFF
_M16 = 0xFFFF
# Philox4x32 round multipliers and Weyl key increments (published constants).
_PHILOX_M0 = 0xD2511F53
_PHILOX_M1 = 0xCD9E8D57
_PHILOX_W0 = 0x9E3779B9
_PHILOX_W1 = 0xBB67AE85

# Stream identifiers (second key word); one per independent random field.
STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
STREAM_MEAN = {STREAM_Q: 11, STREAM_K: 12, STREAM_V: 13}
STREAM_DRIFT = {STREAM_Q: 21, STREAM_K: 22, STREAM_V: 23}
STREAM_CENTRES = 31
STREAM_CLUSTER_ID = 32


def _mulhilo(a: torch.Tensor, m: int):
    """(hi, lo) 32-bit halves of a * m for 0 <= a, m < 2^32, without overflow."""
    m_lo = m & _M16
    m_hi = m >> 16
    t_lo = a * m_lo                      # < 2^48
    t_hi = a * m_hi                      # < 2^48
    mid = t_lo + ((t_hi & _M16) << 16)   # < 2^49
    lo = mid & _M32
    hi = (t_hi >> 16) + (mid >> 32)
    return hi & _M32, lo


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds.  Counters are int64 tensors holding uint32."""
    k0 &= _M32
    k1 &= _M32
    for _ in range(10):
        hi0, lo0 = _mulhilo(c0, _PHILOX_M0)
        hi1, lo1 = _mulhilo(c2, _PHILOX_M1)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
        k0 = (k0 + _PHILOX_W0) & _M32
        k1 = (k1 + _PHILOX_W1) & _M32
    return c0, c1, c2, c3


def _box_muller(x0, x1):
    u1 = (x0.to(torch.float64) + 1.0) * (1.0 / 4294967296.0)   # (0, 1]
    u2 = x1.to(torch.float64) * (1.0 / 4294967296.0)           # [0, 1)
    r = torch.sqrt(-2.0 * torch.log(u1))
    t = (2.0 * math.pi) * u2
    return r * torch.cos(t), r * torch.sin(t)


def normal_field(seed: int, stream: int, frames, heads, n_tokens: int, d: int,
                 device="cpu", token_offset: int = 0) -> torch.Tensor:
    """Standard normals, float64, shape [len(heads), len(frames), n_tokens, d].

    Counter = (channel // 4, token, frame, head); key = (seed, stream).
    ``frames`` and ``heads`` are absolute indices (sequences of ints).
    """
    assert d % 4 == 0
    f = torch.as_tensor(list(frames), dtype=torch.int64, device=device)
    h = torch.as_tensor(list(heads), dtype=torch.int64, device=device)
    t = torch.arange(token_offset, token_offset + n_tokens, dtype=torch.int64, device=device)
    c = torch.arange(d // 4, dtype=torch.int64, device=device)
    shape = (h.numel(), f.numel(), n_tokens, d // 4)
    c0 = c.view(1, 1, 1, -1).expand(shape)
    c1 = t.view(1, 1, -1, 1).expand(shape)
    c2 = f.view(1, -1, 1, 1).expand(shape)
    c3 = h.view(-1, 1, 1, 1).expand(shape)
    x0, x1, x2, x3 = philox4x32_10(c0, c1, c2, c3, seed, stream)
    n0, n1 = _box_muller(x0, x1)
    n2, n3 = _box_muller(x2, x3)
    out = torch.stack((n0, n1, n2, n3), dim=-1)           # [..., d/4, 4]
    return out.reshape(h.numel(), f.numel(), n_tokens, d)


def uniform_u32(seed: int, stream: int, frames, heads, n_tokens: int,
                device="cpu") -> torch.Tensor:
    """One uint32 (in int64) per (head, frame, token): first Philox output word."""
    f = torch.as_tensor(list(frames), dtype=torch.int64, device=device)
    h = torch.as_tensor(list(heads), dtype=torch.int64, device=device)
    t = torch.arange(n_tokens, dtype=torch.int64, device=device)
    shape = (h.numel(), f.numel(), n_tokens)
    c0 = torch.zeros(shape, dtype=torch.int64, device=device)
    c1 = t.view(1, 1, -1).expand(shape)
    c2 = f.view(1, -1, 1).expand(shape)
    c3 = h.view(-1, 1, 1).expand(shape)
    x0, _, _, _ = philox4x32_10(c0, c1, c2, c3, seed, stream)
    return x0


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """float64 -> float32 -> bf16, each step round-to-nearest-even."""
    return x.to(torch.float32).to(torch.bfloat16)

"""Seeded, counter-based synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the method (no attention, no importance, no selection).  It only
turns (seed, stream, element index) into numbers, and it does so with integer operations plus one
float32 multiply and one round-to-nearest-even cast to bfloat16.  Every operation used is exact or
IEEE-rounded elementwise, so the same call gives bit-identical tensors on the CPU and on a CUDA device.
That lets a test regenerate any slice of a multi-GB device tensor on the host.

Generator (stated here because both sides depend on it):

* ``mix32`` is a 32-bit integer finaliser of the xorshift-multiply kind (shift 16, multiply by
  0x7feb352d, shift 15, multiply by 0x846ca68b, shift 16).  Multiplications are carried out modulo
  2**32 on int64 tensors by splitting the left operand into 16-bit halves, so no int64 product ever
  overflows.
* For element counter ``n`` of stream ``s`` under seed ``seed``: two keyed rounds over the low and
  high 32 bits of ``n`` give a word ``a``, and one more keyed round gives ``b``.  The four 16-bit
  halves of ``a`` and ``b`` are uniform integers u1..u4 in [0, 65536).
* An approximately standard normal value is the centred Irwin-Hall sum of four uniforms:
  ``z = (u1 + u2 + u3 + u4 - 131070) * (sqrt(3) / 65536)``.  The integer sum is exact, its
  conversion to float32 is exact (|sum| < 2**24), the multiply is one float32 rounding, and the
  cast to bfloat16 is round-to-nearest-even.  The distribution has mean 0, variance 1 and support
  [-2*sqrt(3), 2*sqrt(3)]: a bounded stand-in for N(0, 1).
"""
from __future__ import annotations

import math

import torch

M32 = 0xFFFFFFFF
_C1 = 0x7FEB352D
_C2 = 0x846CA68B
_NORMAL_CENTER = 2 * 65535
_NORMAL_SCALE = math.sqrt(3.0) / 65536.0
DEFAULT_CHUNK = 1 << 25


def _mulmod32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 x in [0, 2**32) and a constant c < 2**32, without int64 overflow."""
    lo = (x & 0xFFFF) * c                      # < 2**48
    hi = (((x >> 16) * c) & 0xFFFF) << 16      # < 2**32
    return (lo + hi) & M32


def _mix32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * _C1) & M32
    x ^= x >> 15
    x = (x * _C2) & M32
    x ^= x >> 16
    return x


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mulmod32(x, _C1)
    x = x ^ (x >> 15)
    x = _mulmod32(x, _C2)
    return x ^ (x >> 16)


def stream_id(*parts: int) -> int:
    """Fold a tuple of small non-negative integers (tensor kind, layer, ...) into one 32-bit stream id."""
    h = 0x2545F491
    for p in parts:
        h = _mix32_int(h ^ _mix32_int(int(p) + 0x9E3779B9))
    return h


def _keys(seed: int, stream: int):
    k0 = _mix32_int(int(seed) ^ 0x5BD1E995)
    k1 = _mix32_int(k0 ^ int(stream))
    k2 = _mix32_int(k1 + 0x27D4EB2F)
    k3 = _mix32_int(k2 ^ 0x165667B1)
    return k1, k2, k3


def hash_words(seed: int, stream: int, counters: torch.Tensor):
    """Two independent 32-bit words (int64 tensors in [0, 2**32)) for each int64 counter."""
    k1, k2, k3 = _keys(seed, stream)
    lo = counters & M32
    hi = counters >> 32
    a = _mix32(lo ^ k1)
    a = _mix32((a + hi + k2) & M32)
    b = _mix32(a ^ k3)
    return a, b


def uint32_at(seed: int, stream: int, counters: torch.Tensor) -> torch.Tensor:
    """Uniform 32-bit integers (as int64) for the given counters."""
    a, _ = hash_words(seed, stream, counters)
    return a


def _normal_f32_at(seed: int, stream: int, counters: torch.Tensor) -> torch.Tensor:
    a, b = hash_words(seed, stream, counters)
    s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16) - _NORMAL_CENTER
    scale = torch.tensor(_NORMAL_SCALE, dtype=torch.float32, device=counters.device)
    return s.to(torch.float32) * scale


def normal_f32_at(seed: int, stream: int, counters: torch.Tensor) -> torch.Tensor:
    """Float32 Irwin-Hall normals (before the bfloat16 cast) for the given int64 counters."""
    return _normal_f32_at(seed, stream, counters)


def normal_bf16_at(seed: int, stream: int, counters: torch.Tensor) -> torch.Tensor:
    """Bfloat16 normals for the given int64 counters (same device as ``counters``)."""
    return _normal_f32_at(seed, stream, counters).to(torch.bfloat16)


def normal_bf16(seed: int, stream: int, shape, device="cpu", offset: int = 0, out: torch.Tensor | None = None,
                chunk: int = DEFAULT_CHUNK) -> torch.Tensor:
    """A bfloat16 tensor of ``shape`` whose element with row-major linear index i uses counter offset + i.

    Generated in chunks so that multi-GB device tensors need only bounded temporaries.
    """
    shape = tuple(int(s) for s in shape)
    numel = 1
    for s in shape:
        numel *= s
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    dev = flat.device
    for start in range(0, numel, chunk):
        stop = min(numel, start + chunk)
        ctr = torch.arange(offset + start, offset + stop, dtype=torch.int64, device=dev)
        flat[start:stop] = normal_bf16_at(seed, stream, ctr)
    return out


def normal_bf16_rows(seed: int, stream: int, full_shape, index_prefix, device="cpu") -> torch.Tensor:
    """Regenerate the sub-tensor ``full[index_prefix]`` (a tuple of leading integer indices) of a tensor
    that ``normal_bf16(seed, stream, full_shape)`` would produce, without building the full tensor."""
    full_shape = tuple(int(s) for s in full_shape)
    strides = [1] * len(full_shape)
    for i in range(len(full_shape) - 2, -1, -1):
        strides[i] = strides[i + 1] * full_shape[i + 1]
    base = 0
    for i, ix in enumerate(index_prefix):
        base += int(ix) * strides[i]
    sub_shape = full_shape[len(index_prefix):]
    n = 1
    for s in sub_shape:
        n *= s
    ctr = torch.arange(base, base + n, dtype=torch.int64, device=device)
    return normal_bf16_at(seed, stream, ctr).view(sub_shape)


def distinct_positions(seed: int, stream: int, n_pos: int, count: int) -> torch.Tensor:
    """``count`` distinct positions in [0, n_pos): the first ``count`` entries of the permutation that
    sorts ``uint32_at(seed, stream, 0..n_pos-1)`` (stable, so equal hashes keep index order)."""
    h = uint32_at(seed, stream, torch.arange(n_pos, dtype=torch.int64))
    order = torch.sort(h, stable=True).indices
    return order[:count].clone()


__all__ = [
    "stream_id", "hash_words", "uint32_at", "normal_f32_at", "normal_bf16_at", "normal_bf16",
    "normal_bf16_rows", "distinct_positions",
]

"""Counter-based seeded random numbers for synthetic inputs.

Every value is a pure function of (seed, stream, index): the 64-bit key
``seed << 56 | stream << 40 | index`` is advanced by the SplitMix64 increment
and passed through the SplitMix64 output mix (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014).  All steps are
integer operations (wrapping 64-bit multiply, xor, logical shift), so the
same call gives bit-identical results on a CPU tensor and on a CUDA tensor.
That is what lets a test regenerate, on the host, exactly the slice of a
weight tensor that a sampled token touches on the GPU.

Two kinds of normal deviates:
  * ``normal``: standardised Irwin-Hall(4) sums of the four 16-bit fields of one
    hash: mean 0, variance 1 (to 1 part in 2^32), support (-2√3, 2√3).  Only
    exact operations (integer sum, power-of-two scaling) and one correctly
    rounded multiply are used, so they are bit-identical across devices; the
    weights are drawn this way, on the device.
  * ``gaussian``: Box-Muller (Box & Muller, "A note on the generation of random
    normal deviates", Ann. Math. Statist. 1958) on the two 32-bit halves of one
    hash, in fp64 on the host: a true N(0,1) with tails to about 6.8 sigma.  Its
    log/cos/sqrt are the host's, so it is always computed on the CPU and copied
    to where it is needed; x and the RMSNorm gammas are drawn this way.
This module holds no arithmetic of the latent-MoE block.
"""
from __future__ import annotations

import math

import torch

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _s64(u: int) -> int:
    """Two's-complement view of a 64-bit unsigned constant as a signed int64."""
    u &= (1 << 64) - 1
    return u - (1 << 64) if u >= (1 << 63) else u


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns (torch's >> is arithmetic)."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def mix64(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output function on int64 bit patterns (wrapping arithmetic)."""
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


def mix64_int(z: int) -> int:
    """Pure-Python SplitMix64 output function, for cross-checking the tensor path."""
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * _M1) & m
    z = ((z ^ (z >> 27)) * _M2) & m
    return z ^ (z >> 31)


def hash64(seed: int, stream: int, index: torch.Tensor) -> torch.Tensor:
    """Hash of (seed, stream, index) as int64 bit patterns; index < 2^40."""
    assert 0 <= seed < 256 and 0 <= stream < 65536
    key = _s64((seed << 56) | (stream << 40))
    return mix64((index.to(torch.int64) | key) + _s64(_GOLDEN))


def hash64_int(seed: int, stream: int, index: int) -> int:
    return mix64_int(((seed << 56) | (stream << 40) | index) + _GOLDEN)


def _irwin_hall4(h: torch.Tensor) -> torch.Tensor:
    """Standardised sum of the four 16-bit fields of h, exact in fp64 up to the last multiply."""
    s = (h & 0xFFFF) + (_lsr(h, 16) & 0xFFFF) + (_lsr(h, 32) & 0xFFFF) + _lsr(h, 48)
    u = (s.to(torch.float64) + 2.0) / 65536.0 - 2.0  # exact: in (-2, 2), variance 1/3
    return u


def _chunk(device) -> int:
    # host: cache-sized pieces (the int64 temporaries then stay in cache); device: large
    return 1 << 18 if torch.device(device).type == "cpu" else 1 << 26


def normal(seed: int, stream: int, start: int, count: int, std: float,
           device="cpu") -> torch.Tensor:
    """fp64 deviates with mean 0 and standard deviation ``std`` for indices [start, start+count)."""
    out = torch.empty(count, dtype=torch.float64, device=device)
    c = _chunk(device)
    for s0 in range(0, count, c):
        n = min(c, count - s0)
        idx = torch.arange(start + s0, start + s0 + n, dtype=torch.int64, device=device)
        u = _irwin_hall4(hash64(seed, stream, idx))
        out[s0:s0 + n] = u * (math.sqrt(3.0) * std)  # one correctly rounded multiply
    return out


def gaussian(seed: int, stream: int, start: int, count: int, std: float) -> torch.Tensor:
    """fp64 N(0, std^2) deviates (host) for indices [start, start+count): Box-Muller on the hash,
    u1 = (hi32 + 0.5) / 2^32 and u2 = (lo32 + 0.5) / 2^32, z = sqrt(-2 ln u1) cos(2 pi u2)."""
    out = torch.empty(count, dtype=torch.float64)
    c = _chunk("cpu")
    for s0 in range(0, count, c):
        n = min(c, count - s0)
        idx = torch.arange(start + s0, start + s0 + n, dtype=torch.int64)
        h = hash64(seed, stream, idx)
        u1 = (_lsr(h, 32).to(torch.float64) + 0.5) * (1.0 / 4294967296.0)
        u2 = ((h & 0xFFFFFFFF).to(torch.float64) + 0.5) * (1.0 / 4294967296.0)
        out[s0:s0 + n] = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2) * std
    return out


def uniform_bits(seed: int, stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Raw int64 hash values for indices [start, start+count)."""
    out = torch.empty(count, dtype=torch.int64, device=device)
    c = _chunk(device)
    for s0 in range(0, count, c):
        n = min(c, count - s0)
        idx = torch.arange(start + s0, start + s0 + n, dtype=torch.int64, device=device)
        out[s0:s0 + n] = hash64(seed, stream, idx)
    return out


def permutation(seed: int, stream: int, n: int) -> torch.Tensor:
    """A seeded permutation of range(n): indices sorted by their hash (stable)."""
    h = uniform_bits(seed, stream, 0, n)
    # Sort on the top 62 bits as a non-negative key so the order is the unsigned order.
    key = _lsr(h, 2)
    return torch.sort(key, stable=True).indices

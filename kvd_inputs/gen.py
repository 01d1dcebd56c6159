"""Counter-based random numbers for synthetic decode-attention inputs.

Every value is a pure function of (seed, stream tags, element index).  The
hash is the splitmix64 finaliser evaluated with wrapping 64-bit integer
arithmetic, and a normal variate is an exact lookup into a fixed
inverse-CDF table, so the same call gives bit-identical tensors on the CPU
and on a CUDA device.  That lets a host-side checker regenerate any slice of
a multi-GiB device workload without copying it back.

This module holds no attention arithmetic: only random numbers.
"""

from __future__ import annotations

import statistics

import torch

_MASK64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _s64(x: int) -> int:
    """Python int -> the signed 64-bit integer with the same bit pattern."""
    x &= _MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def mix64(x: int) -> int:
    """splitmix64 finaliser on a Python int (unsigned 64-bit result)."""
    z = (x + _GOLDEN) & _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, *tags) -> int:
    """Fold a seed and a tuple of int/str tags into one 64-bit stream key."""
    k = mix64(int(seed) & _MASK64)
    for t in tags:
        if isinstance(t, str):
            v = 0
            for ch in t.encode():
                v = (v * 131 + ch) & _MASK64
        else:
            v = int(t) & _MASK64
        k = mix64(k ^ v)
    return k


def _lshr(z: torch.Tensor, s: int) -> torch.Tensor:
    return torch.bitwise_right_shift(z, s) & ((1 << (64 - s)) - 1)


def hash_index(key: int, idx: torch.Tensor) -> torch.Tensor:
    """splitmix64(key + idx) elementwise on an int64 tensor (wrapping)."""
    z = idx + _s64(key + _GOLDEN)
    z = torch.bitwise_xor(z, _lshr(z, 30)) * _s64(_M1)
    z = torch.bitwise_xor(z, _lshr(z, 27)) * _s64(_M2)
    return torch.bitwise_xor(z, _lshr(z, 31))


_TABLE_BITS = 16
_tables: dict = {}


def _normal_table(device) -> torch.Tensor:
    dev = torch.device(device)
    t = _tables.get(dev)
    if t is None:
        n = 1 << _TABLE_BITS
        nd = statistics.NormalDist()
        vals = [nd.inv_cdf((i + 0.5) / n) for i in range(n)]
        t = torch.tensor(vals, dtype=torch.float64).to(torch.float32).to(dev)
        _tables[dev] = t
    return t


def index_range(start: int, count: int, device) -> torch.Tensor:
    return torch.arange(start, start + count, dtype=torch.int64, device=device)


def normal(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Standard-normal float32 variates (65,536-level inverse-CDF quantiles)."""
    h = hash_index(key, idx)
    return _normal_table(idx.device)[_lshr(h, 64 - _TABLE_BITS)]


def uniform(key: int, idx: torch.Tensor) -> torch.Tensor:
    """float32 uniform on [0, 1) with 24 random bits (exactly representable)."""
    h = hash_index(key, idx)
    return _lshr(h, 40).to(torch.float32) * (1.0 / (1 << 24))


def permutation(key: int, n: int, device="cpu") -> torch.Tensor:
    """A seeded permutation of range(n): argsort of hashed keys (ties by index)."""
    h = hash_index(key, index_range(0, n, device))
    # Sort on the CPU so CPU and CUDA callers get the same permutation.
    order = torch.sort(h.cpu(), stable=True).indices
    return order.to(device)


def choose(key: int, population: int, k: int) -> torch.Tensor:
    """k distinct values from range(population), uniformly, as a sorted int64 tensor."""
    if k > population:
        raise ValueError("k > population")
    return torch.sort(permutation(key, population)[:k]).values

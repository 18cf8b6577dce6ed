"""Seeded synthetic inputs for the dense GEMM workloads.

This module is shared by the CPU oracle checks and by the CUDA path (tests and
bench).  It draws numbers and rounds them to storage formats; it holds none of
the GEMM arithmetic.

Generator
---------
Counter-based SplitMix64 (Steele, Lea & Flood, "Fast Splittable Pseudorandom
Number Generators", OOPSLA 2014; the 64-bit finaliser constants are the ones
Vigna publishes with ``splitmix64.c``).  Value ``i`` of stream ``seed`` is

    state = (seed * 2**40 + i + 1) * GAMMA  (mod 2**64)
    out   = mix64(state)

which is exactly output number ``seed * 2**40 + i`` of the sequential
SplitMix64 generator started from state 0, so the published first outputs of
that generator (0xE220A8397B1DCDAF, ...) pin this implementation.

Distributions
-------------
* ``uniform``:  u = ((out >> 40) + 0.5) * 2**-24 in (0, 1), then lo + (hi-lo)*u.
  For (lo, hi) = (-1, 1) every value is an odd multiple of 2**-24, hence exact
  in fp32 (and in fp64).
* ``normal``:   Box-Muller in fp64 from two uniforms drawn at counters 2i and
  2i+1 of the stream.
* ``small_ints``: integers in [lo, hi] from the top bits (used by the
  bit-exactness tests: every partial sum stays an integer below 2**24).

Rounding to storage formats is round-to-nearest-even: fp64 -> fp32 (numpy),
fp32 -> bf16 (bit arithmetic below), fp64 -> fp16 (numpy).

Seeds per workload follow ``seed = 1000 * workload_id + role`` with roles
A=1, B=2, C=3, bias=4.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

ROLE_A, ROLE_B, ROLE_C, ROLE_BIAS = 1, 2, 3, 4


def seed_for(workload_id: int, role: int) -> int:
    """Seed of one operand of one workload: 1000 * workload + role."""
    return 1000 * int(workload_id) + int(role)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def raw64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n raw 64-bit outputs of stream ``seed`` starting at counter ``offset``."""
    if seed < 0 or seed >= (1 << 24):
        raise ValueError("seed must be in [0, 2**24)")
    if n < 0 or offset < 0 or offset + n > (1 << 40):
        raise ValueError("counter range out of [0, 2**40)")
    with np.errstate(over="ignore"):
        c = np.arange(n, dtype=np.uint64)
        c += np.uint64((int(seed) << 40) + int(offset) + 1)
        c *= GAMMA
        return _mix64(c)


def _u01(bits: np.ndarray) -> np.ndarray:
    return ((bits >> np.uint64(40)).astype(np.float64) + 0.5) * (2.0 ** -24)


def uniform(seed: int, shape, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """fp64 array of i.i.d. Uniform(lo, hi) values, C order over ``shape``."""
    n = int(np.prod(shape, dtype=np.int64))
    u = _u01(raw64(seed, n))
    return (lo + (hi - lo) * u).reshape(shape)


def normal(seed: int, shape) -> np.ndarray:
    """fp64 array of i.i.d. N(0, 1) values (Box-Muller), C order over ``shape``."""
    n = int(np.prod(shape, dtype=np.int64))
    bits = raw64(seed, 2 * n)
    u1 = _u01(bits[0::2])
    u2 = _u01(bits[1::2])
    r = np.sqrt(-2.0 * np.log(u1))
    return (r * np.cos(2.0 * np.pi * u2)).reshape(shape)


def small_ints(seed: int, shape, lo: int = -8, hi: int = 8) -> np.ndarray:
    """fp64 array of i.i.d. integers uniform on [lo, hi]."""
    n = int(np.prod(shape, dtype=np.int64))
    span = np.uint64(hi - lo + 1)
    v = (raw64(seed, n) >> np.uint64(11)) % span
    return (v.astype(np.float64) + lo).reshape(shape)


# ----------------------------------------------------------------------------
# storage formats (round to nearest even)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of fp32 values, round-to-nearest-even.

    NaN inputs are not expected from the generators and are rejected.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if np.isnan(x).any():
        raise ValueError("NaN in generator output")
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE) bit patterns."""
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32))


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp16 (RNE) bit patterns."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def to_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact), for building test inputs."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values to the storage dtype ('bf16' | 'f16' -> uint16 bits, 'f32')."""
    if dtype == "bf16":
        return to_bf16_bits(x)
    if dtype == "f16":
        return to_f16_bits(x)
    if dtype == "f32":
        return to_f32(x)
    raise ValueError(f"unknown dtype {dtype!r}")

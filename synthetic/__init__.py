"""Seeded synthetic inputs shared by the tests and the benchmark.

This module holds no arithmetic of the optimizer: it only draws the
parameters and gradients that both the CUDA library and the CPU oracle are
fed.  Values are a pure function of (seed, stream, step, index), so any
element can be drawn on its own, on the host (numpy, here) or on the device
(``synthetic/gen.cu``, the same definition), and the two agree bit for bit:

* counter hash: the SplitMix64 output function (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014), applied to
  ``key + (index + 1) * 0x9E3779B97F4A7C15``;
* approximately normal value: the sum of the four 16-bit lanes of one hash
  word minus its mean (an Irwin-Hall sum of four uniforms; exact small
  integer), times a float32 scale ``sigma / sqrt((2^32 - 1) / 3)`` rounded
  once; one correctly rounded float32 multiply, so numpy and CUDA agree;
* outliers: a second stream picks an element with probability ``frac``
  (top 32 bits of its hash below ``round(frac * 2^32)``) and multiplies it by
  ``mult`` (one float32 multiply).

The values are bounded at about +-3.46 sigma (four uniforms), which is the
stand-in used for the pages' "N(0, sigma)" draws.
"""
from __future__ import annotations

import math

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
IH_STD = math.sqrt(((1 << 32) - 1) / 3.0)  # std of the 4-lane sum

STREAM_W = 0        # initial weights
STREAM_G = 1        # gradient values
STREAM_OUTLIER = 2  # gradient outlier selection

CHUNK = 1 << 22


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2^64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int, step: int) -> int:
    """64-bit key of one (seed, stream, step) triple."""
    k = mix64_int(seed)
    k = mix64_int(k ^ (stream & MASK64))
    k = mix64_int(k ^ (step & MASK64))
    return k


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def hash_words(key: int, idx: np.ndarray) -> np.ndarray:
    """hash(key, i) for int64 indices idx, as uint64."""
    i = idx.astype(np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (i + np.uint64(1)) * np.uint64(GOLDEN)
    return _mix64(z)


def normal_scale(sigma: float) -> np.float32:
    return np.float32(sigma / IH_STD)


def outlier_threshold(frac: float) -> int:
    t = int(round(frac * 4294967296.0))
    return max(0, min(t, 0xFFFFFFFF))


def _values(key, scale, okey, othr, omul, idx):
    h = hash_words(key, idx)
    s = ((h & np.uint64(0xFFFF)) + ((h >> np.uint64(16)) & np.uint64(0xFFFF))
         + ((h >> np.uint64(32)) & np.uint64(0xFFFF)) + (h >> np.uint64(48)))
    x = (s.astype(np.int64) - 131070).astype(np.float32) * np.float32(scale)
    if othr:
        pick = (hash_words(okey, idx) >> np.uint64(32)) < np.uint64(othr)
        x = np.where(pick, x * np.float32(omul), x).astype(np.float32)
    return x.astype(np.float32, copy=False)


def draw(seed: int, stream: int, step: int, sigma: float, n: int = None,
         idx=None, outlier_frac: float = 0.0, outlier_mult: float = 1.0,
         out: np.ndarray = None) -> np.ndarray:
    """float32 values of one stream at indices ``idx`` (or 0..n-1)."""
    key = stream_key(seed, stream, step)
    okey = stream_key(seed, STREAM_OUTLIER, step)
    othr = outlier_threshold(outlier_frac)
    scale = normal_scale(sigma)
    if idx is not None:
        idx = np.asarray(idx, dtype=np.int64)
        return _values(key, scale, okey, othr, outlier_mult, idx)
    if out is None:
        out = np.empty(n, np.float32)
    for lo in range(0, n, CHUNK):
        hi = min(n, lo + CHUNK)
        out[lo:hi] = _values(key, scale, okey, othr, outlier_mult,
                             np.arange(lo, hi, dtype=np.int64))
    return out


def weights(seed: int, n: int = None, sigma: float = 0.02, idx=None):
    return draw(seed, STREAM_W, 0, sigma, n=n, idx=idx)


def grads(seed: int, step: int, sigma: float, n: int = None, idx=None,
          outlier_frac: float = 0.0, outlier_mult: float = 1.0):
    return draw(seed, STREAM_G, step, sigma, n=n, idx=idx,
                outlier_frac=outlier_frac, outlier_mult=outlier_mult)


def device_args(seed: int, stream: int, step: int, sigma: float,
                outlier_frac: float = 0.0, outlier_mult: float = 1.0):
    """Arguments of the device twin ``synth_fill`` for the same draw."""
    return dict(key=stream_key(seed, stream, step),
                scale=float(normal_scale(sigma)),
                okey=stream_key(seed, STREAM_OUTLIER, step),
                othr=outlier_threshold(outlier_frac),
                omul=float(np.float32(outlier_mult)))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns of float32 inputs (nearest, ties to even): how
    the 16-bit gradients of the mixed-precision tests are prepared."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns of float32 inputs (numpy's conversion)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)

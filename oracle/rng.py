"""Seeded random streams used to draw the method's random matrices (oracle side).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

The pages say only that the rotation and the projection are random and seeded
([BLOG] §1.2).  Two independent implementations (this oracle and the library's C++ host
code) must draw the same matrices, so both implement one published counter-based
generator from its definition:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014; the 64-bit finaliser constants as published by S. Vigna in splitmix64.c).
  Output i (i = 0, 1, ...) of the stream with seed s is mix(s + (i+1)*0x9E3779B97F4A7C15)
  where mix(z) = z ^= z>>30, z *= 0xBF58476D1CE4E5B9, z ^= z>>27, z *= 0x94D049BB133111EB,
  z ^= z>>31 (all mod 2^64).
* A uniform double u = (x >> 11) * 2^-53 in [0, 1).
* Box-Muller (1958) on consecutive pairs (u1, u2): with w = 1 - u1 in (0, 1],
  rad = sqrt(-2 ln w), theta = 2 pi u2, the pair yields rad*cos(theta) then rad*sin(theta).

Stream assignment (a reading; the pages fix none): the rotation's Gaussian matrix uses the
stream seeded with 2*seed, the QJL matrix S the stream seeded with 2*seed + 1 (mod 2^64).
"""
import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed, count, start=0):
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream seeded with ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed % (1 << 64)) + i * GOLDEN_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniforms(seed, count):
    """``count`` doubles in [0, 1) from the top 53 bits of each SplitMix64 output."""
    x = splitmix64(seed, count)
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def gaussians(seed, count):
    """``count`` standard normal doubles by Box-Muller on consecutive uniform pairs."""
    npairs = (count + 1) // 2
    u = uniforms(seed, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(1.0 - u1))
    theta = 2.0 * np.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = rad * np.cos(theta)
    out[1::2] = rad * np.sin(theta)
    return out[:count]


def rotation_stream_seed(seed):
    return (2 * int(seed)) % (1 << 64)


def projection_stream_seed(seed):
    return (2 * int(seed) + 1) % (1 << 64)

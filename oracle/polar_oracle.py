"""Float64 CPU oracle for the recursive polar-angle quantizer ("PolarQuant")
of "TurboQuant: 3-Bit Compression with Zero Overhead" (cneuralnets), Part 1
("The Mathematics of Recursive Polar Transformation" and "The Quantization
Step").

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the test-suite, the smoke check and the CPU-baseline leg of the
benchmark do.  It shares no code with the CUDA library; both sides receive
the same seeded inputs and nothing else.

The method, in the page's order, for a vector x of d = 2^k values:

1. Level 1 pairs coordinates (x_{2i}, x_{2i+1}) (0-based) into a radius
   sqrt(x_{2i}^2 + x_{2i+1}^2) and an angle atan2(x_{2i+1}, x_{2i}).  Each
   further level pairs the previous level's radii the same way, until one
   radius is left (the vector's L2 norm) beside d - 1 angles.
2. Every angle is rounded on one uniform grid of 2^b points spanning
   [-pi, pi]: index round((theta + pi) / (2 pi) * (2^b - 1)), value
   index / (2^b - 1) * 2 pi - pi.  No scale is stored.
3. Decoding walks the tree from the root down: a radius r with angle theta
   gives the two children r cos(theta) and r sin(theta).

Readings where the page is silent or loose (also listed in the design notes):
* The radius is stored as fp16 (round to nearest even), like every other
  norm of this codec; decoding uses the stored fp16 radius.
* All levels use the [-pi, pi] grid of the page's quantiser, although the
  page notes that angles above level 1 lie in [0, pi/2].
* Exact ties of the rounding go to the even index (round half to even).
* atan2 of a (0, 0) pair is 0 (IEEE: atan2(+0, +0) = +0).
* Storage: the d - 1 angle indices level by level (the d/2 of level 1 first,
  the root's last), then one 0 index, packed as d codes of b bits with the
  codec's own packed layout (``tq_oracle.pack_codes``); the radius is one
  fp16 per vector.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import tq_oracle as O


def levels(d: int) -> int:
    k = int(round(math.log2(d)))
    if 1 << k != d or d < 2:
        raise ValueError("d must be a power of two >= 2")
    return k


def polar_transform(x: np.ndarray):
    """x [N, d] -> (radius [N], angles [N, d-1]), angles level by level."""
    x = np.asarray(x, dtype=np.float64)
    N, d = x.shape
    levels(d)
    r = x
    angles = []
    while r.shape[1] > 1:
        a, b = r[:, 0::2], r[:, 1::2]
        angles.append(np.arctan2(b, a))
        r = np.sqrt(a * a + b * b)
    return r[:, 0], np.concatenate(angles, axis=1)


def angle_index(theta: np.ndarray, bits: int) -> np.ndarray:
    """Index of the grid point an angle rounds to (half to even)."""
    steps = (1 << bits) - 1
    return np.rint((np.asarray(theta, dtype=np.float64) + math.pi) / (2 * math.pi) * steps).astype(np.int64)


def angle_value(idx: np.ndarray, bits: int) -> np.ndarray:
    steps = (1 << bits) - 1
    return np.asarray(idx, dtype=np.float64) / steps * 2 * math.pi - math.pi


def tie_distance(theta: np.ndarray, bits: int) -> np.ndarray:
    """Distance of the scaled angle from the nearest rounding tie (in units
    of grid steps): where it is tiny, float32 and float64 may round apart."""
    steps = (1 << bits) - 1
    t = (np.asarray(theta, dtype=np.float64) + math.pi) / (2 * math.pi) * steps
    return np.abs(t - np.floor(t) - 0.5)


def polar_encode(x: np.ndarray, bits: int):
    """x [N, d] -> (indices [N, d-1] int64, radius [N] float16)."""
    r, th = polar_transform(x)
    return angle_index(th, bits), r.astype(np.float16)


def polar_inverse(radius: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """The tree from the root down: radius [N], angles [N, d-1] -> [N, d]."""
    radius = np.asarray(radius, dtype=np.float64)
    angles = np.asarray(angles, dtype=np.float64)
    N, dm1 = angles.shape
    d = dm1 + 1
    k = levels(d)
    offs = [0]
    for lv in range(1, k + 1):
        offs.append(offs[-1] + (d >> lv))
    r = radius.reshape(N, 1)
    for lv in range(k, 0, -1):
        th = angles[:, offs[lv - 1]:offs[lv]]        # level lv: d / 2^lv angles
        child = np.empty((N, 2 * r.shape[1]))
        child[:, 0::2] = r * np.cos(th)
        child[:, 1::2] = r * np.sin(th)
        r = child
    return r


def polar_decode(idx: np.ndarray, radius16: np.ndarray, bits: int) -> np.ndarray:
    return polar_inverse(np.asarray(radius16, dtype=np.float16).astype(np.float64), angle_value(idx, bits))


def pack_polar(idx: np.ndarray, bits: int) -> np.ndarray:
    """indices [N, d-1] -> uint8 [N, d*bits/8] (a trailing 0 index)."""
    idx = np.asarray(idx, dtype=np.int64)
    N = idx.shape[0]
    return O.pack_codes(np.concatenate([idx, np.zeros((N, 1), dtype=np.int64)], axis=1), bits)


def unpack_polar(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    return O.unpack_codes(packed, bits, d)[:, :d - 1]

"""Float64 CPU oracle for the TurboQuant / PolarQuant KV-cache codec and for
attention over the decoded cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the test-suite, the smoke check and the CPU-baseline leg of the
benchmark do.  It shares no code with the CUDA library (no kernels, headers,
tables or generators); both sides receive the same seeded inputs and nothing
else.

Everything is computed in numpy float64, step by step, in the order the
source pages describe the method:

* "TurboQuant From Scratch on Real KV Tensors" (sotaaz.com), section 2
  "The Algorithm in 60 Lines": norm split, rotation y = H.D.u, Lloyd-Max
  scalar quantisation for N(0, 1/d), un-rotation, optional QJL residual and
  optional norm correction; section 7 "Finding 4: Block-32": every 32-value
  block rotated and quantised on its own, with its own norm.
* "turboquant-pytorch" README, QJL estimator formula: the inner
  product estimator <q,k_mse> + ||r|| sqrt(pi/2)/m <Sq, sign(Sr)>.
* llama.cpp-turboquant "docs/turboquant.md", "How it works" (encode/decode
  pipeline) and "GGML Types" (14-byte turbo3 / 18-byte turbo4 blocks of 32
  values, i.e. the bytes per element the packed layout here keeps).

Readings where the pages are silent (each also listed in the design notes):
* Codebook target distribution: Gaussian N(0, 1/blk), blk = rotation block
  (codebook 0); codebook 1 is the exact Beta law of a rotated unit-vector
  coordinate (a listed variant of the llama.cpp page).
* Sign vector D: splitmix64 stream seeded with ``sign_seed``; D_i = -1 when
  the top bit of the i-th output is set.
* Bucketize ties go to the lower code (code = #{k : y > beta_k}).
* Codes are decided from the unrounded norm; the stored scale is the fp16
  (round-to-nearest-even) value; decoding uses the stored fp16 scale.
* Zero block: u = 0, every y = 0, scale 0; the decoded block is exactly 0;
  with QJL its residual is taken as 0 (rho = 0, every sign bit 1).
* QJL sign(0) is taken as +1 (stored bit 1).
* QJL scale constant sqrt(pi/2)/m with S entries N(0,1), m rows.
* Norm correction with QJL: the QJL term is added before renormalising.
* Packed bit layout: defined in ``pack_codes`` below (the pages fix only the
  bytes per element).
"""
from __future__ import annotations

import math
from statistics import NormalDist

import numpy as np

MASK64 = (1 << 64) - 1
QJL_CONST = math.sqrt(math.pi / 2.0)


# --------------------------------------------------------------------------
# S1  sign vector D
# --------------------------------------------------------------------------
def splitmix64_stream(seed: int, count: int) -> list[int]:
    """``count`` successive outputs of splitmix64 (Steele, Lea, Flood 2014,
    "Fast splittable pseudorandom number generators") started from state
    ``seed``.  Written from the published definition: the state advances by
    the golden-ratio increment and each output is the state passed through
    the variant-13 mixer."""
    state = seed & MASK64
    out = []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        z = z ^ (z >> 31)
        out.append(z)
    return out


def sign_vector(seed: int, d: int) -> np.ndarray:
    """D in {-1,+1}^d: the random diagonal of the randomized Hadamard
    transform (TurboQuant From Scratch, section 2, step 2: D holds random
    signs).  D_i = -1 when bit 63 of the i-th splitmix64 output is set."""
    return np.array([-1.0 if (z >> 63) else 1.0 for z in splitmix64_stream(seed, d)])


# --------------------------------------------------------------------------
# S3  orthonormal Walsh-Hadamard transform
# --------------------------------------------------------------------------
def hadamard_matrix(n: int) -> np.ndarray:
    """Orthonormal Sylvester-ordered Walsh-Hadamard matrix,
    H[i, k] = (-1)^popcount(i & k) / sqrt(n).  This is the closed form of the
    butterfly in TurboQuant From Scratch, section 2 (``fwht``: pairs (a+b,
    a-b) at strides 1, 2, 4, ..., scaled by 1/sqrt(d))."""
    if n <= 0 or n & (n - 1):
        raise ValueError("Hadamard size must be a power of two")
    i = np.arange(n)
    parity = np.zeros((n, n), dtype=np.int64)
    x = i[:, None] & i[None, :]
    while np.any(x):
        parity ^= x & 1
        x = x >> 1
    return np.where(parity == 1, -1.0, 1.0) / math.sqrt(n)


# --------------------------------------------------------------------------
# S0  Lloyd-Max codebook for N(0, 1/blk)
# --------------------------------------------------------------------------
_STD = NormalDist()


def _phi(t: float) -> float:
    if math.isinf(t):
        return 0.0
    return math.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)


def _Phi_diff(a: float, b: float) -> float:
    """P(a < Z <= b) for standard normal Z, accurate in both tails."""
    if a >= 0.0:
        return 0.5 * (math.erfc(a / math.sqrt(2.0)) - math.erfc(b / math.sqrt(2.0)))
    if b <= 0.0:
        return 0.5 * (math.erfc(-b / math.sqrt(2.0)) - math.erfc(-a / math.sqrt(2.0)))
    return 0.5 * (math.erf(b / math.sqrt(2.0)) - math.erf(a / math.sqrt(2.0)))


_CODEBOOK_CACHE: dict = {}


def lloyd_max_codebook(bits: int, blk: int, max_iter: int = 1000000):
    """Lloyd-Max scalar quantiser for N(0, sigma^2 = 1/blk) with 2^bits
    levels (TurboQuant From Scratch, section 2, step 3: the codebook is solved once
    per bit width for N(0, 1/d); turboquant-pytorch README, lloyd_max.py).

    Start from the quantiles sigma * Phi^-1((k + 1/2) / 2^bits), then
    alternate the two optimality conditions: boundaries are midpoints of
    neighbouring centroids, centroids are conditional means of their cell,
    c_k = sigma (phi(a) - phi(b)) / (Phi(b) - Phi(a)) with a, b the cell
    edges in units of sigma.  The iteration converges linearly, so it runs
    to the fixed point itself: until the centroids stop moving, or the step
    is below 1e-15 sigma and no longer shrinks (rounding-level oscillation).
    Returns (centroids ascending, boundaries), float64."""
    key = (bits, blk)
    if key in _CODEBOOK_CACHE:
        c, b = _CODEBOOK_CACHE[key]
        return c.copy(), b.copy()
    K = 1 << bits
    sigma = 1.0 / math.sqrt(blk)
    c = [_STD.inv_cdf((k + 0.5) / K) for k in range(K)]   # in units of sigma
    if K > 16:
        # 256 levels: Lloyd's linear convergence is too slow in pure Python;
        # Newton's method on the same fixed point (see _lloyd_max_newton)
        c = _lloyd_max_newton(c)
        max_iter = 0
    last = math.inf
    for _ in range(max_iter):
        edges = [-math.inf] + [0.5 * (c[k] + c[k + 1]) for k in range(K - 1)] + [math.inf]
        new = []
        for k in range(K):
            a, b = edges[k], edges[k + 1]
            new.append((_phi(a) - _phi(b)) / _Phi_diff(a, b))
        delta = max(abs(x - y) for x, y in zip(new, c))
        c = new
        if delta == 0.0 or (delta < 1e-15 and delta >= last):
            break
        last = delta
    # N(0, sigma^2) is symmetric, so is its Lloyd-Max codebook: remove the
    # rounding-level asymmetry so that the middle boundary is exactly 0.
    c = [0.5 * (c[k] - c[K - 1 - k]) for k in range(K)]
    cent = np.array(c) * sigma
    bnd = 0.5 * (cent[1:] + cent[:-1])
    _CODEBOOK_CACHE[key] = (cent.copy(), bnd.copy())
    return cent, bnd


def _lloyd_max_newton(c: list) -> list:
    """The Lloyd-Max fixed point for N(0, 1) by Newton's method: the
    residual F_k = m_k - c_k, with m_k = (phi(l) - phi(u)) / P the mean of
    cell [l, u] (midpoints of the neighbouring centroids) and P its mass, has
    a tridiagonal Jacobian: dm/du = phi(u) (u - m) / P, dm/dl = phi(l) (m - l)
    / P, each edge moving by half of either neighbour's step.  Solved by the
    Thomas algorithm until the step is at rounding level."""
    K = len(c)
    c = list(c)
    last = math.inf
    for _ in range(200):
        edges = [-math.inf] + [0.5 * (c[k] + c[k + 1]) for k in range(K - 1)] + [math.inf]
        lo, di, up, rhs = [0.0] * K, [0.0] * K, [0.0] * K, [0.0] * K
        for k in range(K):
            l, u = edges[k], edges[k + 1]
            P = _Phi_diff(l, u)
            m = (_phi(l) - _phi(u)) / P
            dmu = 0.0 if math.isinf(u) else _phi(u) * (u - m) / P
            dml = 0.0 if math.isinf(l) else _phi(l) * (m - l) / P
            lo[k] = 0.5 * dml
            up[k] = 0.5 * dmu
            di[k] = 0.5 * dml + 0.5 * dmu - 1.0
            rhs[k] = -(m - c[k])
        # Thomas algorithm
        for k in range(1, K):
            w = lo[k] / di[k - 1]
            di[k] -= w * up[k - 1]
            rhs[k] -= w * rhs[k - 1]
        step = [0.0] * K
        step[K - 1] = rhs[K - 1] / di[K - 1]
        for k in range(K - 2, -1, -1):
            step[k] = (rhs[k] - up[k] * step[k + 1]) / di[k]
        c = [c[k] + step[k] for k in range(K)]
        moved = max(abs(x) for x in step)
        if moved == 0.0 or (moved < 1e-15 and moved >= last):
            break
        last = moved
    return c


def _beta_cell(alpha: float, e0: np.ndarray, e1: np.ndarray):
    """Mass and first moment of the cells [e0, e1] under the law of one
    coordinate of a uniformly random unit vector in R^blk, alpha = (blk-1)/2:
    (x + 1)/2 ~ Beta(alpha, alpha), density (1 - x^2)^(alpha-1) / B(1/2, alpha).
    The mass is the regularised incomplete beta function (scipy), taken
    from the nearer end of [-1, 1]; the moment is exact:
    int x (1 - x^2)^(alpha-1) dx = -(1 - x^2)^alpha / (2 alpha)."""
    from scipy import special
    z0, z1 = (1.0 + e0) / 2.0, (1.0 + e1) / 2.0
    upper = e0 >= 0.0
    low = special.betainc(alpha, alpha, z1) - special.betainc(alpha, alpha, z0)
    high = special.betainc(alpha, alpha, 1.0 - z0) - special.betainc(alpha, alpha, 1.0 - z1)
    mass = np.where(upper, high, low)
    norm = special.beta(0.5, alpha)
    mom = (np.power(np.clip(1.0 - e0 * e0, 0.0, None), alpha) -
           np.power(np.clip(1.0 - e1 * e1, 0.0, None), alpha)) / (2.0 * alpha * norm)
    return mass, mom


def lloyd_max_beta_codebook(bits: int, blk: int):
    """Lloyd-Max quantiser with 2^bits levels for the exact law of one
    coordinate of a rotated unit vector in R^blk, (x + 1)/2 ~
    Beta((blk-1)/2, (blk-1)/2) (llama.cpp-turboquant "How it works": the
    Beta((d-1)/2, (d-1)/2) codebook).  The fixed point of "boundaries =
    midpoints, centroids = conditional means", solved by a root finder on
    step(c) - c from the scaled Gaussian codebook, then polished with plain
    steps until they stop moving.  blk >= 2 (blk = 3: the uniform law on
    [-1, 1]).  Returns (centroids ascending, boundaries), float64."""
    from scipy import optimize
    key = ("beta", bits, blk)
    if key in _CODEBOOK_CACHE:
        c, b = _CODEBOOK_CACHE[key]
        return c.copy(), b.copy()
    K = 1 << bits
    alpha = 0.5 * (blk - 1)

    def step(c):
        edges = np.clip(np.concatenate([[-1.0], 0.5 * (c[1:] + c[:-1]), [1.0]]), -1.0, 1.0)
        mass, mom = _beta_cell(alpha, edges[:-1], edges[1:])
        return mom / mass

    c0, _ = lloyd_max_codebook(bits, max(blk, 1))
    c0 = np.clip(c0, -1.0 + 1.0 / K, 1.0 - 1.0 / K)
    import warnings
    with warnings.catch_warnings():   # fsolve reports the rounding floor as slow progress
        warnings.simplefilter("ignore", RuntimeWarning)
        c = optimize.fsolve(lambda v: step(v) - v, c0, xtol=1e-13)
    last = math.inf
    for _ in range(2000):
        new = step(c)
        delta = float(np.max(np.abs(new - c)))
        c = new
        if delta == 0.0 or (delta < 1e-17 and delta >= last):
            break
        last = delta
    c = 0.5 * (c - c[::-1])
    bnd = 0.5 * (c[1:] + c[:-1])
    _CODEBOOK_CACHE[key] = (c.copy(), bnd.copy())
    return c, bnd


def codebook_for(L) -> tuple:
    """The codebook a layout selects: Gaussian N(0, 1/blk) (codebook 0) or
    the exact Beta law (codebook 1)."""
    if getattr(L, "codebook", 0) == 1:
        return lloyd_max_beta_codebook(L.bits, L.blk)
    return lloyd_max_codebook(L.bits, L.blk)


def relative_distortion(bits: int) -> float:
    """D_b = E[(Z - Q(Z))^2] / sigma^2 of the Lloyd-Max quantiser, computed
    from the optimality conditions as 1 - sum_k P_k c_k^2 / sigma^2."""
    cent, bnd = lloyd_max_codebook(bits, 1)
    edges = [-math.inf] + list(bnd) + [math.inf]
    s = 0.0
    for k, ck in enumerate(cent):
        s += _Phi_diff(edges[k], edges[k + 1]) * ck * ck
    return 1.0 - s


# --------------------------------------------------------------------------
# Layout description (the oracle's own copy; the library has its own)
# --------------------------------------------------------------------------
class Layout:
    """Codec settings of one cache (K or V): head_dim d, rotation/norm
    block blk (d for one norm per vector, 32 for block-32), MSE bits,
    QJL rows m (0 = none, requires blk == d), norm correction flag, and the
    seed of the sign vector."""

    def __init__(self, head_dim, block, bits, qjl_m=0, norm_correct=0, sign_seed=1, codebook=0):
        self.d = int(head_dim)
        self.codebook = int(codebook)
        self.blk = int(block)
        self.bits = int(bits)
        self.m = int(qjl_m)
        self.nc = int(norm_correct)
        self.seed = int(sign_seed)
        if self.d % self.blk or self.blk < 2 or self.blk & (self.blk - 1):
            raise ValueError("block must be a power of two dividing head_dim")
        if not (1 <= self.bits <= 4 or self.bits == 8):
            raise ValueError("bits must be 1..4 or 8")
        if self.bits == 8 and (self.codebook != 0 or qjl_m):
            raise ValueError("8-bit codes take the Gaussian codebook and no QJL")
        if self.m and (self.blk != self.d or self.m % 32):
            raise ValueError("QJL needs block == head_dim and m a multiple of 32")

    @property
    def nb(self):
        return self.d // self.blk

    @property
    def code_bytes(self):
        return self.d * self.bits // 8

    @property
    def qjl_bytes(self):
        return self.m // 8


# --------------------------------------------------------------------------
# S6 QJL correction term (shared by quantise-with-nc and dequantise)
# --------------------------------------------------------------------------
def qjl_term(S: np.ndarray, bits_pm: np.ndarray, rho: np.ndarray) -> np.ndarray:
    """rho * sqrt(pi/2)/m * S^T (2s - 1): the QJL reconstruction of the unit
    residual (TurboQuant From Scratch, section 2, the ``qjl`` branch;
    turboquant-pytorch README, QJL estimator formula).  bits_pm holds
    +-1 per projection row, shape [N, m]; rho shape [N]."""
    m = S.shape[0]
    return (rho[:, None] * (QJL_CONST / m)) * (bits_pm @ S)


# --------------------------------------------------------------------------
# S2-S7  quantise
# --------------------------------------------------------------------------
def quantize(x, L: Layout, S=None):
    """Encode rows of x ([N, d], any float dtype, promoted exactly to
    float64).  Returns a dict with
      codes  int64 [N, d]  code index per rotated coordinate (block-major)
      y      float64 [N, d]  rotated unit-block coordinates (for tie checks)
      scale  float16 [N, nb]
      qjl    uint8 [N, m]  (0/1, only with QJL) and proj float64 [N, m]
      rho    float16 [N]   (only with QJL)
    """
    x = np.asarray(x, dtype=np.float64)
    N, d = x.shape
    assert d == L.d
    D = sign_vector(L.seed, d)
    H = hadamard_matrix(L.blk)
    cent, bnd = codebook_for(L)
    codes = np.zeros((N, d), dtype=np.int64)
    y_all = np.zeros((N, d))
    scale = np.zeros((N, L.nb))
    u_all = np.zeros((N, d))
    for j in range(L.nb):
        sl = slice(j * L.blk, (j + 1) * L.blk)
        xb = x[:, sl]
        n = np.sqrt(np.sum(xb * xb, axis=1))                 # S2 norm split
        safe = np.where(n > 0, n, 1.0)
        u = np.where(n[:, None] > 0, xb / safe[:, None], 0.0)
        y = (D[sl][None, :] * u) @ H.T                        # S3 y = H (D u)
        code = np.searchsorted(bnd, y, side="left")           # S4 #{k: y > beta_k}
        codes[:, sl] = code
        y_all[:, sl] = y
        u_all[:, sl] = u
        if L.nc and not L.m:                                   # S5 norm correction
            cn = np.sqrt(np.sum(cent[code] ** 2, axis=1))
            scale[:, j] = np.where(cn > 0, n / np.where(cn > 0, cn, 1.0), 0.0)
        else:
            scale[:, j] = n
    out = {"codes": codes, "y": y_all}
    if L.m:                                                    # S6 QJL residual
        if S is None:
            raise ValueError("QJL layout needs S")
        S = np.asarray(S, dtype=np.float64)
        assert S.shape == (L.m, d)
        u_mse = (cent[codes] @ H) * D[None, :]               # D (H c)
        # a zero vector has no direction: its residual is taken as 0
        r = np.where(scale[:, :1] > 0, u_all - u_mse, 0.0)
        rho = np.sqrt(np.sum(r * r, axis=1))
        proj = r @ S.T
        s = (proj >= 0).astype(np.uint8)
        out["qjl"] = s
        out["proj"] = proj
        rho16 = rho.astype(np.float16)
        out["rho"] = rho16
        if L.nc:
            corr = qjl_term(S, 2.0 * s - 1.0, rho16.astype(np.float64))
            tot = np.sqrt(np.sum((u_mse + corr) ** 2, axis=1))
            n = scale[:, 0]
            scale[:, 0] = np.where(tot > 0, n / np.where(tot > 0, tot, 1.0), 0.0)
    out["scale"] = scale.astype(np.float16)
    return out


# --------------------------------------------------------------------------
# S7  packed layout (32-code groups, little endian 32-bit words)
# --------------------------------------------------------------------------
def _group_words(g: np.ndarray, bits: int) -> list:
    """Words of one 32-code group.  g: [N, 32] int codes.  Word w, nibble k
    (bits 4k..4k+3) is defined per bit width as
      b=4: code(8w+k)                                       (4 words)
      b=3: bits 0-2 = code(8w+k), bit 3 = bit w of code(24+k) (3 words)
      b=2: bits 0-1 = code(8w+k), bits 2-3 = code(16+8w+k)  (2 words)
      b=1: bit p = code(8p+k)                                (1 word)
    so every word holds whole codes in nibble positions."""
    N = g.shape[0]
    words = []
    for w in range(bits):
        acc = np.zeros(N, dtype=np.uint64)
        for k in range(8):
            if bits == 4:
                nib = g[:, 8 * w + k]
            elif bits == 3:
                nib = g[:, 8 * w + k] | (((g[:, 24 + k] >> w) & 1) << 3)
            elif bits == 2:
                nib = g[:, 8 * w + k] | (g[:, 16 + 8 * w + k] << 2)
            else:
                nib = g[:, k] | (g[:, 8 + k] << 1) | (g[:, 16 + k] << 2) | (g[:, 24 + k] << 3)
            acc |= (nib.astype(np.uint64) & np.uint64(0xF)) << np.uint64(4 * k)
        words.append(acc.astype(np.uint32))
    return words


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes [N, d] -> uint8 [N, d*bits/8]: 32-code groups in coordinate
    order, each group 4*bits bytes of little-endian words (see
    ``_group_words``).  Same bytes per element as the turbo3/turbo4 GGML
    blocks of llama.cpp-turboquant (12 and 16 code bytes per 32 values)."""
    codes = np.asarray(codes, dtype=np.int64)
    N, d = codes.shape
    if bits == 8:   # one byte per code, in coordinate order
        return codes.astype(np.uint8)
    out = np.zeros((N, d * bits // 8), dtype=np.uint8)
    gb = 4 * bits
    for gi in range(d // 32):
        words = _group_words(codes[:, 32 * gi:32 * gi + 32], bits)
        for w, word in enumerate(words):
            for byte in range(4):
                out[:, gi * gb + 4 * w + byte] = ((word >> np.uint32(8 * byte)) & np.uint32(0xFF)).astype(np.uint8)
    return out


def unpack_codes(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Inverse of ``pack_codes``."""
    packed = np.asarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    if bits == 8:
        return packed[:, :d].astype(np.int64)
    codes = np.zeros((N, d), dtype=np.int64)
    gb = 4 * bits
    for gi in range(d // 32):
        base = 32 * gi
        for w in range(bits):
            o = gi * gb + 4 * w
            word = (packed[:, o].astype(np.int64) | (packed[:, o + 1].astype(np.int64) << 8)
                    | (packed[:, o + 2].astype(np.int64) << 16) | (packed[:, o + 3].astype(np.int64) << 24))
            for k in range(8):
                nib = (word >> (4 * k)) & 0xF
                if bits == 4:
                    codes[:, base + 8 * w + k] = nib
                elif bits == 3:
                    codes[:, base + 8 * w + k] = nib & 7
                    codes[:, base + 24 + k] |= ((nib >> 3) & 1) << w
                elif bits == 2:
                    codes[:, base + 8 * w + k] = nib & 3
                    codes[:, base + 16 + 8 * w + k] = (nib >> 2) & 3
                else:
                    for p in range(4):
                        codes[:, base + 8 * p + k] = (nib >> p) & 1
    return codes


def pack_qjl(s: np.ndarray) -> np.ndarray:
    """QJL sign bits [N, m] (0/1) -> uint8 [N, m/8]: m/32 little-endian
    32-bit words, bit i of word w = s[32w + i]."""
    s = np.asarray(s, dtype=np.uint8)
    N, m = s.shape
    out = np.zeros((N, m // 8), dtype=np.uint8)
    for i in range(m):
        out[:, i // 8] |= (s[:, i] << (i % 8)).astype(np.uint8)
    return out


def unpack_qjl(packed: np.ndarray, m: int) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    return np.stack([(packed[:, i // 8] >> (i % 8)) & 1 for i in range(m)], axis=1).astype(np.uint8)


def encode(x, L: Layout, S=None):
    """Quantise then pack: returns (codes_packed, scales fp16, qjl_packed or
    None, rho fp16 or None) - the four arrays the packed cache stores."""
    q = quantize(x, L, S)
    codes = pack_codes(q["codes"], L.bits)
    qjl = pack_qjl(q["qjl"]) if L.m else None
    return codes, q["scale"], qjl, (q["rho"] if L.m else None)


# --------------------------------------------------------------------------
# S8  dequantise
# --------------------------------------------------------------------------
def dequantize(codes_packed, scales, L: Layout, qjl_packed=None, rho=None, S=None):
    """x~ = scale * (D (H c) [+ rho sqrt(pi/2)/m S^T (2s-1)]) per block
    (TurboQuant From Scratch, section 2: un-rotate ``fwht(yq) * sign``, add
    the QJL term, multiply by the norm; llama.cpp-turboquant "How it works",
    Decode: unpack -> centroid lookup -> inverse FWHT -> x norm).  Uses the
    stored fp16 scale and fp16 rho."""
    codes = unpack_codes(codes_packed, L.bits, L.d)
    N = codes.shape[0]
    D = sign_vector(L.seed, L.d)
    H = hadamard_matrix(L.blk)
    cent, _ = codebook_for(L)
    sc = np.asarray(scales, dtype=np.float16).astype(np.float64).reshape(N, L.nb)
    out = np.zeros((N, L.d))
    for j in range(L.nb):
        sl = slice(j * L.blk, (j + 1) * L.blk)
        out[:, sl] = (cent[codes[:, sl]] @ H) * D[sl][None, :]   # H symmetric: H c
    if L.m:
        s = unpack_qjl(qjl_packed, L.m).astype(np.float64)
        out = out + qjl_term(np.asarray(S, dtype=np.float64), 2.0 * s - 1.0,
                             np.asarray(rho, dtype=np.float16).astype(np.float64).reshape(N))
    for j in range(L.nb):
        sl = slice(j * L.blk, (j + 1) * L.blk)
        out[:, sl] *= sc[:, j:j + 1]
    return out


# --------------------------------------------------------------------------
# GGML-style blocks (llama.cpp-turboquant "GGML Types": 32 values per block,
# a 2-byte norm then the packed codes, 14 bytes at 3 bits, 18 at 4 bits; the
# "How it works" section: the norm of a 128-value rotation chunk is stored in
# each of its 32-value blocks)
# --------------------------------------------------------------------------
def block_bytes(bits: int) -> int:
    return 2 + 4 * bits


def to_blocks(codes_packed: np.ndarray, scales: np.ndarray, L: Layout) -> np.ndarray:
    """codes [N, d*bits/8] + scales fp16 [N, d/blk] -> uint8 [N, d/32 *
    (2 + 4 bits)]: block j = the fp16 norm of the rotation block holding
    values 32j .. 32j+31 (little-endian), then group j's packed code bytes."""
    codes_packed = np.asarray(codes_packed, dtype=np.uint8)
    sc = np.asarray(scales, dtype=np.float16).reshape(codes_packed.shape[0], L.nb)
    N = codes_packed.shape[0]
    bb, gb = block_bytes(L.bits), 4 * L.bits
    out = np.zeros((N, (L.d // 32) * bb), dtype=np.uint8)
    for j in range(L.d // 32):
        norm = sc[:, (32 * j) // L.blk].view(np.uint16)
        out[:, j * bb] = (norm & 0xFF).astype(np.uint8)
        out[:, j * bb + 1] = (norm >> 8).astype(np.uint8)
        out[:, j * bb + 2:(j + 1) * bb] = codes_packed[:, j * gb:(j + 1) * gb]
    return out


def from_blocks(blocks: np.ndarray, L: Layout):
    """Inverse of ``to_blocks``: the norm of a rotation block is read from its
    first 32-value block."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    N = blocks.shape[0]
    bb, gb = block_bytes(L.bits), 4 * L.bits
    codes = np.zeros((N, L.d * L.bits // 8), dtype=np.uint8)
    sc = np.zeros((N, L.nb), dtype=np.uint16)
    for j in range(L.d // 32):
        codes[:, j * gb:(j + 1) * gb] = blocks[:, j * bb + 2:(j + 1) * bb]
        if (32 * j) % L.blk == 0:
            sc[:, (32 * j) // L.blk] = blocks[:, j * bb].astype(np.uint16) | (blocks[:, j * bb + 1].astype(np.uint16) << 8)
    return codes, sc.view(np.float16)


# --------------------------------------------------------------------------
# S9-S14  attention over the decoded cache (no Hadamard-domain shortcut)
# --------------------------------------------------------------------------
def softmax_rows(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def decode_attention(q, Kd, Vd, kv_len=None, softmax_scale=None):
    """One query per (batch, q-head) over explicitly decoded K~, V~.
    q [B, Hq, d]; Kd, Vd [B, Hkv, S, d] float64; kv_len [B] (None: all S).
    q-head h reads KV head floor(h / (Hq/Hkv)); scores scaled by 1/sqrt(d)
    (cneuralnets "TurboQuant: 3-Bit Compression with Zero Overhead",
    Part 3, standard 1/sqrt(d_k) scaling); plain max-subtracted softmax."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    Hkv = Kd.shape[1]
    g = Hq // Hkv
    sc = 1.0 / math.sqrt(d) if not softmax_scale or softmax_scale <= 0 else softmax_scale
    out = np.zeros((B, Hq, d))
    for b in range(B):
        n = Kd.shape[2] if kv_len is None else int(kv_len[b])
        for h in range(Hq):
            kh = h // g
            if n == 0:
                continue
            s = Kd[b, kh, :n] @ q[b, h] * sc
            p = softmax_rows(s[None, :])[0]
            out[b, h] = p @ Vd[b, kh, :n]
    return out


def prefill_attention(q, Kd, Vd, ctx, causal=True, softmax_scale=None, rows=None, group=None):
    """Tq queries per (batch, q-head) at positions ctx-Tq .. ctx-1 over the
    decoded cache positions [0, ctx).  With ``causal`` query i attends to
    positions <= ctx - Tq + i (bottom-right aligned mask).

    ``rows`` (query indices) restricts the result to those queries, at their
    own positions.  ``group`` = (first q-head, count) restricts it to q-heads
    that share one KV head, which Kd and Vd then hold alone ([B, 1, S, d])."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, Tq, d = q.shape
    sc = 1.0 / math.sqrt(d) if not softmax_scale or softmax_scale <= 0 else softmax_scale
    rows = np.arange(Tq) if rows is None else np.asarray(rows)
    if group is None:
        heads = list(range(Hq))
        g = Hq // Kd.shape[1]
        kv_of = [h // g for h in heads]
    else:
        heads = list(range(group[0], group[0] + group[1]))
        kv_of = [0] * len(heads)
    out = np.zeros((B, len(heads), len(rows), d))
    for b in range(B):
        for j, h in enumerate(heads):
            kh = kv_of[j]
            s = q[b, h, rows] @ Kd[b, kh, :ctx].T * sc        # [rows, ctx]
            if causal:
                pos = ctx - Tq + rows
                mask = np.arange(ctx)[None, :] > pos[:, None]
                s = np.where(mask, -np.inf, s)
            p = softmax_rows(s)
            out[b, j] = p @ Vd[b, kh, :ctx]
    return out


def qjl_score_estimate(q, k_mse, rho, s_bits, S, knorm):
    """turboquant-pytorch README, QJL estimator formula, scaled by the key
    norm: <q,k> ~ ||k|| (<q,u_mse> + rho sqrt(pi/2)/m <Sq, 2s-1>).  Used only
    to check that decoding-then-dot equals the estimator."""
    m = S.shape[0]
    return knorm * (q @ k_mse + rho * QJL_CONST / m * ((S @ q) @ (2.0 * s_bits - 1.0)))

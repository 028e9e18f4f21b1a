"""Pins for the float64 oracle: checks against what the source pages print,
closed forms, textbook values, brute force and invariants.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

from oracle import tq_oracle as O
from turboquant_kv_cache_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- signs
def test_splitmix64_known_answers():
    # Published first outputs of splitmix64 from state 0 (reference C
    # implementation by S. Vigna, prng.di.unimi.it).
    assert O.splitmix64_stream(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_sign_vector_top_bit_rule():
    D = O.sign_vector(0, 3)
    assert list(D) == [-1.0, 1.0, 1.0]
    D = O.sign_vector(1, 256)
    assert set(np.unique(D)) <= {-1.0, 1.0}
    assert 80 < np.sum(D > 0) < 176            # roughly balanced


# ---------------------------------------------------------------- Hadamard
def _sylvester(n):
    H = np.array([[1.0]])
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H / math.sqrt(n)


def _butterfly(v):
    """Walsh-Hadamard by butterflies on the last axis, as in the
    ``fwht`` listing of TurboQuant From Scratch, section 2."""
    v = np.array(v, dtype=np.float64, copy=True)
    n = v.shape[-1]
    h = 1
    while h < n:
        for start in range(0, n, 2 * h):
            a = v[..., start:start + h].copy()
            b = v[..., start + h:start + 2 * h].copy()
            v[..., start:start + h] = a + b
            v[..., start + h:start + 2 * h] = a - b
        h *= 2
    return v / math.sqrt(n)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 32, 64, 128, 256])
def test_hadamard_closed_form(n):
    H = O.hadamard_matrix(n)
    assert np.array_equal(H, _sylvester(n))
    assert np.allclose(H @ H, np.eye(n), atol=1e-15)
    assert np.array_equal(H, H.T)
    x = np.random.default_rng(n).standard_normal((5, n))
    assert np.allclose(np.linalg.norm(x @ H.T, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    assert np.allclose(_butterfly(x), x @ H.T, atol=1e-14)


def test_rotation_order_is_sign_then_hadamard():
    # y = H (D u): the sign vector multiplies u before the transform.
    L = O.Layout(64, 32, 3, sign_seed=5)
    x = inputs.gaussian((7, 64), 99, np.float64)
    q = O.quantize(x, L)
    D = O.sign_vector(5, 64)
    for j in range(2):
        sl = slice(32 * j, 32 * j + 32)
        u = x[:, sl] / np.linalg.norm(x[:, sl], axis=1, keepdims=True)
        assert np.allclose(q["y"][:, sl], _butterfly(u * D[sl]), atol=1e-14)


# ---------------------------------------------------------------- codebook
def test_codebook_textbook_values():
    g = _golden("textbook_lloyd_max.json")
    for bits, ref in g["levels"].items():
        c, b = O.lloyd_max_codebook(int(bits), 1)
        K = len(c)
        assert np.allclose(c[K // 2:], ref["outputs"], atol=g["tolerance"])
        assert np.allclose(b[K // 2 - 1:], ref["thresholds"], atol=g["tolerance"])


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("blk", [32, 64, 128, 256])
def test_codebook_symmetry_and_scaling(bits, blk):
    c, b = O.lloyd_max_codebook(bits, blk)
    assert np.allclose(c, -c[::-1], atol=1e-15)
    assert np.all(np.diff(c) > 0)
    c1, _ = O.lloyd_max_codebook(bits, 1)
    assert np.allclose(c, c1 / math.sqrt(blk), rtol=1e-13)
    assert np.allclose(b, 0.5 * (c[1:] + c[:-1]), rtol=0, atol=1e-16)


def test_codebook_one_bit_closed_form():
    c, b = O.lloyd_max_codebook(1, 128)
    s = 1 / math.sqrt(128)
    assert np.allclose(c, [-s * math.sqrt(2 / math.pi), s * math.sqrt(2 / math.pi)], rtol=1e-13)
    assert abs(O.relative_distortion(1) - (1 - 2 / math.pi)) < 1e-12


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codebook_centroid_condition_quadrature(bits):
    integrate = pytest.importorskip("scipy.integrate")
    c, b = O.lloyd_max_codebook(bits, 1)
    edges = [-np.inf] + list(b) + [np.inf]
    pdf = lambda t: math.exp(-t * t / 2) / math.sqrt(2 * math.pi)
    for k in range(len(c)):
        mass = integrate.quad(pdf, edges[k], edges[k + 1], epsabs=1e-14)[0]
        mom = integrate.quad(lambda t: t * pdf(t), edges[k], edges[k + 1], epsabs=1e-14)[0]
        assert abs(mom / mass - c[k]) < 1e-9


def test_distortion_matches_page_figures():
    g = _golden("pages_codec_figures.json")["lloyd_max_relative_distortion"]
    for bits, val in zip(g["bits"], g["values"]):
        assert abs(O.relative_distortion(bits) - val) / val < 0.01


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_distortion_monte_carlo(bits):
    c, b = O.lloyd_max_codebook(bits, 1)
    z = np.random.default_rng(bits).standard_normal(2_000_000)
    mse = np.mean((z - c[np.searchsorted(b, z)]) ** 2)
    assert abs(mse - O.relative_distortion(bits)) / O.relative_distortion(bits) < 0.01


# ---------------------------------------------------------------- brute force
def _all_codevectors(n, bits):
    K = 1 << bits
    idx = np.indices([K] * n).reshape(n, -1).T
    return idx


@pytest.mark.parametrize("d,bits", [(4, 1), (4, 2), (4, 3), (8, 2)])
def test_bucketize_is_nearest_codeword(d, bits):
    L = O.Layout(d, d, bits, sign_seed=3)
    c, _ = O.lloyd_max_codebook(bits, d)
    D = O.sign_vector(3, d)
    H = _sylvester(d)
    allc = _all_codevectors(d, bits)
    recon = (c[allc] @ H.T) * D[None, :]           # D H c for every code vector
    x = inputs.gaussian((40, d), 7 + d + bits, np.float64)
    u = x / np.linalg.norm(x, axis=1, keepdims=True)
    q = O.quantize(x, L)
    for i in range(x.shape[0]):
        dist = np.sum((recon - u[i]) ** 2, axis=1)
        best = allc[np.argmin(dist)]
        assert np.array_equal(best, q["codes"][i])


# ---------------------------------------------------------------- MSE
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_unit_vector_mse_matches_page_table(bits):
    g = _golden("pages_codec_figures.json")["unit_vector_mse"]
    i = g["bits"].index(bits)
    x = inputs.unit_vectors(g["n_vectors"], g["d"], seed=2024, dtype=np.float64)
    L = O.Layout(128, 128, bits)
    codes, scale, _, _ = O.encode(x, L)
    xr = O.dequantize(codes, scale, L)
    u = x / np.linalg.norm(x, axis=1, keepdims=True)
    ur = xr / scale.astype(np.float64)
    mse = np.mean(np.sum((u - ur) ** 2, axis=1))
    assert abs(mse - g["measured"][i]) / g["measured"][i] < 0.05
    bound = math.sqrt(3) * math.pi / 2 * 4.0 ** (-bits)
    assert abs(bound - g["upper_bound"][i]) <= 0.0006      # the bound column's formula
    assert mse < bound


# ---------------------------------------------------------------- QJL
def test_qjl_term_unbiased_over_projections():
    d, m, n_seeds = 64, 32, 10000
    rng = np.random.default_rng(11)
    q = rng.standard_normal(d)
    r = 0.3 * rng.standard_normal(d)
    est = np.empty(n_seeds)
    for s0 in range(0, n_seeds, 500):
        S = rng.standard_normal((500, m, d))
        for t in range(500):
            sb = (S[t] @ r >= 0).astype(np.float64)
            corr = O.qjl_term(S[t], (2 * sb - 1)[None, :], np.array([np.linalg.norm(r)]))
            est[s0 + t] = corr[0] @ q
    true = q @ r
    var_theory = (math.pi / 2 * (q @ q) * (r @ r) - true ** 2) / m
    se = math.sqrt(var_theory / n_seeds)
    assert abs(est.mean() - true) < 4 * se
    assert abs(est.var() / var_theory - 1) < 0.1


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_inner_product_bias_and_correlation(bits):
    g = _golden("pages_codec_figures.json")["qjl_inner_product"]
    i = g["bits"].index(bits)
    d = m = g["d"]
    n = g["n_pairs"]
    k = inputs.unit_vectors(n, d, seed=500 + bits, dtype=np.float64)
    q = inputs.unit_vectors(n, d, seed=600 + bits, dtype=np.float64)
    S = inputs.qjl_matrix(m, d, 7).astype(np.float64)
    L = O.Layout(d, d, bits - 1, qjl_m=m)                 # (b-1)-bit MSE + 1-bit QJL
    codes, scale, qjl, rho = O.encode(k, L, S)
    kr = O.dequantize(codes, scale, L, qjl, rho, S)
    true = np.sum(q * k, axis=1)
    est = np.sum(q * kr, axis=1)
    err = est - true
    assert abs(err.mean()) < 3 * err.std() / math.sqrt(n)
    corr = np.corrcoef(true, est)[0, 1]
    D = O.relative_distortion(bits - 1)
    closed = math.sqrt((1 / d) / (1 / d + math.pi / 2 * D / m))
    assert abs(corr - closed) < 0.02
    assert abs(corr - g["correlation"][i]) < 0.03
    assert abs(err.mean() - g["bias"][i]) < 0.005


def test_dequant_dot_equals_qjl_estimator():
    d = m = 128
    L = O.Layout(d, d, 2, qjl_m=m)
    k = inputs.gaussian((20, d), 41, np.float64)
    q = inputs.gaussian((20, d), 42, np.float64)
    S = inputs.qjl_matrix(m, d, 7).astype(np.float64)
    codes, scale, qjl, rho = O.encode(k, L, S)
    kr = O.dequantize(codes, scale, L, qjl, rho, S)
    c, _ = O.lloyd_max_codebook(2, d)
    D = O.sign_vector(1, d)
    u_mse = (c[O.unpack_codes(codes, 2, d)] @ _sylvester(d).T) * D
    s = O.unpack_qjl(qjl, m).astype(np.float64)
    for i in range(20):
        ref = O.qjl_score_estimate(q[i], u_mse[i], float(rho[i]), s[i], S, float(scale[i, 0]))
        assert abs(ref - q[i] @ kr[i]) < 1e-9 * max(1.0, abs(ref))


# ---------------------------------------------------------------- norm correction
@pytest.mark.parametrize("qjl", [0, 128])
def test_norm_correction_restores_norm(qjl):
    d = 128
    L = O.Layout(d, d, 2, qjl_m=qjl, norm_correct=1)
    x = inputs.gaussian((50, d), 77, np.float64) * 3.0
    S = inputs.qjl_matrix(128, d, 7).astype(np.float64) if qjl else None
    codes, scale, qb, rho = O.encode(x, L, S)
    xr = O.dequantize(codes, scale, L, qb, rho, S)
    n = np.linalg.norm(x, axis=1)
    assert np.allclose(np.linalg.norm(xr, axis=1), n, rtol=2e-3)
    L0 = O.Layout(d, d, 2, qjl_m=qjl, norm_correct=0)
    codes0, scale0, qb0, rho0 = O.encode(x, L0, S)
    assert np.array_equal(codes0, codes)
    xr0 = O.dequantize(codes0, scale0, L0, qb0, rho0, S)
    if not qjl:   # plain MSE reconstruction is shorter on average: sqrt(1 - D_2)
        ratio = np.mean(np.linalg.norm(xr0, axis=1) / n)
        assert abs(ratio - math.sqrt(1 - O.relative_distortion(2))) < 0.02


def test_block32_norms_per_block():
    L = O.Layout(128, 32, 3)
    x = inputs.gaussian((10, 128), 5, np.float64)
    x[:, 32:64] *= 100.0
    q = O.quantize(x, L)
    for j in range(4):
        nj = np.linalg.norm(x[:, 32 * j:32 * j + 32], axis=1)
        assert np.allclose(q["scale"][:, j].astype(np.float64), nj, rtol=1e-3)


# ---------------------------------------------------------------- zero / packing
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_zero_vector(bits):
    L = O.Layout(64, 32, bits)
    x = np.zeros((2, 64))
    codes, scale, _, _ = O.encode(x, L)
    assert np.all(O.unpack_codes(codes, bits, 64) == (1 << (bits - 1)) - 1)
    assert np.all(scale == 0)
    assert np.all(O.dequantize(codes, scale, L) == 0.0)
    Lq = O.Layout(64, 64, bits, qjl_m=32)
    S = inputs.qjl_matrix(32, 64, 3)
    codes, scale, qb, rho = O.encode(x, Lq, S)
    assert np.all(O.unpack_qjl(qb, 32) == 1) and np.all(rho == 0)
    assert np.all(O.dequantize(codes, scale, Lq, qb, rho, S) == 0.0)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_pack_roundtrip(bits, d):
    codes = np.random.default_rng(bits * d).integers(0, 1 << bits, size=(17, d))
    p = O.pack_codes(codes, bits)
    assert p.shape == (17, d * bits // 8)
    assert np.array_equal(O.unpack_codes(p, bits, d), codes)
    # every bit of the packed bytes carries information: distinct codes
    # give distinct bytes (the map is a bijection on 32-code groups)
    flips = codes.copy()
    flips[:, 5] ^= 1
    assert not np.array_equal(O.pack_codes(flips, bits), p)


def _known_answer_codes(entry):
    i = np.arange(32)
    b = entry["bits"]
    if b == 3:
        return np.where(i < 24, i % 8, 7 - (i - 24))
    if b == 4:
        return i % 16
    if b == 2:
        return (i // 8) % 4 if "//" in entry["codes"] else i % 4
    return np.isin(i, [0, 9, 18, 27]).astype(np.int64)


def test_pack_known_answers():
    """Bytes worked out by hand from the layout definition in include/tq.h
    (not from the oracle): a misread of the definition shared by the oracle
    and the kernels would fail here."""
    g = _golden("packed_layout_known_answers.json")
    for e in g["groups"]:
        exp = np.array([int(x, 16) for x in e["bytes"]], dtype=np.uint8)
        codes = _known_answer_codes(e)
        assert np.array_equal(O.pack_codes(codes[None], e["bits"])[0], exp), e["bits"]
        assert np.array_equal(O.unpack_codes(exp[None], e["bits"], 32)[0], codes), e["bits"]
    q = g["qjl"]
    s = np.zeros((1, q["m"]), dtype=np.uint8)
    s[0, q["ones_at"]] = 1
    exp = np.array([int(x, 16) for x in q["bytes"]], dtype=np.uint8)
    assert np.array_equal(O.pack_qjl(s)[0], exp)
    assert np.array_equal(O.unpack_qjl(exp[None], q["m"])[0], s[0])


def test_prefill_attention_restriction():
    """The sampled form (query rows, one GQA group) equals the matching
    slice of the full result."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 8, 9, 16))
    Kd, Vd = rng.standard_normal((1, 2, 30, 16)), rng.standard_normal((1, 2, 30, 16))
    full = O.prefill_attention(q, Kd, Vd, 27, causal=True)
    rows = np.array([0, 4, 8])
    part = O.prefill_attention(q, Kd[:, 1:2], Vd[:, 1:2], 27, causal=True, rows=rows, group=(4, 4))
    assert np.allclose(part, full[:, 4:8][:, :, rows], atol=1e-13)


def test_qjl_pack_roundtrip():
    s = np.random.default_rng(0).integers(0, 2, size=(9, 128)).astype(np.uint8)
    assert np.array_equal(O.unpack_qjl(O.pack_qjl(s), 128), s)


def test_bytes_per_element_and_cache_size():
    g = _golden("pages_codec_figures.json")
    for name, bits in (("turbo3", 3), ("turbo4", 4)):
        L = O.Layout(256, 32, bits)
        per_elem = (L.code_bytes + 2 * L.nb) / L.d
        assert per_elem == g["bytes_per_element"][name]["bytes_per_element"]
        blk = g["bytes_per_element"][name]
        assert per_elem == blk["block_bytes"] / blk["block_values"]
    c = g["kv_cache_mib_131072"]
    elems = 2 * c["layers"] * c["kv_heads"] * c["head_dim"] * c["context"]   # K and V
    assert elems * 2 / 2 ** 20 == c["f16_mib"]
    assert elems * 0.5625 / 2 ** 20 == c["turbo4_mib"]
    assert elems * 0.4375 / 2 ** 20 == c["turbo3_mib"]


# ---------------------------------------------------------------- attention
def _loop_attention(qv, K, V, n, scale):
    s = [scale * sum(qv[i] * K[t][i] for i in range(len(qv))) for t in range(n)]
    mx = max(s)
    e = [math.exp(v - mx) for v in s]
    tot = sum(e)
    return [sum(e[t] * V[t][i] for t in range(n)) / tot for i in range(len(qv))]


def test_decode_attention_against_loops():
    B, Hq, Hkv, S, d = 2, 4, 2, 9, 8
    rng = np.random.default_rng(3)
    q = rng.standard_normal((B, Hq, d))
    K = rng.standard_normal((B, Hkv, S, d))
    V = rng.standard_normal((B, Hkv, S, d))
    kv_len = [9, 5]
    out = O.decode_attention(q, K, V, kv_len)
    for b in range(B):
        for h in range(Hq):
            ref = _loop_attention(q[b, h], K[b, h // 2], V[b, h // 2], kv_len[b], 1 / math.sqrt(d))
            assert np.allclose(out[b, h], ref, atol=1e-13)


def test_prefill_attention_against_loops():
    B, Hq, Hkv, ctx, Tq, d = 1, 4, 1, 11, 4, 8
    rng = np.random.default_rng(4)
    q = rng.standard_normal((B, Hq, Tq, d))
    K = rng.standard_normal((B, Hkv, ctx, d))
    V = rng.standard_normal((B, Hkv, ctx, d))
    out = O.prefill_attention(q, K, V, ctx, causal=True)
    for h in range(Hq):
        for i in range(Tq):
            n = ctx - Tq + i + 1
            ref = _loop_attention(q[0, h, i], K[0, 0], V[0, 0], n, 1 / math.sqrt(d))
            assert np.allclose(out[0, h, i], ref, atol=1e-13)
    full = O.prefill_attention(q, K, V, ctx, causal=False)
    assert np.allclose(full[0, :, -1], out[0, :, -1], atol=1e-13)


def test_attention_degenerate_cases():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 2, 8))
    V = rng.standard_normal((1, 1, 6, 8))
    K = np.repeat(rng.standard_normal((1, 1, 1, 8)), 6, axis=2)
    out = O.decode_attention(q, K, V)
    assert np.allclose(out[0, 0], V[0, 0].mean(axis=0), atol=1e-14)
    out1 = O.decode_attention(q, K, V, kv_len=[1])
    assert np.allclose(out1[0, 1], V[0, 0, 0], atol=1e-15)


# ---------------------------------------------------------------- Beta codebook
def test_beta_codebook_uniform_law_closed_form():
    """blk = 3: one coordinate of a random unit vector in R^3 is uniform on
    [-1, 1] (Archimedes), and the Lloyd-Max quantiser of a uniform law is
    the uniform one: centroids -1 + (2k + 1)/K."""
    for bits in (1, 2, 3, 4):
        K = 1 << bits
        c, b = O.lloyd_max_beta_codebook(bits, 3)
        assert np.max(np.abs(c - (-1.0 + (2.0 * np.arange(K) + 1.0) / K))) < 1e-12
        assert np.max(np.abs(b - (-1.0 + 2.0 * np.arange(1, K) / K))) < 1e-12


def test_beta_codebook_is_the_fixed_point_by_quadrature():
    """Centroids equal the conditional means of their cells under the density
    (1 - x^2)^((blk-3)/2), computed here by plain trapezoid quadrature (no
    incomplete beta function), and the codebook is symmetric."""
    for blk, bits in ((32, 3), (64, 4), (256, 2)):
        c, b = O.lloyd_max_beta_codebook(bits, blk)
        assert np.allclose(c, -c[::-1], atol=1e-15)
        edges = np.concatenate([[-1.0], b, [1.0]])
        for k in range(len(c)):
            x = np.linspace(edges[k], edges[k + 1], 200001)
            f = np.power(np.clip(1.0 - x * x, 0.0, None), 0.5 * (blk - 3))
            assert abs(np.trapezoid(x * f, x) / np.trapezoid(f, x) - c[k]) < 1e-9 * max(1.0, abs(c[k]) * 10)


def test_beta_codebook_tends_to_gaussian():
    """As blk grows, sqrt(blk) x a rotated coordinate tends to N(0, 1): the
    scaled Beta codebook approaches the Gaussian one, monotonically."""
    g, _ = O.lloyd_max_codebook(3, 1)
    errs = []
    for blk in (32, 256, 4096):
        c, _ = O.lloyd_max_beta_codebook(3, blk)
        errs.append(np.max(np.abs(c * np.sqrt(blk) - g)))
    assert errs[0] > errs[1] > errs[2]
    assert errs[2] < 2e-3


# ---------------------------------------------------------------- GGML-style blocks
def test_block_bytes_are_the_pages_ggml_types():
    """14 bytes per 32 values at 3 bits and 18 at 4 bits (llama.cpp-turboquant
    'GGML Types'), i.e. the pages' 0.4375 and 0.5625 bytes per element."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_codec_figures.json")))
    b = g["bytes_per_element"]
    assert O.block_bytes(3) == b["turbo3"]["block_bytes"] and O.block_bytes(4) == b["turbo4"]["block_bytes"]
    assert O.block_bytes(3) / 32 == b["turbo3"]["bytes_per_element"]


@pytest.mark.parametrize("d,blk,bits", [(128, 128, 3), (256, 128, 4), (128, 32, 3), (64, 64, 2), (128, 128, 1)])
def test_blocks_round_trip_and_replicate_the_norm(d, blk, bits):
    L = O.Layout(d, blk, bits, 0, 0, 1)
    x = np.random.default_rng(d + blk + bits).standard_normal((40, d))
    codes, scales, _, _ = O.encode(x, L)
    blocks = O.to_blocks(codes, scales, L)
    assert blocks.shape == (40, (d // 32) * O.block_bytes(bits))
    c2, s2 = O.from_blocks(blocks, L)
    assert np.array_equal(c2, codes) and np.array_equal(s2.view(np.uint16), scales.view(np.uint16))
    # every 32-value block of a rotation block carries that block's norm
    bb = O.block_bytes(bits)
    for j in range(d // 32):
        norm = blocks[:, j * bb].astype(np.uint16) | (blocks[:, j * bb + 1].astype(np.uint16) << 8)
        assert np.array_equal(norm.view(np.float16), scales.reshape(40, L.nb)[:, (32 * j) // blk])


# ---------------------------------------------------------------- 8-bit codes
def test_8bit_codebook_near_panter_dite():
    """High-resolution theory (Panter and Dite, 1951): the optimal quantiser of
    N(0, 1) at b bits has relative distortion -> (pi sqrt(3) / 2) 4^-b from
    below; the Lloyd-Max ratio is 0.53, 0.69, 0.81, 0.89 at 1-4 bits and must be
    within 2% of 1 at 8 bits."""
    pd = math.pi * math.sqrt(3) / 2 * 4.0 ** -8
    r = O.relative_distortion(8) / pd
    assert 0.98 < r < 1.0, r


def test_8bit_codebook_centroid_condition_by_quadrature():
    """Every centroid is the mean of its cell, checked by numerical
    integration (scipy quad), independent of the solver; symmetric codebook."""
    from scipy import integrate
    c, b = O.lloyd_max_codebook(8, 1)
    assert len(c) == 256 and np.allclose(c, -c[::-1], atol=0, rtol=0)
    phi = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    edges = [-math.inf] + list(b) + [math.inf]
    for k in (0, 1, 60, 127, 128, 200, 254, 255):
        lo, hi = edges[k], edges[k + 1]
        mass = integrate.quad(phi, lo, hi, epsabs=0, epsrel=1e-13)[0]
        first = integrate.quad(lambda x: x * phi(x), lo, hi, epsabs=0, epsrel=1e-13)[0]
        assert abs(first / mass - c[k]) < 1e-9, (k, first / mass, c[k])


def test_8bit_codes_pack_as_bytes():
    codes = np.random.default_rng(8).integers(0, 256, size=(10, 128))
    packed = O.pack_codes(codes, 8)
    assert packed.shape == (10, 128) and np.array_equal(O.unpack_codes(packed, 8, 128), codes)

"""GPU quantise / dequantise kernels against the float64 oracle, through
the C ABI."""
import numpy as np
import pytest
import torch

from oracle import tq_oracle as O
from turboquant_kv_cache_gb300 import inputs

from _parity import (DEQ_RTOL, compare_codes, compare_qjl, compare_scales, fp16_ulp_diff, rel_l2, to_np,
                     upload_packed)

pytestmark = pytest.mark.gpu


def _x(n, d, seed, dtype, heavy=False):
    x = (inputs.student_t((n, d), seed, 4.0, np.float32) if heavy else inputs.gaussian((n, d), seed, np.float32))
    x[3] = 0.0                       # a zero vector
    x[5] *= 300.0                    # a large one
    if n > 40:
        x[40, :32] = 0.0             # a zero 32-block inside a nonzero vector
    return x.astype(dtype)


CASES = [
    # d, block, bits, dtype, nc, qjl_m
    (128, 128, 3, np.float32, 0, 0),     # unit-vector round trip shape
    (128, 32, 3, np.float16, 0, 0),      # turbo3
    (128, 32, 4, np.float16, 0, 0),      # turbo4
    (64, 64, 4, np.float16, 0, 0),       # Llama-1B per-vector
    (64, 32, 4, np.float16, 0, 0),       # Llama-1B block-32
    (256, 32, 4, np.float16, 0, 0),      # d256 turbo4
    (256, 32, 3, np.float16, 0, 0),
    (256, 256, 2, np.float16, 0, 0),
    (128, 64, 1, np.float32, 0, 0),
    (128, 128, 2, np.float16, 1, 0),     # norm correction
    (64, 32, 3, np.float32, 1, 0),
    (128, 128, 2, np.float16, 0, 128),   # QJL keys
    (128, 128, 3, np.float32, 0, 64),
    (64, 64, 1, np.float16, 0, 32),
    (256, 256, 2, np.float16, 0, 256),
    (128, 128, 2, np.float16, 1, 128),   # QJL + norm correction
    (128, 32, 8, np.float16, 0, 0),      # 8-bit keys (k8v4)
    (64, 64, 8, np.float32, 0, 0),
    (256, 256, 8, np.float16, 1, 0),     # 8 bits + norm correction
]


@pytest.mark.parametrize("d,blk,bits,dt,nc,m", CASES)
def test_quantize_matches_oracle(tqlib, d, blk, bits, dt, nc, m):
    from turboquant_kv_cache_gb300 import binding as tb
    n = 1037                                   # ragged: not a multiple of any tile
    x = _x(n, d, 100 + d + bits + m, dt, heavy=(d == 256))
    S = inputs.qjl_matrix(m, d, 7) if m else None
    L = tb.make_layout(d, blk, bits, m, nc, 1)
    Lo = O.Layout(d, blk, bits, m, nc, 1)
    xg = torch.from_numpy(x).cuda()
    Sg = torch.from_numpy(S).cuda() if m else None
    pk = tb.tq_quantize_kv(L, xg, S=Sg)
    torch.cuda.synchronize()
    oq = O.quantize(x, Lo, S)
    n_code, rows = compare_codes(to_np(pk.codes), oq, Lo)
    assert n_code <= max(5, n * d // 10000)
    if not m or not nc:
        compare_scales(to_np(pk.scales)[~rows], oq["scale"][~rows])
    else:  # QJL + nc: the scale depends on every sign bit too
        compare_scales(to_np(pk.scales)[~rows], oq["scale"][~rows], max_frac=2e-2)
    if m:
        compare_qjl(to_np(pk.qjl), oq, Lo, rows)
        assert fp16_ulp_diff(to_np(pk.rnorm)[~rows], oq["rho"][~rows]).max() <= 1
    assert np.all(to_np(pk.scales)[3] == 0)


@pytest.mark.parametrize("d,blk,bits,dt,nc,m", CASES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_dequantize_matches_oracle(tqlib, d, blk, bits, dt, nc, m, out_dtype):
    from turboquant_kv_cache_gb300 import binding as tb
    n = 517
    x = _x(n, d, 200 + d + bits, np.float32)
    S = inputs.qjl_matrix(m, d, 9) if m else None
    Lo = O.Layout(d, blk, bits, m, nc, 3)
    codes, scales, qb, rho = O.encode(x, Lo, S)
    ref = O.dequantize(codes, scales, Lo, qb, rho, S)
    L = tb.make_layout(d, blk, bits, m, nc, 3)
    pk = upload_packed(tb, L, Lo, codes, scales, qb, rho, (n,), S=torch.from_numpy(S).cuda() if m else None)
    out = tb.tq_dequantize_kv(pk, out_dtype)
    torch.cuda.synchronize()
    got = to_np(out.float())
    err = rel_l2(got, ref)
    tol = DEQ_RTOL if out_dtype == torch.float16 else 1e-5
    assert err.max() < tol, err.max()
    assert np.all(got[3] == 0)


def _golden(name):
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


@pytest.mark.parametrize("idx", range(5))
def test_dequantize_reads_known_answer_bytes(tqlib, idx):
    """The GPU reads the hand-derived bytes of the packed layout
    (tests/golden/packed_layout_known_answers.json, worked out from the
    definition in include/tq.h) as the codes they encode: dequantising
    records made of those groups gives scale * D (H c(code)) per 32-block,
    formed here from the oracle's signs, Hadamard matrix and codebook."""
    from turboquant_kv_cache_gb300 import binding as tb
    e = _golden("packed_layout_known_answers.json")["groups"][idx]
    bits, d = e["bits"], 128
    i = np.arange(32)
    if bits == 3:
        codes = np.where(i < 24, i % 8, 7 - (i - 24))
    elif bits == 4:
        codes = i % 16
    elif bits == 2:
        codes = (i // 8) % 4 if "//" in e["codes"] else i % 4
    else:
        codes = np.isin(i, [0, 9, 18, 27]).astype(np.int64)
    group = np.array([int(x, 16) for x in e["bytes"]], dtype=np.uint8)
    n = 3
    rec = np.tile(group, (n, d // 32))                          # every 32-block of every record
    scales = np.array([[1.0, 0.5, 2.0, 0.25]] * n, dtype=np.float16) * np.arange(1, n + 1, dtype=np.float16)[:, None]
    L = tb.make_layout(d, 32, bits, 0, 0, 7)
    Lo = O.Layout(d, 32, bits, 0, 0, 7)
    pk = tb.PackedKV(L, (n,))
    pk.codes.copy_(torch.from_numpy(rec))
    pk.scales.copy_(torch.from_numpy(scales))
    got = to_np(tb.tq_dequantize_kv(pk, torch.float32))
    cent, _ = O.codebook_for(Lo)
    H = O.hadamard_matrix(32)
    D = O.sign_vector(7, d)
    ref = np.zeros((n, d))
    for r in range(n):
        for j in range(d // 32):
            ref[r, 32 * j:32 * j + 32] = float(scales[r, j]) * D[32 * j:32 * j + 32] * (H @ np.asarray(cent)[codes])
    assert np.abs(got - ref).max() < 1e-5 * max(1.0, np.abs(ref).max())


def test_roundtrip_unit_vectors_mse(tqlib):
    """4096 unit vectors, d=128, 3 bits: GPU quantise -> GPU dequantise MSE
    against the oracle's closed-form distortion (3-bit: 0.0345)."""
    from turboquant_kv_cache_gb300 import binding as tb
    w = inputs.unit_roundtrip_workload()
    x = torch.from_numpy(w["x"]).cuda()
    L = tb.make_layout(128, 128, 3, 0, 0, 1)
    pk = tb.tq_quantize_kv(L, x)
    xr = tb.tq_dequantize_kv(pk, torch.float32)
    mse = float(((xr - x) ** 2).sum(dim=1).mean())
    assert abs(mse - O.relative_distortion(3)) / O.relative_distortion(3) < 0.05


def test_quantize_row_stride_and_alignment(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    base = torch.from_numpy(inputs.gaussian((64, 256), 5, np.float16)).cuda()
    x = base[:, :128]                          # row stride 256 elements
    L = tb.make_layout(128, 32, 3, 0, 0, 1)
    a = tb.tq_quantize_kv(L, x)
    b = tb.tq_quantize_kv(L, x.contiguous())
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    with pytest.raises(tb.TQError) as e:
        tb.tq_quantize_kv(L, base.reshape(-1)[1:1 + 128 * 63].reshape(63, 128))
    assert e.value.status == -3


APPEND_CASES = [
    # d, block, bits, dtype, nc, qjl_m  (fast, general and QJL quantise kernels)
    (128, 32, 3, np.float16, 0, 0),
    (64, 64, 4, np.float16, 0, 0),
    (128, 64, 1, np.float32, 0, 0),
    (128, 128, 2, np.float16, 1, 0),
    (128, 128, 2, np.float16, 0, 128),
    (128, 128, 3, np.float32, 0, 64),
    (128, 32, 8, np.float16, 0, 0),
]


@pytest.mark.parametrize("d,blk,bits,dt,nc,m", APPEND_CASES)
def test_append_into_cache_matches_oracle(tqlib, d, blk, bits, dt, nc, m):
    """tq_append_kv writes token j of (b, h) to slot pos[b] + j of a
    [B, H, S_cap] cache: the records equal tq_quantize_kv of the same rows
    (and the oracle), slots past S_cap and every other slot stay as they
    were."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, H, n_new, S_cap = 3, 2, 5, 40
    pos = np.array([0, 17, 37], dtype=np.int32)          # the last batch runs past the end
    x = _x(B * H * n_new, d, 300 + d + bits + m, dt).reshape(B, H, n_new, d)
    S = inputs.qjl_matrix(m, d, 7) if m else None
    L = tb.make_layout(d, blk, bits, m, nc, 1)
    Lo = O.Layout(d, blk, bits, m, nc, 1)
    Sg = torch.from_numpy(S).cuda() if m else None
    cache = tb.PackedKV(L, (B, H, S_cap), device="cuda", S=Sg)
    cache.codes.fill_(0xA5)
    cache.scales.view(torch.int16).fill_(0x1357)
    if m:
        cache.qjl.fill_(0x5A)
        cache.rnorm.view(torch.int16).fill_(0x2468)
    before = {k: to_np(v).copy() for k, v in (("codes", cache.codes), ("scales", cache.scales),
                                              ("qjl", cache.qjl), ("rnorm", cache.rnorm)) if v is not None}
    xg = torch.from_numpy(x).cuda()
    tb.tq_append_kv(cache, xg, torch.from_numpy(pos).cuda())
    ref = tb.tq_quantize_kv(L, xg.reshape(-1, d), S=Sg)
    torch.cuda.synchronize()
    written = np.zeros((B, H, S_cap), dtype=bool)
    rows, slots = [], []
    for b in range(B):
        for h in range(H):
            for j in range(n_new):
                s = pos[b] + j
                if s < S_cap:
                    written[b, h, s] = True
                    rows.append((b * H + h) * n_new + j)
                    slots.append((b, h, s))
    rows = np.array(rows)
    sl = tuple(np.array(slots).T)
    got = {k: to_np(v) for k, v in (("codes", cache.codes), ("scales", cache.scales),
                                    ("qjl", cache.qjl), ("rnorm", cache.rnorm)) if v is not None}
    refs = {k: to_np(v) for k, v in (("codes", ref.codes), ("scales", ref.scales),
                                     ("qjl", ref.qjl), ("rnorm", ref.rnorm)) if v is not None}
    for k in got:
        assert np.array_equal(got[k][sl], refs[k][rows]), k          # same kernel, same records
        assert np.array_equal(got[k][~written], before[k][~written]), k   # nothing else touched
    oq = O.quantize(x.reshape(-1, d)[rows], Lo, S)
    n_code, bad = compare_codes(got["codes"][sl], oq, Lo)
    assert n_code <= 5
    compare_scales(got["scales"][sl][~bad], oq["scale"][~bad], max_frac=2e-2 if (m and nc) else 1e-3)


def test_append_no_tokens_and_errors(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    L = tb.make_layout(128, 32, 3)
    cache = tb.PackedKV(L, (2, 2, 8), device="cuda")
    cache.codes.fill_(7)
    x = torch.zeros((2, 2, 0, 128), dtype=torch.float16, device="cuda")
    tb.tq_append_kv(cache, x, torch.zeros(2, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert bool((cache.codes == 7).all())
    with pytest.raises(ValueError):
        tb.tq_append_kv(cache, torch.zeros((2, 2, 1, 128), dtype=torch.float16, device="cuda"),
                        torch.zeros(2, dtype=torch.int64, device="cuda"))


BETA_CASES = [
    # d, block, bits, dtype, nc, qjl_m with the exact Beta codebook (kind 1)
    (128, 32, 3, np.float16, 0, 0),      # fast quantise kernel
    (64, 64, 4, np.float16, 0, 0),
    (256, 256, 2, np.float32, 1, 0),     # general kernel, norm correction
    (128, 128, 2, np.float16, 0, 128),   # QJL kernel
]


@pytest.mark.parametrize("d,blk,bits,dt,nc,m", BETA_CASES)
def test_beta_codebook_quantize_dequantize(tqlib, d, blk, bits, dt, nc, m):
    from turboquant_kv_cache_gb300 import binding as tb
    n = 777
    x = _x(n, d, 400 + d + bits + m, dt)
    S = inputs.qjl_matrix(m, d, 7) if m else None
    L = tb.make_layout(d, blk, bits, m, nc, 1, codebook=tb.CODEBOOK_BETA)
    Lo = O.Layout(d, blk, bits, m, nc, 1, codebook=1)
    Sg = torch.from_numpy(S).cuda() if m else None
    pk = tb.tq_quantize_kv(L, torch.from_numpy(x).cuda(), S=Sg)
    torch.cuda.synchronize()
    oq = O.quantize(x, Lo, S)
    n_code, rows = compare_codes(to_np(pk.codes), oq, Lo)
    assert n_code <= 5
    compare_scales(to_np(pk.scales)[~rows], oq["scale"][~rows], max_frac=2e-2 if (m and nc) else 1e-3)
    # the oracle's own encoding decoded on the GPU
    codes, scales, qb, rho = O.encode(x.astype(np.float64), Lo, S)
    ref = O.dequantize(codes, scales, Lo, qb, rho, S)
    up = upload_packed(tb, L, Lo, codes, scales, qb, rho, (n,), S=Sg)
    got = to_np(tb.tq_dequantize_kv(up, torch.float32))
    assert rel_l2(got, ref).max() < 1e-5


@pytest.mark.parametrize("d,blk,bits,cb", [(128, 128, 3, 1), (256, 128, 4, 1), (128, 32, 3, 0), (64, 64, 2, 0),
                                           (128, 128, 1, 1), (128, 32, 8, 0)])
def test_ggml_blocks_match_oracle(tqlib, d, blk, bits, cb):
    """tq_to_blocks / tq_from_blocks against the oracle's block bytes, byte
    for byte, on the library's own quantisation of seeded vectors (the
    128-chunk Beta layout is the llama.cpp-turboquant arrangement)."""
    from turboquant_kv_cache_gb300 import binding as tb
    L = tb.make_layout(d, blk, bits, 0, 0, 1, codebook=cb)
    Lo = O.Layout(d, blk, bits, 0, 0, 1, codebook=cb)
    x = torch.from_numpy(inputs.gaussian((3, 5, 70, d), 77)).cuda()
    pk = tb.tq_quantize_kv(L, x)
    blocks = tb.tq_to_blocks(pk)
    torch.cuda.synchronize()
    codes = pk.codes.reshape(-1, pk.codes.shape[-1]).cpu().numpy()
    scales = pk.scales.reshape(-1, pk.scales.shape[-1]).cpu().numpy()
    want = O.to_blocks(codes, scales, Lo)
    got = blocks.reshape(-1, (d // 32) * (2 + 4 * bits)).cpu().numpy()
    assert np.array_equal(got, want)
    back = tb.tq_from_blocks(L, blocks)
    torch.cuda.synchronize()
    assert torch.equal(back.codes, pk.codes) and torch.equal(back.scales, pk.scales)

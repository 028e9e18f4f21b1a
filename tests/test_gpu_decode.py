"""Fused decode attention (tq_decode_attn) against the oracle: the oracle
encodes the seeded K/V itself, the GPU attends over those packed bytes, and
the oracle attends over its own explicit dequantisation (no Hadamard-domain
shortcut), so the rotated-domain identities of the kernel are checked too."""
import math

import numpy as np
import pytest
import torch

from oracle import tq_oracle as O
from turboquant_kv_cache_gb300 import inputs

from _parity import ATTN_ATOL, to_np, upload_packed

pytestmark = pytest.mark.gpu


def _encode_cache(x, Lo, S=None):
    """x [B, H, S, d] -> oracle packed arrays and its dequantised cache."""
    B, H, Sc, d = x.shape
    flat = x.reshape(-1, d)
    codes, scales, qb, rho = O.encode(flat, Lo, S)
    deq = O.dequantize(codes, scales, Lo, qb, rho, S).reshape(B, H, Sc, d)
    return (codes, scales, qb, rho), deq


def _run(tb, cfgK, cfgV, B, Hq, Hkv, S_cap, ctx, d, kv_len=None, n_split=0, seed=0, heavy_k=False, S=None):
    Lk = O.Layout(d, *cfgK)
    Lv = O.Layout(d, *cfgV)
    k = (inputs.student_t((B, Hkv, S_cap, d), seed + 1, 4.0, np.float16) if heavy_k
         else inputs.gaussian((B, Hkv, S_cap, d), seed + 1))
    v = inputs.gaussian((B, Hkv, S_cap, d), seed + 2)
    q = inputs.gaussian((B, Hq, d), seed + 3)
    (kc, ks, kq, kr), kd = _encode_cache(k, Lk, S)
    (vc, vs, _, _), vd = _encode_cache(v, Lv)
    Sg = torch.from_numpy(S).cuda() if S is not None else None
    K = upload_packed(tb, tb.make_layout(d, *cfgK), Lk, kc, ks, kq, kr, (B, Hkv, S_cap), S=Sg)
    V = upload_packed(tb, tb.make_layout(d, *cfgV), Lv, vc, vs, None, None, (B, Hkv, S_cap))
    kvl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    out = tb.tq_decode_attn(K, V, torch.from_numpy(q).cuda(), ctx=ctx, kv_len=kvl, n_split=n_split)
    torch.cuda.synchronize()
    lens = kv_len if kv_len is not None else [ctx] * B
    ref = O.decode_attention(q, kd, vd, lens)
    return to_np(out.float()), ref, vd


CASES = [
    # name, K (block, bits, m, nc, seed), V (...), B, Hq, Hkv, S_cap, ctx, d
    ("turbo3_d128_gqa4", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 2, 8, 2, 700, 650, 128),
    ("turbo4k_turbo3v_d256", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 1, 8, 2, 530, 513, 256),
    ("pervec_d64_mha", (64, 4, 0, 0, 5), (32, 3, 0, 0, 6), 2, 2, 2, 300, 300, 64),
    ("pervec_nc_d128_gqa2", (128, 3, 0, 1, 2), (128, 2, 0, 1, 3), 1, 4, 2, 257, 257, 128),
    ("block64_d256_gqa8", (64, 3, 0, 0, 1), (64, 4, 0, 0, 2), 1, 8, 1, 200, 190, 256),
    ("bits1_d128", (32, 1, 0, 0, 1), (32, 2, 0, 0, 1), 1, 4, 1, 100, 97, 128),
    # exact Beta codebooks (codebook kind 1): the tensor-core and CUDA-core paths
    ("beta_turbo3_d128_gqa4", (32, 3, 0, 0, 1, 1), (32, 3, 0, 0, 1, 1), 2, 8, 2, 700, 650, 128),
    ("beta_pervec_d64", (64, 4, 0, 0, 5, 1), (64, 2, 0, 0, 6, 1), 1, 2, 2, 300, 280, 64),
    # 8-bit keys (one byte per code) beside 4- and 3-bit values
    ("k8v4_d128_gqa4", (32, 8, 0, 0, 1), (32, 4, 0, 0, 1), 2, 8, 2, 700, 650, 128),
    ("k8v4_d128_gqa4_long", (32, 8, 0, 0, 2), (32, 4, 0, 0, 3), 1, 8, 2, 2048, 2000, 128),
    ("k8v4_pervec_d64_mha", (64, 8, 0, 0, 5), (64, 4, 0, 0, 6), 1, 2, 2, 300, 280, 64),
    ("k8nc_v3_d256_gqa8", (256, 8, 0, 1, 2), (32, 3, 0, 0, 3), 1, 8, 1, 200, 190, 256),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,d", CASES)
@pytest.mark.parametrize("n_split", [0, 1, 7])
def test_decode_matches_oracle(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, d, n_split):
    from turboquant_kv_cache_gb300 import binding as tb
    got, ref, _ = _run(tb, cK, cV, B, Hq, Hkv, S_cap, ctx, d, n_split=n_split, heavy_k=(d == 256))
    err = np.abs(got - ref).max()
    assert err < ATTN_ATOL, (name, err)


TC_CASES = [
    # name, B, Hq, Hkv, S_cap, ctx, kv_len, n_split, heavy_k
    ("long_many_tiles", 2, 8, 2, 4100, 4097, None, 0, False),
    ("heavy_tailed_keys", 1, 8, 2, 3000, 2999, None, 3, True),
    ("ragged_splits", 3, 12, 3, 2050, 2050, [2050, 1000, 63], 6, False),
    ("odd_scap_generic_path", 1, 4, 1, 333, 333, None, 0, False),
]


@pytest.mark.parametrize("name,B,Hq,Hkv,S_cap,ctx,kv_len,n_split,heavy", TC_CASES)
def test_decode_turbo3_tensor_core_path(tqlib, name, B, Hq, Hkv, S_cap, ctx, kv_len, n_split, heavy):
    """turbo3 K/V, d=128, GQA 4: the shape of the fused tensor-core kernel."""
    from turboquant_kv_cache_gb300 import binding as tb
    got, ref, _ = _run(tb, (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), B, Hq, Hkv, S_cap, ctx, 128, kv_len=kv_len,
                       n_split=n_split, seed=7, heavy_k=heavy)
    err = np.abs(got - ref).max()
    assert err < ATTN_ATOL, (name, err)


def test_decode_qjl_keys(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    S = inputs.qjl_matrix(128, 128, 7)
    got, ref, _ = _run(tb, (128, 2, 128, 0, 1), (128, 3, 0, 0, 1), 2, 8, 2, 400, 391, 128, S=S)
    assert np.abs(got - ref).max() < ATTN_ATOL


def test_decode_ragged_kv_len_and_empty(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    got, ref, _ = _run(tb, (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 3, 8, 2, 520, 500, 128,
                       kv_len=[500, 37, 0], n_split=5)
    assert np.abs(got - ref).max() < ATTN_ATOL
    assert np.all(got[2] == 0)


def test_decode_single_token_returns_value(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    got, ref, vd = _run(tb, (32, 3, 0, 0, 1), (32, 4, 0, 0, 1), 1, 4, 1, 64, 1, 128)
    assert np.abs(got[0] - vd[0, 0, 0][None, :]).max() < ATTN_ATOL


def test_decode_workspace_errors(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    L = tb.make_layout(128, 32, 3)
    K = tb.PackedKV(L, (1, 1, 64))
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(tb.TQError) as e:
        tb.tq_decode_attn(K, K, q, ctx=64, workspace=small)
    assert e.value.status == -4
    with pytest.raises(tb.TQError) as e:
        tb.tq_decode_attn(K, K, q, ctx=65)
    assert e.value.status == -1


TC_LAYOUT_CASES = [
    # name, K (block, bits, m, nc, seed), V, B, Hq, Hkv, S_cap, ctx, kv_len, n_split, d, heavy_k
    ("d256_turbo4k_turbo3v", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 1, 8, 2, 3000, 2999, None, 0, 256, True),
    ("d256_turbo3_ragged", (32, 3, 0, 0, 1), (32, 3, 0, 0, 2), 2, 8, 2, 1030, 1029, [1029, 77], 4, 256, False),
    ("d256_bits2k", (32, 2, 0, 0, 3), (32, 3, 0, 0, 1), 1, 4, 1, 600, 600, None, 2, 256, False),
    ("d128_turbo4k", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 1, 8, 2, 1500, 1499, None, 0, 128, True),
    ("d128_bits2k_block32", (32, 2, 0, 0, 4), (32, 3, 0, 0, 1), 2, 8, 2, 900, 899, [899, 450], 3, 128, False),
    ("d128_turbo3k_pervec_v", (32, 3, 0, 0, 1), (128, 3, 0, 0, 2), 1, 8, 2, 1000, 1000, None, 0, 128, False),
    ("d128_pervec_2bit_k", (128, 2, 0, 0, 1), (128, 3, 0, 0, 1), 2, 8, 2, 1000, 999, [999, 1], 0, 128, True),
    ("d128_pervec_2bit_k_v32", (128, 2, 0, 0, 2), (32, 3, 0, 0, 1), 1, 4, 1, 800, 777, None, 4, 128, False),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,kv_len,n_split,d,heavy", TC_LAYOUT_CASES)
def test_decode_tensor_core_layouts(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, kv_len, n_split, d, heavy):
    """Every layout combination of the tensor-core decode kernel (GQA 4),
    several tiles, partial last steps, ragged lengths and split counts."""
    from turboquant_kv_cache_gb300 import binding as tb
    got, ref, _ = _run(tb, cK, cV, B, Hq, Hkv, S_cap, ctx, d, kv_len=kv_len, n_split=n_split, seed=11,
                       heavy_k=heavy)
    err = np.abs(got - ref).max()
    assert err < ATTN_ATOL, (name, err)


AUTO_SPLIT_CASES = [
    # the library's own split count (n_split 0) on the tensor-core kernel:
    # name, K (block, bits, m, nc, seed), V, B, Hq, Hkv, S_cap, ctx, kv_len, heavy_k
    ("turbo3_ragged", (32, 3, 0, 0, 1), (32, 3, 0, 0, 2), 3, 12, 3, 2050, 2050, [2050, 1000, 63], False),
    ("empty_and_short_units", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 3, 8, 2, 600, 600, [500, 0, 129], False),
    ("one_partial_step", (32, 3, 0, 0, 3), (32, 3, 0, 0, 4), 2, 8, 2, 100, 100, None, False),
    ("more_units_than_sms", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 16, 32, 8, 300, 300, None, False),
    ("turbo4k_heavy", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 1, 8, 2, 3000, 2999, None, True),
    ("bits2k", (32, 2, 0, 0, 5), (32, 3, 0, 0, 6), 2, 4, 1, 1030, 1029, [1029, 640], False),
    ("beta_codebook", (32, 3, 0, 0, 1, 1), (32, 3, 0, 0, 1, 1), 2, 8, 2, 1500, 1400, None, False),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,kv_len,heavy", AUTO_SPLIT_CASES)
def test_decode_auto_splits(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, kv_len, heavy):
    """Ragged and empty (batch, KV head) units, a single partial step, more
    units than SMs and every K width, at the library's own split count."""
    from turboquant_kv_cache_gb300 import binding as tb
    got, ref, _ = _run(tb, cK, cV, B, Hq, Hkv, S_cap, ctx, 128, kv_len=kv_len, n_split=0, seed=21, heavy_k=heavy)
    err = np.abs(got - ref).max()
    assert err < ATTN_ATOL, (name, err)
    if kv_len is not None and 0 in kv_len:
        assert np.all(got[kv_len.index(0)] == 0)


def test_decode_qjl_keys_long_ragged(tqlib):
    """QJL keys (2-bit + m=128 signs) with 3-bit per-vector values over many
    tiles, ragged lengths and splits: the tensor-core QJL path."""
    from turboquant_kv_cache_gb300 import binding as tb
    S = inputs.qjl_matrix(128, 128, 7)
    got, ref, _ = _run(tb, (128, 2, 128, 0, 1), (128, 3, 0, 0, 1), 2, 8, 2, 2000, 1999, 128,
                       kv_len=[1999, 333], n_split=5, S=S)
    assert np.abs(got - ref).max() < ATTN_ATOL


def test_append_and_decode_replay_in_a_cuda_graph(tqlib):
    """tq_append_kv + tq_decode_attn captured once in a CUDA graph and
    replayed with new inputs give the same bytes as the calls issued one by
    one (nothing in the calls allocates, synchronises or reads host state)."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, Hq, Hkv, d, S_cap = 2, 8, 2, 128, 512
    L = tb.make_layout(d, 32, 3, 0, 0, 1)
    k0 = torch.from_numpy(inputs.gaussian((B, Hkv, S_cap, d), 71)).cuda()
    v0 = torch.from_numpy(inputs.gaussian((B, Hkv, S_cap, d), 72)).cuda()

    def fresh():
        return tb.tq_quantize_kv(L, k0), tb.tq_quantize_kv(L, v0)

    def run(K, V, q, kn, vn, pos, ws, out):
        tb.tq_append_kv(K, kn, pos)
        tb.tq_append_kv(V, vn, pos)
        tb.tq_decode_attn(K, V, q, ctx=S_cap, workspace=ws, out=out)

    q = torch.empty((B, Hq, d), dtype=torch.float16, device="cuda")
    kn = torch.empty((B, Hkv, 1, d), dtype=torch.float16, device="cuda")
    vn = torch.empty_like(kn)
    pos = torch.full((B,), S_cap - 1, dtype=torch.int32, device="cuda")
    need, _ = tb.tq_decode_workspace_bytes(B, Hq, Hkv, d, S_cap, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    Kg, Vg = fresh()
    run(Kg, Vg, q.normal_(), kn.normal_(), vn.normal_(), pos, ws, out)   # warm-up outside capture
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(Kg, Vg, q, kn, vn, pos, ws, out)
    for seed in (5, 6):
        torch.manual_seed(seed)
        q.normal_(); kn.normal_(); vn.normal_()
        Ke, Ve = fresh()
        oe = torch.empty_like(q)
        run(Ke, Ve, q, kn, vn, pos, ws.clone(), oe)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, oe)
        assert torch.equal(Kg.codes[:, :, S_cap - 1], Ke.codes[:, :, S_cap - 1])


WINDOW_CASES = [
    # fp16 residual window: name, K (block, bits, m, nc, seed), V, B, Hq, Hkv, S_cap, ctx, kv_len, d, W_cap,
    # win_len (None: every batch W_cap), qjl
    ("turbo3_d128_tc", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 2, 8, 2, 700, 650, [650, 300], 128, 128, [128, 5],
     False),
    ("empty_cache_or_window", (32, 3, 0, 0, 1), (32, 3, 0, 0, 2), 3, 8, 2, 300, 300, [0, 300, 0], 128, 40,
     [40, 0, 0], False),
    ("pervec_d64_cuda_core", (64, 4, 0, 0, 5), (64, 3, 0, 0, 6), 2, 2, 2, 200, 190, None, 64, 64, None, False),
    ("d256_turbo4k_tc", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 1, 8, 2, 530, 513, None, 256, 32, [17], False),
    ("block64_v_gqa8", (64, 3, 0, 0, 1), (64, 4, 0, 0, 2), 1, 8, 1, 200, 190, None, 256, 96, None, False),
    ("qjl_keys", (128, 2, 128, 0, 1), (128, 3, 0, 0, 1), 2, 8, 2, 400, 391, [391, 100], 128, 64, [64, 33], True),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,kv_len,d,W_cap,win_len,qjl", WINDOW_CASES)
def test_decode_with_fp16_window(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, kv_len, d, W_cap, win_len, qjl):
    """tq_decode_attn_window against the oracle's attention over the
    decoded cache tokens followed by the exact fp16 window tokens."""
    from turboquant_kv_cache_gb300 import binding as tb
    S = inputs.qjl_matrix(128, 128, 7) if qjl else None
    Lk, Lv = O.Layout(d, *cK), O.Layout(d, *cV)
    k = inputs.gaussian((B, Hkv, S_cap, d), 41)
    v = inputs.gaussian((B, Hkv, S_cap, d), 42)
    q = inputs.gaussian((B, Hq, d), 43)
    kw = inputs.gaussian((B, Hkv, W_cap, d), 44)
    vw = inputs.gaussian((B, Hkv, W_cap, d), 45)
    (kc, ks, kq, kr), kd = _encode_cache(k, Lk, S)
    (vc, vs, _, _), vd = _encode_cache(v, Lv)
    Sg = torch.from_numpy(S).cuda() if S is not None else None
    K = upload_packed(tb, tb.make_layout(d, *cK), Lk, kc, ks, kq, kr, (B, Hkv, S_cap), S=Sg)
    V = upload_packed(tb, tb.make_layout(d, *cV), Lv, vc, vs, None, None, (B, Hkv, S_cap))
    kvl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    wl = torch.tensor(win_len, dtype=torch.int32, device="cuda") if win_len is not None else None
    out = tb.tq_decode_attn_window(K, V, torch.from_numpy(q).cuda(), torch.from_numpy(kw).cuda(),
                                   torch.from_numpy(vw).cuda(), ctx=ctx, kv_len=kvl, win_len=wl)
    torch.cuda.synchronize()
    lens = kv_len if kv_len is not None else [ctx] * B
    wls = win_len if win_len is not None else [W_cap] * B
    n_all = [lens[b] + wls[b] for b in range(B)]
    Kc = np.zeros((B, Hkv, max(max(n_all), 1), d))
    Vc = np.zeros_like(Kc)
    for b in range(B):
        Kc[b, :, :lens[b]] = kd[b, :, :lens[b]]
        Vc[b, :, :lens[b]] = vd[b, :, :lens[b]]
        Kc[b, :, lens[b]:n_all[b]] = kw[b, :, :wls[b]].astype(np.float64)
        Vc[b, :, lens[b]:n_all[b]] = vw[b, :, :wls[b]].astype(np.float64)
    ref = O.decode_attention(q, Kc, Vc, n_all)
    got = to_np(out.float())
    err = np.abs(got - ref).max()
    assert err < ATTN_ATOL, (name, err)
    for b in range(B):
        if n_all[b] == 0:
            assert np.all(got[b] == 0)


def test_decode_window_argument_errors(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    L = tb.make_layout(128, 32, 3)
    K = tb.PackedKV(L, (1, 2, 64))
    q = torch.zeros(1, 8, 128, dtype=torch.float16, device="cuda")
    kw = torch.zeros(1, 2, 16, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(tb.TQError) as e:   # more window tokens than slots
        tb.tq_decode_attn_window(K, K, q, kw, kw, ctx=64, win=17)
    assert e.value.status == -1
    with pytest.raises(ValueError):
        tb.tq_decode_attn_window(K, K, q, kw, kw[:, :, :8], ctx=64)


QJL_V_CASES = [
    # QJL residual on V: name, K (block, bits, m, nc, seed), V, B, Hq, Hkv, S_cap, ctx, kv_len, d
    ("v2bit_qjl_gqa4", (32, 3, 0, 0, 1), (128, 2, 128, 0, 2), 2, 8, 2, 400, 391, [391, 100], 128),
    ("qjl_k_and_v", (128, 2, 128, 0, 1), (128, 2, 128, 0, 3), 2, 8, 2, 300, 300, None, 128),
    ("v3bit_qjl64_nc_d64", (64, 3, 0, 0, 4), (64, 3, 64, 1, 5), 1, 2, 2, 260, 257, None, 64),
    ("v1bit_qjl_d256_gqa8", (32, 4, 0, 0, 1), (256, 1, 128, 0, 6), 1, 8, 1, 150, 150, None, 256),
    # on the tensor-core decode (4 q heads per KV head, head_dim 128, 2-bit per-vector K with or without
    # QJL, 2/3-bit per-vector V with m = 128, row pitches a multiple of 16 bytes): ragged lengths, one
    # empty row, several steps per split
    ("qjl_k_and_v_tc", (128, 2, 128, 0, 1), (128, 2, 128, 0, 3), 2, 8, 2, 320, 300, [300, 177], 128),
    ("v2bit_qjl_kpv2_tc", (128, 2, 0, 0, 1), (128, 2, 128, 0, 2), 1, 16, 4, 400, 391, None, 128),
    ("v3bit_qjl_tc", (128, 2, 128, 0, 1), (128, 3, 128, 0, 5), 2, 4, 1, 256, 256, [256, 0], 128),
    ("v3bit_qjl_nokq_long_tc", (128, 2, 0, 0, 4), (128, 3, 128, 0, 6), 1, 8, 2, 2048, 2000, None, 128),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,kv_len,d", QJL_V_CASES)
@pytest.mark.parametrize("n_split", [0, 5])
def test_decode_qjl_values(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, kv_len, d, n_split):
    """Values with a QJL residual: the oracle dequantises V with its QJL term
    (rho sqrt(pi/2)/m S^T (2s - 1), times the norm) and attends; the kernel
    sums the signs per split and applies S^T once."""
    from turboquant_kv_cache_gb300 import binding as tb
    Lk, Lv = O.Layout(d, *cK), O.Layout(d, *cV)
    Sk = inputs.qjl_matrix(Lk.m, d, 7) if Lk.m else None
    Sv = inputs.qjl_matrix(Lv.m, d, 8)
    k = inputs.gaussian((B, Hkv, S_cap, d), 51)
    v = inputs.gaussian((B, Hkv, S_cap, d), 52)
    q = inputs.gaussian((B, Hq, d), 53)
    (kc, ks, kq, kr), kd = _encode_cache(k, Lk, Sk)
    (vc, vs, vq, vr), vd = _encode_cache(v, Lv, Sv)
    K = upload_packed(tb, tb.make_layout(d, *cK), Lk, kc, ks, kq, kr, (B, Hkv, S_cap),
                      S=torch.from_numpy(Sk).cuda() if Sk is not None else None)
    V = upload_packed(tb, tb.make_layout(d, *cV), Lv, vc, vs, vq, vr, (B, Hkv, S_cap), S=torch.from_numpy(Sv).cuda())
    kvl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    out = tb.tq_decode_attn(K, V, torch.from_numpy(q).cuda(), ctx=ctx, kv_len=kvl, n_split=n_split)
    torch.cuda.synchronize()
    ref = O.decode_attention(q, kd, vd, kv_len if kv_len is not None else [ctx] * B)
    err = np.abs(to_np(out.float()) - ref).max()
    assert err < ATTN_ATOL, (name, err)


BLOCK_CASES = [
    # name, K (block, bits, m, nc, seed[, codebook]), V (...), B, Hq, Hkv, S_cap, ctx, kv_len, d
    # the llama.cpp arrangement: 128-value chunks, Beta codebook of a chunk, 14/18-byte blocks
    ("llama_turbo3_d128_gqa4", (128, 3, 0, 0, 1, 1), (128, 3, 0, 0, 2, 1), 2, 8, 2, 300, 290, None, 128),
    ("llama_turbo4_d256_halves_gqa8", (128, 4, 0, 0, 3, 1), (128, 4, 0, 0, 4, 1), 1, 8, 1, 150, 150, None, 256),
    ("b32_turbo4k_turbo3v_d256_gqa2", (32, 4, 0, 0, 1), (32, 3, 0, 0, 2), 1, 4, 2, 200, 199, None, 256),
    ("b64_2bit_nc_k_1bit_v_d64_mha", (64, 2, 0, 1, 5), (32, 1, 0, 0, 6), 2, 2, 2, 100, 97, [97, 0], 64),
    # on the tensor-core decode (4 q heads per KV head, 32-value blocks, 3-bit V, 16-byte row pitch): the
    # same kernel as the packed layout, so the two outputs are the same bytes
    ("b32_turbo3_d128_gqa4_tc", (32, 3, 0, 0, 1), (32, 3, 0, 0, 2), 2, 8, 2, 320, 300, [300, 177], 128),
    ("b32_turbo4k_turbo3v_d256_gqa4_tc", (32, 4, 0, 0, 1), (32, 3, 0, 0, 2), 1, 16, 4, 200, 199, None, 256),
    ("b32_2bit_k_d128_gqa4_tc", (32, 2, 0, 0, 3), (32, 3, 0, 0, 4), 1, 4, 1, 96, 96, [0], 128),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,kv_len,d", BLOCK_CASES)
@pytest.mark.parametrize("n_split", [0, 3])
def test_decode_over_blocks(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, kv_len, d, n_split):
    """tq_decode_attn_blocks reads the oracle's own block bytes (its
    quantisation, its to_blocks): the result matches the oracle's attention
    over its dequantised cache, and the packed-layout decode of the same codes."""
    from turboquant_kv_cache_gb300 import binding as tb
    Lk, Lv = O.Layout(d, *cK), O.Layout(d, *cV)
    k = inputs.gaussian((B, Hkv, S_cap, d), 31)
    v = inputs.gaussian((B, Hkv, S_cap, d), 32)
    q = inputs.gaussian((B, Hq, d), 33)
    (kc, ks, _, _), kd = _encode_cache(k, Lk)
    (vc, vs, _, _), vd = _encode_cache(v, Lv)
    kb = O.to_blocks(kc, ks, Lk).reshape(B, Hkv, S_cap, d // 32, 2 + 4 * Lk.bits)
    vb = O.to_blocks(vc, vs, Lv).reshape(B, Hkv, S_cap, d // 32, 2 + 4 * Lv.bits)
    tLk, tLv = tb.make_layout(d, *cK), tb.make_layout(d, *cV)
    kvl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    qg = torch.from_numpy(q).cuda()
    got = tb.tq_decode_attn_blocks(tLk, torch.from_numpy(kb).cuda(), tLv, torch.from_numpy(vb).cuda(), qg,
                                   ctx=ctx, kv_len=kvl, n_split=n_split)
    K = upload_packed(tb, tLk, Lk, kc, ks, None, None, (B, Hkv, S_cap))
    V = upload_packed(tb, tLv, Lv, vc, vs, None, None, (B, Hkv, S_cap))
    packed = tb.tq_decode_attn(K, V, qg, ctx=ctx, kv_len=kvl, n_split=n_split)
    torch.cuda.synchronize()
    lens = kv_len if kv_len is not None else [ctx] * B
    ref = O.decode_attention(q, kd, vd, lens)
    got = to_np(got.float())
    assert np.abs(got - ref).max() < ATTN_ATOL, (name, np.abs(got - ref).max())
    if name.endswith("_tc"):
        assert np.array_equal(got, to_np(packed.float())), name
    else:
        assert np.abs(got - to_np(packed.float())).max() <= 1e-3
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(got[b] == 0)

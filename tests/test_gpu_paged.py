"""Paged caches: the same packed records scattered into pages (shuffled
page order, spare pages, page sizes from 32 to 512 tokens) must give the
same bytes out of every kernel as the contiguous cache they came from:
decode on the tensor-core and CUDA-core paths, QJL keys, the static decode,
prefill, and tq_append_kv writing new tokens across page boundaries."""
import numpy as np
import pytest
import torch

from oracle import tq_oracle as O
from turboquant_kv_cache_gb300 import inputs

from _parity import ATTN_ATOL, to_np, upload_packed

pytestmark = pytest.mark.gpu


def _page_table(B, pages_per_seq, spare, seed):
    """A shuffled page table [B, pages_per_seq] over B * pages_per_seq +
    spare pages (the spare ones stay unused)."""
    n_pages = B * pages_per_seq + spare
    perm = np.random.default_rng(seed).permutation(n_pages)[:B * pages_per_seq]
    return torch.from_numpy(perm.reshape(B, pages_per_seq).astype(np.int32)).cuda(), n_pages


def _to_paged(tb, C, table, n_pages, page_size, S=None):
    """Scatter a contiguous [B, H, S_cap] PackedKV into pages."""
    B, H, S_cap = C.lead_shape
    pps = table.shape[1]
    P = tb.PackedKV(C.layout, (n_pages, H, page_size), S=S if S is not None else C.S, page_table=table)
    tab = table.cpu().numpy()
    for name in ("codes", "scales", "qjl", "rnorm"):
        src, dst = getattr(C, name), getattr(P, name)
        if src is None:
            continue
        dst.zero_()
        for b in range(B):
            for j in range(pps):
                lo, hi = j * page_size, min((j + 1) * page_size, S_cap)
                if lo < hi:
                    dst[int(tab[b, j]), :, :hi - lo] = src[b, :, lo:hi]
    return P


def _cache(tb, cfg, B, H, S_cap, d, seed, S=None, heavy=False):
    L = O.Layout(d, *cfg)
    x = (inputs.student_t((B, H, S_cap, d), seed, 4.0, np.float16) if heavy
         else inputs.gaussian((B, H, S_cap, d), seed))
    c, s, qb, rho = O.encode(x.reshape(-1, d), L, S)
    Sg = torch.from_numpy(S).cuda() if S is not None else None
    return upload_packed(tb, tb.make_layout(d, *cfg), L, c, s, qb, rho, (B, H, S_cap), S=Sg)


DECODE_CASES = [
    # name, K (block, bits, m, nc, seed), V, B, Hq, Hkv, S_cap, ctx, kv_len, n_split, d, page_size, qjl
    ("tc_turbo3_d128_p32", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 2, 8, 2, 2048, 2000, [2000, 777], 0, 128, 32, False),
    ("tc_turbo3_d128_p96_split_kernel", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 2, 8, 2, 960, 900, [900, 500], 3, 128,
     96, False),
    ("tc_turbo3_d128_p128_empty_batch", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 3, 8, 2, 1024, 1000, [1000, 130, 0], 0, 128,
     128, False),
    ("tc_turbo4k_d128_p256", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 2, 8, 2, 2048, 2048, None, 0, 128, 256,
     False),
    ("tc_turbo3_d128_p256", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 3, 8, 2, 4096, 4096, [4096, 1, 2500], 5, 128, 256,
     False),
    ("tc_d256_turbo4k_p64", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 1, 8, 2, 1536, 1500, None, 0, 256, 64, False),
    ("tc_qjl_keys_p128", (128, 2, 128, 0, 1), (128, 3, 0, 0, 1), 2, 8, 2, 1024, 1000, [1000, 333], 3, 128, 128,
     True),
    # QJL on the values too: the tensor-core kernel's sign and rho streams come from the pages as well
    ("tc_qjl_keys_values_p64", (128, 2, 128, 0, 1), (128, 2, 128, 0, 3), 2, 8, 2, 1024, 1000, [1000, 333], 0, 128,
     64, True),
    ("cuda_core_pervec_d64_p32", (64, 4, 0, 0, 5), (64, 3, 0, 0, 6), 2, 2, 2, 320, 300, [300, 31], 0, 64, 32, False),
    ("cuda_core_gqa2_d128_p512", (32, 3, 0, 0, 1), (32, 2, 0, 0, 2), 1, 4, 2, 1024, 1024, None, 2, 128, 512, False),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,kv_len,n_split,d,page_size,qjl", DECODE_CASES)
def test_paged_decode_matches_contiguous(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, kv_len, n_split, d,
                                         page_size, qjl):
    from turboquant_kv_cache_gb300 import binding as tb
    S = inputs.qjl_matrix(cK[2], d, 7) if qjl else None
    Sv = inputs.qjl_matrix(cV[2], d, 8) if cV[2] else None
    K = _cache(tb, cK, B, Hkv, S_cap, d, 101, S=S, heavy=(d == 256))
    V = _cache(tb, cV, B, Hkv, S_cap, d, 102, S=Sv)
    table, n_pages = _page_table(B, S_cap // page_size, 3, 5)
    Kp = _to_paged(tb, K, table, n_pages, page_size)
    Vp = _to_paged(tb, V, table, n_pages, page_size)
    q = torch.from_numpy(inputs.gaussian((B, Hq, d), 103)).cuda()
    kvl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    ref = tb.tq_decode_attn(K, V, q, ctx=ctx, kv_len=kvl, n_split=n_split)
    got = tb.tq_decode_attn(Kp, Vp, q, ctx=ctx, kv_len=kvl, n_split=n_split)
    stat = tb.tq_decode_attn_static(Kp, Vp, q, ctx=ctx, kv_len=kvl, n_split=n_split)
    torch.cuda.synchronize()
    assert torch.equal(got, ref), name
    assert torch.equal(stat, ref), name


def test_paged_decode_matches_oracle(tqlib):
    """The paged tensor-core decode against the oracle directly (not only
    against the contiguous kernel)."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, Hq, Hkv, S_cap, d, ps = 2, 8, 2, 1024, 128, 64
    Lo = O.Layout(d, 32, 3, 0, 0, 1)
    k = inputs.gaussian((B, Hkv, S_cap, d), 111)
    v = inputs.gaussian((B, Hkv, S_cap, d), 112)
    q = inputs.gaussian((B, Hq, d), 113)
    kc, ks, _, _ = O.encode(k.reshape(-1, d), Lo)
    vc, vs, _, _ = O.encode(v.reshape(-1, d), Lo)
    kd = O.dequantize(kc, ks, Lo).reshape(B, Hkv, S_cap, d)
    vd = O.dequantize(vc, vs, Lo).reshape(B, Hkv, S_cap, d)
    Lc = tb.make_layout(d, 32, 3, 0, 0, 1)
    K = upload_packed(tb, Lc, Lo, kc, ks, None, None, (B, Hkv, S_cap))
    V = upload_packed(tb, Lc, Lo, vc, vs, None, None, (B, Hkv, S_cap))
    table, n_pages = _page_table(B, S_cap // ps, 0, 9)
    Kp, Vp = _to_paged(tb, K, table, n_pages, ps), _to_paged(tb, V, table, n_pages, ps)
    lens = [1000, 515]
    out = tb.tq_decode_attn(Kp, Vp, torch.from_numpy(q).cuda(), ctx=1000,
                            kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    ref = O.decode_attention(q, kd, vd, lens)
    assert np.abs(to_np(out.float()) - ref).max() < ATTN_ATOL


PREFILL_CASES = [
    # name, K, V, B, Hq, Hkv, S_cap, ctx, Tq, d, page_size
    ("d128_q100_p32", (32, 3, 0, 0, 1), (32, 3, 0, 0, 1), 2, 8, 2, 640, 600, 100, 128, 32),
    ("d256_q64_p128", (32, 4, 0, 0, 1), (32, 3, 0, 0, 1), 1, 8, 2, 1024, 1000, 64, 256, 128),
    ("d64_q5_p64", (64, 4, 0, 0, 2), (64, 3, 0, 0, 3), 2, 2, 2, 256, 200, 5, 64, 64),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,Tq,d,page_size", PREFILL_CASES)
@pytest.mark.parametrize("causal", [True, False])
def test_paged_prefill_matches_contiguous(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, Tq, d, page_size, causal):
    from turboquant_kv_cache_gb300 import binding as tb
    K = _cache(tb, cK, B, Hkv, S_cap, d, 121, heavy=(d == 256))
    V = _cache(tb, cV, B, Hkv, S_cap, d, 122)
    table, n_pages = _page_table(B, S_cap // page_size, 2, 13)
    Kp = _to_paged(tb, K, table, n_pages, page_size)
    Vp = _to_paged(tb, V, table, n_pages, page_size)
    q = torch.from_numpy(inputs.gaussian((B, Hq, Tq, d), 123)).cuda()
    ref = tb.tq_prefill_attn(K, V, q, ctx, causal=causal)
    got = tb.tq_prefill_attn(Kp, Vp, q, ctx, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(got, ref), name


@pytest.mark.parametrize("cfg,d,n_new,page_size,qjl", [
    ((32, 3, 0, 0, 1), 128, 1, 32, False),
    ((32, 3, 0, 0, 1), 128, 70, 32, False),     # crosses several pages
    ((32, 4, 0, 0, 1), 256, 33, 64, False),
    ((128, 2, 128, 0, 1), 128, 40, 32, True),  # QJL keys
    ((64, 3, 0, 0, 2), 64, 9, 128, False),
])
def test_paged_append_matches_contiguous(tqlib, cfg, d, n_new, page_size, qjl):
    """tq_append_kv into a paged cache writes the same records as into the
    contiguous cache, each at its page's row; nothing else changes."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, H, S_cap = 3, 2, 4 * page_size
    S = torch.from_numpy(inputs.qjl_matrix(cfg[2], d, 17)).cuda() if qjl else None
    L = tb.make_layout(d, *cfg)
    C = tb.PackedKV(L, (B, H, S_cap), S=S)
    for t in (C.codes, C.scales, C.qjl, C.rnorm):
        if t is not None:
            t.zero_()
    table, n_pages = _page_table(B, S_cap // page_size, 2, 21)
    P = _to_paged(tb, C, table, n_pages, page_size, S=S)
    x = torch.from_numpy(inputs.gaussian((B, H, n_new, d), 22)).cuda()
    pos = torch.tensor([0, page_size - 1 if n_new < S_cap - page_size else 0, S_cap - n_new],
                       dtype=torch.int32, device="cuda")
    tb.tq_append_kv(C, x, pos)
    tb.tq_append_kv(P, x, pos)
    torch.cuda.synchronize()
    want = _to_paged(tb, C, table, n_pages, page_size, S=S)
    for name in ("codes", "scales", "qjl", "rnorm"):
        a, b = getattr(P, name), getattr(want, name)
        if a is not None:
            assert torch.equal(a, b), name


def test_paged_append_then_decode(tqlib):
    """A paged cache filled token by token (as a decoder does) and read back
    by decode equals the contiguous cache filled by one quantise."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, Hq, Hkv, d, ps, n_tok = 2, 8, 2, 128, 32, 100
    L = tb.make_layout(d, 32, 3, 0, 0, 1)
    k = torch.from_numpy(inputs.gaussian((B, Hkv, n_tok, d), 31)).cuda()
    v = torch.from_numpy(inputs.gaussian((B, Hkv, n_tok, d), 32)).cuda()
    table, n_pages = _page_table(B, 4, 1, 33)
    Kp = tb.PackedKV(L, (n_pages, Hkv, ps), page_table=table)
    Vp = tb.PackedKV(L, (n_pages, Hkv, ps), page_table=table)
    for t in range(n_tok):
        pos = torch.full((B,), t, dtype=torch.int32, device="cuda")
        tb.tq_append_kv(Kp, k[:, :, t:t + 1], pos)
        tb.tq_append_kv(Vp, v[:, :, t:t + 1], pos)
    Kc, Vc = tb.tq_quantize_kv(L, k), tb.tq_quantize_kv(L, v)
    q = torch.from_numpy(inputs.gaussian((B, Hq, d), 34)).cuda()
    got = tb.tq_decode_attn(Kp, Vp, q, ctx=n_tok)
    ref = tb.tq_decode_attn(Kc, Vc, q, ctx=n_tok)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


def test_paged_argument_errors(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    L = tb.make_layout(128, 32, 3)
    table = torch.zeros(1, 2, dtype=torch.int32, device="cuda")
    K = tb.PackedKV(L, (2, 1, 64), page_table=table)
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(tb.TQError) as e:  # ctx beyond pages_per_seq * page_size
        tb.tq_decode_attn(K, K, q, ctx=129)
    assert e.value.status == -1
    C = tb.PackedKV(L, (1, 1, 128))
    with pytest.raises(tb.TQError) as e:  # K paged, V contiguous
        tb.tq_decode_attn(K, C, q, ctx=64)
    assert e.value.status == -1
    with pytest.raises(ValueError):  # more sequences than the page table holds
        tb.tq_decode_attn(K, K, torch.zeros(2, 4, 128, dtype=torch.float16, device="cuda"), ctx=64)
    with pytest.raises(ValueError):
        tb.PackedKV(L, (2, 1, 64), page_table=table.to(torch.int64))

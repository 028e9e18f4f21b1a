"""tq_decode_attn_static: decode attention for callers that cannot allocate
device memory (their memory belongs to a host runtime's own pool, or an
allocation's implicit synchronisation is not acceptable on their hot path).
Its split partials live in the library's own fixed device array instead of a
caller workspace.  Given the same split count it runs the same kernels on
the same inputs as tq_decode_attn, so its output must be the same bytes.

This file is collected last on purpose; it must pass alone in a fresh
process as well as after every other test."""
import ctypes

import numpy as np
import pytest
import torch

from turboquant_kv_cache_gb300 import inputs

pytestmark = pytest.mark.gpu


def _cache(tb, L, B, Hkv, S_cap, d, seed, S=None):
    x = torch.from_numpy(inputs.gaussian((B, Hkv, S_cap, d), seed)).cuda()
    return tb.tq_quantize_kv(L, x, S=S)


def _page_table(B, pps, seed):
    """A shuffled page table [B, pps] over B * pps + 2 pages (two spare)."""
    n_pages = B * pps + 2
    perm = np.random.default_rng(seed).permutation(n_pages)[:B * pps].reshape(B, pps)
    return torch.from_numpy(perm.astype(np.int32)).cuda(), perm, n_pages


def _to_paged(tb, C, table, perm, n_pages, page_size):
    """The records of a contiguous [B, H, S_cap] cache scattered into the
    pages of one table (K and V of a call share their table)."""
    B, H, S_cap = C.lead_shape
    pps = S_cap // page_size
    P = tb.PackedKV(C.layout, (n_pages, H, page_size), S=C.S, page_table=table)
    for name in ("codes", "scales", "qjl", "rnorm"):
        src, dst = getattr(C, name), getattr(P, name)
        if src is None:
            continue
        dst.zero_()
        for b in range(B):
            for j in range(pps):
                dst[int(perm[b, j]), :, :] = src[b, :, j * page_size:(j + 1) * page_size]
    return P


CASES = [
    # name, K (block, bits, m), V (block, bits), B, Hq, Hkv, S_cap, ctx, d, n_split, page_size
    ("tc_turbo3_gqa4", (32, 3, 0), (32, 3), 2, 8, 2, 700, 650, 128, 0, 0),
    ("tc_turbo4k_d256_gqa4", (32, 4, 0), (32, 3), 1, 16, 4, 2100, 2048, 256, 9, 0),
    ("cuda_core_gqa2", (32, 3, 0), (32, 3), 2, 4, 2, 800, 777, 128, 0, 0),
    ("cuda_core_gqa8", (64, 4, 0), (64, 2), 1, 16, 2, 640, 600, 64, 5, 0),
    ("qjl_keys_m128", (128, 2, 128), (128, 3), 2, 8, 2, 512, 500, 128, 3, 0),
    ("paged_tc_turbo3", (32, 3, 0), (32, 3), 2, 8, 2, 1024, 1000, 128, 0, 128),
]


@pytest.mark.parametrize("name,cK,cV,B,Hq,Hkv,S_cap,ctx,d,n_split,page_size", CASES)
def test_static_decode_matches_workspace_decode(tqlib, name, cK, cV, B, Hq, Hkv, S_cap, ctx, d, n_split, page_size):
    """Two calls in a row (the array keeps the first call's partials) give
    exactly the bytes of the workspace decode with the same split count."""
    from turboquant_kv_cache_gb300 import binding as tb
    Lk = tb.make_layout(d, cK[0], cK[1], cK[2], 0, 1)
    Lv = tb.make_layout(d, cV[0], cV[1], 0, 0, 1)
    S = torch.from_numpy(inputs.qjl_matrix(cK[2], d, 7)).cuda() if cK[2] else None
    K = _cache(tb, Lk, B, Hkv, S_cap, d, 41, S=S)
    V = _cache(tb, Lv, B, Hkv, S_cap, d, 42)
    if page_size:
        table, perm, n_pages = _page_table(B, S_cap // page_size, 3)
        K = _to_paged(tb, K, table, perm, n_pages, page_size)
        V = _to_paged(tb, V, table, perm, n_pages, page_size)
    kv_len = torch.tensor([ctx - 7 * b for b in range(B)], dtype=torch.int32, device="cuda")
    for call in range(2):
        q = torch.from_numpy(inputs.gaussian((B, Hq, d), 43 + call)).cuda()
        ref = tb.tq_decode_attn(K, V, q, ctx=ctx, kv_len=kv_len, n_split=n_split)
        got = tb.tq_decode_attn_static(K, V, q, ctx=ctx, kv_len=kv_len, n_split=n_split)
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all(), (name, call)
        assert torch.equal(got, ref), (name, call, (got.float() - ref.float()).abs().max().item())


def test_static_decode_refuses_oversized_partials(tqlib):
    """64 x 8 heads split 4096 ways needs more than the fixed array holds:
    refused with TQ_ERR_WORKSPACE before anything is launched."""
    from turboquant_kv_cache_gb300 import binding as tb
    L = tb.make_layout(128, 32, 3, 0, 0, 1)
    K = tb.PackedKV(L, (1, 1, 8))
    q = torch.zeros(64, 8, 128, dtype=torch.float16, device="cuda")
    need, _ = tb.tq_decode_workspace_bytes(64, 8, 1, 128, 8, 4096)
    assert need > (8 << 20)
    with pytest.raises(tb.TQError) as e:
        _static_raw(tb, tqlib, K, q, 64, 8, 1, 8, 4096)
    assert e.value.status == -4


def _static_raw(tb, lib, K, q, B, Hq, Hkv, ctx, n_split):
    kv = K.view()
    out = torch.empty_like(q)
    st = lib.tq_decode_attn_static(ctypes.byref(kv), ctypes.byref(kv), ctypes.c_void_p(q.data_ptr()), B, Hq, Hkv,
                                   K.lead_shape[2], None, ctx, 0.0, ctypes.c_void_p(out.data_ptr()), n_split,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != 0:
        raise tb.TQError(st, "tq_decode_attn_static")
    return out

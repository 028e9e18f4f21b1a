"""tq_decode_attn_static: decode attention for callers that cannot allocate
device memory (their memory belongs to a host runtime's own pool, or an
allocation's implicit synchronisation is not acceptable on their hot path).
Its split partials live in the library's own fixed device array instead of a
caller workspace.  This file is collected last on purpose; it must pass
alone in a fresh process as well as after every other test."""
import ctypes

import pytest
import torch

from turboquant_kv_cache_gb300 import inputs

from _parity import ATTN_ATOL

pytestmark = pytest.mark.gpu


def _cache(tb, L, B, Hkv, S_cap, d, seed):
    x = torch.from_numpy(inputs.gaussian((B, Hkv, S_cap, d), seed)).cuda()
    return tb.tq_quantize_kv(L, x)


@pytest.mark.parametrize("B,Hq,Hkv,S_cap,ctx,d,n_split", [
    (2, 8, 2, 700, 650, 128, 0),
    (1, 16, 4, 2100, 2048, 256, 9),
])
def test_static_decode_matches_workspace_decode(tqlib, B, Hq, Hkv, S_cap, ctx, d, n_split):
    from turboquant_kv_cache_gb300 import binding as tb
    Lk = tb.make_layout(d, 32, 4 if d == 256 else 3, 0, 0, 1)
    Lv = tb.make_layout(d, 32, 3, 0, 0, 1)
    K = _cache(tb, Lk, B, Hkv, S_cap, d, 41)
    V = _cache(tb, Lv, B, Hkv, S_cap, d, 42)
    kv_len = torch.tensor([ctx - 7 * b for b in range(B)], dtype=torch.int32, device="cuda")
    for call in range(2):                      # two calls in a row share the array
        q = torch.from_numpy(inputs.gaussian((B, Hq, d), 43 + call)).cuda()
        ref = tb.tq_decode_attn(K, V, q, ctx=ctx, kv_len=kv_len, n_split=n_split)
        got = tb.tq_decode_attn_static(K, V, q, ctx=ctx, kv_len=kv_len, n_split=n_split)
        torch.cuda.synchronize()
        err = (got.float() - ref.float()).abs().max().item()
        assert err < ATTN_ATOL, (call, err)
        assert torch.isfinite(got.float()).all()


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

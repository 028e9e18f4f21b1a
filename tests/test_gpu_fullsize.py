"""Full-size parity: the benchmark's workloads at their full sizes, launched
as bench.py launches them (same shapes, split counts and workspace), checked
against the oracle on sampled outputs.

The caches are filled on the GPU (tq_quantize_kv of seeded device data)
except the sampled (batch, KV head) slices, which hold the oracle's own
encoding of seeded host rows; the sampled output rows read only those
slices, so every byte the oracle compares against is its own.  The other
slices only give the launch its full size."""
import numpy as np
import pytest
import torch

from oracle import tq_oracle as O
from turboquant_kv_cache_gb300 import inputs

from _parity import ATTN_ATOL, to_np

pytestmark = pytest.mark.gpu


def _fill_gpu(tb, L, lead, seed, S=None, heavy=False):
    """A cache of lead shape [B, H, T] quantised on the GPU from seeded
    device draws, one batch row at a time."""
    B, H, T = lead
    d = L.head_dim
    C = tb.PackedKV(L, lead, S=S)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    for b in range(B):
        x = torch.randn((H, T, d), generator=g, device="cuda", dtype=torch.float32)
        if heavy:   # Student-t(4) from normal / sqrt(chi2_4 / 4)
            chi = torch.randn((4, H, T, d), generator=g, device="cuda").pow(2).sum(0) / 4.0
            x = x / chi.sqrt()
        part = tb.tq_quantize_kv(L, x.half(), S=S)
        for name in ("codes", "scales", "qjl", "rnorm"):
            if getattr(C, name) is not None:
                getattr(C, name)[b].copy_(getattr(part, name))
    return C


def _plant(C, Lo, b, h, x, S=None):
    """Overwrite slice (b, h) of a cache with the oracle's encoding of x
    [T, d]; returns the oracle's decoded slice [T, d] (float64)."""
    codes, scales, qb, rho = O.encode(x, Lo, S)
    C.codes[b, h].copy_(torch.from_numpy(codes))
    C.scales[b, h].copy_(torch.from_numpy(scales))
    if Lo.m:
        C.qjl[b, h].copy_(torch.from_numpy(qb))
        C.rnorm[b, h].copy_(torch.from_numpy(rho))
    return O.dequantize(codes, scales, Lo, qb, rho, S)


def test_headline_decode_full_size(tqlib):
    """Qwen3-8B-shaped turbo3 decode, B=8, Hq=32, Hkv=8, d=128, ctx=32768,
    with the library's own split count and an explicit workspace (the timed
    call); slices (0, 0) and (7, 5) against the oracle."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, Hq, Hkv, d, ctx = 8, 32, 8, 128, 32768
    L = tb.make_layout(d, 32, 3, 0, 0, 1)
    Lo = O.Layout(d, 32, 3, 0, 0, 1)
    K = _fill_gpu(tb, L, (B, Hkv, ctx), 1)
    V = _fill_gpu(tb, L, (B, Hkv, ctx), 2)
    q = inputs.gaussian((B, Hq, d), 10)
    samples = [(0, 0), (7, 5)]
    dec = {}
    for i, (b, h) in enumerate(samples):
        kd = _plant(K, Lo, b, h, inputs.gaussian((ctx, d), 900 + 2 * i))
        vd = _plant(V, Lo, b, h, inputs.gaussian((ctx, d), 901 + 2 * i))
        dec[(b, h)] = (kd, vd)
    ws_bytes, _ = tb.tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = tb.tq_decode_attn(K, V, torch.from_numpy(q).cuda(), ctx=ctx, workspace=ws)
    got = to_np(out.float())
    g = Hq // Hkv
    for (b, h), (kd, vd) in dec.items():
        ref = O.decode_attention(q[b:b + 1, h * g:(h + 1) * g], kd[None, None], vd[None, None])[0]
        err = np.abs(got[b, h * g:(h + 1) * g] - ref).max()
        assert err < ATTN_ATOL, ((b, h), err)


@pytest.fixture(scope="module")
def d256_caches(tqlib):
    """The head_dim-256 / 131072-context workload (B=1, Hq=16, Hkv=4; turbo4
    K with Student-t(4) keys, turbo3 V), slice (0, 3) planted by the oracle."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, Hkv, d, ctx = 1, 4, 256, 131072
    Lk, Lv = tb.make_layout(d, 32, 4, 0, 0, 1), tb.make_layout(d, 32, 3, 0, 0, 1)
    Lko, Lvo = O.Layout(d, 32, 4, 0, 0, 1), O.Layout(d, 32, 3, 0, 0, 1)
    K = _fill_gpu(tb, Lk, (B, Hkv, ctx), 3, heavy=True)
    V = _fill_gpu(tb, Lv, (B, Hkv, ctx), 4)
    kd = _plant(K, Lko, 0, 3, inputs.student_t((ctx, d), 930, 4.0))
    vd = _plant(V, Lvo, 0, 3, inputs.gaussian((ctx, d), 931))
    return K, V, kd, vd


def test_d256_decode_full_size(tqlib, d256_caches):
    """One decode query per head over 131072 tokens (the library's own split
    count and workspace, as timed); q-heads 12-15 (KV head 3)."""
    from turboquant_kv_cache_gb300 import binding as tb
    K, V, kd, vd = d256_caches
    q = inputs.gaussian((1, 16, 256), 32)
    got = to_np(tb.tq_decode_attn(K, V, torch.from_numpy(q).cuda(), ctx=131072).float())
    ref = O.decode_attention(q[:, 12:16], kd[None, None], vd[None, None])
    assert np.abs(got[:, 12:16] - ref).max() < ATTN_ATOL


def test_d256_prefill_full_size(tqlib, d256_caches):
    """The 512-query causal prefill chunk at positions 130560..131071 over the
    same cache (tensor-core prefill, its own split count); q-heads 12-15 on
    sampled query rows (first, last, and spread between)."""
    from turboquant_kv_cache_gb300 import binding as tb
    K, V, kd, vd = d256_caches
    ctx, Tq = 131072, 512
    qp = inputs.gaussian((1, 16, Tq, 256), 33)
    got = to_np(tb.tq_prefill_attn(K, V, torch.from_numpy(qp).cuda(), ctx, causal=True).float())
    rows = np.array([0, 1, 63, 64, 127, 128, 200, 255, 256, 383, 384, 447, 500, 510, 511])
    ref = O.prefill_attention(qp, kd[None, None], vd[None, None], ctx, causal=True, rows=rows, group=(12, 4))
    err = np.abs(got[:, 12:16][:, :, rows] - ref).max()
    assert err < ATTN_ATOL, err


def test_qjl_keys_decode_full_size(tqlib):
    """QJL-key decode: B=4, Hq=32, Hkv=8, d=128, ctx=16384, K 2-bit + QJL
    m=128 (S seed 7), V 3-bit, one norm per vector; slice (2, 6)."""
    from turboquant_kv_cache_gb300 import binding as tb
    B, Hq, Hkv, d, ctx = 4, 32, 8, 128, 16384
    S = inputs.qjl_matrix(128, d, 7)
    Sg = torch.from_numpy(S).cuda()
    Lk, Lv = tb.make_layout(d, 128, 2, 128, 0, 1), tb.make_layout(d, 128, 3, 0, 0, 1)
    Lko, Lvo = O.Layout(d, 128, 2, 128, 0, 1), O.Layout(d, 128, 3, 0, 0, 1)
    K = _fill_gpu(tb, Lk, (B, Hkv, ctx), 5, S=Sg)
    V = _fill_gpu(tb, Lv, (B, Hkv, ctx), 6)
    kd = _plant(K, Lko, 2, 6, inputs.gaussian((ctx, d), 940), S)
    vd = _plant(V, Lvo, 2, 6, inputs.gaussian((ctx, d), 941))
    q = inputs.gaussian((B, Hq, d), 20)
    got = to_np(tb.tq_decode_attn(K, V, torch.from_numpy(q).cuda(), ctx=ctx).float())
    ref = O.decode_attention(q[2:3, 24:28], kd[None, None], vd[None, None])
    assert np.abs(got[2:3, 24:28] - ref).max() < ATTN_ATOL

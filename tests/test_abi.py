"""The C ABI without a GPU: the library loads, exports every function the
header declares, and its host-side calls agree with the oracle."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from oracle import tq_oracle as O
from turboquant_kv_cache_gb300 import binding as tb

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tq.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(tqlib):
    names = _declared()
    assert "tq_quantize_kv" in names and "tq_decode_attn" in names and "tq_prefill_attn" in names
    for n in names:
        assert hasattr(tqlib, n), n


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("block", [32, 64, 128, 256])
def test_codebook_matches_oracle(tqlib, bits, block):
    c, b = tb.tq_codebook(bits, block, f64=True)
    oc, ob = O.lloyd_max_codebook(bits, block)
    assert np.max(np.abs(np.array(c) - oc)) < 1e-12
    assert np.max(np.abs(np.array(b) - ob)) < 1e-12
    cf, bf = tb.tq_codebook(bits, block)
    assert np.array_equal(np.array(cf, dtype=np.float32), oc.astype(np.float32))
    assert np.array_equal(np.array(bf, dtype=np.float32), ob.astype(np.float32))


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("block", [32, 64, 128, 256])
def test_beta_codebook_matches_oracle(tqlib, bits, block):
    c, b = tb.tq_codebook_kind(bits, block, tb.CODEBOOK_BETA)
    oc, ob = O.lloyd_max_beta_codebook(bits, block)
    assert np.max(np.abs(np.array(c) - oc)) < 1e-12
    assert np.max(np.abs(np.array(b) - ob)) < 1e-12
    g, _ = tb.tq_codebook_kind(bits, block, tb.CODEBOOK_GAUSSIAN)
    assert g == tb.tq_codebook(bits, block, f64=True)[0]


def test_codebook_kind_rules(tqlib):
    c = (ctypes.c_double * 16)()
    assert tqlib.tq_codebook_kind(3, 32, 2, c, None) == -1
    assert tqlib.tq_codebook_kind(3, 16, 1, c, None) == -2
    assert tqlib.tq_codebook_kind(3, 512, 1, c, None) == -2
    assert tqlib.tq_layout_sizes(ctypes.byref(tb.make_layout(128, 32, 3, codebook=1)), None, None, None) == 0
    assert tqlib.tq_layout_sizes(ctypes.byref(tb.make_layout(128, 32, 3, codebook=2)), None, None, None) == -1


@pytest.mark.parametrize("seed", [0, 1, 7, 2 ** 63 + 5])
def test_signs_match_oracle(tqlib, seed):
    assert tb.tq_signs(seed, 256) == [int(v) for v in O.sign_vector(seed, 256)]


def test_layout_sizes(tqlib):
    assert tb.tq_layout_sizes(tb.make_layout(128, 32, 3)) == (48, 4, 0)
    assert tb.tq_layout_sizes(tb.make_layout(256, 32, 4)) == (128, 8, 0)
    assert tb.tq_layout_sizes(tb.make_layout(128, 128, 2, qjl_m=128)) == (32, 1, 16)
    L = O.Layout(128, 32, 3)
    assert tb.tq_layout_sizes(tb.make_layout(128, 32, 3))[0] == L.code_bytes


@pytest.mark.parametrize("args,status", [
    ((96, 32, 3), -2), ((128, 16, 3), -2), ((128, 48, 3), -2), ((128, 32, 5), -2), ((128, 32, 0), -2),
])
def test_invalid_layouts_rejected(tqlib, args, status):
    L = tb.make_layout(*args)
    assert tqlib.tq_layout_sizes(ctypes.byref(L), None, None, None) == status


def test_qjl_layout_rules(tqlib):
    assert tqlib.tq_layout_sizes(ctypes.byref(tb.make_layout(128, 32, 2, qjl_m=128)), None, None, None) == -2
    assert tqlib.tq_layout_sizes(ctypes.byref(tb.make_layout(128, 128, 2, qjl_m=48)), None, None, None) == -2
    assert tqlib.tq_layout_sizes(ctypes.byref(tb.make_layout(128, 128, 2, qjl_m=512)), None, None, None) == -2


def test_8bit_layout_rules(tqlib):
    """One byte per code: Gaussian codebook only, no QJL, d code bytes; the
    decode takes 8-bit keys but not 8-bit values, the prefill neither."""
    assert tb.tq_layout_sizes(tb.make_layout(128, 32, 8)) == (128, 4, 0)
    assert tb.tq_layout_sizes(tb.make_layout(64, 64, 8)) == (64, 1, 0)
    sizes = lambda L: tqlib.tq_layout_sizes(ctypes.byref(L), None, None, None)
    assert sizes(tb.make_layout(128, 32, 8, codebook=1)) == -2
    assert sizes(tb.make_layout(128, 128, 8, qjl_m=128)) == -2
    for bits in (5, 6, 7, 9):
        assert sizes(tb.make_layout(128, 32, bits)) == -2
    with pytest.raises(ValueError):
        O.Layout(128, 32, 8, codebook=1)
    P16 = ctypes.c_void_p(16)
    L4, L8 = tb.make_layout(128, 32, 4), tb.make_layout(128, 32, 8)
    Lq = tb.make_layout(128, 128, 2, qjl_m=128)
    view = lambda L: tb.tq_kv_view(16, 16, 16, 16, 16, L, None, 0, 0)

    def dec(K, V):
        return tqlib.tq_decode_attn(ctypes.byref(K), ctypes.byref(V), P16, 1, 4, 1, 128, None, 64, 0.0, P16, P16,
                                    1 << 20, 0, None)

    assert dec(view(L4), view(L8)) == -2        # 8-bit values
    assert dec(view(L8), view(Lq)) == -2        # QJL values beside 8-bit keys
    assert tqlib.tq_prefill_attn(ctypes.byref(view(L8)), ctypes.byref(view(L4)), P16, 1, 4, 1, 16, 128, 64, 1,
                                 0.0, P16, P16, 1 << 20, None) == -2


def test_host_side_argument_checks_need_no_gpu(tqlib):
    L = tb.make_layout(128, 32, 3)
    # zero vectors: nothing to do
    assert tqlib.tq_quantize_kv(ctypes.byref(L), None, 0, 0, 128, None, None, None, None, None, None) == 0
    # missing buffers / bad stride / misaligned pointers are refused before any launch
    assert tqlib.tq_quantize_kv(ctypes.byref(L), None, 0, 4, 128, None, None, None, None, None, None) == -1
    assert tqlib.tq_quantize_kv(ctypes.byref(L), ctypes.c_void_p(16), 0, 4, 64, None,
                                ctypes.c_void_p(16), ctypes.c_void_p(16), None, None, None) == -1
    assert tqlib.tq_quantize_kv(ctypes.byref(L), ctypes.c_void_p(18), 0, 4, 128, None,
                                ctypes.c_void_p(16), ctypes.c_void_p(16), None, None, None) == -3
    assert tqlib.tq_quantize_kv(ctypes.byref(L), ctypes.c_void_p(16), 2, 4, 128, None,
                                ctypes.c_void_p(16), ctypes.c_void_p(16), None, None, None) == -1
    bad = tb.tq_layout(128, 32, 3, 0, 0, 7, 1)  # no such codebook kind
    assert tqlib.tq_layout_sizes(ctypes.byref(bad), None, None, None) == -1


def test_append_argument_checks_need_no_gpu(tqlib):
    L = tb.make_layout(128, 32, 3)
    P16 = ctypes.c_void_p(16)
    NP = (None, 0, 0)  # contiguous cache: no page table

    def app(x, dt, B, H, n, stride, pos, S_cap, paging=NP, codes=P16, scales=P16):
        return tqlib.tq_append_kv(ctypes.byref(L), x, dt, B, H, n, stride, pos, S_cap, *paging, None, codes,
                                  scales, None, None, None)

    # no tokens: nothing to do, even without buffers
    assert app(None, 0, 2, 8, 0, 128, None, 64, codes=None, scales=None) == 0
    # negative sizes, a missing position array or S_cap 0 are refused
    assert app(P16, 0, -1, 8, 1, 128, P16, 64) == -1
    assert app(P16, 0, 2, 8, 1, 128, None, 64) == -1
    assert app(P16, 0, 2, 8, 1, 128, P16, 0) == -1
    # then the quantise checks: misaligned rows, bad stride
    assert app(ctypes.c_void_p(18), 0, 2, 8, 1, 128, P16, 64) == -3
    assert app(P16, 0, 2, 8, 1, 64, P16, 64) == -1
    # paging: a table needs a page size that is a positive multiple of 32 and
    # pages_per_seq * page_size >= S_cap
    assert app(P16, 0, 2, 8, 1, 128, P16, 64, (P16, 0, 4)) == -1
    assert app(P16, 0, 2, 8, 1, 128, P16, 64, (P16, 48, 2)) == -1
    assert app(P16, 0, 2, 8, 1, 128, P16, 64, (P16, 32, 1)) == -1


def test_paging_checks_need_no_gpu(tqlib):
    """A page table with a page size that is not a positive multiple of 32,
    too few pages for S_cap, or K and V views that disagree on paging are
    refused before anything reaches the device."""
    L = tb.make_layout(128, 32, 3)
    P16 = ctypes.c_void_p(16)

    def view(pt, ps, pps):
        return tb.tq_kv_view(16, 16, None, None, None, L, pt, ps, pps)

    def dec(K, V, S_cap=128):
        return tqlib.tq_decode_attn(ctypes.byref(K), ctypes.byref(V), P16, 1, 4, 1, S_cap, None, 64, 0.0, P16,
                                    P16, 1 << 20, 0, None)

    def pre(K, V, S_cap=128):
        return tqlib.tq_prefill_attn(ctypes.byref(K), ctypes.byref(V), P16, 1, 4, 1, 8, S_cap, 64, 1, 0.0, P16,
                                     P16, 1 << 20, None)

    for f in (dec, pre):
        assert f(view(16, 48, 4), view(16, 48, 4)) == -1   # page size not a multiple of 32
        assert f(view(16, 0, 4), view(16, 0, 4)) == -1
        assert f(view(16, 32, 3), view(16, 32, 3)) == -1   # 96 slots < S_cap 128
        assert f(view(16, 32, 4), view(32, 32, 4)) == -1   # K and V tables differ
        assert f(view(16, 32, 4), view(None, 0, 0)) == -1  # K paged, V contiguous
        assert f(view(16, 64, 2), view(16, 32, 4)) == -1


def test_window_decode_checks_need_no_gpu(tqlib):
    L = tb.make_layout(128, 32, 3)
    P16 = ctypes.c_void_p(16)
    K = tb.tq_kv_view(16, 16, None, None, None, L, None, 0, 0)

    def win(kw, vw, W_cap, win_n):
        return tqlib.tq_decode_attn_window(ctypes.byref(K), ctypes.byref(K), P16, 1, 4, 1, 128, None, 64, kw, vw,
                                           W_cap, None, win_n, 0.0, P16, P16, 1 << 20, 0, None)

    assert win(None, P16, 16, 8) == -1            # missing window array
    assert win(P16, P16, 16, 17) == -1            # more window tokens than slots
    assert win(P16, P16, -1, 0) == -1
    assert win(ctypes.c_void_p(20), P16, 16, 8) == -3   # not 8-byte aligned
    # one split slot more than the plain decode
    nb, ns = tb.tq_decode_workspace_bytes(8, 32, 8, 128, 32768, 9)
    assert tb.tq_decode_window_workspace_bytes(8, 32, 8, 128, 32768, 9) == _decode_ws(8, 32, 128, 10)


def test_block_conversion_checks_need_no_gpu(tqlib):
    L = tb.make_layout(128, 128, 3, 0, 0, 1, codebook=1)
    Lq = tb.make_layout(128, 128, 2, 128, 0, 1)
    P16 = ctypes.c_void_p(16)
    assert tqlib.tq_to_blocks(ctypes.byref(L), None, None, 0, None, None) == 0
    assert tqlib.tq_to_blocks(ctypes.byref(Lq), P16, P16, 4, P16, None) == -2   # QJL: no block form
    assert tqlib.tq_to_blocks(ctypes.byref(L), ctypes.c_void_p(18), P16, 4, P16, None) == -3
    assert tqlib.tq_from_blocks(ctypes.byref(L), ctypes.c_void_p(17), 4, P16, P16, None) == -3
    assert tqlib.tq_from_blocks(ctypes.byref(L), P16, -1, P16, P16, None) == -1


def test_block_decode_checks_need_no_gpu(tqlib):
    L = tb.make_layout(128, 128, 3, codebook=1)
    Lq = tb.make_layout(128, 128, 2, qjl_m=128)
    L8 = tb.make_layout(128, 32, 8)
    P16 = ctypes.c_void_p(16)

    def dec(Lk, kb, Lv, Hq=4, Hkv=1, ws=P16, ws_bytes=1 << 20):
        return tqlib.tq_decode_attn_blocks(ctypes.byref(Lk), kb, ctypes.byref(Lv), P16, P16, 1, Hq, Hkv, 128, None,
                                           64, 0.0, P16, ws, ws_bytes, 0, None)

    assert dec(Lq, P16, L) == -2          # blocks carry no QJL data
    assert dec(L, P16, L8) == -2          # 8-bit codes: packed layout only
    assert dec(L, P16, L, Hq=6, Hkv=2) == -2   # group of 3
    assert dec(L, None, L) == -1
    assert dec(L, ctypes.c_void_p(17), L) == -3   # blocks are 2-byte aligned
    assert dec(L, P16, L, ws=None) == -4
    assert dec(L, P16, L, ws_bytes=64) == -4


def test_polar_checks_need_no_gpu(tqlib):
    cb = ctypes.c_int64()
    assert tqlib.tq_polar_code_bytes(128, 3, ctypes.byref(cb)) == 0 and cb.value == 48
    assert tqlib.tq_polar_code_bytes(96, 3, ctypes.byref(cb)) == -2      # not a power of two
    assert tqlib.tq_polar_code_bytes(128, 5, ctypes.byref(cb)) == -2
    P16 = ctypes.c_void_p(16)
    # no vectors: nothing to do, even without buffers
    assert tqlib.tq_polar_quantize(None, 0, 0, 128, 128, 3, None, None, None) == 0
    assert tqlib.tq_polar_dequantize(None, None, 0, 128, 3, None, 0, None) == 0
    # bad stride, bad dtype, misaligned codes or radius
    assert tqlib.tq_polar_quantize(P16, 0, 4, 128, 64, 3, P16, P16, None) == -1
    assert tqlib.tq_polar_quantize(P16, 5, 4, 128, 128, 3, P16, P16, None) == -1
    assert tqlib.tq_polar_quantize(P16, 0, 4, 128, 128, 3, ctypes.c_void_p(24), P16, None) == -3
    assert tqlib.tq_polar_dequantize(P16, ctypes.c_void_p(17), 4, 128, 3, P16, 0, None) == -3


def _decode_ws(B, Hq, d, ns):
    # split partials [B*Hq][n_split][d + 4] fp32, rounded up to 256 bytes, then
    # the tensor-core path's S q rows (fp16, m = 128) and row sums of QJL keys
    part = B * Hq * ns * (d + 4) * 4
    return (part + 255) // 256 * 256 + B * Hq * (128 * 2 + 4) + 256


def test_decode_workspace_query(tqlib):
    nb, ns = tb.tq_decode_workspace_bytes(8, 32, 8, 128, 32768, 16)
    assert ns == 16 and nb == _decode_ws(8, 32, 128, 16)
    nb, ns = tb.tq_decode_workspace_bytes(1, 16, 4, 256, 131072, 0)
    assert ns >= 1 and nb == _decode_ws(1, 16, 256, ns)
    # the library's own choice: one wave of the most resident decode CTAs (four
    # per SM; with no device the SM count is taken as 152), never more splits
    # than 256-token slices, so the workspace covers every layout's choice
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    nb, ns = tb.tq_decode_workspace_bytes(4, 32, 8, 128, 16384, 0)
    assert ns == min(4 * sms // 32, 64) and nb == _decode_ws(4, 32, 128, ns)
    nb, ns = tb.tq_decode_workspace_bytes(1, 8, 2, 128, 600, 0)
    assert ns == (600 + 255) // 256
    with pytest.raises(tb.TQError):
        tb.tq_decode_workspace_bytes(2, 6, 4, 128, 100)


def test_strerror_and_version(tqlib):
    assert tb.tq_strerror(0) == "ok"
    assert "workspace" in tb.tq_strerror(-4)
    assert tb.tq_version() >= 100

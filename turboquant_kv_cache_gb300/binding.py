"""Thin Python binding of libtq (the C ABI in include/tq.h).

Argument marshalling only: every function here checks shapes, takes raw
pointers from torch tensors, calls the C entry point of the same name on the
caller's current CUDA stream and raises TQError on a non-zero status.  All
computation happens in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libtq.so")
_lib = None

TQ_F16, TQ_F32 = 0, 1


class TQError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = _load().tq_strerror(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: tq status {status} ({msg})")


class tq_layout(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("block", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("qjl_m", ctypes.c_int32), ("norm_correct", ctypes.c_int32), ("codebook", ctypes.c_int32),
                ("sign_seed", ctypes.c_uint64)]


class tq_kv_view(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("qjl_bits", ctypes.c_void_p),
                ("qjl_rnorm", ctypes.c_void_p), ("S", ctypes.c_void_p), ("layout", tq_layout),
                ("page_table", ctypes.c_void_p), ("page_size", ctypes.c_int32), ("pages_per_seq", ctypes.c_int32)]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"libtq.so not built at {_LIB_PATH}: run `python -m turboquant_kv_cache_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "tq_codebook": (I, [I, I, P, P]),
        "tq_codebook_f64": (I, [I, I, P, P]),
        "tq_codebook_kind": (I, [I, I, I, P, P]),
        "tq_signs": (I, [ctypes.c_uint64, I, P]),
        "tq_layout_sizes": (I, [P, P, P, P]),
        "tq_quantize_kv": (I, [P, P, I, I64, I64, P, P, P, P, P, P]),
        "tq_append_kv": (I, [P, P, I, I, I, I, I64, P, I64, P, I, I, P, P, P, P, P, P]),
        "tq_dequantize_kv": (I, [P, P, P, P, P, P, I64, P, I, P]),
        "tq_decode_attn": (I, [P, P, P, I, I, I, I64, P, I64, ctypes.c_float, P, P, SZ, I, P]),
        "tq_decode_workspace_bytes": (I, [I, I, I, I, I64, I, P, P]),
        "tq_decode_attn_window": (I, [P, P, P, I, I, I, I64, P, I64, P, P, I, P, I, ctypes.c_float, P, P, SZ, I, P]),
        "tq_decode_window_workspace_bytes": (I, [I, I, I, I, I64, I, P]),
        "tq_polar_code_bytes": (I, [I, I, P]),
        "tq_to_blocks": (I, [P, P, P, I64, P, P]),
        "tq_from_blocks": (I, [P, P, I64, P, P, P]),
        "tq_decode_attn_blocks": (I, [P, P, P, P, P, I, I, I, I64, P, I64, ctypes.c_float, P, P, SZ, I, P]),
        "tq_polar_quantize": (I, [P, I, I64, I, I64, I, P, P, P]),
        "tq_polar_dequantize": (I, [P, P, I64, I, I, P, I, P]),
        "tq_decode_attn_static": (I, [P, P, P, I, I, I, I64, P, I64, ctypes.c_float, P, I, P]),
        "tq_prefill_attn": (I, [P, P, P, I, I, I, I, I64, I64, I, ctypes.c_float, P, P, SZ, P]),
        "tq_prefill_workspace_bytes": (I, [I, I, I, I, I, I64, P]),
        "tq_set_wait_limit_ns": (I, [ctypes.c_uint64]),
        "tq_device_status": (I, [I, I, P]),
        "tq_strerror": (ctypes.c_char_p, [I]),
        "tq_version": (I, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def library():
    """The loaded ctypes library (raises if libtq.so is missing)."""
    return _load()


# ------------------------------------------------------------------ helpers
CODEBOOK_GAUSSIAN, CODEBOOK_BETA = 0, 1


def make_layout(head_dim, block, bits, qjl_m=0, norm_correct=0, sign_seed=1, codebook=CODEBOOK_GAUSSIAN):
    return tq_layout(head_dim, block, bits, qjl_m, norm_correct, codebook, sign_seed)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st, where):
    if st != 0:
        raise TQError(st, where)


def _dtype_code(dt):
    if dt == torch.float16:
        return TQ_F16
    if dt == torch.float32:
        return TQ_F32
    raise TypeError(f"unsupported dtype {dt}")


# ------------------------------------------------------------------ host calls
def tq_codebook(bits, block, f64=False):
    """(centroids, boundaries) as Python lists (host call)."""
    lib = _load()
    K = 1 << bits
    T = ctypes.c_double if f64 else ctypes.c_float
    c = (T * K)()
    b = (T * max(K - 1, 1))()
    _check((lib.tq_codebook_f64 if f64 else lib.tq_codebook)(bits, block, c, b), "tq_codebook")
    return list(c), list(b)[:K - 1]


def tq_codebook_kind(bits, block, kind):
    """(centroids, boundaries) in double precision for a codebook kind
    (CODEBOOK_GAUSSIAN or CODEBOOK_BETA)."""
    lib = _load()
    K = 1 << bits
    c = (ctypes.c_double * K)()
    b = (ctypes.c_double * max(K - 1, 1))()
    _check(lib.tq_codebook_kind(bits, block, kind, c, b), "tq_codebook_kind")
    return list(c), list(b)[:K - 1]


def tq_signs(sign_seed, d):
    lib = _load()
    out = (ctypes.c_int8 * d)()
    _check(lib.tq_signs(ctypes.c_uint64(sign_seed), d, out), "tq_signs")
    return list(out)


def tq_layout_sizes(layout):
    lib = _load()
    cb, ns, qb = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib.tq_layout_sizes(ctypes.byref(layout), ctypes.byref(cb), ctypes.byref(ns), ctypes.byref(qb)),
           "tq_layout_sizes")
    return cb.value, ns.value, qb.value


def tq_decode_workspace_bytes(B, Hq, Hkv, head_dim, ctx, n_split=0):
    lib = _load()
    nb, ns = ctypes.c_size_t(), ctypes.c_int()
    _check(lib.tq_decode_workspace_bytes(B, Hq, Hkv, head_dim, ctx, n_split, ctypes.byref(nb), ctypes.byref(ns)),
           "tq_decode_workspace_bytes")
    return nb.value, ns.value


def tq_prefill_workspace_bytes(B, Hq, Hkv, head_dim, Tq, ctx):
    lib = _load()
    nb = ctypes.c_size_t()
    _check(lib.tq_prefill_workspace_bytes(B, Hq, Hkv, head_dim, Tq, ctx, ctypes.byref(nb)),
           "tq_prefill_workspace_bytes")
    return nb.value


# ------------------------------------------------------------------ packed cache
class PackedKV:
    """Device buffers of one packed cache (K or V): codes [N, code_bytes]
    uint8, scales [N, d/block] fp16, and with QJL qjl [N, m/8] uint8, rnorm
    [N] fp16 and the projection S [m, d] fp32.  N may carry leading dims.

    As an attention cache the lead shape is [B, Hkv, S_cap] (contiguous), or
    [num_pages, Hkv, page_size] with page_table an int32 CUDA tensor
    [B, pages_per_seq] (paged: token t of batch b is row t % page_size of
    page page_table[b, t // page_size])."""

    def __init__(self, layout, lead_shape, device="cuda", S=None, page_table=None):
        cb, ns, qb = tq_layout_sizes(layout)
        self.layout = layout
        self.lead_shape = tuple(lead_shape)
        self.page_table = page_table
        if page_table is not None:
            if (page_table.dtype != torch.int32 or page_table.dim() != 2 or not page_table.is_cuda
                    or len(self.lead_shape) != 3):
                raise ValueError("paged cache: lead shape [num_pages, Hkv, page_size] and an int32 CUDA "
                                 "page table [B, pages_per_seq]")
        self.codes = torch.empty(self.lead_shape + (cb,), dtype=torch.uint8, device=device)
        self.scales = torch.empty(self.lead_shape + (ns,), dtype=torch.float16, device=device)
        self.qjl = torch.empty(self.lead_shape + (qb,), dtype=torch.uint8, device=device) if qb else None
        self.rnorm = torch.empty(self.lead_shape, dtype=torch.float16, device=device) if qb else None
        self.S = S

    @property
    def n_vec(self):
        n = 1
        for s in self.lead_shape:
            n *= s
        return n

    @property
    def heads(self):
        return self.lead_shape[1]

    @property
    def batch(self):
        return self.page_table.shape[0] if self.page_table is not None else self.lead_shape[0]

    @property
    def capacity(self):
        """Slots per (batch, head): S_cap."""
        if self.page_table is not None:
            return self.page_table.shape[1] * self.lead_shape[2]
        return self.lead_shape[2]

    def view(self):
        pt = self.page_table
        return tq_kv_view(self.codes.data_ptr(), self.scales.data_ptr(),
                          self.qjl.data_ptr() if self.qjl is not None else None,
                          self.rnorm.data_ptr() if self.rnorm is not None else None,
                          self.S.data_ptr() if self.S is not None else None, self.layout,
                          pt.data_ptr() if pt is not None else None,
                          self.lead_shape[2] if pt is not None else 0, pt.shape[1] if pt is not None else 0)

    def nbytes(self):
        n = self.codes.numel() + 2 * self.scales.numel()
        if self.qjl is not None:
            n += self.qjl.numel() + 2 * self.rnorm.numel()
        return n


# ------------------------------------------------------------------ device calls
def tq_quantize_kv(layout, x, S=None, out=None, stream=None):
    """Quantise x [..., d] (fp16/fp32, CUDA, last dim contiguous) into a
    PackedKV with leading shape x.shape[:-1]."""
    lib = _load()
    d = layout.head_dim
    if x.shape[-1] != d or x.stride(-1) != 1:
        raise ValueError("x must have a contiguous last dimension of head_dim")
    lead = tuple(x.shape[:-1])
    x2 = x.reshape(-1, d)
    if out is None:
        out = PackedKV(layout, lead, device=x.device, S=S)
    n = x2.shape[0]
    st = lib.tq_quantize_kv(ctypes.byref(layout), _ptr(x2), _dtype_code(x.dtype), n, x2.stride(0), _ptr(S),
                            _ptr(out.codes), _ptr(out.scales), _ptr(out.qjl), _ptr(out.rnorm), _stream(stream))
    _check(st, "tq_quantize_kv")
    return out


def tq_append_kv(cache, x, pos, stream=None):
    """Quantise new tokens x [B, H, n_new, d] (fp16/fp32, CUDA, last dim
    contiguous, rows of one (b, h) contiguous) into a PackedKV cache of
    leading shape [B, H, S_cap]: token j of (b, h) lands in slot pos[b] + j
    (pos: int32 CUDA tensor [B]); slots outside [0, S_cap) are skipped."""
    lib = _load()
    layout = cache.layout
    d = layout.head_dim
    if x.dim() != 4 or x.shape[-1] != d or x.stride(-1) != 1:
        raise ValueError("x must be [B, H, n_new, head_dim] with a contiguous last dimension")
    B, H, n_new, _ = x.shape
    if len(cache.lead_shape) != 3 or (cache.batch, cache.heads) != (B, H):
        raise ValueError("cache must have leading shape [B, H, S_cap] (or be paged for B sequences) matching x")
    if pos.dtype != torch.int32 or pos.numel() != B or not pos.is_cuda:
        raise ValueError("pos must be an int32 CUDA tensor of B slot offsets")
    x2 = x.reshape(-1, d)
    pt = cache.page_table
    st = lib.tq_append_kv(ctypes.byref(layout), _ptr(x2), _dtype_code(x.dtype), B, H, n_new, x2.stride(0),
                          _ptr(pos.contiguous()), cache.capacity, _ptr(pt),
                          cache.lead_shape[2] if pt is not None else 0, pt.shape[1] if pt is not None else 0,
                          _ptr(cache.S), _ptr(cache.codes), _ptr(cache.scales), _ptr(cache.qjl), _ptr(cache.rnorm),
                          _stream(stream))
    _check(st, "tq_append_kv")
    return cache


def tq_dequantize_kv(packed, out_dtype=torch.float16, stream=None, out=None):
    lib = _load()
    d = packed.layout.head_dim
    if out is None:
        out = torch.empty(packed.lead_shape + (d,), dtype=out_dtype, device=packed.codes.device)
    elif out.dtype != out_dtype or out.numel() != packed.n_vec * d or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of n_vec x head_dim elements of out_dtype")
    st = lib.tq_dequantize_kv(ctypes.byref(packed.layout), _ptr(packed.codes), _ptr(packed.scales),
                              _ptr(packed.qjl), _ptr(packed.rnorm), _ptr(packed.S), packed.n_vec, _ptr(out),
                              _dtype_code(out_dtype), _stream(stream))
    _check(st, "tq_dequantize_kv")
    return out


def _cache_for(K, V, B):
    """Heads and S_cap of a K/V cache pair read by B sequences."""
    if K.batch < B or V.batch < B or (K.heads, K.capacity) != (V.heads, V.capacity):
        raise ValueError("K and V caches must hold the same heads and slots for at least B sequences")
    return K.heads, K.capacity


def tq_decode_attn(K, V, q, ctx=None, kv_len=None, softmax_scale=0.0, n_split=0, workspace=None, out=None,
                   stream=None):
    """q [B, Hq, d] fp16; K, V PackedKV caches (contiguous [B, Hkv, S_cap]
    or paged with one page table)."""
    lib = _load()
    B, Hq, d = q.shape
    Hkv, S_cap = _cache_for(K, V, B)
    ctx = S_cap if ctx is None else ctx
    need, ns = tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, n_split)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    kv, vv = K.view(), V.view()
    st = lib.tq_decode_attn(ctypes.byref(kv), ctypes.byref(vv), _ptr(q), B, Hq, Hkv, S_cap, _ptr(kv_len), ctx,
                            float(softmax_scale), _ptr(out), _ptr(workspace), workspace.numel(), n_split,
                            _stream(stream))
    _check(st, "tq_decode_attn")
    return out


def tq_decode_attn_static(K, V, q, ctx=None, kv_len=None, softmax_scale=0.0, n_split=0, out=None, stream=None):
    """tq_decode_attn without a workspace: the library's own fixed device
    array holds the split partials (for callers that cannot allocate)."""
    lib = _load()
    B, Hq, d = q.shape
    Hkv, S_cap = _cache_for(K, V, B)
    ctx = S_cap if ctx is None else ctx
    if out is None:
        out = torch.empty_like(q)
    kv, vv = K.view(), V.view()
    st = lib.tq_decode_attn_static(ctypes.byref(kv), ctypes.byref(vv), _ptr(q), B, Hq, Hkv, S_cap, _ptr(kv_len),
                                   ctx, float(softmax_scale), _ptr(out), n_split, _stream(stream))
    _check(st, "tq_decode_attn_static")
    return out


def tq_decode_window_workspace_bytes(B, Hq, Hkv, head_dim, ctx, n_split=0):
    lib = _load()
    nb = ctypes.c_size_t()
    _check(lib.tq_decode_window_workspace_bytes(B, Hq, Hkv, head_dim, ctx, n_split, ctypes.byref(nb)),
           "tq_decode_window_workspace_bytes")
    return nb.value


def tq_decode_attn_window(K, V, q, k_win, v_win, ctx=None, kv_len=None, win_len=None, win=None, softmax_scale=0.0,
                          n_split=0, workspace=None, out=None, stream=None):
    """Decode over the packed cache plus an fp16 residual window: k_win,
    v_win [B, Hkv, W_cap, d] fp16 CUDA (contiguous, unrotated); win_len an
    int32 CUDA tensor [B] of window tokens, or win for every batch (default
    W_cap)."""
    lib = _load()
    B, Hq, d = q.shape
    Hkv, S_cap = _cache_for(K, V, B)
    ctx = S_cap if ctx is None else ctx
    if k_win.shape != v_win.shape or k_win.dim() != 4 or tuple(k_win.shape[:2]) != (B, Hkv) or k_win.shape[3] != d:
        raise ValueError("k_win, v_win must be [B, Hkv, W_cap, head_dim]")
    if k_win.dtype != torch.float16 or v_win.dtype != torch.float16:
        raise ValueError("the window is fp16")
    k_win, v_win = k_win.contiguous(), v_win.contiguous()
    W_cap = k_win.shape[2]
    if win_len is not None and (win_len.dtype != torch.int32 or win_len.numel() != B or not win_len.is_cuda):
        raise ValueError("win_len must be an int32 CUDA tensor of B window lengths")
    win = W_cap if win is None else win
    need = tq_decode_window_workspace_bytes(B, Hq, Hkv, d, ctx, n_split)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    kv, vv = K.view(), V.view()
    st = lib.tq_decode_attn_window(ctypes.byref(kv), ctypes.byref(vv), _ptr(q), B, Hq, Hkv, S_cap, _ptr(kv_len), ctx,
                                   _ptr(k_win), _ptr(v_win), W_cap, _ptr(win_len), win, float(softmax_scale),
                                   _ptr(out), _ptr(workspace), workspace.numel(), n_split, _stream(stream))
    _check(st, "tq_decode_attn_window")
    return out


def tq_to_blocks(pk, stream=None):
    """GGML-style blocks of a PackedKV without QJL: uint8 [..., d/32,
    2 + 4 bits] (fp16 norm of the rotation block, then the packed codes)."""
    lib = _load()
    L = pk.layout
    n = pk.scales.numel() // pk.scales.shape[-1]
    bb = 2 + 4 * L.bits
    out = torch.empty(tuple(pk.lead_shape) + (L.head_dim // 32, bb), dtype=torch.uint8, device=pk.codes.device)
    _check(lib.tq_to_blocks(ctypes.byref(L), _ptr(pk.codes), _ptr(pk.scales), n, _ptr(out), _stream(stream)),
           "tq_to_blocks")
    return out


def tq_decode_attn_blocks(Lk, k_blocks, Lv, v_blocks, q, ctx=None, kv_len=None, softmax_scale=0.0, n_split=0,
                          workspace=None, out=None, stream=None):
    """Decode attention read straight from block-form caches: q [B, Hq, d]
    fp16; k_blocks / v_blocks uint8 [B, Hkv, S_cap, d/32, 2 + 4 bits] (as
    tq_to_blocks gives for a contiguous cache) of layouts Lk / Lv."""
    lib = _load()
    B, Hq, d = q.shape
    for blk, L in ((k_blocks, Lk), (v_blocks, Lv)):
        if blk.dim() != 5 or blk.dtype != torch.uint8 or tuple(blk.shape[3:]) != (L.head_dim // 32, 2 + 4 * L.bits):
            raise ValueError("blocks must be uint8 [B, Hkv, S_cap, head_dim/32, 2 + 4 bits]")
        if not blk.is_contiguous():
            raise ValueError("blocks must be contiguous")
    if tuple(k_blocks.shape[:3]) != tuple(v_blocks.shape[:3]) or k_blocks.shape[0] != B:
        raise ValueError("K and V blocks must share [B, Hkv, S_cap] with q's batch")
    Hkv, S_cap = k_blocks.shape[1], k_blocks.shape[2]
    ctx = S_cap if ctx is None else ctx
    need, ns = tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, n_split)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    st = lib.tq_decode_attn_blocks(ctypes.byref(Lk), _ptr(k_blocks), ctypes.byref(Lv), _ptr(v_blocks), _ptr(q), B,
                                   Hq, Hkv, S_cap, _ptr(kv_len), ctx, float(softmax_scale), _ptr(out),
                                   _ptr(workspace), workspace.numel(), n_split, _stream(stream))
    _check(st, "tq_decode_attn_blocks")
    return out


def tq_from_blocks(layout, blocks, stream=None):
    """Inverse of tq_to_blocks: a PackedKV with leading shape blocks.shape[:-2]."""
    lib = _load()
    lead = tuple(blocks.shape[:-2])
    pk = PackedKV(layout, lead, device=blocks.device)
    n = pk.scales.numel() // pk.scales.shape[-1]
    _check(lib.tq_from_blocks(ctypes.byref(layout), _ptr(blocks), n, _ptr(pk.codes), _ptr(pk.scales),
                              _stream(stream)), "tq_from_blocks")
    return pk


def tq_polar_quantize(x, bits, stream=None):
    """Polar-angle quantise x [..., d] (fp16/fp32, CUDA, last dim
    contiguous): returns (codes uint8 [..., d*bits/8], radius fp16 [...])."""
    lib = _load()
    d = x.shape[-1]
    if x.stride(-1) != 1:
        raise ValueError("x must have a contiguous last dimension")
    lead = tuple(x.shape[:-1])
    x2 = x.reshape(-1, d)
    n = x2.shape[0]
    cb = ctypes.c_int64()
    _check(lib.tq_polar_code_bytes(d, bits, ctypes.byref(cb)), "tq_polar_code_bytes")
    codes = torch.empty(lead + (cb.value,), dtype=torch.uint8, device=x.device)
    radius = torch.empty(lead, dtype=torch.float16, device=x.device)
    st = lib.tq_polar_quantize(_ptr(x2), _dtype_code(x.dtype), n, d, x2.stride(0), bits, _ptr(codes), _ptr(radius),
                               _stream(stream))
    _check(st, "tq_polar_quantize")
    return codes, radius


def tq_polar_dequantize(codes, radius, head_dim, bits, out_dtype=torch.float16, out=None, stream=None):
    lib = _load()
    lead = tuple(radius.shape)
    n = radius.numel()
    if out is None:
        out = torch.empty(lead + (head_dim,), dtype=out_dtype, device=codes.device)
    st = lib.tq_polar_dequantize(_ptr(codes), _ptr(radius), n, head_dim, bits, _ptr(out), _dtype_code(out.dtype),
                                 _stream(stream))
    _check(st, "tq_polar_dequantize")
    return out


def tq_prefill_attn(K, V, q, ctx, causal=True, softmax_scale=0.0, workspace=None, out=None, stream=None):
    """q [B, Hq, Tq, d] fp16 at positions ctx-Tq .. ctx-1."""
    lib = _load()
    B, Hq, Tq, d = q.shape
    Hkv, S_cap = _cache_for(K, V, B)
    need = tq_prefill_workspace_bytes(B, Hq, Hkv, d, Tq, ctx)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    kv, vv = K.view(), V.view()
    st = lib.tq_prefill_attn(ctypes.byref(kv), ctypes.byref(vv), _ptr(q), B, Hq, Hkv, Tq, S_cap, ctx,
                             1 if causal else 0, float(softmax_scale), _ptr(out), _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check(st, "tq_prefill_attn")
    return out


def tq_set_wait_limit_ns(ns):
    """Wait limit (ns) of the library's bounded device-side waits for later
    launches; 0 restores the default (2 s)."""
    _check(_load().tq_set_wait_limit_ns(int(ns)), "tq_set_wait_limit_ns")


def tq_device_status(device=None, clear=False):
    """The library's device status word of `device` (default: the current
    one) after synchronising it: 0 when no launch recorded a failure since
    the last clear, else the first failure (TQ_ERR_TIMEOUT = -6)."""
    if device is None:
        device = torch.cuda.current_device()
    st = ctypes.c_int(0)
    _check(_load().tq_device_status(int(device), 1 if clear else 0, ctypes.byref(st)), "tq_device_status")
    return st.value


def tq_strerror(status):
    return _load().tq_strerror(status).decode()


def tq_version():
    return _load().tq_version()

"""Seeded synthetic inputs shared by the tests, the smoke check and the
benchmark.  This module draws random numbers and shapes them; it holds none
of the codec's arithmetic, so the CUDA path and the CPU oracle can both be
fed from it without sharing any of the method.

Shapes and value distributions follow the workloads the source pages
measure on (real-model KV tensors replaced by seeded synthetic ones):
  * unit vectors d=128 ("turboquant-pytorch" README, synthetic MSE table);
  * Llama-3.2-1B-shaped KV (16 layers, 8 KV heads, head_dim 64) with a few
    outlier channels (TurboQuant From Scratch, K/V norm discussion);
  * Qwen3-8B-shaped decode (32 q-heads / 8 KV-heads, head_dim 128);
  * head_dim 256, 16 q / 4 KV heads, 131072 context with heavy-tailed keys
    (llama.cpp-turboquant, Qwen3.5-9B measurements).
"""
from __future__ import annotations

import numpy as np


def gaussian(shape, seed, dtype=np.float16):
    """i.i.d. N(0,1) drawn in float32 from numpy's PCG64 stream ``seed``,
    then cast to ``dtype``."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape, dtype=np.float32).astype(dtype)


def student_t(shape, seed, nu=4.0, dtype=np.float16):
    """i.i.d. Student-t with ``nu`` degrees of freedom (heavy-tailed keys)."""
    rng = np.random.default_rng(seed)
    return rng.standard_t(nu, size=shape).astype(np.float32).astype(dtype)


def unit_vectors(n, d, seed, dtype=np.float32):
    """n Gaussian rows normalised to unit length in float32."""
    x = gaussian((n, d), seed, np.float32)
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    return x.astype(dtype)


def outlier_kv(layers, heads, seq, d, seed, outlier_seed, n_outlier=4, factor=8.0):
    """[layers, heads, seq, d] fp16 N(0,1); in every (layer, head) the same
    ``n_outlier`` distinct channels (drawn from ``outlier_seed``) are
    multiplied by ``factor`` on every token."""
    x = gaussian((layers, heads, seq, d), seed, np.float32)
    rng = np.random.default_rng(outlier_seed)
    for l in range(layers):
        for h in range(heads):
            ch = rng.choice(d, size=n_outlier, replace=False)
            x[l, h, :, ch] *= factor
    return x.astype(np.float16)


def qjl_matrix(m, d, seed):
    """QJL projection S: [m, d] float32 with N(0,1) entries."""
    return gaussian((m, d), seed, np.float32)


# Workload definitions.  Each returns plain numpy arrays; sizes can be
# overridden so the tests can run the same recipe at small sizes.

def unit_roundtrip_workload(n=4096, d=128, seed=0):
    """4096 random unit vectors, d=128, fp32 (3-bit, one fp16 norm per
    vector, sign seed 1, no QJL)."""
    return {"x": unit_vectors(n, d, seed)}


def llama1b_kv_workload(layers=16, heads=8, seq=2048, d=64):
    """Llama-3.2-1B-shaped K and V with 4 outlier channels per head x8."""
    k = outlier_kv(layers, heads, seq, d, seed=2, outlier_seed=4)
    v = outlier_kv(layers, heads, seq, d, seed=3, outlier_seed=4)
    return {"k": k, "v": v}


def qwen8b_decode_workload(batch=8, hq=32, hkv=8, ctx=32768, d=128, seeds=(10, 11, 12)):
    """Qwen3-8B-shaped decode: q [B,Hq,d], K/V [B,Hkv,ctx,d], fp16 N(0,1)."""
    return {
        "q": gaussian((batch, hq, d), seeds[0]),
        "k": gaussian((batch, hkv, ctx, d), seeds[1]),
        "v": gaussian((batch, hkv, ctx, d), seeds[2]),
    }


def qjl_decode_workload(batch=4, hq=32, hkv=8, ctx=16384, d=128, m=128):
    """Same shape as the Qwen3-8B decode at 16384 context, batch 4, plus the
    Gaussian QJL matrix S (m=128 rows, seed 7)."""
    w = qwen8b_decode_workload(batch, hq, hkv, ctx, d, seeds=(20, 21, 22))
    w["S"] = qjl_matrix(m, d, 7)
    return w


def d256_longctx_workload(batch=1, hq=16, hkv=4, ctx=131072, d=256, tq=512):
    """head_dim 256, 16 q / 4 KV heads, 131072 context; Student-t(4) keys,
    N(0,1) values and queries; one decode query per head plus a 512-query
    prefill chunk."""
    return {
        "k": student_t((batch, hkv, ctx, d), 30),
        "v": gaussian((batch, hkv, ctx, d), 31),
        "q": gaussian((batch, hq, d), 32),
        "q_prefill": gaussian((batch, hq, tq, d), 33),
    }

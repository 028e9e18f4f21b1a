"""Comparison helpers for the GPU-vs-oracle parity tests.

Acceptance rules (the codec's stated tolerances):
  * codes identical except coordinates whose rotated value lies within 1e-5
    of a decision boundary (counted and reported);
  * QJL sign bits identical except where |(S r)_i| < 1e-5, and except in
    vectors that already have a boundary-tie code difference;
  * stored fp16 scales / residual norms within one fp16 ulp;
  * decoded vectors within 1e-3 relative L2;
  * attention outputs within 2e-3 absolute.
"""
import os

import numpy as np
import torch

from oracle import tq_oracle as O

TIE = 1e-5
ATTN_ATOL = 2e-3
DEQ_RTOL = 1e-3

# Boundary-tie mismatches seen by the comparisons below, one entry per call:
# (test id, kind, mismatches, compared); printed at the end of the session.
TIE_LOG = []


def _log_ties(kind, n_bad, n_total):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" (")[0]
    TIE_LOG.append((test, kind, int(n_bad), int(n_total)))


def fp16_ulp_diff(a, b):
    """Distance in fp16 ulps between two fp16 arrays (same sign assumed)."""
    ai = np.asarray(a, dtype=np.float16).view(np.int16).astype(np.int64)
    bi = np.asarray(b, dtype=np.float16).view(np.int16).astype(np.int64)
    return np.abs(ai - bi)


def compare_codes(gpu_packed, oq, L):
    """Returns (n_mismatch, vectors_with_mismatch).  Asserts every mismatch is
    a boundary tie and off by one level."""
    gcodes = O.unpack_codes(gpu_packed, L.bits, L.d)
    ocodes = oq["codes"]
    diff = gcodes != ocodes
    if diff.any():
        _, bnd = O.codebook_for(L)
        y = oq["y"][diff]
        near = np.min(np.abs(y[:, None] - bnd[None, :]), axis=1) < TIE
        assert near.all(), f"{(~near).sum()} code mismatches away from a boundary"
        assert np.all(np.abs(gcodes[diff] - ocodes[diff]) == 1)
    _log_ties("codes", diff.sum(), diff.size)
    return int(diff.sum()), np.any(diff, axis=1)


def compare_scales(gpu, ref, max_frac=1e-3):
    d = fp16_ulp_diff(gpu, ref)
    assert d.max() <= 1, f"scale off by {d.max()} ulp"
    assert (d > 0).mean() <= max_frac
    return int((d > 0).sum())


def compare_qjl(gpu_bits, oq, L, skip_rows):
    g = O.unpack_qjl(gpu_bits, L.m)
    o = oq["qjl"]
    diff = (g != o)
    diff[skip_rows] = False
    if diff.any():
        assert np.all(np.abs(oq["proj"][diff]) < TIE), "QJL sign mismatch away from zero"
    _log_ties("qjl", diff.sum(), diff.size)
    return int(diff.sum())


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    num = np.linalg.norm(a - b, axis=-1)
    den = np.maximum(np.linalg.norm(b, axis=-1), 1e-30)
    return np.where(np.linalg.norm(b, axis=-1) == 0, num, num / den)


def to_np(t):
    return t.detach().cpu().numpy()


def upload_packed(binding, L_c, L_o, codes, scales, qjl, rho, lead, S=None, device="cuda"):
    """Build a PackedKV on the device holding oracle-encoded arrays."""
    pk = binding.PackedKV(L_c, lead, device=device, S=S)
    pk.codes.copy_(torch.from_numpy(codes.reshape(pk.codes.shape)))
    pk.scales.copy_(torch.from_numpy(scales.reshape(pk.scales.shape)))
    if L_o.m:
        pk.qjl.copy_(torch.from_numpy(qjl.reshape(pk.qjl.shape)))
        pk.rnorm.copy_(torch.from_numpy(rho.reshape(pk.rnorm.shape)))
    return pk

"""The polar-angle quantizer's kernels (tq_polar_quantize /
tq_polar_dequantize) against the oracle (oracle/polar_oracle.py): angle
indices bit-exact except where the oracle's scaled angle sits within 1e-5
grid steps of a rounding tie, the fp16 radius exact except next to an fp16
rounding midpoint, the decoded vectors within 1e-5 relative L2 (fp32
trigonometry against float64)."""
import numpy as np
import pytest
import torch

from oracle import polar_oracle as P
from turboquant_kv_cache_gb300 import inputs

from _parity import to_np

pytestmark = pytest.mark.gpu

TIE = 1e-5


def _radius_tie(x):
    """Vectors whose float64 norm lies next to an fp16 rounding midpoint."""
    n = np.linalg.norm(np.asarray(x, dtype=np.float64), axis=1)
    lo = n.astype(np.float16).astype(np.float64)
    nxt = np.nextafter(n.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    prv = np.nextafter(n.astype(np.float16), np.float16(-np.inf)).astype(np.float64)
    mid = np.minimum(np.abs(n - (lo + nxt) / 2), np.abs(n - (lo + prv) / 2))
    return mid <= 1e-6 * np.maximum(n, 1e-30)


def _inputs(n, d, seed, dtype):
    x = inputs.gaussian((n, d), seed, np.float32 if dtype == torch.float32 else np.float16)
    x[3] = 0                       # a zero vector
    x[5, : d // 2] = 0             # zero pairs and a zero subtree
    x[7, 1::2] = 0                 # every level-1 pair on the axis
    return x


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_polar_quantize_matches_oracle(tqlib, d, bits, dtype):
    from turboquant_kv_cache_gb300 import binding as tb
    n = 1003                                       # not a multiple of the CTA's 4 vectors
    x = _inputs(n, d, 60 + d + bits, dtype)
    codes, radius = tb.tq_polar_quantize(torch.from_numpy(x).cuda(), bits)
    torch.cuda.synchronize()
    idx_ref, r_ref = P.polar_encode(x.astype(np.float64), bits)
    _, theta = P.polar_transform(x.astype(np.float64))
    full = P.O.unpack_codes(to_np(codes), bits, d)
    assert np.all(full[:, d - 1] == 0)
    idx = full[:, :d - 1]
    bad = idx != idx_ref
    assert not np.any(bad & (P.tie_distance(theta, bits) > TIE)), int(np.sum(bad))
    r_gpu = to_np(radius)
    rbad = r_gpu != r_ref
    assert not np.any(rbad & ~_radius_tie(x)), int(np.sum(rbad))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 3, 4])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_polar_dequantize_matches_oracle(tqlib, d, bits, out_dtype):
    from turboquant_kv_cache_gb300 import binding as tb
    n = 517
    x = _inputs(n, d, 90 + d + bits, torch.float16).astype(np.float64)
    idx, r16 = P.polar_encode(x, bits)
    codes = torch.from_numpy(P.pack_polar(idx, bits)).cuda()
    radius = torch.from_numpy(r16).cuda()
    out = tb.tq_polar_dequantize(codes, radius, d, bits, out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = P.polar_decode(idx, r16, bits)
    got = to_np(out.float()).astype(np.float64)
    nrm = np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    rel = np.linalg.norm(got - ref, axis=1) / nrm
    tol = 1e-5 if out_dtype == torch.float32 else 1e-3
    assert np.all(rel[nrm > 1e-20] < tol), rel.max()
    assert np.all(got[3] == 0)                       # the zero vector


def test_polar_empty_and_errors(tqlib):
    from turboquant_kv_cache_gb300 import binding as tb
    x = torch.zeros(0, 128, dtype=torch.float16, device="cuda")
    codes, radius = tb.tq_polar_quantize(x, 3)
    assert codes.shape == (0, 48) and radius.shape == (0,)
    with pytest.raises(tb.TQError) as e:
        tb.tq_polar_quantize(torch.zeros(4, 96, dtype=torch.float16, device="cuda"), 3)
    assert e.value.status == -2

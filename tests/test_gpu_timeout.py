"""Bounded device-side waits.  With the wait limit set far below any real
wait (1 ns), the fast quantiser and the tensor-core prefill record
TQ_ERR_TIMEOUT in the device status word while their outputs stay exactly
those of an ordinary launch (a wait past the limit is reported and goes on;
only the hard bound stops a CTA).  With the default limit restored the status
stays clean and the context is still usable."""
import numpy as np
import pytest
import torch

from oracle import tq_oracle as O
from turboquant_kv_cache_gb300 import inputs

from _parity import upload_packed

pytestmark = pytest.mark.gpu

TQ_ERR_TIMEOUT = -6


@pytest.fixture
def tb(tqlib):
    from turboquant_kv_cache_gb300 import binding
    torch.cuda.synchronize()
    binding.tq_set_wait_limit_ns(0)
    binding.tq_device_status(clear=True)
    yield binding
    binding.tq_set_wait_limit_ns(0)
    binding.tq_device_status(clear=True)


@pytest.mark.parametrize("block,bits", [(32, 3), (64, 4)])
def test_quantize_reports_timeout_and_stays_exact(tb, block, bits):
    L = tb.make_layout(128, block, bits, 0, 0, 1)
    x = torch.from_numpy(inputs.gaussian((40000, 128), 70)).cuda().half()
    ref = tb.tq_quantize_kv(L, x)
    assert tb.tq_device_status(clear=True) == 0
    tb.tq_set_wait_limit_ns(1)
    got = tb.tq_quantize_kv(L, x)
    assert tb.tq_device_status(clear=True) == TQ_ERR_TIMEOUT
    assert torch.equal(got.codes, ref.codes) and torch.equal(got.scales, ref.scales)
    tb.tq_set_wait_limit_ns(0)
    again = tb.tq_quantize_kv(L, x)
    assert tb.tq_device_status() == 0
    assert torch.equal(again.codes, ref.codes)


def test_prefill_reports_timeout_and_stays_exact(tb):
    d, B, Hq, Hkv, S_cap, ctx, Tq = 128, 1, 8, 2, 700, 650, 256
    Lk = O.Layout(d, 32, 3, 0, 0, 1)
    k = inputs.gaussian((B, Hkv, S_cap, d), 71)
    v = inputs.gaussian((B, Hkv, S_cap, d), 72)
    kc, ks, _, _ = O.encode(k.reshape(-1, d), Lk)
    vc, vs, _, _ = O.encode(v.reshape(-1, d), Lk)
    K = upload_packed(tb, tb.make_layout(d, 32, 3, 0, 0, 1), Lk, kc, ks, None, None, (B, Hkv, S_cap))
    V = upload_packed(tb, tb.make_layout(d, 32, 3, 0, 0, 1), Lk, vc, vs, None, None, (B, Hkv, S_cap))
    q = torch.from_numpy(inputs.gaussian((B, Hq, Tq, d), 73)).cuda()
    ref = tb.tq_prefill_attn(K, V, q, ctx, causal=True)
    assert tb.tq_device_status(clear=True) == 0
    tb.tq_set_wait_limit_ns(1)
    got = tb.tq_prefill_attn(K, V, q, ctx, causal=True)
    assert tb.tq_device_status(clear=True) == TQ_ERR_TIMEOUT
    assert torch.equal(got, ref)
    tb.tq_set_wait_limit_ns(0)
    again = tb.tq_prefill_attn(K, V, q, ctx, causal=True)
    assert tb.tq_device_status() == 0
    assert torch.equal(again, ref)
    assert np.isfinite(again.float().cpu().numpy()).all()

"""ra_forward_host: the forward on host tensors (H2D copies, the kernel, D2H
copies on one stream) gives the same bits as ra_forward on device tensors."""
import numpy as np
import pytest

from helpers import inputs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def test_forward_host_equals_device_forward(ra):
    import torch
    B, Hq, Hkv, S, N, D = 1, 4, 2, 2048, 4, 128
    q, k, v = inputs(8200, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out0, lse0 = ra.forward(tq, tk, tv, N, causal=True, striped=1)
    ra.check()
    hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
                  for x in (q, k, v))
    out_h = torch.empty(hq.shape, dtype=torch.int16).pin_memory()
    lse_h = torch.empty((B, Hq, S), dtype=torch.float32).pin_memory()
    stage = [torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv),
             torch.empty_like(tq), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")]
    P = ra._ptr
    side = torch.cuda.Stream()
    rc = ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), P(lse_h), *[P(x) for x in stage], B,
                            Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16, ra._stream_handle(side))
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(ra._stream_handle(side)) == ra.RA_OK
    assert torch.equal(out_h, out0.view(torch.int16).cpu())
    assert torch.equal(lse_h, lse0.cpu())
    # without lse
    out_h.zero_()
    rc = ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), None, *[P(x) for x in stage[:4]], None,
                            B, Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16, ra._stream_handle(side))
    assert rc == ra.RA_OK
    assert ra.ra_check(ra._stream_handle(side)) == ra.RA_OK
    assert torch.equal(out_h, out0.view(torch.int16).cpu())
    # an lse pair with one side missing is refused before anything is enqueued
    assert ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), P(lse_h), *[P(x) for x in stage[:4]],
                              None, B, Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16,
                              None) == ra.RA_ERR_INVALID_ARG

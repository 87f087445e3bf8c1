"""Failure detection on the GPU without a fault: the tensor-core kernel's
bounded waits.  ra_watchdog_selftest withholds each CTA's first K-tile copy,
so the waits that need it run out after a short limit; the kernel must
report RA_ERR_TIMEOUT through ra_check, return promptly, and leave the
context usable -- a normal forward right after it must still match the
oracle."""
import time

import numpy as np
import pytest

from helpers import assert_close, from_device, inputs, reference, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def test_withheld_copy_times_out_and_context_stays_usable(ra):
    import torch
    B, Hq, Hkv, S, N, D = 1, 2, 1, 512, 2, 128
    q, k, v = inputs(31, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out = torch.empty_like(tq)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    stream = ra._stream_handle(None)
    assert ra.ra_check(stream) == ra.RA_OK  # clean start

    t0 = time.time()
    rc = ra.ra_watchdog_selftest(ra._ptr(tq), ra._ptr(tk), ra._ptr(tv), ra._ptr(out),
                                 ra._ptr(lse), B, Hq, Hkv, S, D, N, 1, 1, 0.0, 20_000_000, stream)
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(stream) == ra.RA_ERR_TIMEOUT
    assert time.time() - t0 < 30.0
    assert ra.ra_check(stream) == ra.RA_OK  # the status word was cleared

    # the context still works: a normal forward is correct
    out2, lse2 = ra.forward(tq, tk, tv, N, causal=True, striped=True)
    ra.check()
    ro, rl = reference(q, k, v, N, True, True, "bf16")
    assert_close(from_device(out2), from_device(lse2), ro, rl, "bf16", "after the self test")


def test_selftest_argument_checks(ra):
    """Refused on the host; the buffers are real and large enough anyway."""
    import torch
    q = torch.zeros((1, 1, 256, 128), dtype=torch.bfloat16, device="cuda")
    k, v, o = torch.zeros_like(q), torch.zeros_like(q), torch.zeros_like(q)
    P = [ra._ptr(x) for x in (q, k, v, o)]
    assert ra.ra_watchdog_selftest(*P, None, 1, 1, 1, 256, 128, 2, 1, 0, 0.0, 10,
                                   None) == ra.RA_ERR_INVALID_ARG    # limit below 1e5 cycles
    q96 = torch.zeros((1, 1, 256, 96), dtype=torch.bfloat16, device="cuda")
    P96 = [ra._ptr(x) for x in (q96, torch.zeros_like(q96), torch.zeros_like(q96),
                                torch.zeros_like(q96))]
    assert ra.ra_watchdog_selftest(*P96, None, 1, 1, 1, 256, 96, 2, 1, 0, 0.0, 1_000_000,
                                   None) == ra.RA_ERR_UNSUPPORTED   # D = 96
    torch.cuda.synchronize()


@pytest.mark.parametrize("which", [0, 1])
def test_backward_kernels_time_out_cleanly(ra, which):
    """The same check for the backward's dq (which = 0) and dk/dv (which = 1)
    kernels: the first K (resp. Q) tile is never loaded, the kernel reports
    RA_ERR_TIMEOUT, and a normal backward right after it is still correct."""
    import torch
    from helpers import assert_grad_close, backward_reference, delta_error_bounds, grad_inputs
    B, Hq, Hkv, S, N, D = 1, 2, 1, 512, 2, 128
    q, k, v = inputs(32 + which, B, Hq, Hkv, S, D, "bf16")
    dout = grad_inputs(32 + which, B, Hq, S, D, "bf16")
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, N, causal=True, striped=True)
    ra.check()
    rc, need = ra.ra_backward_workspace(B, Hq, S, D)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
    stream = ra._stream_handle(None)
    P = ra._ptr
    t0 = time.time()
    rc = ra.ra_watchdog_selftest_backward(P(tq), P(tk), P(tv), P(out), P(lse), P(tg), P(dq),
                                          P(dk), P(dv), P(ws), need, B, Hq, Hkv, S, D, N, 1, 1,
                                          0.0, 20_000_000, which, stream)
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(stream) == ra.RA_ERR_TIMEOUT
    assert time.time() - t0 < 30.0
    assert ra.ra_check(stream) == ra.RA_OK
    assert ra.ra_watchdog_selftest_backward(P(tq), P(tk), P(tv), P(out), P(lse), P(tg), P(dq),
                                            P(dk), P(dv), P(ws), need, B, Hq, Hkv, S, D, N, 1,
                                            1, 0.0, 20_000_000, 2, stream) == ra.RA_ERR_INVALID_ARG
    grads = ra.backward(tq, tk, tv, out, lse, tg, N, causal=True, striped=True, kernel="tc")
    ra.check()
    ref = backward_reference(q, k, v, dout, N, True, True, "bf16")
    bq, bk = delta_error_bounds(q, k, v, dout, N, True, True, "bf16")
    for name, g, r, e in zip(("dq", "dk", "dv"), grads, ref, (bq, bk, None)):
        assert_grad_close(from_device(g), r, "bf16", name, e)

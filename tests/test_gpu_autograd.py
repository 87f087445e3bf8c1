"""The autograd wrapper (ra.attention): its forward is ra.forward's output
bit for bit, the gradients torch computes through it are ra.backward's bit
for bit, and both agree with the oracle."""
import pytest

from helpers import (assert_close, assert_grad_close, backward_reference, delta_error_bounds,
                     from_device, grad_inputs, inputs, reference, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout", [
    (1, 4, 2, 1024, 4, 128, True, 1),   # causal striped GQA
    (2, 2, 2, 512, 2, 64, False, 0),    # non-causal, D = 64
])
def test_autograd_matches_backward_and_oracle(ra, B, Hq, Hkv, S, N, D, causal, layout):
    import torch
    q, k, v = inputs(9900 + S + D, B, Hq, Hkv, S, D, "bf16")
    dout = grad_inputs(9900 + S + D, B, Hq, S, D, "bf16")
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    lq, lk, lv = (t.clone().requires_grad_(True) for t in (tq, tk, tv))
    out = ra.attention(lq, lk, lv, N, causal=causal, striped=layout)
    out.backward(tg)
    ra.check()
    ref_out, ref_lse = ra.forward(tq, tk, tv, N, causal=causal, striped=layout)
    grads = ra.backward(tq, tk, tv, ref_out, ref_lse, tg, N, causal=causal, striped=layout)
    ra.check()
    bits = lambda x: x.view(torch.int16)
    assert torch.equal(bits(out.detach()), bits(ref_out))
    for got, want in zip((lq.grad, lk.grad, lv.grad), grads):
        assert torch.equal(bits(got), bits(want))
    ro, rl = reference(q, k, v, N, causal, layout, "bf16")
    assert_close(from_device(out.detach()), from_device(ref_lse), ro, rl, "bf16", "autograd forward")
    ref = backward_reference(q, k, v, dout, N, causal, layout, "bf16")
    bq, bk = delta_error_bounds(q, k, v, dout, N, causal, layout, "bf16")
    for name, g, r, e in zip(("dq", "dk", "dv"), (lq.grad, lk.grad, lv.grad), ref, (bq, bk, None)):
        assert_grad_close(from_device(g), r, "bf16", name, e)

"""Memory-safety checks of the kernels' stores, in place of a sanitizer.

Every output buffer (out, lse; dq, dk, dv and the backward's workspace) is
allocated inside a larger block: 64 KiB before it and 64 KiB after it are
filled with a byte pattern, and so is the buffer itself.  After the call the
bands must hold the pattern byte for byte (no store before or past a buffer),
and every element of the buffer must hold the oracle's value within the
usual tolerances (no row left unwritten, none overwritten with another row's
data).  The shapes have partial last tiles (shards of 200, 250 and 8000
rows, whose last tiles hold 72, 122 and 64 rows), several batch entries and
heads, and every kernel family: the tensor-core forward and backward and the
SIMT forward and backward.
"""
import numpy as np
import pytest

from helpers import (assert_close, assert_grad_close, backward_reference, delta_error_bounds,
                     from_device, grad_inputs, inputs, reference, to_device)

pytestmark = pytest.mark.gpu

PAD = 1 << 16
BYTE = 0xA5


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


class Guarded:
    """A tensor of `shape` and `dtype` inside a block whose PAD bytes on
    either side, and the tensor itself, start as the byte pattern."""

    def __init__(self, shape, dtype):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.raw = torch.full((2 * PAD + n,), BYTE, dtype=torch.uint8, device="cuda")
        self.t = self.raw[PAD:PAD + n].view(dtype).view(shape)

    def bands_intact(self):
        return bool((self.raw[:PAD] == BYTE).all()) and bool((self.raw[PAD + self.n:] == BYTE).all())


CASES = [
    # B, Hq, Hkv, S, N, D, causal, layout, kernel, dtype
    (2, 4, 2, 600, 3, 128, True, 1, "tc", "bf16"),       # Sb = 200, GQA head pairing
    (2, 3, 3, 1000, 4, 128, True, 0, "tc", "bf16"),      # Sb = 250, MHA query-tile pairing
    (1, 2, 1, 16000, 2, 128, True, 1, "tc", "bf16"),     # Sb = 8000
    (2, 2, 2, 500, 2, 64, False, 0, "tc", "bf16"),       # Sb = 250, D = 64, non-causal
    (2, 2, 1, 600, 3, 100, True, 1, "simt", "bf16"),     # SIMT, D = 100 padded to 128
    (2, 3, 1, 750, 3, 64, True, 0, "simt", "f32"),       # SIMT fp32, Sb = 250
]


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout,kernel,dt", CASES)
def test_forward_and_backward_stay_inside_their_buffers(ra, B, Hq, Hkv, S, N, D, causal, layout,
                                                        kernel, dt):
    import torch
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    rdt = ra.RA_BF16 if dt == "bf16" else ra.RA_F32
    kcode = ra.RA_KERNEL_TC if kernel == "tc" else ra.RA_KERNEL_SIMT
    q, k, v = inputs(9300 + S + D, B, Hq, Hkv, S, D, dt)
    dout = grad_inputs(9300 + S + D, B, Hq, S, D, dt)
    tq, tk, tv, tg = (to_device(x, dt) for x in (q, k, v, dout))
    P = ra._ptr
    st = ra._stream_handle(None)

    out = Guarded((B, Hq, S, D), tdt)
    lse = Guarded((B, Hq, S), torch.float32)
    rc = ra.ra_forward_ex(P(tq), P(tk), P(tv), P(out.t), P(lse.t), B, Hq, Hkv, S, D, N,
                          int(causal), layout, 0.0, rdt, kcode, st)
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(st) == ra.RA_OK
    assert out.bands_intact() and lse.bands_intact()
    ro, rl = reference(q, k, v, N, causal, layout, dt)
    assert_close(from_device(out.t), from_device(lse.t), ro, rl, dt, "guarded forward")

    rc, need = ra.ra_backward_workspace(B, Hq, S, D)
    assert rc == ra.RA_OK
    ws = Guarded((need,), torch.uint8)
    grads = [Guarded((B, Hq, S, D), tdt), Guarded((B, Hkv, S, D), tdt),
             Guarded((B, Hkv, S, D), tdt)]
    rc = ra.ra_backward_ex(P(tq), P(tk), P(tv), P(out.t), P(lse.t), P(tg),
                           *[P(g.t) for g in grads], P(ws.t), need, B, Hq, Hkv, S, D, N,
                           int(causal), layout, 0.0, rdt, kcode, st)
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(st) == ra.RA_OK
    for name, g in zip(("dq", "dk", "dv", "workspace"), grads + [ws]):
        assert g.bands_intact(), name
    ref = backward_reference(q, k, v, dout, N, causal, layout, dt)
    bq, bk = delta_error_bounds(q, k, v, dout, N, causal, layout, dt)
    for name, g, r, e in zip(("dq", "dk", "dv"), grads, ref, (bq, bk, None)):
        assert_grad_close(from_device(g.t), r, dt, f"guarded {name}", e)

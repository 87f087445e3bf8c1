"""GPU parity of the backward (ra_backward through the C ABI) against the
oracle's gradients.

The forward runs first through the library (its out and lse feed the
backward, as in training); the oracle computes dq, dk, dv from the inputs
alone by the plain chain rule in float64.  Shapes span several tiles, a
ragged last tile, GQA groups, every layout and causal/non-causal.  Bounds:
tests/helpers.py TOL_BWD (row-wise and normwise).
"""
import numpy as np
import pytest

from helpers import (assert_grad_close, backward_reference, delta_error_bounds, from_device,
                     grad_inputs, inputs, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def run_backward(ra, seed, B, Hq, Hkv, S, N, D, causal, layout, dtype, kernel, scale=None):
    q, k, v = inputs(seed, B, Hq, Hkv, S, D, dtype)
    dout = grad_inputs(seed, B, Hq, S, D, dtype)
    tq, tk, tv, tg = (to_device(x, dtype) for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, N, causal=causal, striped=layout, scale=scale)
    dq, dk, dv = ra.backward(tq, tk, tv, out, lse, tg, N, causal=causal, striped=layout,
                             scale=scale, kernel=kernel)
    ra.check()
    ref = backward_reference(q, k, v, dout, N, causal, layout, dtype, scale)
    bq, bk = delta_error_bounds(q, k, v, dout, N, causal, layout, dtype, scale)
    return [from_device(x) for x in (dq, dk, dv)], ref, (bq, bk, None)


SIMT_F32 = [
    # B, Hq, Hkv, S, N, D, causal, layout
    (1, 1, 1, 32, 4, 16, False, 0),     # the glossary page's toy shape
    (1, 1, 1, 32, 4, 16, True, 1),
    (2, 4, 2, 96, 3, 24, True, 1),
    (1, 3, 1, 200, 5, 64, True, 0),
    (1, 2, 2, 384, 2, 128, False, 0),
    (1, 2, 1, 256, 4, 32, True, 2),
    (1, 1, 1, 7, 1, 5, True, 0),
    (1, 1, 1, 1, 1, 8, True, 1),
    # register-blocked kernels: several 64-row blocks, ragged shards, zigzag
    (1, 2, 1, 1000, 4, 128, True, 1),   # Sb = 250
    (2, 4, 2, 640, 5, 64, False, 0),    # Sb = 128
    (1, 2, 2, 512, 4, 32, True, 2),     # zigzag
    # head dimensions padded up to the tiled kernels' 128 / 32 variants: the
    # partial-vector staging and the padded columns of the epilogue
    (1, 2, 1, 300, 3, 100, True, 0),    # D = 100 in the 128 variant, GQA
    (1, 4, 2, 256, 2, 20, True, 1),     # D = 20 in the 32 variant, GQA
    (1, 2, 2, 192, 3, 4, False, 0),     # D = 4, the smallest
]


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout", SIMT_F32)
def test_simt_backward_f32(ra, B, Hq, Hkv, S, N, D, causal, layout):
    got, ref, ext = run_backward(ra, 7100 + S + D, B, Hq, Hkv, S, N, D, causal, layout, "f32",
                                 "simt")
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, ext):
        assert_grad_close(g, r, "f32", name, e)


SIMT_BF16 = [
    (1, 4, 2, 1024, 4, 128, True, 1),
    (1, 2, 2, 512, 2, 64, False, 0),
    (1, 2, 1, 1000, 4, 128, True, 0),   # Sb = 250: ragged
    (1, 2, 1, 1024, 4, 128, True, 2),
]


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout", SIMT_BF16)
def test_simt_backward_bf16(ra, B, Hq, Hkv, S, N, D, causal, layout):
    got, ref, ext = run_backward(ra, 7200 + S + D, B, Hq, Hkv, S, N, D, causal, layout, "bf16",
                                 "simt")
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, ext):
        fro, worst = assert_grad_close(g, r, "bf16", name, e)
        print(f"simt bf16 {S} {N} {layout} {name}: normwise {fro:.2e} worst row {worst:.2e}")


def test_backward_scale_argument(ra):
    got, ref, ext = run_backward(ra, 7300, 1, 2, 1, 256, 2, 64, True, 1, "f32", "simt",
                                 scale=0.05)
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, ext):
        assert_grad_close(g, r, "f32", name, e)


def test_backward_workspace_and_argument_checks(ra):
    import torch
    rc, need = ra.ra_backward_workspace(1, 2, 256, 64)
    assert rc == ra.RA_OK and need == 256 * 2 * 4
    q = torch.zeros((1, 2, 256, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 2, 256), dtype=torch.float32, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    P = ra._ptr
    args = [P(q), P(k), P(k), P(q), P(lse), P(q), P(q.clone()), P(k.clone()), P(k.clone()),
            P(ws)]
    common = (1, 2, 1, 256, 64, 2, 1, 1, 0.0, ra.RA_BF16, None)
    assert ra.ra_backward(*args, need - 16, *common) == ra.RA_ERR_CAPACITY
    bad = list(args)
    bad[4] = None
    assert ra.ra_backward(*bad, need, *common) == ra.RA_ERR_INVALID_ARG
    torch.cuda.synchronize()


TC_BF16 = [
    # B, Hq, Hkv, S, N, D, causal, layout
    (1, 2, 2, 256, 1, 128, False, 0),    # one ring device, two tiles
    (1, 4, 2, 1024, 4, 128, True, 1),    # GQA, striped
    (1, 2, 1, 1024, 2, 128, True, 0),    # contiguous
    (1, 2, 1, 2048, 4, 128, True, 2),    # zigzag: four tiles per shard
    (2, 3, 1, 768, 2, 128, True, 1),     # odd GQA group, B = 2
    (1, 2, 2, 1000, 4, 128, True, 1),    # Sb = 250: ragged last tile, striped
    (1, 2, 1, 1000, 4, 128, True, 0),    # ragged, contiguous
    (1, 1, 1, 200, 2, 128, False, 0),    # one partial tile per shard
    (1, 1, 1, 128, 1, 128, True, 0),     # a single tile
    (2, 2, 2, 512, 1, 128, False, 0),    # B = 2, one ring device, no GQA
    (1, 8, 1, 1024, 8, 128, True, 1),    # GQA group of 8, one tile per shard
    (1, 2, 1, 2048, 16, 128, True, 0),   # 16 shards of one tile, contiguous
    (1, 2, 1, 2048, 16, 128, True, 1),   # 16 shards of one tile, striped
    (1, 2, 1, 130, 1, 128, True, 1),     # Sb = 130: ragged, one ring device
    (2, 2, 2, 1536, 3, 128, True, 2),    # zigzag, B = 2, two tiles per chunk
    (1, 4, 2, 1024, 4, 64, True, 1),     # D = 64: one box per tile, striped GQA
    (1, 2, 2, 512, 2, 64, False, 0),     # D = 64, non-causal
    (1, 2, 1, 1000, 4, 64, True, 0),     # D = 64, ragged
    (1, 2, 1, 2048, 4, 64, True, 2),     # D = 64, zigzag
]


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout", TC_BF16)
def test_tc_backward_bf16(ra, B, Hq, Hkv, S, N, D, causal, layout):
    got, ref, ext = run_backward(ra, 7400 + S + Hq, B, Hq, Hkv, S, N, D, causal, layout, "bf16",
                                 "tc")
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, ext):
        fro, worst = assert_grad_close(g, r, "bf16", name, e)
        print(f"tc bf16 {S} {N} {layout} {name}: normwise {fro:.2e} worst row {worst:.2e}")


def test_tc_backward_custom_scale(ra):
    got, ref, ext = run_backward(ra, 7600, 1, 4, 2, 1024, 4, 128, True, 1, "bf16", "tc",
                                 scale=0.05)
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, ext):
        assert_grad_close(g, r, "bf16", name, e)


def test_tc_backward_is_deterministic(ra):
    """No atomics: two calls on the same inputs give the same bits."""
    import torch
    B, Hq, Hkv, S, N, D = 1, 4, 2, 2048, 4, 128
    q, k, v = inputs(7500, B, Hq, Hkv, S, D, "bf16")
    dout = grad_inputs(7500, B, Hq, S, D, "bf16")
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, N, causal=True, striped=1)
    a = ra.backward(tq, tk, tv, out, lse, tg, N, causal=True, striped=1, kernel="tc")
    b = ra.backward(tq, tk, tv, out, lse, tg, N, causal=True, striped=1, kernel="tc")
    ra.check()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))

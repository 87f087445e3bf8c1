"""Seeded random shapes through the tensor-core kernels, forward and
backward, against the oracle: batch 1-2, GQA groups 1-4, 1-6 ring devices,
shards of any size (ragged last tiles included; zigzag with whole-tile
chunks), every layout, causal or not, D = 64 or 128.  The shapes are drawn
once from a fixed seed, so a failure names a reproducible case."""
import numpy as np
import pytest

from helpers import (assert_close, assert_grad_close, backward_reference, delta_error_bounds,
                     from_device, grad_inputs, inputs, reference, to_device)

pytestmark = pytest.mark.gpu


def _draw(n, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        B = int(rng.integers(1, 3))
        Hkv = int(rng.integers(1, 3))
        g = int(rng.choice([1, 2, 3, 4]))
        N = int(rng.integers(1, 7))
        layout = int(rng.integers(0, 3))
        causal = bool(rng.integers(0, 2)) or layout != 0
        D = int(rng.choice([64, 128]))
        if layout == 2:
            Sb = 256 * int(rng.integers(1, 4))            # zigzag chunks of whole tiles
        else:
            Sb = int(rng.integers(1, 700))
        cases.append((B, Hkv * g, Hkv, N * Sb, N, D, causal, layout))
    return cases


CASES = _draw(16)


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_random_shape_forward_and_backward(ra, case):
    B, Hq, Hkv, S, N, D, causal, layout = case
    seed = 5000 + S + 3 * Hq + D
    q, k, v = inputs(seed, B, Hq, Hkv, S, D, "bf16")
    dout = grad_inputs(seed, B, Hq, S, D, "bf16")
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, N, causal=causal, striped=layout, kernel="tc")
    grads = ra.backward(tq, tk, tv, out, lse, tg, N, causal=causal, striped=layout, kernel="tc")
    ra.check()
    ro, rl = reference(q, k, v, N, causal, layout, "bf16")
    assert_close(from_device(out), from_device(lse), ro, rl, "bf16", f"forward {case}")
    ref = backward_reference(q, k, v, dout, N, causal, layout, "bf16")
    bq, bk = delta_error_bounds(q, k, v, dout, N, causal, layout, "bf16")
    for name, g_, r, e in zip(("dq", "dk", "dv"), grads, ref, (bq, bk, None)):
        assert_grad_close(from_device(g_), r, "bf16", f"{name} {case}", e)

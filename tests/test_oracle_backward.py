"""Pins for the oracle's gradients, each against something other than itself.

* central finite differences of the forward definition (itself pinned by
  brute force in test_oracle.py) on tiny inputs;
* a library routine: torch's scaled_dot_product_attention on CPU in float64,
  differentiated by autograd;
* closed forms: with every value row equal, O is that row whatever the
  scores, so dQ = dK = 0; with Q = 0 the weights are uniform over the visible
  keys, so dV_u is a plain average of dO over the rows that see u, and dK = 0;
* invariants: adding a constant to a row's scores changes nothing, so the
  key gradients sum to zero over keys; every row's weights sum to one, so the
  value gradients sum to the sum of dO;
* the ring-order backward equals the plain gradients for every layout.
"""
import math

import numpy as np
import pytest

import oracle


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def loss(q, k, v, dout, causal, scale=None):
    o, _ = oracle.full_attention(q, k, v, causal, scale)
    return float((o * dout).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 2), (3, 1)])
def test_gradients_match_finite_differences(causal, Hq, Hkv):
    B, S, D = 1, 7, 3
    q, k, v = rnd((B, Hq, S, D), 11), rnd((B, Hkv, S, D), 12), rnd((B, Hkv, S, D), 13)
    dout = rnd((B, Hq, S, D), 14)
    scale = 0.7
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, causal, scale, chunk=3)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"], dout, causal, scale)
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"], dout, causal, scale)
            fd[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, fd, rtol=0, atol=2e-8, err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 1)])
def test_gradients_match_torch_autograd(causal, Hq, Hkv):
    torch = pytest.importorskip("torch")
    B, S, D = 2, 40, 16
    q, k, v = rnd((B, Hq, S, D), 21), rnd((B, Hkv, S, D), 22), rnd((B, Hkv, S, D), 23)
    dout = rnd((B, Hq, S, D), 24)
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, causal, chunk=16)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    g = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1), is_causal=causal)
    o.backward(torch.tensor(dout, dtype=torch.float64))
    for mine, lib in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine, lib.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_value_rows_give_zero_query_and_key_gradients(causal):
    B, Hq, Hkv, S, D = 1, 2, 1, 24, 8
    q, k = rnd((B, Hq, S, D), 31), rnd((B, Hkv, S, D), 32)
    v = np.broadcast_to(rnd((1, 1, 1, D), 33), (B, Hkv, S, D)).copy()
    dout = rnd((B, Hq, S, D), 34)
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, causal)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv).max() > 0.1


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_closed_form(causal):
    """Q = 0: row t weighs its n_t visible keys equally (n_t = t + 1 causal,
    S otherwise), so dV_u = sum over rows t that see u of dO_t / n_t; the
    key gradient is scale * dS^T Q = 0."""
    B, Hq, Hkv, S, D = 1, 3, 1, 20, 4
    q = np.zeros((B, Hq, S, D))
    k, v = rnd((B, Hkv, S, D), 41), rnd((B, Hkv, S, D), 42)
    dout = rnd((B, Hq, S, D), 43)
    _, dk, dv = oracle.attention_backward(q, k, v, dout, causal)
    want = np.zeros((S, D))
    for h in range(Hq):
        for u in range(S):
            for t in range(S):
                if causal and t < u:
                    continue
                want[u] += dout[0, h, t] / ((t + 1) if causal else S)
    np.testing.assert_allclose(dv[0, 0], want, rtol=0, atol=1e-12)
    assert np.abs(dk).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sums_over_keys(causal):
    B, Hq, Hkv, S, D = 2, 4, 2, 33, 6
    q, k, v = rnd((B, Hq, S, D), 51), rnd((B, Hkv, S, D), 52), rnd((B, Hkv, S, D), 53)
    dout = rnd((B, Hq, S, D), 54)
    _, dk, dv = oracle.attention_backward(q, k, v, dout, causal, chunk=10)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-11)
    want = dout.reshape(B, Hkv, Hq // Hkv, S, D).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), want, rtol=0, atol=1e-11)


@pytest.mark.parametrize("N", [1, 2, 4])
@pytest.mark.parametrize("causal,layout", [(False, 0), (True, 0), (True, 1), (True, 2)])
def test_ring_backward_equals_plain(N, causal, layout):
    B, Hq, Hkv, S, D = 1, 4, 2, 48, 8
    q, k, v = rnd((B, Hq, S, D), 61), rnd((B, Hkv, S, D), 62), rnd((B, Hkv, S, D), 63)
    dout = rnd((B, Hq, S, D), 64)
    ref = oracle.attention_backward(q, k, v, dout, causal, chunk=20)
    sm = [oracle.to_shard_major(x, N, layout) for x in (q, k, v, dout)]
    got = oracle.ring_attention_backward(*sm, N, causal, layout)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(oracle.to_token_order(g, N, layout), r, rtol=0, atol=1e-11)


@pytest.mark.parametrize("N", [1, 3, 4])
@pytest.mark.parametrize("causal,layout", [(False, 0), (True, 0), (True, 1), (True, 2)])
def test_ring_steps_sum_to_the_plain_gradients(N, causal, layout):
    """The one-step function a device applies (ring_step_backward_block), run
    for every device i and step s with block j = (i - s) mod N, each device
    seeing only its own shard and the block it holds, adds up to the plain
    gradients (pinned above by finite differences and autograd)."""
    if layout == 2 and N == 3:
        N = 2  # zigzag needs an even number of chunks per shard below
    B, Hq, Hkv, S, D = 2, 4, 2, 48, 8
    q, k, v = rnd((B, Hq, S, D), 65), rnd((B, Hkv, S, D), 66), rnd((B, Hkv, S, D), 67)
    dout = rnd((B, Hq, S, D), 68)
    ref = oracle.attention_backward(q, k, v, dout, causal, chunk=20)
    o, lse = oracle.full_attention(q, k, v, causal)
    delta = (dout * o).sum(axis=-1)
    sm = [oracle.to_shard_major(x, N, layout) for x in (q, k, v, dout)]
    lse_sm = oracle.to_shard_major(lse[..., None], N, layout)[..., 0]
    delta_sm = oracle.to_shard_major(delta[..., None], N, layout)[..., 0]
    Sb = S // N
    sh = lambda x, i: x[:, :, i * Sb:(i + 1) * Sb]
    dq = np.zeros_like(sm[0])
    dk = np.zeros_like(sm[1])
    dv = np.zeros_like(sm[2])
    for s in range(N):
        for i in range(N):
            j = (i - s) % N
            a, b, c = oracle.ring_step_backward_block(
                sh(sm[0], i), sh(sm[1], j), sh(sm[2], j), sh(sm[3], i), sh(lse_sm, i),
                sh(delta_sm, i), N, i, j, causal, layout)
            dq[:, :, i * Sb:(i + 1) * Sb] += a
            dk[:, :, j * Sb:(j + 1) * Sb] += b
            dv[:, :, j * Sb:(j + 1) * Sb] += c
    for got, want in zip((dq, dk, dv), ref):
        np.testing.assert_allclose(oracle.to_token_order(got, N, layout), want, rtol=0,
                                   atol=1e-11)


def test_ring_backward_scale_argument():
    """Scaling q by r and the scale by 1/r leaves every score unchanged; by
    the chain rule dQ then scales by 1/r while dK and dV are unchanged."""
    B, Hq, Hkv, S, D, N = 1, 2, 1, 16, 4, 4
    q, k, v = rnd((B, Hq, S, D), 71), rnd((B, Hkv, S, D), 72), rnd((B, Hkv, S, D), 73)
    dout = rnd((B, Hq, S, D), 74)
    r = 0.3 / (1 / math.sqrt(D))
    a = oracle.ring_attention_backward(q, k, v, dout, N, True, 1, scale=0.3)
    b = oracle.ring_attention_backward(q * r, k, v, dout, N, True, 1)  # default 1/sqrt(D)
    np.testing.assert_allclose(a[0], b[0] * r, rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[2], b[2], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,layout", [(False, 0), (True, 1), (True, 2)])
def test_backward_rows_equal_the_full_gradient(causal, layout):
    """The per-row dq (used on sampled rows at full size) equals the rows of
    the plain gradient, rows taken in shard-major order with their token
    positions."""
    B, Hq, Hkv, S, D, N = 1, 2, 1, 64, 8, 4
    q, k, v = rnd((B, Hq, S, D), 81), rnd((B, Hkv, S, D), 82), rnd((B, Hkv, S, D), 83)
    dout = rnd((B, Hq, S, D), 84)
    dq, _, _ = oracle.attention_backward(q, k, v, dout, causal)
    pos = oracle.positions(S, N, layout)
    sm = [oracle.to_shard_major(x, N, layout) for x in (q, k, v, dout)]
    dq_sm = oracle.to_shard_major(dq, N, layout)
    rows = [0, 5, 17, 40, 63]
    for h in range(Hq):
        got = oracle.attention_backward_rows(sm[0][0, h, rows], pos[rows], sm[3][0, h, rows],
                                             sm[1][0, 0], sm[2][0, 0], pos, causal,
                                             1 / math.sqrt(D))
        np.testing.assert_allclose(got, dq_sm[0, h, rows], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_score_closed_form_equals_the_full_gradient(causal):
    """With K = 0 the prefix-sum closed form (used at full size) equals the
    plain gradient."""
    B, Hq, Hkv, S, D = 2, 4, 2, 50, 6
    q, v = rnd((B, Hq, S, D), 91), rnd((B, Hkv, S, D), 92)
    dout = rnd((B, Hq, S, D), 93)
    k = np.zeros((B, Hkv, S, D))
    _, dk, dv = oracle.attention_backward(q, k, v, dout, causal)
    rows = [0, 1, 13, 49]
    dk_cf, dv_cf = oracle.backward_uniform_scores(q, v, dout, causal, dk_rows=rows)
    np.testing.assert_allclose(dv_cf, dv, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk_cf, dk[:, :, rows], rtol=0, atol=1e-12)
    dk_all, _ = oracle.backward_uniform_scores(q, v, dout, causal)
    np.testing.assert_allclose(dk_all, dk, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_rows_match_torch_autograd(causal):
    """dk, dv of chosen key rows (used on sampled key rows at full size),
    summed over the query heads of a GQA group, against torch autograd of the
    whole problem.  Under the causal mask only the queries at or after the
    earliest chosen key are passed, which must be enough."""
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, S, D = 1, 4, 2, 40, 16
    q, k, v = rnd((B, Hq, S, D), 31), rnd((B, Hkv, S, D), 32), rnd((B, Hkv, S, D), 33)
    dout = rnd((B, Hq, S, D), 34)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    g = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1), is_causal=causal)
    o.backward(torch.tensor(dout, dtype=torch.float64))
    keys = [25, 26, 31, 39] if causal else [0, 7, 25, 39]
    t0 = keys[0] if causal else 0
    pos = np.arange(S)
    for kvh in range(Hkv):
        dk = np.zeros((len(keys), D))
        dv = np.zeros((len(keys), D))
        for h in range(kvh * g, (kvh + 1) * g):
            a, b = oracle.attention_backward_key_rows(
                q[0, h, t0:], pos[t0:], dout[0, h, t0:], k[0, kvh], v[0, kvh], pos, keys,
                causal, 1 / math.sqrt(D), chunk=7)
            dk += a
            dv += b
        np.testing.assert_allclose(dk, tk.grad[0, kvh, keys].numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dv, tv.grad[0, kvh, keys].numpy(), rtol=0, atol=1e-11)


def test_ring_step_backward_scale_argument():
    """The one-step function under a scale argument: scaling q by r and the
    scale by 1/r leaves P unchanged, so dq scales by 1/r and dk, dv do not
    change (the chain rule through s = scale q.k)."""
    B, Hq, Hkv, Sb, D, N, i, j = 1, 2, 1, 8, 4, 4, 2, 1
    q, k, v = rnd((B, Hq, Sb, D), 81), rnd((B, Hkv, Sb, D), 82), rnd((B, Hkv, Sb, D), 83)
    dout = rnd((B, Hq, Sb, D), 84)
    lse, delta = rnd((B, Hq, Sb), 85) + 3.0, rnd((B, Hq, Sb), 86)
    r = 0.3 / (1 / math.sqrt(D))
    a = oracle.ring_step_backward_block(q, k, v, dout, lse, delta, N, i, j, True, 1, scale=0.3)
    b = oracle.ring_step_backward_block(q * r, k, v, dout, lse, delta, N, i, j, True, 1)
    np.testing.assert_allclose(a[0], b[0] * r, rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[2], b[2], rtol=0, atol=1e-12)
    # a block no query of the shard sees (contiguous causal, j > i) adds nothing
    z = oracle.ring_step_backward_block(q, k, v, dout, lse, delta, N, 1, 3, True, 0)
    assert all(not x.any() for x in z)

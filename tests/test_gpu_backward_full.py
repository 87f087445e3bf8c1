"""Backward parity at full size, launched the way the bench launches it
(ra.backward over the whole workload, tensor-core path).

* noncausal_8k (B=1, 8 heads, S=8192, N=8): every element of dq, dk and dv
  against the oracle's gradient.
* gqa_128k (the bench workload: 32 query heads on 8 KV heads, S=131072 in
  16 striped shards, causal):
  - random inputs: stratified sampled rows of dq against the per-row oracle,
    and dk, dv of sampled key rows (among the last 1024 tokens, whose
    gradients need at most 1024 query rows per head) against the oracle;
  - uniform scores (K = 0, random q, v, dout): every row of dv and sampled
    rows of dk against the oracle's prefix-sum closed form, and dq exactly 0.
    All tiles, masks and ring steps run; only the score values are trivial.
* long_1m (8 query heads on one KV head, S=1048576 in 64 striped shards):
  every gradient element written, and stratified dq rows against the oracle.
Bounds: tests/helpers.py TOL_BWD plus the delta term of delta_error_bounds.
"""
import math

import numpy as np
import pytest

import oracle
import ragen
from ragen import WORKLOADS

from helpers import (TOL_BWD, assert_grad_close, backward_reference, delta_error_bounds,
                     from_device, grad_inputs, inputs, key_rows_delta_bound, sample_rows,
                     to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def test_backward_noncausal_8k_every_element(ra):
    wl = WORKLOADS["noncausal_8k"]
    q, k, v = inputs(wl.seed, wl.B, wl.Hq, wl.Hkv, wl.S, wl.D, "bf16")
    dout = grad_inputs(wl.seed, wl.B, wl.Hq, wl.S, wl.D, "bf16")
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, wl.N, causal=wl.causal, striped=wl.striped)
    got = ra.backward(tq, tk, tv, out, lse, tg, wl.N, causal=wl.causal, striped=wl.striped)
    ra.check()
    ref = backward_reference(q, k, v, dout, wl.N, wl.causal, wl.striped, "bf16")
    bq, bk = delta_error_bounds(q, k, v, dout, wl.N, wl.causal, wl.striped, "bf16")
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, (bq, bk, None)):
        fro, worst = assert_grad_close(from_device(g), r, "bf16", name, e)
        print(f"noncausal_8k {name}: normwise {fro:.2e}")


def _host_inputs(wl, tensors):
    """The workload's bf16 tensors from the generator, as uint16 host arrays."""
    qs, kvs = wl.shapes()
    shapes = {ragen.TENSOR_Q: qs, ragen.TENSOR_K: kvs, ragen.TENSOR_V: kvs, ragen.TENSOR_DO: qs}
    return [ragen.normal_bf16(wl.seed, t, int(np.prod(shapes[t]))).reshape(shapes[t])
            for t in tensors]


@pytest.fixture(scope="module")
def gqa_128k_grads(ra):
    """The bench workload's forward and backward on random inputs (host
    arrays of the inputs, device gradients)."""
    wl = WORKLOADS["gqa_128k"]
    q, k, v, dout = _host_inputs(wl, (ragen.TENSOR_Q, ragen.TENSOR_K, ragen.TENSOR_V,
                                      ragen.TENSOR_DO))
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, wl.N, causal=wl.causal, striped=wl.striped)
    dq, dk, dv = ra.backward(tq, tk, tv, out, lse, tg, wl.N, causal=wl.causal,
                             striped=wl.striped)
    ra.check()
    del tq, tk, tv, tg, out, lse
    return wl, (q, k, v, dout), (dq, dk, dv)


def test_backward_gqa_128k_sampled_dk_dv_rows(gqa_128k_grads):
    """Random inputs: dk and dv of sampled key rows against the oracle.  A
    key's gradient needs every query row that sees it, each with its full
    softmax, so the sample is taken among the last 1024 tokens (seen by at
    most 1024 queries per head): they lie in the last key tile of every one
    of the 16 shards, visited by query tiles of every shard.  Two KV heads,
    each summing its four query heads."""
    wl, (q, k, v, dout), (dq, dk, dv) = gqa_128k_grads
    S, N, D = wl.S, wl.N, wl.D
    g = wl.Hq // wl.Hkv
    sc = 1.0 / math.sqrt(D)
    pos = oracle.positions(S, N, wl.striped)
    inv = np.empty(S, dtype=np.int64)
    inv[pos] = np.arange(S)            # token t sits at shard-major row inv[t]
    rng = np.random.default_rng(wl.seed + 5)
    keys = sorted({S - 1024, S - 1} | set(rng.integers(S - 1024, S, 30).tolist()))
    t0 = keys[0]
    tok = np.arange(S)
    qs, _ = wl.shapes()
    for kvh in (0, wl.Hkv - 1):
        K = oracle.to_token_order(oracle.bf16_bits_to_f64(k[0, kvh]), N, wl.striped)
        V = oracle.to_token_order(oracle.bf16_bits_to_f64(v[0, kvh]), N, wl.striped)
        dk_ref = np.zeros((len(keys), D))
        dv_ref = np.zeros((len(keys), D))
        extra = np.zeros(len(keys))
        for h in range(kvh * g, (kvh + 1) * g):
            Qw = oracle.to_token_order(oracle.bf16_bits_to_f64(q[0, h]), N, wl.striped)[t0:]
            dOw = oracle.to_token_order(oracle.bf16_bits_to_f64(dout[0, h]), N, wl.striped)[t0:]
            a, b = oracle.attention_backward_key_rows(Qw, tok[t0:], dOw, K, V, tok, keys,
                                                      wl.causal, sc)
            dk_ref += a
            dv_ref += b
            extra += key_rows_delta_bound(Qw, tok[t0:], dOw, K, V, tok, keys, wl.causal, sc)
        rows = torch_rows(dk, 0, kvh, inv[keys])
        assert_grad_close(rows, dk_ref, "bf16", f"dk kv head {kvh}", np.sqrt(extra))
        assert_grad_close(torch_rows(dv, 0, kvh, inv[keys]), dv_ref, "bf16",
                          f"dv kv head {kvh}")


def torch_rows(t, b, h, rows):
    import torch
    return t[b, h][torch.as_tensor(np.asarray(rows), device=t.device)].double().cpu().numpy()


def test_backward_gqa_128k_sampled_dq_rows(gqa_128k_grads):
    wl, (q, k, v, dout), (dq, dk, dv) = gqa_128k_grads
    _check_dq_rows(wl, q, k, v, dout, dq, 96)


def test_backward_long_1m_sampled_dq_rows(ra):
    """1M tokens (8 query heads on one KV head, 64 striped shards): the dq
    kernel's query tiles enter the ring at block N-1 here (its concurrent
    blocks exceed the L2).  NaN-filled gradients must be written everywhere,
    and stratified dq rows match the per-row oracle."""
    import torch
    wl = WORKLOADS["long_1m"]
    q, k, v, dout = _host_inputs(wl, (ragen.TENSOR_Q, ragen.TENSOR_K, ragen.TENSOR_V,
                                      ragen.TENSOR_DO))
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, wl.N, causal=wl.causal, striped=wl.striped)
    nan = float("nan")
    dq = torch.full_like(tq, nan)
    dk = torch.full_like(tk, nan)
    dv = torch.full_like(tv, nan)
    ra.backward(tq, tk, tv, out, lse, tg, wl.N, causal=wl.causal, striped=wl.striped,
                dq=dq, dk=dk, dv=dv)
    ra.check()
    del tq, tk, tv, tg, out, lse
    for t in (dq, dk, dv):
        flat = t.view(-1, wl.D)
        for r0 in range(0, flat.shape[0], 1 << 22):
            assert bool(torch.isfinite(flat[r0:r0 + (1 << 22)]).all())
    _check_dq_rows(wl, q, k, v, dout, dq, 48)


def _check_dq_rows(wl, q, k, v, dout, dq, n_rows):
    """Sampled dq rows against the per-row oracle, within TOL_BWD plus the
    delta term of each row's error bound."""
    rows = sample_rows(wl.seed + 1, wl.B, wl.Hq, wl.S, wl.N, n_rows)
    g = wl.Hq // wl.Hkv
    sc = 1.0 / math.sqrt(wl.D)
    pos = oracle.positions(wl.S, wl.N, wl.striped)
    lam, u = 8.0, 2.0 ** -9
    errs, bounds, norms = [], [], []
    cache = {}
    for (b, h, p) in rows:
        if (b, h // g) not in cache:
            cache.clear()
            cache[(b, h // g)] = (oracle.bf16_bits_to_f64(k[b, h // g]),
                                  oracle.bf16_bits_to_f64(v[b, h // g]))
        K, V = cache[(b, h // g)]
        qr = oracle.bf16_bits_to_f64(q[b, h, p])[None]
        gr = oracle.bf16_bits_to_f64(dout[b, h, p])[None]
        ref = oracle.attention_backward_rows(qr, pos[[p]], gr, K, V, pos, wl.causal, sc)[0]
        # the delta term of delta_error_bounds for this row
        o, l = oracle.attend_rows(qr, pos[[p]], K, V, pos, wl.causal, sc)
        P = np.exp(np.where(pos <= pos[p], (qr @ K.T)[0] * sc, -np.inf) - l[0])
        var_o = o[0] ** 2 + (P ** 2) @ (V ** 2)
        dd = lam * u * math.sqrt(float((gr[0] ** 2 * var_o).sum()))
        extra = sc * dd * float(np.linalg.norm(P @ K))
        got = from_device(dq[b, h, p])
        errs.append(float(np.linalg.norm(got - ref)))
        bounds.append(extra)
        norms.append(float(np.linalg.norm(ref)))
    norms = np.array(norms)
    tol = TOL_BWD["bf16"]
    bound = tol["row_rtol"] * norms + tol["row_atol"] * float(np.median(norms)) + \
        tol["floor"] + np.array(bounds)
    errs = np.array(errs)
    worst = int(np.argmax(errs - bound))
    assert (errs <= bound).all(), (rows[worst], errs[worst], bound[worst], norms[worst])
    print(f"{wl.name} dq: {len(rows)} rows, worst error/|row| "
          f"{float((errs / np.maximum(norms, 1e-30)).max()):.2e}")


def test_backward_gqa_128k_uniform_scores(ra):
    """K = 0: every score is zero, each row weighs its visible keys equally."""
    import torch
    wl = WORKLOADS["gqa_128k"]
    q, v, dout = _host_inputs(wl, (ragen.TENSOR_Q, ragen.TENSOR_V, ragen.TENSOR_DO))
    k = np.zeros_like(v)
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, wl.N, causal=wl.causal, striped=wl.striped)
    dq, dk, dv = ra.backward(tq, tk, tv, out, lse, tg, wl.N, causal=wl.causal,
                             striped=wl.striped)
    ra.check()
    assert int(torch.count_nonzero(dq)) == 0
    g = wl.Hq // wl.Hkv
    S, N, D = wl.S, wl.N, wl.D
    sc = 1.0 / math.sqrt(D)
    pos = oracle.positions(S, N, wl.striped)
    inv = np.empty(S, dtype=np.int64)
    inv[pos] = np.arange(S)            # token t sits at shard-major row inv[t]
    rng = np.random.default_rng(wl.seed + 2)
    dk_tok = sorted({0, 1, 127, 128, S - 1} | set(rng.integers(0, S, 27).tolist()))
    n = np.arange(1, S + 1, dtype=np.float64)
    lam, u = 8.0, 2.0 ** -9
    tol = TOL_BWD["bf16"]
    dv_h = from_device(dv)
    dk_h = from_device(dk)
    for b in range(wl.B):
        for kvh in range(wl.Hkv):
            hs = slice(kvh * g, (kvh + 1) * g)
            to_tok = lambda x: oracle.to_token_order(oracle.bf16_bits_to_f64(x), N, wl.striped)
            Q, V, dO = to_tok(q[b:b + 1, hs]), to_tok(v[b:b + 1, kvh:kvh + 1]), \
                to_tok(dout[b:b + 1, hs])
            dk_ref, dv_ref = oracle.backward_uniform_scores(Q, V, dO, wl.causal, dk_rows=dk_tok)
            # every dv row, in token order
            got_dv = dv_h[b, kvh][inv]
            assert_grad_close(got_dv, dv_ref[0, 0], "bf16", f"dv kv head {kvh}")
            # sampled dk rows with the delta term (P = 1/n_t, O_t = prefix mean of v)
            vbar = np.cumsum(V[0, 0], axis=0) / n[:, None]
            v2 = np.cumsum(V[0, 0] ** 2, axis=0) / n[:, None] ** 2
            extra = np.zeros(len(dk_tok))
            for hh in range(g):
                dd = lam * u * np.sqrt((dO[0, hh] ** 2 * (vbar ** 2 + v2)).sum(axis=1))
                w = (sc * dd * np.linalg.norm(Q[0, hh], axis=1) / n) ** 2
                suffix = np.cumsum(w[::-1])[::-1]
                extra += suffix[dk_tok]
            got_dk = dk_h[b, kvh][inv[dk_tok]]
            assert_grad_close(got_dk, dk_ref[0, 0], "bf16", f"dk kv head {kvh}",
                              np.sqrt(extra))

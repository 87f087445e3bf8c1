"""Test-side glue: seeded inputs from ragen, torch device copies, oracle
references in shard-major order, and error metrics.  Shares no code with the
CUDA path (which it reaches only through the C-ABI binding)."""
from __future__ import annotations

import math

import numpy as np

import oracle
import ragen

# tolerances: fp32 path max-abs 1e-5; bf16 path max-abs 2e-2 and mean-abs 2e-3
# on the output (bf16 output upcast to float64 vs the float64 oracle); lse
# max-abs 1e-4 (fp32) / 2e-3 (bf16)
TOL = {"f32": dict(max_abs=1e-5, mean_abs=1e-5, lse=1e-4),
       "bf16": dict(max_abs=2e-2, mean_abs=2e-3, lse=2e-3)}


# Gradient tolerance, per tensor (dq, dk or dv) against the float64 oracle:
#   every row:  |got_row - ref_row| <= row_rtol |ref_row| + row_atol median_row|ref|
#                                      + floor
#   the tensor: |got - ref|_F       <= fro * |ref|_F
# fp32: the SIMT kernel's fp32 sums of up to S terms, about 1e-6 relative.
# bf16: each output element is rounded once (2^-9 relative) and the
# tensor-core kernel also rounds P and dS to bf16 before its products, another
# 2^-9 per term with random sign, so a row's relative error stays near 2^-8;
# the bounds give that a factor 4 (normwise 2^-7) to 8 (per row 2^-5).  The
# median term covers rows whose exact gradient vanishes (the first causal
# row's dq is exactly zero); the floor covers a tensor whose rows all vanish
# (one token), where what is left is the rounding of dP - delta, about
# eps |dout| |v| scale |k| (1e-6 in fp32 at these sizes).  A key tile missing
# from or doubled in the fold moves the rows it feeds by well over 2^-5 at the
# tested sizes.
# On top of this, every row of dq and dk gets the effect of delta_t = dO_t.O_t
# being formed from the stored output (rounded to the output dtype) rather
# than the exact one; where a row's weights concentrate on one key,
# dP - delta cancels and this term dominates (see ``delta_error_bounds``).
TOL_BWD = {"f32": dict(row_rtol=1e-4, row_atol=1e-5, floor=1e-5, fro=1e-5),
           "bf16": dict(row_rtol=2.0 ** -5, row_atol=2.0 ** -7, floor=1e-3, fro=2.0 ** -7)}


def gen(seed, shape, dtype, tensor_id):
    n = int(np.prod(shape))
    if dtype == "bf16":
        return ragen.normal_bf16(seed, tensor_id, n).reshape(shape)
    return ragen.normal_f32(seed, tensor_id, n).reshape(shape)


def inputs(seed, B, Hq, Hkv, S, D, dtype):
    return (gen(seed, (B, Hq, S, D), dtype, ragen.TENSOR_Q),
            gen(seed, (B, Hkv, S, D), dtype, ragen.TENSOR_K),
            gen(seed, (B, Hkv, S, D), dtype, ragen.TENSOR_V))


def to_f64(a, dtype):
    return oracle.bf16_bits_to_f64(a) if dtype == "bf16" else np.asarray(a, np.float64)


def to_device(a, dtype, device="cuda"):
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def from_device(t):
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def reference(q, k, v, N, causal, striped, dtype, scale=None):
    """Oracle O and lse for shard-major inputs, returned shard-major (float64).

    Uses the plain full-attention definition on token-order tensors."""
    qf, kf, vf = (oracle.to_token_order(to_f64(x, dtype), N, striped) for x in (q, k, v))
    o, lse = oracle.full_attention(qf, kf, vf, causal, scale)
    return (oracle.to_shard_major(o, N, striped),
            oracle.to_shard_major(lse[..., None], N, striped)[..., 0])


def errors(got, want):
    d = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    return float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0


def assert_close(out, lse, ref_o, ref_lse, dtype, what=""):
    tol = TOL[dtype]
    mx, mean = errors(out, ref_o)
    assert mx <= tol["max_abs"] and mean <= tol["mean_abs"], \
        f"{what}: out max-abs {mx:.3e} mean-abs {mean:.3e} (tol {tol})"
    if lse is not None:
        lmx, _ = errors(lse, ref_lse)
        assert lmx <= tol["lse"], f"{what}: lse max-abs {lmx:.3e}"
    return mx, mean


def sample_rows(seed, B, Hq, S, N, n_rows):
    """Stratified query-row sample (b, h, shard-major row): every head and
    shard, the first and last row of every shard, then uniform rows."""
    rng = np.random.default_rng(seed)
    Sb = S // N
    picks = set()
    for b in range(B):
        for h in range(Hq):
            for i in range(N):
                picks.add((b, h, i * Sb))
                picks.add((b, h, i * Sb + Sb - 1))
    picks = sorted(picks)
    if len(picks) > n_rows // 2:
        idx = rng.choice(len(picks), n_rows // 2, replace=False)
        picks = [picks[i] for i in sorted(idx)]
    while len(picks) < n_rows:
        picks.append((int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(S))))
    return sorted(set(picks))


def _kv_token_order(seed, S, D, N, layout, Hkv, b, kvh):
    """k and v of one (batch, KV head) slice, regenerated and put in token
    order (float64, [S, D] each)."""
    base = (b * Hkv + kvh) * S * D
    kk = oracle.bf16_bits_to_f64(ragen.normal_bf16(seed, ragen.TENSOR_K, S * D, start=base))
    vv = oracle.bf16_bits_to_f64(ragen.normal_bf16(seed, ragen.TENSOR_V, S * D, start=base))
    return (oracle.to_token_order(kk.reshape(S, D), N, layout),
            oracle.to_token_order(vv.reshape(S, D), N, layout))


def sampled_reference(seed, wl_shapes, rows, causal, striped, N, scale=None,
                      max_elems=1 << 25):
    """Oracle O, lse for sampled shard-major query rows of a bf16 workload,
    regenerating only what is needed (the sampled q rows, full k/v of the
    kv heads involved) from the counter-based generator.

    Each row is the plain definition (``oracle.attend_rows``) against the keys
    of its KV head in token order.  Rows are taken in order of position, so
    under the causal mask a group of rows needs only the keys up to its
    largest position (the others are invisible to all of them); groups are
    sized to keep the score block under ``max_elems`` entries."""
    (B, Hq, S, D), (_, Hkv, _, _) = wl_shapes
    g = Hq // Hkv
    sc = 1.0 / math.sqrt(D) if not scale else scale
    pos = oracle.positions(S, N, striped)
    out_o = np.empty((len(rows), D))
    out_l = np.empty(len(rows))
    by_kv = {}
    for n, (b, h, p) in enumerate(rows):
        by_kv.setdefault((b, h // g), []).append(n)
    for (b, kvh), idxs in by_kv.items():
        kk, vv = _kv_token_order(seed, S, D, N, striped, Hkv, b, kvh)
        idxs = np.array(sorted(idxs, key=lambda n: pos[rows[n][2]]))
        qrows = [(rows[n][0] * Hq + rows[n][1]) * S + rows[n][2] for n in idxs]
        qq = oracle.bf16_bits_to_f64(ragen.normal_bf16_rows(seed, ragen.TENSOR_Q, qrows, D))
        qpos = pos[[rows[n][2] for n in idxs]]
        c0 = 0
        while c0 < len(idxs):
            # rows in this group: as many as fit the score block
            c1 = c0 + 1
            while c1 < len(idxs) and (c1 + 1 - c0) * (
                    (int(qpos[c1]) + 1) if causal else S) <= max_elems:
                c1 += 1
            hi = int(qpos[c1 - 1]) + 1 if causal else S
            o, l = oracle.attend_rows(qq[c0:c1], qpos[c0:c1], kk[:hi], vv[:hi],
                                      np.arange(hi), causal, sc)
            out_o[idxs[c0:c1]] = o
            out_l[idxs[c0:c1]] = l
            c0 = c1
    return out_o, out_l


def slice_reference(seed, wl, b, h):
    """Oracle O [S, D] and lse [S] of every row of one (batch, query head)
    slice of a bf16 workload, shard-major, from regenerated inputs: the plain
    definition (``oracle.full_attention``) in token order."""
    S, D, N = wl.S, wl.D, wl.N
    g = wl.Hq // wl.Hkv
    base = (b * wl.Hq + h) * S * D
    qq = oracle.bf16_bits_to_f64(ragen.normal_bf16(seed, ragen.TENSOR_Q, S * D, start=base))
    qq = oracle.to_token_order(qq.reshape(S, D), N, wl.striped)
    kk, vv = _kv_token_order(seed, S, D, N, wl.striped, wl.Hkv, b, h // g)
    o, lse = oracle.full_attention(qq[None, None], kk[None, None], vv[None, None], wl.causal)
    return (oracle.to_shard_major(o[0, 0], N, wl.striped),
            oracle.to_shard_major(lse[0, 0][:, None], N, wl.striped)[:, 0])


def grad_inputs(seed, B, Hq, S, D, dtype):
    """dL/dout for the backward tests: N(0, 1) with tensor id TENSOR_DO."""
    return gen(seed, (B, Hq, S, D), dtype, ragen.TENSOR_DO)


def backward_reference(q, k, v, dout, N, causal, layout, dtype, scale=None):
    """Oracle dq, dk, dv for shard-major inputs, returned shard-major (float64),
    from the plain gradient definition on token-order tensors."""
    qf, kf, vf, gf = (oracle.to_token_order(to_f64(x, dtype), N, layout) for x in (q, k, v, dout))
    grads = oracle.attention_backward(qf, kf, vf, gf, causal, scale)
    return tuple(oracle.to_shard_major(g, N, layout) for g in grads)


def delta_error_bounds(q, k, v, dout, N, causal, layout, dtype, scale=None, lam=8.0):
    """Per-row bounds (shard-major [B, H, S]) on how far dq and dk move when
    delta_t = dO_t . O_t uses the stored output instead of the exact one.

    The stored output differs from the exact O by its rounding to the output
    dtype (at most u |O_td|, u = 2^-9 for bf16 and 2^-24 for fp32) and by the
    forward's rounding of each weight P_tu to that dtype before the P.V
    product (sum_u e_u P_tu v_ud with |e_u| <= u).  These are sums of
    independent roundings of random sign, so their size is taken as lam
    standard deviations of such a sum (the probabilistic rounding-error
    analysis of Higham and Mary, SIAM J. Sci. Comput. 2019), lam = 8:
        |d delta_t| <= lam u sqrt(sum_d dout_td^2 (O_td^2 + sum_u P_tu^2 v_ud^2)).
    Since dS_tu = P_tu (dP_tu - delta_t), a change of delta_t moves
        dq_t by exactly scale d delta_t sum_u P_tu k_u,
        dk_u by scale sum_t P_tu d delta_t q_t, whose terms have independent
             signs: scale sqrt(sum_t (P_tu |d delta_t| |q_t|)^2);
    dv does not involve delta.  O, lse and P come from the oracle."""
    u = 2.0 ** -9 if dtype == "bf16" else 2.0 ** -24
    qf, kf, vf, gf = (oracle.to_token_order(to_f64(x, dtype), N, layout) for x in (q, k, v, dout))
    B, Hq, S, D = qf.shape
    g = Hq // kf.shape[1]
    sc = 1.0 / math.sqrt(D) if not scale else scale
    o, lse = oracle.full_attention(qf, kf, vf, causal, scale)
    bq = np.zeros((B, Hq, S))
    bk2 = np.zeros((B, kf.shape[1], S))
    pos = np.arange(S)
    for b in range(B):
        for h in range(Hq):
            K, V = kf[b, h // g], vf[b, h // g]
            for r0 in range(0, S, 256):
                r1 = min(S, r0 + 256)
                s = (qf[b, h, r0:r1] @ K.T) * sc - lse[b, h, r0:r1, None]
                if causal:
                    s = np.where(pos[None, :] <= pos[r0:r1, None], s, -np.inf)
                P = np.exp(s)
                var_o = o[b, h, r0:r1] ** 2 + (P ** 2) @ (V ** 2)
                dd = lam * u * np.sqrt((gf[b, h, r0:r1] ** 2 * var_o).sum(axis=1))
                bq[b, h, r0:r1] = sc * dd * np.linalg.norm(P @ K, axis=1)
                w = dd * np.linalg.norm(qf[b, h, r0:r1], axis=1)
                bk2[b, h // g] += ((sc * P * w[:, None]) ** 2).sum(axis=0)
    to_sm = lambda x: oracle.to_shard_major(x[..., None], N, layout)[..., 0]
    return to_sm(bq), to_sm(np.sqrt(bk2))


def assert_grad_close(got, ref, dtype, what="", extra=None):
    """The row-wise and normwise gradient bounds of TOL_BWD, plus ``extra``
    (per row, e.g. from ``delta_error_bounds``) when given."""
    tol = TOL_BWD[dtype]
    got = np.asarray(got, np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    ext = np.zeros(len(ref)) if extra is None else np.asarray(extra, np.float64).reshape(-1)
    assert np.isfinite(got).all(), f"{what}: non-finite gradient"
    err = np.linalg.norm(got - ref, axis=1)
    nrm = np.linalg.norm(ref, axis=1)
    bound = tol["row_rtol"] * nrm + tol["row_atol"] * float(np.median(nrm)) + tol["floor"] + ext
    worst = int(np.argmax(err - bound))
    assert (err <= bound).all(), \
        f"{what}: row {worst} error {err[worst]:.3e} > bound {bound[worst]:.3e} (|ref| {nrm[worst]:.3e})"
    total = float(np.linalg.norm(got - ref))
    fro = total / max(float(np.linalg.norm(ref)), 1e-300)
    assert total <= tol["fro"] * float(np.linalg.norm(ref)) + float(np.linalg.norm(ext)) + \
        tol["floor"], f"{what}: normwise error {fro:.3e} > {tol['fro']:.3e}"
    # worst relative row error, over rows whose reference is not (near) zero:
    # a causal first row's dq is exactly 0 (it sees only its own key)
    live = nrm > 1e-6 * max(float(np.median(nrm)), 1e-300)
    return fro, float((err[live] / nrm[live]).max()) if live.any() else 0.0


def slice_token_order(seed, tensor_id, shape, b, h, N, layout):
    """One (batch, head) slice [S, D] of a generated bf16 tensor of shape
    [B, H, S, D], as float64 in token order."""
    _, H, S, D = shape
    x = oracle.bf16_bits_to_f64(ragen.normal_bf16(seed, tensor_id, S * D,
                                                  start=(b * H + h) * S * D))
    return oracle.to_token_order(x.reshape(S, D), N, layout)


def key_rows_delta_bound(qw, qpos, dow, k, v, kpos, keys, causal, scale, lam=8.0,
                         u=2.0 ** -9, chunk=256):
    """Per chosen key row, the squared delta term of ``delta_error_bounds``
    for one query head: sum over the query rows t that see key c of
    (scale P_tc |d delta_t| |q_t|)^2, with |d delta_t| <=
    lam u sqrt(sum_d dO_td^2 (O_td^2 + sum_u P_tu^2 v_ud^2)).  qw, dow hold
    every query row that sees a chosen key (token order)."""
    keys = np.asarray(keys, np.int64)
    out = np.zeros(len(keys))
    for r0 in range(0, len(qw), chunk):
        q, do, qp = qw[r0:r0 + chunk], dow[r0:r0 + chunk], qpos[r0:r0 + chunk]
        s = (q @ k.T) * scale
        if causal:
            s = np.where(np.asarray(kpos)[None, :] <= qp[:, None], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        P = e / e.sum(axis=1, keepdims=True)
        o = P @ v
        var_o = o ** 2 + (P ** 2) @ (v ** 2)
        dd = lam * u * np.sqrt((do ** 2 * var_o).sum(axis=1))
        w = scale * dd * np.linalg.norm(q, axis=1)
        out += ((P[:, keys] * w[:, None]) ** 2).sum(axis=0)
    return out

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


def sampled_reference(seed, wl_shapes, rows, causal, striped, N, scale=None):
    """Oracle O, lse for sampled shard-major query rows of a bf16 workload,
    regenerating only what is needed (the sampled q rows, full k/v of the
    kv heads involved) from the counter-based generator."""
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
        base = (b * Hkv + kvh) * S * D
        kk = oracle.bf16_bits_to_f64(ragen.normal_bf16(seed, ragen.TENSOR_K, S * D, start=base))
        vv = oracle.bf16_bits_to_f64(ragen.normal_bf16(seed, ragen.TENSOR_V, S * D, start=base))
        kk, vv = kk.reshape(S, D), vv.reshape(S, D)
        qrows = [(rows[n][0] * Hq + rows[n][1]) * S + rows[n][2] for n in idxs]
        qq = oracle.bf16_bits_to_f64(ragen.normal_bf16_rows(seed, ragen.TENSOR_Q, qrows, D))
        qpos = pos[[rows[n][2] for n in idxs]]
        for c0 in range(0, len(idxs), 32):  # bounds the [rows, S] score matrix
            sl = slice(c0, c0 + 32)
            o, l = oracle.attend_rows(qq[sl], qpos[sl], kk, vv, pos, causal, sc)
            out_o[idxs[sl]] = o
            out_l[idxs[sl]] = l
    return out_o, out_l

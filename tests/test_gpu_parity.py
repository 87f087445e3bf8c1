"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Element by element on small shapes that span several tiles (plus ragged and
degenerate cases); on sampled rows (stratified over heads and shards, each
row computed by the oracle from regenerated inputs) at the full sizes of the
named workloads, launched exactly as the bench launches them.  Tolerances:
fp32 max-abs 1e-5; bf16 max-abs 2e-2 and mean-abs 2e-3; lse 1e-4 / 2e-3.
Schedules (fold order) and the stripe permutation are compared bit for bit.
"""
import math

import numpy as np
import pytest

import oracle
import ragen
from ragen import WORKLOADS

from helpers import (TOL, assert_close, errors, from_device, inputs, reference, sample_rows,
                     sampled_reference, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def run(ra, q, k, v, N, causal, striped, dtype, kernel="auto", scale=None):
    tq, tk, tv = (to_device(x, dtype) for x in (q, k, v))
    out, lse = ra.forward(tq, tk, tv, N, causal=causal, striped=striped, scale=scale,
                          kernel=kernel)
    ra.check()
    return from_device(out), from_device(lse)


# ------------------------------------------------------------------ fp32 path
def test_toy_f32_workload(ra):
    """The glossary page's toy shape: N=4 devices x 8 tokens, D=16, fp32."""
    wl = WORKLOADS["toy_f32"]
    q, k, v = inputs(wl.seed, wl.B, wl.Hq, wl.Hkv, wl.S, wl.D, "f32")
    out, lse = run(ra, q, k, v, wl.N, wl.causal, wl.striped, "f32")
    ro, rl = reference(q, k, v, wl.N, wl.causal, wl.striped, "f32")
    assert_close(out, lse, ro, rl, "f32", "toy")


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,striped", [
    (1, 1, 1, 32, 4, 16, True, False),
    (1, 1, 1, 32, 4, 16, True, True),
    (2, 4, 2, 96, 3, 24, True, True),
    (1, 3, 1, 200, 5, 64, True, False),
    (1, 2, 2, 384, 2, 128, False, False),
    (1, 2, 1, 256, 8, 200, True, True),
    (1, 1, 1, 7, 1, 5, True, False),
    (1, 1, 1, 1, 1, 8, True, True),
    # register-blocked kernel (D % 4 == 0, D <= 128): several 64-row blocks and
    # 32-key chunks, ragged shards, every layout, D padded up to 32/64/128
    (1, 2, 1, 1000, 4, 128, True, True),    # Sb = 250
    (2, 2, 2, 640, 5, 32, False, False),    # Sb = 128
    (1, 4, 2, 512, 4, 64, True, 2),         # zigzag
    (1, 2, 1, 300, 3, 100, True, False),    # D = 100 in the 128 variant; Sb = 100
    (1, 1, 1, 96, 2, 4, True, True),        # D = 4, smallest
])
def test_simt_f32_grid(ra, B, Hq, Hkv, S, N, D, causal, striped):
    q, k, v = inputs(11 + S + D, B, Hq, Hkv, S, D, "f32")
    out, lse = run(ra, q, k, v, N, causal, striped, "f32")
    ro, rl = reference(q, k, v, N, causal, striped, "f32")
    assert_close(out, lse, ro, rl, "f32", "simt f32")


# ------------------------------------------------------------------ bf16 tensor-core path
TC_GRID = [
    # B, Hq, Hkv, S, N, D, causal, striped
    (1, 1, 1, 128, 1, 128, False, False),
    (1, 1, 1, 128, 1, 128, True, False),
    (1, 2, 1, 512, 2, 128, True, False),
    (1, 2, 1, 512, 2, 128, True, True),
    (1, 4, 2, 1024, 4, 128, True, True),
    (2, 2, 2, 768, 3, 128, True, False),   # MHA: query-tile pairing, odd tiles per shard
    (1, 3, 1, 768, 2, 128, True, True),    # odd GQA group -> tile pairing, 3 tiles per shard
    (1, 8, 1, 1024, 8, 128, True, True),   # one tile per shard
    (1, 2, 2, 1024, 2, 64, True, False),
    (1, 4, 4, 1024, 4, 64, True, True),
    (1, 2, 1, 1536, 3, 64, False, False),
    (1, 4, 2, 2048, 4, 128, False, False),
    (1, 4, 2, 2048, 4, 128, True, 2),      # zigzag, GQA head pairing
    (2, 2, 2, 1536, 3, 128, True, 2),      # zigzag, MHA tile pairing, 2 tiles per chunk
    (1, 2, 1, 1024, 2, 64, True, 2),
    # ragged: the last tile of every shard is partial
    (1, 2, 1, 600, 3, 128, True, False),     # Sb = 200
    (1, 4, 2, 1200, 4, 128, True, True),     # Sb = 300, striped
    (2, 2, 2, 1000, 2, 128, True, False),    # Sb = 500, MHA tile pairing
    (1, 2, 2, 520, 2, 64, False, False),     # Sb = 260, non-causal, D = 64
    (1, 2, 1, 130, 1, 128, True, True),      # Sb = 130, one ring device
]


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,striped", TC_GRID)
def test_tc_bf16_grid(ra, B, Hq, Hkv, S, N, D, causal, striped):
    q, k, v = inputs(101 + S + 7 * N + D, B, Hq, Hkv, S, D, "bf16")
    out, lse = run(ra, q, k, v, N, causal, striped, "bf16", kernel="tc")
    ro, rl = reference(q, k, v, N, causal, striped, "bf16")
    assert_close(out, lse, ro, rl, "bf16", "tc")


# Non-causal problems with between one and two work items per SM run as
# stream-K (fixed contiguous work ranges per CTA; an item cut between two CTAs
# is combined from the tail's partial); these shapes have 256 items.
STREAMK_GRID = [
    (2, 8, 8, 4096, 2, 64),      # MHA: query-tile pairs
    (1, 8, 2, 8192, 4, 128),     # GQA: head pairs
    (2, 8, 8, 3800, 2, 128),     # ragged (Sb = 1900), odd tile count: a pair with one tile
]


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D", STREAMK_GRID)
def test_streamk_matches_oracle(ra, B, Hq, Hkv, S, N, D):
    import torch
    q, k, v = inputs(401 + S + N + D, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out, lse = ra.forward(tq, tk, tv, N, causal=False)
    out2, lse2 = ra.forward(tq, tk, tv, N, causal=False)
    whole_o, whole_l = ra.forward(tq, tk, tv, N, causal=False, kernel="tc")
    ra.check()
    # the cut items' halves are combined in a fixed order: the same bits on every call
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)
    ro, rl = reference(q, k, v, N, False, False, "bf16")
    assert_close(from_device(out), from_device(lse), ro, rl, "bf16", "stream-K")
    assert not torch.equal(out.view(torch.int16), whole_o.view(torch.int16)), \
        "expected this few-item problem to run as stream-K"


def test_tc_custom_scale_and_no_lse(ra):
    import torch
    B, Hq, Hkv, S, N, D = 1, 2, 1, 512, 2, 128
    q, k, v = inputs(5, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out, lse = ra.forward(tq, tk, tv, N, causal=True, striped=True, scale=0.2, want_lse=False)
    ra.check()
    assert lse is None
    ro, rl = reference(q, k, v, N, True, True, "bf16", scale=0.2)
    assert_close(from_device(out), None, ro, rl, "bf16", "scale 0.2")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("causal,striped", [(True, False), (True, True), (False, False), (True, 2)])
def test_simt_bf16_matches_oracle(ra, causal, striped):
    B, Hq, Hkv, S, N, D = 1, 2, 1, 640, 5, 96  # outside the tensor-core envelope
    q, k, v = inputs(77, B, Hq, Hkv, S, D, "bf16")
    out, lse = run(ra, q, k, v, N, causal, striped, "bf16")
    ro, rl = reference(q, k, v, N, causal, striped, "bf16")
    assert_close(out, lse, ro, rl, "bf16", "simt bf16")


# ------------------------------------------------------------------ schedule, permutation, merge
@pytest.mark.parametrize("Hq,Hkv,S,N,causal,striped", [
    (2, 1, 1024, 4, True, False),
    (2, 1, 1024, 4, True, True),
    (2, 2, 768, 2, True, False),
    (3, 1, 768, 2, True, True),
    (2, 1, 512, 2, False, False),
    (2, 1, 1024, 2, True, 2),
    (2, 2, 1536, 3, True, 2),
    (2, 1, 600, 3, True, True),   # ragged shards
    (2, 2, 1000, 2, True, False),
])
def test_fold_log_is_the_bruteforce_schedule(ra, Hq, Hkv, S, N, causal, striped):
    """Bit-exact: the order in which the kernel folded every query tile equals
    the oracle's brute-force schedule (and ra_plan)."""
    import torch
    B, D = 1, 128
    q, k, v = inputs(3, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out, lse, log, counts = ra.fold_log(tq, tk, tv, N, causal, striped)
    ra.check()
    log, counts = log.cpu().numpy(), counts.cpu().numpy()
    ref = oracle.fold_schedule(S, N, causal, striped, 128, 128)
    by_tile = {}
    for (i, qt, s, j, kt, kind) in ref:
        by_tile.setdefault((i, qt), []).append((s, j, kt, kind))
    nt = -(-(S // N) // 128)
    for b in range(B):
        for h in range(Hq):
            for i in range(N):
                for qt in range(nt):
                    u = ((b * Hq + h) * N + i) * nt + qt
                    got = [tuple(x) for x in log[u, :counts[u]].tolist()]
                    assert got == by_tile[(i, qt)], (h, i, qt)
                    assert got == ra.plan(S, N, causal, striped, i, qt)
    ro, rl = reference(q, k, v, N, causal, striped, "bf16")
    assert_close(from_device(out), from_device(lse), ro, rl, "bf16", "logging variant")


@pytest.mark.parametrize("S,N,D,dt,layout", [(4096, 8, 128, "bf16", 1), (96, 3, 16, "f32", 1),
                                             (130, 5, 6, "bf16", 1), (4096, 8, 128, "bf16", 2),
                                             (120, 3, 6, "bf16", 2), (64, 4, 16, "f32", 2)])
def test_stripe_permutation_bitexact(ra, S, N, D, dt, layout):
    import torch
    x = np.asarray(inputs(9, 2, 3, 1, S, D, dt)[0])
    tx = to_device(x, dt)
    if layout == 1:
        sm = ra.stripe(tx, N)
        back = ra.stripe(sm, N, inverse=True)
    else:
        sm = ra.relayout(tx, N, layout)
        back = ra.relayout(sm, N, layout, inverse=True)
    torch.cuda.synchronize()
    perm = oracle.stripe_perm(S, N, layout)
    got = sm.cpu().view(torch.int16 if dt == "bf16" else torch.int32).numpy()
    want = x.view(np.int16 if dt == "bf16" else np.int32)[..., perm, :]
    assert np.array_equal(got, want)
    assert torch.equal(back, tx)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_merge_two_ring_halves(ra, dt):
    """ra_merge against the oracle's log-sum-exp merge on random partials,
    including rows where one or both partials are empty (lse = -inf)."""
    import torch
    rows, D = 3000, 128
    rng = np.random.default_rng(1)
    oa, ob = rng.standard_normal((rows, D)), rng.standard_normal((rows, D))
    la, lb = rng.standard_normal(rows) * 3, rng.standard_normal(rows) * 3
    la[::7] = -np.inf
    lb[::11] = -np.inf
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    toa = torch.tensor(oa, dtype=tdt, device="cuda")
    tob = torch.tensor(ob, dtype=tdt, device="cuda")
    tla = torch.tensor(la, dtype=torch.float32, device="cuda")
    tlb = torch.tensor(lb, dtype=torch.float32, device="cuda")
    ref_o, ref_l = oracle.merge(from_device(toa), from_device(tla), from_device(tob),
                                from_device(tlb))
    ra.merge(toa, tla, tob, tlb)
    ra.check()
    got_o, got_l = from_device(toa), from_device(tla)
    tol = 2e-2 if dt == "bf16" else 1e-5
    assert np.nanmax(np.abs(got_o - ref_o)) <= tol
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(got_l))
    assert np.abs(got_l[fin] - ref_l[fin]).max() <= 1e-5


def test_merge_of_kernel_partials_is_full_attention(ra):
    """ra_merge on two kernel results over disjoint key sets == one pass over
    the union (non-causal: keys split by shard halves via two separate calls)."""
    import torch
    B, H, S, D = 1, 2, 512, 128
    q, k, v = inputs(21, B, H, H, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    half = S // 2
    # each call sees only half of the keys (non-causal, N=1 over the half)
    k1, v1 = tk[:, :, :half].contiguous(), tv[:, :, :half].contiguous()
    k2, v2 = tk[:, :, half:].contiguous(), tv[:, :, half:].contiguous()
    # queries: all rows; keys: half -> need equal S for q and k, so split queries too
    outs = []
    for (kk, vv) in ((k1, v1), (k2, v2)):
        o_parts, l_parts = [], []
        for qs in (tq[:, :, :half].contiguous(), tq[:, :, half:].contiguous()):
            o, l = ra.forward(qs, kk, vv, 1, causal=False)
            o_parts.append(o)
            l_parts.append(l)
        outs.append((torch.cat(o_parts, 2).contiguous(), torch.cat(l_parts, 2).contiguous()))
    (oa, la), (ob, lb) = outs
    ra.merge(oa, la, ob, lb)
    ra.check()
    ro, rl = reference(q, k, v, 1, False, False, "bf16")
    assert_close(from_device(oa), from_device(la), ro, rl, "bf16", "merged halves")


# ------------------------------------------------------------------ Ulysses exchange
@pytest.mark.parametrize("N,B,H,S,D,dt", [(4, 2, 8, 512, 128, "bf16"), (2, 1, 4, 96, 16, "f32"),
                                          (3, 1, 6, 30, 6, "bf16")])
def test_ulysses_exchange_bitexact(ra, N, B, H, S, D, dt):
    import torch
    x = np.asarray(inputs(13, N * B, H, 1, S // N, D, dt)[0]).reshape(N, B, H, S // N, D)
    tx = to_device(x, dt)
    y = ra.ulysses_exchange(tx, N)
    back = ra.ulysses_exchange(y, N, inverse=True)
    torch.cuda.synchronize()
    view = torch.int16 if dt == "bf16" else torch.int32
    want = oracle.ulysses_exchange(x.view(np.int16 if dt == "bf16" else np.int32), N)
    assert np.array_equal(y.cpu().view(view).numpy(), want)
    assert torch.equal(back, tx)


@pytest.mark.parametrize("causal", [True, False])
def test_ulysses_attention_equals_full_attention(ra, causal):
    """Sequence-sharded inputs -> exchange -> ra_forward per device over its
    heads -> inverse exchange == full attention."""
    import torch
    N, B, H, S, D = 4, 1, 8, 2048, 128
    q, k, v = inputs(57, B, H, H, S, D, "bf16")
    seq = [to_device(np.ascontiguousarray(
        x.reshape(B, H, N, S // N, D).transpose(2, 0, 1, 3, 4)), "bf16") for x in (q, k, v)]
    hs = [ra.ulysses_exchange(x, N) for x in seq]
    outs = torch.empty_like(hs[0])
    for d in range(N):
        o_d, _ = ra.forward(hs[0][d], hs[1][d], hs[2][d], 1, causal=causal, out=outs[d])
    back = ra.ulysses_exchange(outs, N, inverse=True)
    ra.check()
    o = from_device(back).transpose(1, 2, 0, 3, 4).reshape(B, H, S, D)
    ro, rl = reference(q, k, v, 1, causal, False, "bf16")
    assert_close(o, None, ro, rl, "bf16", "ulysses")


# ------------------------------------------------------------------ named workloads
def _device_inputs(wl):
    """Generate a workload's q, k, v straight into pinned host memory, copy to
    the device (bf16)."""
    import torch
    out = []
    for tid, shape in zip((ragen.TENSOR_Q, ragen.TENSOR_K, ragen.TENSOR_V),
                          (wl.shapes()[0], wl.shapes()[1], wl.shapes()[1])):
        h = torch.empty(shape, dtype=torch.int16, pin_memory=True)
        ragen.normal_bf16(wl.seed, tid, h.numel(), out=h.numpy().reshape(-1).view(np.uint16))
        out.append(h.to("cuda", non_blocking=True).view(torch.bfloat16))
    torch.cuda.synchronize()
    return out


def test_noncausal_8k_every_row(ra):
    wl = WORKLOADS["noncausal_8k"]
    q, k, v = inputs(wl.seed, wl.B, wl.Hq, wl.Hkv, wl.S, wl.D, "bf16")
    out, lse = run(ra, q, k, v, wl.N, wl.causal, wl.striped, "bf16")
    ro, rl = reference(q, k, v, wl.N, wl.causal, wl.striped, "bf16")
    assert_close(out, lse, ro, rl, "bf16", wl.name)


# Full-size workloads, launched as the bench launches them: a stratified row
# sample (every head and shard, each shard's first and last row), plus every
# row of chosen (batch, head) slices, or of a slice's first shards.
FULL_SIZE = [
    # name, sampled rows, whole (b, h) slices, (heads, shards) checked on every row
    ("causal_32k_contig", 768, [(b, h) for b in (0, 1) for h in (0, 31)], None),
    ("causal_32k_striped", 768, [(b, h) for b in (0, 1) for h in (0, 31)], None),
    ("causal_32k_zigzag", 768, [(0, 0), (1, 31)], None),
    ("gqa_128k", 4096, [], ((0, 31), (0, 1))),
    ("gqa_128k_ragged", 768, [], None),
    ("long_1m", 4096, [], None),
    # the common ring entry: every row of one head in the first and last shards
    ("long_shards_384k", 1024, [], ((1,), (0, 15))),
]


@pytest.mark.parametrize("name,n_rows,slices,shard_rows", FULL_SIZE)
def test_full_size_rows(ra, name, n_rows, slices, shard_rows):
    import torch
    from helpers import slice_reference
    wl = WORKLOADS[name]
    tq, tk, tv = _device_inputs(wl)
    # NaN-filled outputs: every query row of every head must be written (the
    # persistent work order covers each query tile exactly once)
    out = torch.full_like(tq, float("nan"))
    lse = torch.full((wl.B, wl.Hq, wl.S), float("nan"), device="cuda")
    ra.forward(tq, tk, tv, wl.N, causal=wl.causal, striped=wl.striped, out=out, lse=lse)
    ra.check()
    del tq, tk, tv
    assert bool(torch.isfinite(lse).all()), f"{wl.name}: unwritten lse rows"
    for r0 in range(0, out.numel() // wl.D, 1 << 22):
        assert bool(torch.isfinite(out.view(-1, wl.D)[r0:r0 + (1 << 22)]).all()), wl.name

    def gather(rows):
        idx = torch.tensor([(b * wl.Hq + h) * wl.S + p for (b, h, p) in rows], device="cuda")
        return (out.view(-1, wl.D)[idx].double().cpu().numpy(),
                lse.view(-1)[idx].double().cpu().numpy())

    rows = sample_rows(wl.seed + 1, wl.B, wl.Hq, wl.S, wl.N, n_rows)
    ro, rl = sampled_reference(wl.seed, wl.shapes(), rows, wl.causal, wl.striped, wl.N)
    mx, mean = assert_close(*gather(rows), ro, rl, "bf16", f"{wl.name} sampled")
    print(f"{wl.name}: {len(rows)} sampled rows max-abs {mx:.2e} mean-abs {mean:.2e}")
    for (b, h) in slices:
        ro, rl = slice_reference(wl.seed, wl, b, h)
        got_o = out[b, h].double().cpu().numpy()
        got_l = lse[b, h].double().cpu().numpy()
        mx, mean = assert_close(got_o, got_l, ro, rl, "bf16", f"{wl.name} b={b} h={h}")
        print(f"{wl.name}: every row of b={b} h={h} max-abs {mx:.2e} mean-abs {mean:.2e}")
    if shard_rows:
        heads, shards = shard_rows
        rows = [(0, h, i * wl.Sb + r) for h in heads for i in shards for r in range(wl.Sb)]
        ro, rl = sampled_reference(wl.seed, wl.shapes(), rows, wl.causal, wl.striped, wl.N)
        mx, mean = assert_close(*gather(rows), ro, rl, "bf16", f"{wl.name} shards {shards}")
        print(f"{wl.name}: every row of heads {heads} in shards {shards} ({len(rows)} rows) "
              f"max-abs {mx:.2e} mean-abs {mean:.2e}")


def test_empty_problems_leave_the_stream_usable(ra):
    """B == 0 or S == 0 through the binding: empty outputs, no error, and the
    next real call on the same stream still matches the oracle."""
    import torch
    for shape_q, shape_kv in (((0, 2, 256, 128), (0, 1, 256, 128)),
                              ((1, 2, 0, 128), (1, 1, 0, 128))):
        for dt in (torch.bfloat16, torch.float32):
            q = torch.empty(shape_q, dtype=dt, device="cuda")
            k = torch.empty(shape_kv, dtype=dt, device="cuda")
            out, lse = ra.forward(q, k, k, 2, causal=True, striped=True)
            assert out.shape == q.shape and lse.shape == shape_q[:3]
            if dt == torch.bfloat16:
                dq, dk, dv = ra.backward(q, k, k, out, lse, q, 2, causal=True, striped=True)
                assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == k.shape
    ra.check()
    q, k, v = inputs(9100, 1, 2, 1, 512, 128, "bf16")
    got = run(ra, q, k, v, 2, True, 1, "bf16")
    assert_close(*got, *reference(q, k, v, 2, True, 1, "bf16"), "bf16")

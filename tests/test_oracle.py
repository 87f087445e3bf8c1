"""Pins for the CPU oracle: each checks it against something other than itself.

* brute force on tiny inputs (pure-Python loops, no matrix ops);
* closed forms (Q = 0 gives the mean of the visible values and lse = ln count;
  V = 1 gives O = 1; a dominant key gives that key's value);
* a library routine (torch scaled_dot_product_attention on CPU in float64);
* the pages' worked example (the glossary page's four-device toy);
* the pages' central claim (ring order == full attention), invariances
  (permutation equivariance without a mask, striped vs contiguous);
* the log-sum-exp merge identity;
* tile-count closed forms for the fold schedule and exact pair coverage.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle.attention import FULL, INCL, STRICT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def brute(q, k, v, causal, scale):
    """Pure-Python triple loop over token-order [S, D] inputs of one head."""
    S, D = len(q), len(q[0])
    out, lses = [], []
    for t in range(S):
        sc = []
        for u in range(S):
            if causal and u > t:
                continue
            sc.append((u, scale * sum(q[t][d] * k[u][d] for d in range(D))))
        mx = max(x for _, x in sc)
        w = [(u, math.exp(x - mx)) for u, x in sc]
        z = sum(x for _, x in w)
        out.append([sum(wu * v[u][d] for u, wu in w) / z for d in range(len(v[0]))])
        lses.append(mx + math.log(z))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 2), (3, 1)])
def test_full_matches_brute_force(causal, Hq, Hkv):
    S, D = 12, 5
    q, k, v = rnd((1, Hq, S, D), 1), rnd((1, Hkv, S, D), 2), rnd((1, Hkv, S, D), 3)
    o, lse = oracle.full_attention(q, k, v, causal, chunk=5)
    g = Hq // Hkv
    for h in range(Hq):
        ob, lb = brute(q[0, h].tolist(), k[0, h // g].tolist(), v[0, h // g].tolist(),
                       causal, 1 / math.sqrt(D))
        np.testing.assert_allclose(o[0, h], ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("striped", [False, True, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_matches_brute_force(causal, striped):
    S, D, N = 16, 4, 4
    q, k, v = rnd((1, 2, S, D), 4), rnd((1, 1, S, D), 5), rnd((1, 1, S, D), 6)
    qs, ks, vs = (oracle.to_shard_major(x, N, striped) for x in (q, k, v))
    o_sm, lse_sm = oracle.ring_attention(qs, ks, vs, N, causal, striped)
    o = oracle.to_token_order(o_sm, N, striped)
    lse = oracle.to_token_order(lse_sm[..., None], N, striped)[..., 0]
    for h in range(2):
        ob, lb = brute(q[0, h].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), causal, 0.5)
        np.testing.assert_allclose(o[0, h], ob, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse[0, h], lb, atol=1e-12, rtol=0)


@pytest.mark.parametrize("striped", [False, True, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_closed_form(causal, striped):
    """Q = 0 makes every visible key equally likely: O is the mean of the
    visible values (the prefix mean under the causal mask) and lse = ln(count)."""
    S, D, N = 24, 8, 4
    q = np.zeros((1, 1, S, D))
    k, v = rnd((1, 1, S, D), 7), rnd((1, 1, S, D), 8)
    qs, ks, vs = (oracle.to_shard_major(x, N, striped) for x in (q, k, v))
    o_sm, lse_sm = oracle.ring_attention(qs, ks, vs, N, causal, striped)
    o = oracle.to_token_order(o_sm, N, striped)[0, 0]
    lse = oracle.to_token_order(lse_sm[..., None], N, striped)[0, 0, :, 0]
    o_f, lse_f = oracle.full_attention(q, k, v, causal)
    for t in range(S):
        cnt = t + 1 if causal else S
        exp_o = v[0, 0, :cnt].mean(axis=0)
        np.testing.assert_allclose(o[t], exp_o, atol=1e-13)
        np.testing.assert_allclose(o_f[0, 0, t], exp_o, atol=1e-13)
        assert abs(lse[t] - math.log(cnt)) < 1e-13
        assert abs(lse_f[0, 0, t] - math.log(cnt)) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    """V = 1: attention weights of every row sum to 1, so O = 1 exactly-ish."""
    S, D, N = 32, 8, 4
    q, k = rnd((2, 2, S, D), 9) * 3, rnd((2, 2, S, D), 10) * 3
    v = np.ones((2, 2, S, D))
    for striped in (False, True):
        o, _ = oracle.ring_attention(q, k, v, N, causal, striped)
        np.testing.assert_allclose(o, 1.0, atol=1e-13)
    o, _ = oracle.full_attention(q, k, v, causal)
    np.testing.assert_allclose(o, 1.0, atol=1e-13)


def test_dominant_key_selects_its_value():
    """k_u = c * q_t with large c: row t attends (almost) only to key u."""
    S, D = 16, 8
    q, k, v = rnd((1, 1, S, D), 11), rnd((1, 1, S, D), 12) * 0.01, rnd((1, 1, S, D), 13)
    t, u = 11, 4
    k[0, 0, u] = 200.0 * q[0, 0, t]
    o, lse = oracle.full_attention(q, k, v, causal=True)
    np.testing.assert_allclose(o[0, 0, t], v[0, 0, u], atol=1e-9)
    expect = 200.0 * float(q[0, 0, t] @ q[0, 0, t]) / math.sqrt(D)
    assert abs(lse[0, 0, t] - expect) < 1e-6
    o2, _ = oracle.ring_attention(q, k, v, 4, True, False)
    np.testing.assert_allclose(o2[0, 0, t], v[0, 0, u], atol=1e-9)


@pytest.mark.parametrize("causal", [False, True])
def test_library_sdpa_crosscheck(causal):
    """torch's CPU scaled_dot_product_attention in float64 (GQA by repeating kv heads)."""
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, S, D = 2, 4, 2, 40, 16
    q, k, v = rnd((B, Hq, S, D), 14), rnd((B, Hkv, S, D), 15), rnd((B, Hkv, S, D), 16)
    o, _ = oracle.full_attention(q, k, v, causal, chunk=16)
    tk = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=1)
    tv = torch.from_numpy(v).repeat_interleave(Hq // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), tk, tv, is_causal=causal).numpy()
    np.testing.assert_allclose(o, ref, atol=1e-12, rtol=0)
    for striped in (False, True, 2):
        qs, ks, vs = (oracle.to_shard_major(x, 5, striped) for x in (q, k, v))
        o_sm, _ = oracle.ring_attention(qs, ks, vs, 5, causal, striped)
        np.testing.assert_allclose(oracle.to_token_order(o_sm, 5, striped), ref, atol=1e-12)


@pytest.mark.parametrize("N", [1, 2, 3, 8])
@pytest.mark.parametrize("causal,striped", [(False, False), (True, False), (True, True), (True, 2)])
def test_ring_equals_full(N, causal, striped):
    """The pages' central claim: the ring-order blockwise fold equals full attention."""
    S, D = 48, 8
    q, k, v = rnd((1, 4, S, D), 17), rnd((1, 2, S, D), 18), rnd((1, 2, S, D), 19)
    o_f, lse_f = oracle.full_attention(q, k, v, causal)
    qs, ks, vs = (oracle.to_shard_major(x, N, striped) for x in (q, k, v))
    o_sm, lse_sm = oracle.ring_attention(qs, ks, vs, N, causal, striped)
    np.testing.assert_allclose(oracle.to_token_order(o_sm, N, striped), o_f, atol=1e-12)
    lse_tok = oracle.to_token_order(lse_sm[..., None], N, striped)[..., 0]
    np.testing.assert_allclose(lse_tok, lse_f, atol=1e-12)


def test_permutation_equivariance_noncausal():
    """Without a mask: permuting keys/values jointly changes nothing, and
    permuting queries permutes the output rows."""
    S, D = 32, 8
    q, k, v = rnd((1, 1, S, D), 20), rnd((1, 1, S, D), 21), rnd((1, 1, S, D), 22)
    pq = np.random.default_rng(0).permutation(S)
    pk = np.random.default_rng(1).permutation(S)
    o, lse = oracle.ring_attention(q, k, v, 4, False, False)
    o2, lse2 = oracle.ring_attention(q[..., pq, :], k[..., pk, :], v[..., pk, :], 4, False, False)
    np.testing.assert_allclose(o2, o[..., pq, :], atol=1e-12)
    np.testing.assert_allclose(lse2, lse[..., pq], atol=1e-12)


@pytest.mark.parametrize("layout", [1, 2])
def test_striped_and_zigzag_equal_contiguous_after_unpermuting(layout):
    S, D, N = 64, 8, 8
    q, k, v = rnd((1, 2, S, D), 23), rnd((1, 1, S, D), 24), rnd((1, 1, S, D), 25)
    o_c, lse_c = oracle.ring_attention(q, k, v, N, True, False)  # token order == contiguous
    qs, ks, vs = (oracle.to_shard_major(x, N, layout) for x in (q, k, v))
    o_s, lse_s = oracle.ring_attention(qs, ks, vs, N, True, layout)
    np.testing.assert_allclose(oracle.to_token_order(o_s, N, layout), o_c, atol=1e-12)
    np.testing.assert_allclose(oracle.to_token_order(lse_s[..., None], N, layout)[..., 0], lse_c,
                               atol=1e-12)


def test_zigzag_positions_example():
    """2N chunks of Sb/2 tokens; device i holds chunk i then chunk 2N-1-i."""
    # N=4, S=16: chunks of 2 tokens; device 0 holds chunks 0 and 7, device 3 chunks 3 and 4
    assert oracle.positions(16, 4, 2).tolist() == [0, 1, 14, 15, 2, 3, 12, 13,
                                                   4, 5, 10, 11, 6, 7, 8, 9]
    assert oracle.positions(4, 1, 2).tolist() == [0, 1, 2, 3]
    # every device owns the same number of visible causal pairs (the point of the layout)
    S, N = 64, 4
    pos = oracle.positions(S, N, 2).reshape(N, -1)
    work = [sum(int(t) + 1 for t in dev) for dev in pos]
    assert len(set(work)) == 1
    with pytest.raises(ValueError):
        oracle.positions(12, 4, 2)  # odd shard size


def test_stripe_permutation_examples():
    """token t sits on device t mod N at local row t div N."""
    assert oracle.stripe_perm(8, 4).tolist() == [0, 4, 1, 5, 2, 6, 3, 7]
    assert oracle.stripe_perm(6, 2).tolist() == [0, 2, 4, 1, 3, 5]
    assert oracle.stripe_perm(5, 1).tolist() == [0, 1, 2, 3, 4]
    x = rnd((2, 3, 24, 2), 26)
    for striped in (False, True):
        np.testing.assert_array_equal(
            oracle.to_token_order(oracle.to_shard_major(x, 4, striped), 4, striped), x)


def test_merge_identity():
    """merge(partial over keys A, partial over keys B) == result over A u B."""
    S, D = 20, 6
    q, k, v = rnd((S, D), 27), rnd((S, D), 28), rnd((S, D), 29)
    pos = np.arange(S)
    rng = np.random.default_rng(3)
    maskA = rng.random(S) < 0.5
    A, Bm = np.where(maskA)[0], np.where(~maskA)[0]
    oa, la = oracle.attend_rows(q, pos, k[A], v[A], A, True, 0.4)
    ob, lb = oracle.attend_rows(q, pos, k[Bm], v[Bm], Bm, True, 0.4)
    o, l = oracle.merge(oa, la, ob, lb)
    of, lf = oracle.attend_rows(q, pos, k, v, pos, True, 0.4)
    np.testing.assert_allclose(o, of, atol=1e-12)
    np.testing.assert_allclose(l, lf, atol=1e-12)
    # some rows saw nothing in A or in B (lse = -inf partials)
    assert np.isneginf(la).any() or np.isneginf(lb).any()
    # both empty -> (0, -inf); commutative
    z, zl = oracle.merge(np.zeros((1, D)), [-np.inf], np.zeros((1, D)), [-np.inf])
    assert np.all(z == 0) and np.isneginf(zl).all()
    o2, l2 = oracle.merge(ob, lb, oa, la)
    np.testing.assert_allclose(o2, o, atol=1e-15)
    np.testing.assert_allclose(l2, l, atol=1e-15)


def test_toy_worked_example():
    """The glossary page's four-device simulation: blockwise == full at atol 1e-5."""
    torch = pytest.importorskip("torch")
    with open(os.path.join(GOLDEN, "toy_glossary_page.json")) as f:
        g = json.load(f)
    n, blk, dim = g["n_devices"], g["block"], g["dim"]
    torch.manual_seed(g["torch_seed"])
    q, k, v = torch.randn(3, n * blk, dim)
    full = (torch.softmax(q @ k.T / dim ** 0.5, dim=-1) @ v).numpy()
    toy = oracle.toy_ring_no_max(q.numpy(), k.numpy(), v.numpy(), n)
    assert np.allclose(toy, full, atol=g["atol"]) == g["matches_full_attention"]
    ring, _ = oracle.ring_attention(q.numpy()[None, None], k.numpy()[None, None],
                                    v.numpy()[None, None], n, False, False)
    assert np.allclose(ring[0, 0], full, atol=g["atol"]) == g["matches_full_attention"]
    np.testing.assert_allclose(ring[0, 0], toy, atol=1e-12)
    assert [blk, blk] == g["largest_score_block_per_device"]
    assert [n * blk, n * blk] == g["full_score_matrix"]


# ----------------------------------------------------------------- schedule
def _covered_pairs(S, N, causal, striped, T, sched):
    pos = oracle.positions(S, N, striped)
    Sb = S // N
    cover = np.zeros((S, S), dtype=np.int64)
    for (i, qt, s, j, kt, kind) in sched:
        assert j == (i - s) % N
        r = np.arange(i * Sb + qt * T, i * Sb + (qt + 1) * T)
        c = np.arange(j * Sb + kt * T, j * Sb + (kt + 1) * T)
        rl, cl = np.arange(T)[:, None], np.arange(T)[None, :]
        vis = {FULL: np.ones((T, T), bool), INCL: cl <= rl, STRICT: cl < rl}[kind]
        cover[np.ix_(r, c)] += vis
    want = (pos[None, :] <= pos[:, None]) if causal else np.ones((S, S), bool)
    return cover, want


@pytest.mark.parametrize("causal,striped", [(False, False), (True, False), (True, True),
                                            (True, 2)])
def test_schedule_covers_each_visible_pair_once(causal, striped):
    S, N, T = 256, 4, 16
    sched = oracle.fold_schedule(S, N, causal, striped, T, T)
    cover, want = _covered_pairs(S, N, causal, striped, T, sched)
    np.testing.assert_array_equal(cover, want.astype(np.int64))
    # fold order: ring steps ascending, key tiles ascending within a step
    by_tile = {}
    for e in sched:
        by_tile.setdefault(e[:2], []).append((e[2], e[4]))
    for lst in by_tile.values():
        assert lst == sorted(lst)


def test_schedule_tile_counts_closed_form():
    """Live tiles per (b, h): contiguous causal n(n+1)/2 with n = S/T; striped
    causal N^2 * m(m+1)/2 with m = Sb/T; non-causal (S/T)^2."""
    S, N, T = 2048, 8, 32
    n, m = S // T, S // N // T
    assert len(oracle.fold_schedule(S, N, True, False, T, T)) == n * (n + 1) // 2
    assert len(oracle.fold_schedule(S, N, True, True, T, T)) == N * N * m * (m + 1) // 2
    assert len(oracle.fold_schedule(S, N, False, False, T, T)) == n * n
    # zigzag: chunk pairs are full or diagonal, never strict -> the contiguous count
    zz = oracle.fold_schedule(S, N, True, 2, T, T)
    assert len(zz) == n * (n + 1) // 2 and all(e[5] != STRICT for e in zz)
    # the 32K-token, 8-device layouts at 128-token tiles, from one query shard per
    # kind of pair to keep it fast: shard 3 (contiguous) sees 3 full blocks + diagonal
    S, N, T = 32768, 8, 128
    m = S // N // T
    c3 = oracle.fold_schedule(S, N, True, False, T, T, i_list=[3])
    assert len(c3) == 3 * m * m + m * (m + 1) // 2
    s3 = oracle.fold_schedule(S, N, True, True, T, T, i_list=[3], qt_list=[0, 5, 31])
    assert len(s3) == sum(N * (qt + 1) for qt in (0, 5, 31))
    kinds = {(e[3] <= 3, e[4] == e[1]): e[5] for e in s3}
    assert kinds[(True, True)] == INCL and kinds[(False, True)] == STRICT
    assert kinds[(True, False)] == FULL and kinds[(False, False)] == FULL
    # and the per-(b, h) totals of the 32K layouts follow from the formulas above
    assert 8 * m * (m + 1) // 2 + 28 * m * m == 32896
    assert N * N * m * (m + 1) // 2 == 33792


# ----------------------------------------------------------------- Ulysses exchange
def test_ulysses_exchange_moves_every_row_to_its_definition():
    """Rows carry their own (device, b, head, local row) coordinates; after the
    exchange each must sit at the head-sharded index the definition gives."""
    N, B, H, Sb = 4, 2, 8, 3
    x = np.zeros((N, B, H, Sb, 4), dtype=np.int64)
    for i in range(N):
        for b in range(B):
            for h in range(H):
                for r in range(Sb):
                    x[i, b, h, r] = (i, b, h, r)
    y = oracle.ulysses_exchange(x, N)
    assert y.shape == (N, B, H // N, N * Sb, 4)
    seen = set()
    for d in range(N):
        for b in range(B):
            for hl in range(H // N):
                for t in range(N * Sb):
                    i, bb, h, r = y[d, b, hl, t]
                    assert (bb, h, i * Sb + r) == (b, d * (H // N) + hl, t)
                    seen.add((i, bb, h, r))
    assert len(seen) == N * B * H * Sb  # a permutation: every row exactly once
    np.testing.assert_array_equal(oracle.ulysses_exchange(y, N, inverse=True), x)


@pytest.mark.parametrize("causal", [False, True])
def test_ulysses_pipeline_equals_full_attention(causal):
    """Exchange, full attention per device over its heads, exchange back ==
    full attention (the other context-parallel scheme reaches the same result)."""
    N, B, H, S, D = 2, 1, 4, 16, 8
    q, k, v = rnd((B, H, S, D), 40), rnd((B, H, S, D), 41), rnd((B, H, S, D), 42)
    seq = [x.reshape(B, H, N, S // N, D).transpose(2, 0, 1, 3, 4) for x in (q, k, v)]
    hs = [oracle.ulysses_exchange(x, N) for x in seq]
    outs = np.stack([oracle.full_attention(hs[0][d], hs[1][d], hs[2][d], causal)[0]
                     for d in range(N)])
    back = oracle.ulysses_exchange(outs, N, inverse=True)  # [N, B, H, Sb, D]
    o = back.transpose(1, 2, 0, 3, 4).reshape(B, H, S, D)
    o_f, _ = oracle.full_attention(q, k, v, causal)
    np.testing.assert_allclose(o, o_f, atol=1e-12)


def test_bf16_upcast_known_words():
    """bfloat16 is the top half of an IEEE binary32 word: sign, 8 exponent
    bits (bias 127), 7 fraction bits.  Known words decoded by hand."""
    words = np.array([0x3F80, 0xC000, 0x3FC0, 0x4049, 0x0000, 0x8000, 0x7F80, 0xFF80,
                      0x0001, 0x0080, 0x7F7F, 0xBE80, 0x4300], dtype=np.uint16)
    want = [1.0, -2.0, 1.5, 3.140625, 0.0, -0.0, math.inf, -math.inf,
            2.0 ** -133,                      # smallest subnormal: 2^-126 * 2^-7
            2.0 ** -126,                      # smallest normal
            (2 - 2.0 ** -7) * 2.0 ** 127,     # largest finite
            -0.25, 128.0]
    got = oracle.bf16_bits_to_f64(words)
    assert got.dtype == np.float64
    for w, g, e in zip(words, got, want):
        assert g == e and math.copysign(1, g) == math.copysign(1, e), (hex(int(w)), g, e)
    assert np.isnan(oracle.bf16_bits_to_f64(np.array([0x7FC0], dtype=np.uint16)))[0]

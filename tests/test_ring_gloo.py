"""The multi-process ring driver (exact_long_context_order_b300.ring) on CPU:
gloo ranks, one query shard each, K/V blocks passed one hop per step.

Each rank's step function is the oracle's fold (the plain definition on the
block's keys, merged into the running state by the log-sum-exp identity),
so what is tested here is the communication half of the method: that at
step s rank r holds block (r - s) mod N -- the block's own data, received
from rank r - 1 -- and that the N folds give full attention for the shard.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shards(seed, B, Hq, Hkv, S, D, N, layout):
    """Token-order float64 q, k, v and their shard-major copies."""
    import oracle
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal(s) for s in ((B, Hq, S, D), (B, Hkv, S, D), (B, Hkv, S, D)))
    return (q, k, v), [oracle.to_shard_major(x, N, layout) for x in (q, k, v)]


def _rank_main(rank, world, port, case, q_out):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from exact_long_context_order_b300.ring import ring_attention
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seed, B, Hq, Hkv, S, D, causal, layout = case
        N = world
        Sb = S // N
        g = Hq // Hkv
        sc = 1.0 / math.sqrt(D)
        _, (qs, ks, vs) = _shards(seed, B, Hq, Hkv, S, D, N, layout)
        sl = lambda x, i: torch.from_numpy(np.ascontiguousarray(x[:, :, i * Sb:(i + 1) * Sb]))
        pos = oracle.positions(S, N, layout)
        seen = []

        def oracle_step(q, k, v, N_, i, j, st_o, st_l, out, lse, first, last, causal_, layout_,
                        scale, stream):
            # the block received must be block j's own data
            assert torch.equal(k, sl(ks, j)) and torch.equal(v, sl(vs, j)), (i, j)
            seen.append(j)
            qp, kp = pos[i * Sb:(i + 1) * Sb], pos[j * Sb:(j + 1) * Sb]
            o = np.zeros((B, Hq, Sb, D))
            l = np.zeros((B, Hq, Sb))
            for b in range(B):
                for h in range(Hq):
                    o[b, h], l[b, h] = oracle.attend_rows(q[b, h].numpy(), qp, k[b, h // g].numpy(),
                                                          v[b, h // g].numpy(), kp, causal_, sc)
            if not first:
                o, l = oracle.merge(st_o, st_l, o, l)
            return (o, l, o, l) if last else (o, l, out, lse)

        trace = []
        out, lse = ring_attention(sl(qs, rank), sl(ks, rank), sl(vs, rank), causal=causal,
                                  layout=layout, step_fn=oracle_step, trace=trace)
        q_out.put((rank, trace, seen, out, lse))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,case", [
    (2, (1, 1, 2, 1, 64, 8, True, 0)),     # contiguous causal: rank 0's second block is empty
    (2, (2, 2, 2, 2, 48, 4, True, 1)),     # striped
    (3, (3, 1, 4, 2, 96, 8, True, 2)),     # zigzag, three ranks, GQA
    (3, (4, 1, 2, 2, 60, 6, False, 0)),    # non-causal
])
def test_ring_over_gloo_ranks_equals_full_attention(world, case):
    import oracle
    seed, B, Hq, Hkv, S, D, causal, layout = case
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, case, q_out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q_out.get(timeout=180) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (q, k, v), _ = _shards(seed, B, Hq, Hkv, S, D, world, layout)
    o_ref, l_ref = oracle.full_attention(q, k, v, causal)
    o_sm = oracle.to_shard_major(o_ref, world, layout)
    l_sm = oracle.to_shard_major(l_ref[..., None], world, layout)[..., 0]
    Sb = S // world
    for rank, trace, seen, out, lse in res:
        want = [(s, (rank - s) % world) for s in range(world)]
        assert trace == want
        assert seen == [j for _, j in want]
        np.testing.assert_allclose(out, o_sm[:, :, rank * Sb:(rank + 1) * Sb], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, l_sm[:, :, rank * Sb:(rank + 1) * Sb], rtol=0, atol=1e-12)


def _rank_backward_main(rank, world, port, case, q_out):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from exact_long_context_order_b300.ring import ring_attention_backward
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seed, B, Hq, Hkv, S, D, causal, layout = case
        N = world
        Sb = S // N
        (q, k, v), (qs, ks, vs) = _shards(seed, B, Hq, Hkv, S, D, N, layout)
        dout = np.random.default_rng(seed + 100).standard_normal((B, Hq, S, D))
        o, lse = oracle.full_attention(q, k, v, causal)
        os_, ls_, ds_ = (oracle.to_shard_major(x, N, layout) for x in (o, lse[..., None], dout))
        ls_ = ls_[..., 0]
        sl = lambda x, i: torch.from_numpy(np.ascontiguousarray(x[:, :, i * Sb:(i + 1) * Sb]))
        seen = []

        def oracle_step(q_, k_, v_, out_, lse_, dout_, N_, i, j, delta, dq_st, dk_st, dv_st,
                        first, last, causal_, layout_, scale, stream):
            # the block and its accumulators received come from block j
            assert torch.equal(k_, sl(ks, j)) and torch.equal(v_, sl(vs, j)), (i, j)
            seen.append(j)
            if first:
                delta = (dout_ * out_).sum(-1)
            a, b, c = oracle.ring_step_backward_block(q_, k_, v_, dout_, lse_, delta, N_, i, j,
                                                      causal_, layout_)
            a, b, c = (torch.from_numpy(x) for x in (a, b, c))
            if not first:
                a, b, c = a + dq_st, b + dk_st, c + dv_st
            return (delta, None, None, None, a, b, c) if last else (delta, a, b, c, None, None,
                                                                    None)

        trace = []
        dq, dk, dv = ring_attention_backward(sl(qs, rank), sl(ks, rank), sl(vs, rank),
                                             sl(os_, rank), sl(ls_, rank), sl(ds_, rank),
                                             causal=causal, layout=layout, step_fn=oracle_step,
                                             trace=trace)
        q_out.put((rank, trace, seen, dq.numpy(), dk.numpy(), dv.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,case", [
    (2, (11, 1, 2, 1, 64, 8, True, 0)),    # contiguous causal
    (3, (12, 1, 4, 2, 96, 8, True, 2)),    # zigzag, three ranks, GQA
    (3, (13, 2, 2, 2, 48, 4, False, 1)),   # non-causal, striped
])
def test_ring_backward_over_gloo_ranks_equals_the_gradients(world, case):
    """The backward ring driver: at step s rank r holds block (r - s) mod N
    with that block's accumulators, and after the ring (and the last hop
    home) each rank has its shard's dq and its own block's dk, dv -- the
    plain gradients."""
    import oracle
    seed, B, Hq, Hkv, S, D, causal, layout = case
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_backward_main, args=(r, world, port, case, q_out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q_out.get(timeout=180) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (q, k, v), _ = _shards(seed, B, Hq, Hkv, S, D, world, layout)
    dout = np.random.default_rng(seed + 100).standard_normal((B, Hq, S, D))
    ref = [oracle.to_shard_major(x, world, layout)
           for x in oracle.attention_backward(q, k, v, dout, causal, chunk=32)]
    Sb = S // world
    for rank, trace, seen, dq, dk, dv in res:
        want = [(s, (rank - s) % world) for s in range(world)]
        assert trace == want
        assert seen == [j for _, j in want]
        for got, r in zip((dq, dk, dv), ref):
            np.testing.assert_allclose(got, r[:, :, rank * Sb:(rank + 1) * Sb], rtol=0,
                                       atol=1e-11)

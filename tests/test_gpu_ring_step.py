"""ra_ring_step (one ring step: a query shard folds one key/value block into
its running state) and the multi-process ring driver, on the GPU, against the
oracle.

* One step with both flags: the state is the block's own partial, the plain
  definition over the block's keys (rows with no visible key: output 0,
  lse -inf), for blocks before, at and after the query shard in every
  layout.
* A ring emulated in one process: for every virtual device i, the N steps
  j = i, i-1, ... (mod N) on buffers holding only shard i and block j equal
  full attention (bf16 tolerances).
* Two processes on the one GPU, each a ring device, exchanging blocks over
  gloo through host memory: full attention for each shard.  Their kernels
  never wait on one another; only the host transfer connects them.
* The backward step (ra_ring_step_backward) the same two ways: an emulated
  ring whose blocks carry their fp32 dk/dv accumulators from device to
  device, and two processes training through the autograd function
  (ring_attention_fn): the gradients of every shard against the oracle's.
"""
import math
import os
import socket

import numpy as np
import pytest

import oracle
from helpers import (assert_close, assert_grad_close, backward_reference, delta_error_bounds,
                     from_device, grad_inputs, inputs, reference, to_device)

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def _shard(t, i, Sb):
    return t[:, :, i * Sb:(i + 1) * Sb].contiguous()


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout,i,j", [
    (1, 2, 1, 1024, 4, 128, True, 0, 2, 1),    # an earlier block: every pair visible
    (1, 2, 1, 1024, 4, 128, True, 0, 2, 2),    # the diagonal block
    (1, 2, 1, 1024, 4, 128, True, 0, 1, 3),    # a later block: nothing visible
    (1, 4, 2, 1024, 4, 128, True, 1, 1, 3),    # striped, later block: row 0 sees nothing
    (1, 4, 2, 1024, 4, 128, True, 1, 3, 0),    # striped, earlier block
    (1, 2, 2, 2048, 4, 128, True, 2, 1, 2),    # zigzag, later block: second chunk only
    (1, 3, 1, 2048, 4, 128, True, 2, 2, 0),    # zigzag, odd group (tile pairs)
    (2, 2, 2, 1000, 4, 64, True, 1, 0, 2),     # ragged shards (Sb = 250), D = 64
    (1, 2, 1, 512, 2, 128, False, 0, 0, 1),    # non-causal
])
def test_one_step_is_the_block_partial(ra, B, Hq, Hkv, S, N, D, causal, layout, i, j):
    import torch
    q, k, v = inputs(9500 + S + 7 * i + j, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    Sb = S // N
    _, _, out, lse = ra.ring_step(_shard(tq, i, Sb), _shard(tk, j, Sb), _shard(tv, j, Sb), N, i,
                                  j, first=True, last=True, causal=causal, layout=layout)
    ra.check()
    pos = oracle.positions(S, N, layout)
    qp, kp = pos[i * Sb:(i + 1) * Sb], pos[j * Sb:(j + 1) * Sb]
    g = Hq // Hkv
    ro = np.zeros((B, Hq, Sb, D))
    rl = np.zeros((B, Hq, Sb))
    f = oracle.bf16_bits_to_f64
    for b in range(B):
        for h in range(Hq):
            ro[b, h], rl[b, h] = oracle.attend_rows(
                f(q[b, h, i * Sb:(i + 1) * Sb]), qp, f(k[b, h // g, j * Sb:(j + 1) * Sb]),
                f(v[b, h // g, j * Sb:(j + 1) * Sb]), kp, causal, 1 / math.sqrt(D))
    got_o, got_l = from_device(out), from_device(lse)
    empty = ~np.isfinite(rl)
    assert np.array_equal(~np.isfinite(got_l), empty)
    assert (got_o[empty] == 0).all()
    assert_close(got_o, np.where(empty, 0, got_l), ro, np.where(empty, 0, rl), "bf16",
                 f"step i={i} j={j}")


def virtual_ring(ra, tq, tk, tv, N, causal, layout, scale=None):
    """Every virtual device's N ring steps on buffers holding only its shard
    and the block it holds at that step; returns the shard-major output and
    lse."""
    import torch
    Sb = tq.shape[2] // N
    outs, lses = [], []
    for i in range(N):
        qi = _shard(tq, i, Sb)
        st_o = st_l = out = lse = None
        for s in range(N):
            j = (i - s) % N
            st_o, st_l, out, lse = ra.ring_step(qi, _shard(tk, j, Sb), _shard(tv, j, Sb), N, i, j,
                                                state_o=st_o, state_lse=st_l, first=s == 0,
                                                last=s == N - 1, causal=causal, layout=layout,
                                                scale=scale)
        outs.append(out)
        lses.append(lse)
    return torch.cat(outs, 2), torch.cat(lses, 2)


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout", [
    (1, 4, 2, 2048, 4, 128, True, 1),      # striped GQA
    (2, 2, 2, 1536, 3, 128, True, 0),      # contiguous: later blocks fold nothing
    (1, 2, 1, 4096, 4, 128, True, 2),      # zigzag
    (1, 3, 1, 1000, 4, 128, True, 1),      # ragged (Sb = 250), odd GQA group
    (1, 2, 2, 1024, 2, 64, False, 0),      # non-causal, D = 64
    (1, 8, 1, 2048, 16, 128, True, 1),     # 16 devices of one tile
])
def test_virtual_ring_equals_full_attention(ra, B, Hq, Hkv, S, N, D, causal, layout):
    q, k, v = inputs(9600 + S + N, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out, lse = virtual_ring(ra, tq, tk, tv, N, causal, layout)
    ra.check()
    ro, rl = reference(q, k, v, N, causal, layout, "bf16")
    assert_close(from_device(out), from_device(lse), ro, rl, "bf16", "virtual ring")


def test_virtual_ring_scale_argument(ra):
    B, Hq, Hkv, S, N, D = 1, 4, 2, 1024, 4, 128
    q, k, v = inputs(9650, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out, lse = virtual_ring(ra, tq, tk, tv, N, True, 1, scale=0.05)
    ra.check()
    ro, rl = reference(q, k, v, N, True, 1, "bf16", scale=0.05)
    assert_close(from_device(out), from_device(lse), ro, rl, "bf16", "scaled virtual ring")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ring_rank(rank, world, port, case, q_out):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    import exact_long_context_order_b300 as ra
    from exact_long_context_order_b300.ring import ring_attention
    from helpers import inputs, to_device
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seed, B, Hq, Hkv, S, D, causal, layout = case
        Sb = S // world
        q, k, v = inputs(seed, B, Hq, Hkv, S, D, "bf16")
        mine = [to_device(np.ascontiguousarray(x[:, :, rank * Sb:(rank + 1) * Sb]), "bf16")
                for x in (q, k, v)]
        trace = []
        out, lse = ring_attention(*mine, causal=causal, layout=layout, trace=trace)
        ra.check()
        q_out.put((rank, trace, out.float().cpu().numpy(), lse.cpu().numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [
    (9700, 1, 4, 2, 2048, 128, True, 1),   # striped
    (9701, 1, 2, 2, 2048, 128, True, 0),   # contiguous
])
def test_two_process_ring_on_one_gpu(cuda_ok, case):
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ring_rank, args=(r, world, port, case, q_out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q_out.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    seed, B, Hq, Hkv, S, D, causal, layout = case
    q, k, v = inputs(seed, B, Hq, Hkv, S, D, "bf16")
    ro, rl = reference(q, k, v, world, causal, layout, "bf16")
    Sb = S // world
    for rank, trace, out, lse in res:
        assert trace == [(s, (rank - s) % world) for s in range(world)]
        assert_close(out, lse, ro[:, :, rank * Sb:(rank + 1) * Sb],
                     rl[:, :, rank * Sb:(rank + 1) * Sb], "bf16", f"rank {rank}")


def virtual_ring_backward(ra, tq, tk, tv, tout, tlse, tg, N, causal, layout, scale=None):
    """The backward ring emulated in one process: at step s device i holds
    block j = (i - s) mod N and that block's accumulators, which the step
    updates and the next device receives.  Returns shard-major dq, dk, dv."""
    import torch
    Sb = tq.shape[2] // N
    sh = lambda t, x: _shard(t, x, Sb)
    delta = [None] * N
    dq_st = [None] * N
    dk_st = [None] * N   # block j's accumulators, wherever the block is
    dv_st = [None] * N
    dq, dk, dv = [None] * N, [None] * N, [None] * N
    for s in range(N):
        for i in range(N):
            j = (i - s) % N
            res = ra.ring_step_backward(sh(tq, i), sh(tk, j), sh(tv, j), sh(tout, i),
                                        tlse[:, :, i * Sb:(i + 1) * Sb].contiguous(), sh(tg, i),
                                        N, i, j, delta=delta[i], dq_state=dq_st[i],
                                        dk_state=dk_st[j], dv_state=dv_st[j], first=s == 0,
                                        last=s == N - 1, causal=causal, layout=layout,
                                        scale=scale)
            delta[i], dq_st[i], dk_st[j], dv_st[j] = res[:4]
            if s == N - 1:
                dq[i], dk[j], dv[j] = res[4:]
    return torch.cat(dq, 2), torch.cat(dk, 2), torch.cat(dv, 2)


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,causal,layout", [
    (1, 4, 2, 2048, 4, 128, True, 1),      # striped GQA
    (2, 2, 2, 1536, 3, 128, True, 0),      # contiguous: later blocks add nothing
    (1, 2, 1, 4096, 4, 128, True, 2),      # zigzag
    (1, 3, 1, 1000, 4, 128, True, 1),      # ragged (Sb = 250), odd GQA group
    (1, 2, 2, 1024, 2, 64, False, 0),      # non-causal, D = 64
    (1, 8, 1, 2048, 16, 128, True, 1),     # 16 devices of one tile
    (1, 2, 1, 512, 1, 128, True, 0),       # one device: first and last step at once
])
def test_virtual_ring_backward_equals_the_gradients(ra, B, Hq, Hkv, S, N, D, causal, layout):
    q, k, v = inputs(9800 + S + N, B, Hq, Hkv, S, D, "bf16")
    dout = grad_inputs(9800 + S + N, B, Hq, S, D, "bf16")
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, N, causal=causal, striped=layout)
    got = virtual_ring_backward(ra, tq, tk, tv, out, lse, tg, N, causal, layout)
    ra.check()
    ref = backward_reference(q, k, v, dout, N, causal, layout, "bf16")
    bq, bk = delta_error_bounds(q, k, v, dout, N, causal, layout, "bf16")
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, (bq, bk, None)):
        fro, worst = assert_grad_close(from_device(g), r, "bf16", f"ring backward {name}", e)
        print(f"ring backward {S} {N} {layout} {name}: normwise {fro:.2e}")


def test_virtual_ring_backward_scale_argument(ra):
    B, Hq, Hkv, S, N, D = 1, 4, 2, 1024, 4, 128
    q, k, v = inputs(9850, B, Hq, Hkv, S, D, "bf16")
    dout = grad_inputs(9850, B, Hq, S, D, "bf16")
    tq, tk, tv, tg = (to_device(x, "bf16") for x in (q, k, v, dout))
    out, lse = ra.forward(tq, tk, tv, N, causal=True, striped=1, scale=0.05)
    got = virtual_ring_backward(ra, tq, tk, tv, out, lse, tg, N, True, 1, scale=0.05)
    ra.check()
    ref = backward_reference(q, k, v, dout, N, True, 1, "bf16", scale=0.05)
    bq, bk = delta_error_bounds(q, k, v, dout, N, True, 1, "bf16", scale=0.05)
    for name, g, r, e in zip(("dq", "dk", "dv"), got, ref, (bq, bk, None)):
        assert_grad_close(from_device(g), r, "bf16", f"scaled ring backward {name}", e)


def _train_rank(rank, world, port, case, q_out):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    import exact_long_context_order_b300 as ra
    from exact_long_context_order_b300.ring import ring_attention_fn
    from helpers import grad_inputs, inputs, to_device
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seed, B, Hq, Hkv, S, D, causal, layout = case
        Sb = S // world
        q, k, v = inputs(seed, B, Hq, Hkv, S, D, "bf16")
        dout = grad_inputs(seed, B, Hq, S, D, "bf16")
        mine = [to_device(np.ascontiguousarray(x[:, :, rank * Sb:(rank + 1) * Sb]), "bf16")
                for x in (q, k, v, dout)]
        lq, lk, lv = (t.clone().requires_grad_(True) for t in mine[:3])
        out = ring_attention_fn(lq, lk, lv, causal=causal, layout=layout)
        out.backward(mine[3])
        ra.check()
        q_out.put((rank, *(t.grad.float().cpu().numpy() for t in (lq, lk, lv))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [
    (9900, 1, 4, 2, 2048, 128, True, 1),   # striped
    (9901, 1, 2, 2, 2048, 128, True, 0),   # contiguous
    (9902, 1, 2, 1, 2048, 128, True, 2),   # zigzag: Sb = 1024, two chunks of 512 per shard
])
def test_two_process_training_step_on_one_gpu(cuda_ok, case):
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_train_rank, args=(r, world, port, case, q_out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q_out.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    seed, B, Hq, Hkv, S, D, causal, layout = case
    q, k, v = inputs(seed, B, Hq, Hkv, S, D, "bf16")
    dout = grad_inputs(seed, B, Hq, S, D, "bf16")
    ref = backward_reference(q, k, v, dout, world, causal, layout, "bf16")
    bq, bk = delta_error_bounds(q, k, v, dout, world, causal, layout, "bf16")
    Sb = S // world
    for rank, dq, dk, dv in res:
        sl = lambda x: x[:, :, rank * Sb:(rank + 1) * Sb]
        for name, g, r, e in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (bq, bk, None)):
            assert_grad_close(g, sl(r), "bf16", f"rank {rank} {name}",
                              None if e is None else sl(e))

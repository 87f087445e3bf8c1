"""Ring attention across processes: one query shard per process, K/V blocks
passed round the ring, one ``ra_ring_step`` kernel call per ring step; and
its backward, one ``ra_ring_step_backward`` call per step, with each block's
gradient accumulators travelling with the block.

The method as the pages describe it for several devices ("Ring Attention"
glossary page, "Como funciona a atencao em anel"; aiunderstanding.org,
"Immersione profonda"): device r of N keeps its query block and starts with
its own key/value block.  At step s it holds block j = (r - s) mod N; it
sends that block to device r + 1 and receives block j - 1 from device r - 1,
while it computes its queries against block j and folds the result into its
running online-softmax state.  After N steps every device has exact
attention for its queries.

Here a device is a process of a ``torch.distributed`` group (rank r holds
shard r of the layouts ``ra_forward`` uses: contiguous, striped or zigzag).
The transfer of the next block is started before the step's kernel and
waited for after it, so it runs while the kernel computes:

* NCCL groups (each rank on its own GPU): the block moves device to device
  with ``batch_isend_irecv`` on NCCL's stream; the receive buffer is the one
  the previous step's kernel read, and NCCL orders the receive after that
  kernel; the next kernel waits for the receive.
* Other backends (gloo) with CUDA tensors: the block is staged through
  pinned host memory (device-to-host copy, gloo send/receive, host-to-device
  copy enqueued behind the step's kernel).
* CPU tensors (gloo): sent and received as they are; the step itself is then
  whatever ``step_fn`` computes (the tests pass a CPU fold).

Only the block moves: the query shard, the running state and the output
stay on their device.  No TMA multicast or remote load is involved; every
kernel reads memory of its own GPU.
"""
from __future__ import annotations

from typing import Callable, Optional


class _Exchange:
    """Moves a list of tensors one hop round the ring: sends ``src`` to rank
    (r + 1) mod N and receives the previous rank's tensors into ``dst``."""

    def __init__(self, group, like):
        import torch
        import torch.distributed as dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        to_global = (lambda r: dist.get_global_rank(group, r)) if group is not None else (
            lambda r: r)
        self.next = to_global((self.rank + 1) % self.world)
        self.prev = to_global((self.rank - 1) % self.world)
        backend = dist.get_backend(group)
        self.on_device = like[0].is_cuda
        self.device_path = self.on_device and backend == "nccl"
        self.staged = self.on_device and not self.device_path
        if self.staged:
            self.h_send = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in like]
            self.h_recv = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in like]

    def start(self, src, dst):
        """Starts the transfer; returns a handle for ``finish``."""
        import torch
        import torch.distributed as dist
        if self.device_path:
            ops = [dist.P2POp(dist.isend, t, self.next, self.group) for t in src] + \
                  [dist.P2POp(dist.irecv, t, self.prev, self.group) for t in dst]
            return ("device", dist.batch_isend_irecv(ops), dst)
        if self.staged:
            for h, t in zip(self.h_send, src):
                h.copy_(t, non_blocking=True)
            torch.cuda.current_stream().synchronize()  # the host copies are complete
            src, recv = self.h_send, self.h_recv
        else:
            recv = dst
        works = [dist.isend(t, self.next, group=self.group) for t in src] + \
                [dist.irecv(t, self.prev, group=self.group) for t in recv]
        return ("host", works, dst)

    def finish(self, handle):
        """Waits for the transfer; the received tensors are then ordered
        before any later work on the current stream."""
        kind, works, dst = handle
        for w in works:
            w.wait()
        if kind == "host" and self.staged:
            for t, h in zip(dst, self.h_recv):
                t.copy_(h, non_blocking=True)  # behind this step's kernel on the stream


def _library_step(q, k, v, N, i, j, state_o, state_lse, out, lse, first, last, causal, layout,
                  scale, stream):
    from . import ring_step
    return ring_step(q, k, v, N, i, j, state_o=state_o, state_lse=state_lse, out=out, lse=lse,
                     first=first, last=last, causal=causal, layout=layout, scale=scale,
                     stream=stream)


def ring_attention(q, k, v, group=None, causal: bool = False, layout=0, scale=None,
                   step_fn: Optional[Callable] = None, out=None, lse=None, stream=None,
                   trace: Optional[list] = None):
    """Exact attention for this rank's query shard over the whole sequence.

    q [B, Hq, Sb, D], k and v [B, Hkv, Sb, D]: this rank's shard r of the
    layout (rank r of the group is ring device r of N = group size).  Returns
    (out, lse) for shard r: out like q, lse float32 [B, Hq, Sb].

    ``step_fn(q, k, v, N, i, j, state_o, state_lse, out, lse, first, last,
    causal, layout, scale, stream)`` folds block j into shard i's state and
    returns (state_o, state_lse, out, lse); by default it is the library's
    ``ra_ring_step`` kernel.  ``trace``, when given, receives (s, j) for
    every step in the order they ran.
    """
    import contextlib

    import torch
    import torch.distributed as dist
    N = dist.get_world_size(group)
    r = dist.get_rank(group)
    step = step_fn or _library_step
    # the kernels and the staging copies all go to one stream: the given one,
    # made current for the call, or the current one
    ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
    with ctx:
        return _ring_loop(q, k, v, group, N, r, step, causal, layout, scale, out, lse, trace)


def _ring_loop(q, k, v, group, N, r, step, causal, layout, scale, out, lse, trace):
    import torch
    cur = [k, v]
    spare = [torch.empty_like(k), torch.empty_like(v)] if N > 1 else None
    ex = _Exchange(group, cur) if N > 1 else None
    state_o = state_lse = None
    for s in range(N):
        j = (r - s) % N
        handle = ex.start(cur, spare) if s < N - 1 else None
        state_o, state_lse, out, lse = step(q, cur[0], cur[1], N, r, j, state_o, state_lse, out,
                                            lse, s == 0, s == N - 1, causal, layout, scale,
                                            None)
        if trace is not None:
            trace.append((s, j))
        if handle is not None:
            ex.finish(handle)
            cur, spare = spare, cur
    return out, lse


def _library_step_backward(q, k, v, out, lse, dout, N, i, j, delta, dq_state, dk_state, dv_state,
                           first, last, causal, layout, scale, stream):
    from . import ring_step_backward
    return ring_step_backward(q, k, v, out, lse, dout, N, i, j, delta=delta, dq_state=dq_state,
                              dk_state=dk_state, dv_state=dv_state, first=first, last=last,
                              causal=causal, layout=layout, scale=scale, stream=stream)


def ring_attention_backward(q, k, v, out, lse, dout, group=None, causal: bool = False,
                            layout=0, scale=None, step_fn: Optional[Callable] = None,
                            stream=None, trace: Optional[list] = None):
    """Gradients (dq, dk, dv) of ``ring_attention`` for this rank's shard.

    q, out, dout [B, Hq, Sb, D], lse [B, Hq, Sb] (the forward's), k, v
    [B, Hkv, Sb, D]: rank r's shard of the layout.  The ring is the
    forward's: at step s rank r holds block j = (r - s) mod N together with
    that block's fp32 accumulators dK_j, dV_j; it adds block j's terms into
    its own dQ_r and its shard's terms into dK_j, dV_j (``ra_ring_step_backward``),
    then passes the block and the accumulators to rank r + 1.  K and V move
    while the step computes; the accumulators move after it (the step
    updates them).  After the last step the block's finished dk, dv (bf16)
    take one more hop, to the rank that owns that block.

    ``step_fn(q, k, v, out, lse, dout, N, i, j, delta, dq_state, dk_state,
    dv_state, first, last, causal, layout, scale, stream)`` returns (delta,
    dq_state, dk_state, dv_state, dq, dk, dv); by default the library's kernel.
    ``trace``, when given, receives (s, j) for every step.
    """
    import contextlib

    import torch
    import torch.distributed as dist
    N = dist.get_world_size(group)
    r = dist.get_rank(group)
    step = step_fn or _library_step_backward
    ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
    with ctx:
        return _ring_backward_loop(q, k, v, out, lse, dout, group, N, r, step, causal, layout,
                                   scale, trace)


def _ring_backward_loop(q, k, v, out, lse, dout, group, N, r, step, causal, layout, scale, trace):
    import torch
    f32 = torch.float32 if k.dtype != torch.float64 else torch.float64
    kv = [k, v]
    acc = [torch.empty(k.shape, dtype=f32, device=k.device),
           torch.empty(v.shape, dtype=f32, device=v.device)]
    spare_kv = [torch.empty_like(k), torch.empty_like(v)] if N > 1 else None
    spare_acc = [torch.empty_like(acc[0]), torch.empty_like(acc[1])] if N > 1 else None
    ex_kv = _Exchange(group, kv) if N > 1 else None
    ex_acc = _Exchange(group, acc) if N > 1 else None
    delta = dq_state = None
    dq = dk = dv = None
    for s in range(N):
        j = (r - s) % N
        first, last = s == 0, s == N - 1
        handle = ex_kv.start(kv, spare_kv) if not last else None
        delta, dq_state, dk_st, dv_st, dq, dk, dv = step(
            q, kv[0], kv[1], out, lse, dout, N, r, j, delta, dq_state, acc[0], acc[1], first,
            last, causal, layout, scale, None)
        if trace is not None:
            trace.append((s, j))
        if not last:
            acc = [dk_st, dv_st]
            h_acc = ex_acc.start(acc, spare_acc)
            ex_kv.finish(handle)
            ex_acc.finish(h_acc)
            kv, spare_kv = spare_kv, kv
            acc, spare_acc = spare_acc, acc
    if N > 1:
        # the finished gradients of block r + 1 go home; block r's come in
        ex_out = _Exchange(group, [dk, dv])
        home = [torch.empty_like(dk), torch.empty_like(dv)]
        ex_out.finish(ex_out.start([dk, dv], home))
        dk, dv = home
    return dq, dk, dv


def _autograd_function():
    import torch

    class RingAttentionFn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, group, causal, layout, scale):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            out, lse = ring_attention(q, k, v, group=group, causal=causal, layout=layout,
                                      scale=scale)
            ctx.save_for_backward(q, k, v, out, lse)
            ctx.cfg = (group, causal, layout, scale)
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            group, causal, layout, scale = ctx.cfg
            dq, dk, dv = ring_attention_backward(q, k, v, out, lse, dout.contiguous(),
                                                 group=group, causal=causal, layout=layout,
                                                 scale=scale)
            return dq, dk, dv, None, None, None, None

    return RingAttentionFn


_FN = []


def ring_attention_fn(q, k, v, group=None, causal: bool = False, layout=0, scale=None):
    """``ring_attention`` with autograd: its backward is ``ring_attention_backward``
    over the same group (every rank must run both, in the same order)."""
    if not _FN:
        _FN.append(_autograd_function())
    return _FN[0].apply(q, k, v, group, causal, layout, scale)

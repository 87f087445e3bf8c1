"""ra_forward_host: the forward on host tensors (H2D copies, the kernel, D2H
copies on one stream) gives the same bits as ra_forward on device tensors."""
import numpy as np
import pytest

from helpers import inputs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def test_forward_host_equals_device_forward(ra):
    import torch
    B, Hq, Hkv, S, N, D = 1, 4, 2, 2048, 4, 128
    q, k, v = inputs(8200, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out0, lse0 = ra.forward(tq, tk, tv, N, causal=True, striped=1)
    ra.check()
    hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
                  for x in (q, k, v))
    out_h = torch.empty(hq.shape, dtype=torch.int16).pin_memory()
    lse_h = torch.empty((B, Hq, S), dtype=torch.float32).pin_memory()
    stage = [torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv),
             torch.empty_like(tq), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")]
    P = ra._ptr
    side = torch.cuda.Stream()
    rc = ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), P(lse_h), *[P(x) for x in stage], B,
                            Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16, ra._stream_handle(side))
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(ra._stream_handle(side)) == ra.RA_OK
    assert torch.equal(out_h, out0.view(torch.int16).cpu())
    assert torch.equal(lse_h, lse0.cpu())
    # without lse
    out_h.zero_()
    rc = ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), None, *[P(x) for x in stage[:4]], None,
                            B, Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16, ra._stream_handle(side))
    assert rc == ra.RA_OK
    assert ra.ra_check(ra._stream_handle(side)) == ra.RA_OK
    assert torch.equal(out_h, out0.view(torch.int16).cpu())
    # an lse pair with one side missing is refused before anything is enqueued
    assert ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), P(lse_h), *[P(x) for x in stage[:4]],
                              None, B, Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16,
                              None) == ra.RA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,dt", [
    (2, 8, 4, 1024, 4, 128, "bf16"),    # 8 (batch, KV head) groups: one per chunk
    (2, 10, 5, 512, 2, 64, "bf16"),     # 10 groups over 8 chunks: uneven chunks
    (1, 12, 4, 1000, 4, 128, "bf16"),   # ragged shards (Sb = 250), 4 groups
    (1, 4, 4, 256, 2, 32, "f32"),       # the SIMT kernel, 4 groups
    # chunk offsets that are not 16-byte multiples (lse: 24 bytes per group;
    # q: 24 bytes per group): the call must run in order, not pipelined
    (1, 4, 4, 6, 2, 16, "bf16"),
    (1, 4, 4, 3, 1, 4, "bf16"),
])
def test_pipelined_forward_host_equals_device_forward(ra, B, Hq, Hkv, S, N, D, dt):
    """With at least four (batch, KV head) groups the call pipelines chunks of
    groups over internal copy and compute streams: same bits as ra.forward."""
    import torch
    q, k, v = inputs(8300 + S + Hq, B, Hq, Hkv, S, D, dt)
    tq, tk, tv = (to_device(x, dt) for x in (q, k, v))
    out0, lse0 = ra.forward(tq, tk, tv, N, causal=True, striped=1)
    ra.check()
    view = np.int16 if dt == "bf16" else np.float32
    hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(x).view(view)).pin_memory()
                  for x in (q, k, v))
    out_h = torch.zeros(hq.shape, dtype=hq.dtype).pin_memory()
    lse_h = torch.zeros((B, Hq, S), dtype=torch.float32).pin_memory()
    stage = [torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv),
             torch.empty_like(tq), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")]
    P = ra._ptr
    dtype = ra.RA_BF16 if dt == "bf16" else ra.RA_F32
    side = torch.cuda.Stream()
    for with_lse in (True, False):
        out_h.zero_()
        lse_args = (P(lse_h), P(stage[4])) if with_lse else (None, None)
        rc = ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), lse_args[0],
                                *[P(x) for x in stage[:4]], lse_args[1], B, Hq, Hkv, S, D, N,
                                1, 1, 0.0, dtype, ra._stream_handle(side))
        assert rc == ra.RA_OK, ra.ra_strerror(rc)
        assert ra.ra_check(ra._stream_handle(side)) == ra.RA_OK
        ref = out0.view(torch.int16) if dt == "bf16" else out0
        assert torch.equal(out_h, ref.cpu())
        if with_lse:
            assert torch.equal(lse_h, lse0.cpu())


def test_pipelined_calls_on_two_streams_reuse_staging_safely(ra):
    """Three calls with different inputs alternate between two caller streams
    and two staging sets, with no host synchronisation between them: call 3
    reuses call 1's staging set, so its uploads must wait for call 1's
    downloads (the call is ordered on its caller's stream).  Every output is
    the device forward of its own inputs."""
    import torch
    B, Hq, Hkv, S, N, D = 1, 8, 4, 1024, 4, 128
    P = ra._ptr
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    stages = [[torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device="cuda"),
               torch.empty((B, Hkv, S, D), dtype=torch.bfloat16, device="cuda"),
               torch.empty((B, Hkv, S, D), dtype=torch.bfloat16, device="cuda"),
               torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device="cuda"),
               torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")] for _ in range(2)]
    calls = []
    for n in range(3):
        q, k, v = inputs(8400 + n, B, Hq, Hkv, S, D, "bf16")
        host = [torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
                for x in (q, k, v)]
        out_h = torch.zeros((B, Hq, S, D), dtype=torch.int16).pin_memory()
        lse_h = torch.zeros((B, Hq, S), dtype=torch.float32).pin_memory()
        calls.append((q, k, v, host, out_h, lse_h))
    torch.cuda.synchronize()
    for n, (q, k, v, host, out_h, lse_h) in enumerate(calls):
        st = streams[n % 2]
        rc = ra.ra_forward_host(*[P(x) for x in host], P(out_h), P(lse_h),
                                *[P(x) for x in stages[n % 2]], B, Hq, Hkv, S, D, N, 1, 1, 0.0,
                                ra.RA_BF16, ra._stream_handle(st))
        assert rc == ra.RA_OK, ra.ra_strerror(rc)
    for st in streams:
        assert ra.ra_check(ra._stream_handle(st)) == ra.RA_OK
    for q, k, v, host, out_h, lse_h in calls:
        tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
        out0, lse0 = ra.forward(tq, tk, tv, N, causal=True, striped=1)
        ra.check()
        assert torch.equal(out_h, out0.view(torch.int16).cpu())
        assert torch.equal(lse_h, lse0.cpu())


def test_forward_host_of_a_stream_k_problem_equals_device_forward(ra):
    """A non-causal problem that ra_forward runs as stream-K (256 items) is
    run whole by ra_forward_host rather than in chunks, so the bits match."""
    import torch
    B, Hq, Hkv, S, N, D = 2, 8, 8, 4096, 2, 64
    q, k, v = inputs(8500, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    out0, lse0 = ra.forward(tq, tk, tv, N, causal=False)
    ra.check()
    hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
                  for x in (q, k, v))
    out_h = torch.zeros(hq.shape, dtype=torch.int16).pin_memory()
    lse_h = torch.zeros((B, Hq, S), dtype=torch.float32).pin_memory()
    stage = [torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv),
             torch.empty_like(tq), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")]
    P = ra._ptr
    side = torch.cuda.Stream()
    rc = ra.ra_forward_host(P(hq), P(hk), P(hv), P(out_h), P(lse_h), *[P(x) for x in stage], B,
                            Hq, Hkv, S, D, N, 0, 0, 0.0, ra.RA_BF16, ra._stream_handle(side))
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(ra._stream_handle(side)) == ra.RA_OK
    assert torch.equal(out_h, out0.view(torch.int16).cpu())
    assert torch.equal(lse_h, lse0.cpu())

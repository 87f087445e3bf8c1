"""CUDA-graph capture of the hot path: ra_forward and ra_backward are
asynchronous on the caller's stream (the work counter is zeroed by a stream
memset, nothing synchronises), so they can be captured once and replayed.
Both are deterministic, so every replay must equal the eager results bit for
bit."""
import pytest

from helpers import grad_inputs, inputs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


def test_forward_and_backward_replay_from_a_cuda_graph(ra):
    import torch
    B, Hq, Hkv, S, N, D = 1, 4, 2, 2048, 4, 128
    q, k, v = (to_device(x, "bf16") for x in inputs(8100, B, Hq, Hkv, S, D, "bf16"))
    dout = to_device(grad_inputs(8100, B, Hq, S, D, "bf16"), "bf16")
    # eager reference (also makes the library's one-time per-device setup
    # happen outside capture)
    out0, lse0 = ra.forward(q, k, v, N, causal=True, striped=1)
    g0 = ra.backward(q, k, v, out0, lse0, dout, N, causal=True, striped=1)
    ra.check()
    rc, need = ra.ra_backward_workspace(B, Hq, S, D)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            ra.forward(q, k, v, N, causal=True, striped=1, out=out, lse=lse, stream=side)
            grads = ra.backward(q, k, v, out, lse, dout, N, causal=True, striped=1,
                                workspace=ws, stream=side)
    for _ in range(3):
        out.zero_()
        for t in grads:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert ra.ra_check(ra._stream_handle(side)) == ra.RA_OK
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse, lse0)
        for a, b in zip(grads, g0):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))

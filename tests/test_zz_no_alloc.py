"""ra_forward_noalloc: the forward entry point for callers that cannot allocate
device memory (a server whose memory pool owns the whole GPU, a framework
caching allocator, code that cannot afford cudaMalloc's synchronisation).

It keeps its scratch -- the tensor-core kernel's work-queue counter -- in a
static device array instead of memory allocated by the library.  The test
calls it twice in a row through the C ABI and checks that both results are
the bits ra_forward computes on the same inputs (the same kernel runs), and
the first against the oracle with the bf16 tolerances of the other GPU tests
(output max-abs 2e-2 and mean-abs 2e-3, lse max-abs 2e-3).  The second call
shows that the shared counter, left at its final count by the first call, is
cleared before the next kernel runs.
"""
import pytest

from helpers import assert_close, from_device, inputs, reference, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra(cuda_ok):
    import exact_long_context_order_b300 as m
    from exact_long_context_order_b300 import build
    build.build()
    m.lib()
    return m


@pytest.mark.parametrize("B,Hq,Hkv,S,N,D,layout", [
    (1, 4, 2, 2048, 4, 128, 1),   # striped GQA, whole tiles
    (2, 3, 3, 1000, 4, 64, 0),    # contiguous MHA, D = 64, ragged shards (Sb = 250)
])
def test_noalloc_matches_forward_on_two_calls(ra, B, Hq, Hkv, S, N, D, layout):
    """Both calls run the tensor-core kernel that ra_forward runs, on the same
    inputs, so their outputs must be the same bits; the first is also checked
    against the oracle at the bf16 tolerances."""
    import torch
    q, k, v = inputs(9001 + S, B, Hq, Hkv, S, D, "bf16")
    tq, tk, tv = (to_device(x, "bf16") for x in (q, k, v))
    stream = ra._stream_handle(None)

    ref_out = torch.empty_like(tq)
    ref_lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    rc = ra.ra_forward(ra._ptr(tq), ra._ptr(tk), ra._ptr(tv), ra._ptr(ref_out), ra._ptr(ref_lse),
                       B, Hq, Hkv, S, D, N, 1, layout, 0.0, ra.RA_BF16, stream)
    assert rc == ra.RA_OK, ra.ra_strerror(rc)
    assert ra.ra_check(stream) == ra.RA_OK

    for call in range(2):
        out = torch.full_like(tq, float("nan"))
        lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
        rc = ra.ra_forward_noalloc(ra._ptr(tq), ra._ptr(tk), ra._ptr(tv), ra._ptr(out),
                                   ra._ptr(lse), B, Hq, Hkv, S, D, N, 1, layout, 0.0, stream)
        assert rc == ra.RA_OK, ra.ra_strerror(rc)
        assert ra.ra_check(stream) == ra.RA_OK
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}"
        assert torch.equal(lse, ref_lse), f"call {call}"
        if call == 0:
            ro, rl = reference(q, k, v, N, True, layout, "bf16")
            assert_close(from_device(out), from_device(lse), ro, rl, "bf16", "noalloc")


def test_noalloc_rejects_shapes_outside_the_tensor_core_kernel(ra):
    """Calls that must be refused on the host.  Every pointer is a real device
    buffer large enough for the problem, so a call that were accepted by
    mistake would still read and write valid memory."""
    import torch

    def bufs(B, H, S, D):
        q = torch.zeros((B, H, S, D), dtype=torch.bfloat16, device="cuda")
        return q, torch.zeros_like(q), torch.zeros_like(q), torch.zeros_like(q)

    q, k, v, o = bufs(1, 1, 256, 96)          # D = 96: no tensor-core kernel
    assert ra.ra_forward_noalloc(ra._ptr(q), ra._ptr(k), ra._ptr(v), ra._ptr(o), None,
                                 1, 1, 1, 256, 96, 2, 1, 0, 0.0, None) == ra.RA_ERR_UNSUPPORTED
    q, k, v, o = bufs(1, 1, 768, 128)         # zigzag with S/N = 384: chunks are not whole tiles
    assert ra.ra_forward_noalloc(ra._ptr(q), ra._ptr(k), ra._ptr(v), ra._ptr(o), None,
                                 1, 1, 1, 768, 128, 2, 1, 2, 0.0, None) == ra.RA_ERR_UNSUPPORTED
    assert ra.ra_forward_noalloc(None, ra._ptr(k), ra._ptr(v), ra._ptr(o), None,
                                 1, 1, 1, 768, 128, 2, 1, 0, 0.0, None) == ra.RA_ERR_INVALID_ARG
    torch.cuda.synchronize()

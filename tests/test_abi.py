"""C-ABI library checks that need no GPU: it loads, exports every function
that include/ra.h declares, rejects bad arguments on the host before touching
a device, and its fold planner equals the oracle's brute-force schedule."""
import ctypes
import os
import re

import pytest

import exact_long_context_order_b300 as ra
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ra_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from exact_long_context_order_b300 import build
    build.build()
    return ra.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"ra_forward", "ra_merge", "ra_plan", "ra_check", "ra_strerror"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in ra._SIGNATURES, n


def test_strerror_and_config(lib):
    assert ra.ra_strerror(ra.RA_OK) == "ok"
    for c in range(1, 8):
        assert ra.ra_strerror(c) and ra.ra_strerror(c) != "unknown status"
    assert ra.ra_strerror(99) == "unknown status"
    assert ra.ra_tile_config() == (128, 128)
    assert ra.ra_version() >= 100


def test_host_validation_rejects_before_any_device_work(lib):
    p = ctypes.c_void_p(16 * 1024)  # never dereferenced: validation fails first
    args = dict(B=1, Hq=2, Hkv=1, S=256, D=128, N=2)

    def call(q=p, k=p, v=p, out=p, **kw):
        a = dict(args, **kw)
        return ra.ra_forward(q, k, v, out, None, a["B"], a["Hq"], a["Hkv"], a["S"], a["D"],
                             a["N"], 1, 0, 0.0, ra.RA_BF16, None)

    assert call(q=None) == ra.RA_ERR_INVALID_ARG
    assert call(S=255) == ra.RA_ERR_INVALID_ARG          # S % N
    assert call(Hq=3, Hkv=2) == ra.RA_ERR_INVALID_ARG    # Hq % Hkv
    assert call(B=-1) == ra.RA_ERR_INVALID_ARG
    assert call(N=0, S=0) == ra.RA_ERR_INVALID_ARG
    assert call(D=512) == ra.RA_ERR_UNSUPPORTED
    p2 = ctypes.c_void_p(16 * 1024)
    assert ra.ra_forward(p2, p2, p2, p2, None, 1, 1, 1, 6, 8, 2, 1, 2, 0.0, ra.RA_BF16,
                         None) == ra.RA_ERR_INVALID_ARG   # zigzag needs an even S/N
    assert ra.ra_forward(p2, p2, p2, p2, None, 1, 1, 1, 8, 8, 2, 1, 3, 0.0, ra.RA_BF16,
                         None) == ra.RA_ERR_INVALID_ARG   # unknown layout
    assert ra.ra_relayout(p2, ctypes.c_void_p(1 << 30), 1, 6, 2, 16, 2, 0,
                          None) == ra.RA_ERR_INVALID_ARG
    assert call(q=ctypes.c_void_p(16 * 1024 + 2)) == ra.RA_ERR_ALIGN
    assert ra.ra_forward_ex(p, p, p, p, None, 1, 1, 1, 256, 128, 2, 0, 0, 0.0, ra.RA_BF16, 7,
                            None) == ra.RA_ERR_INVALID_ARG
    assert ra.ra_forward(p, p, p, p, None, 1, 1, 1, 256, 128, 2, 0, 0, 0.0, 5, None) == \
        ra.RA_ERR_INVALID_ARG
    assert ra.ra_merge(p, p, p, p, 10, 0, ra.RA_BF16, None) == ra.RA_ERR_INVALID_ARG
    assert ra.ra_merge(p, p, p, p, -1, 8, ra.RA_BF16, None) == ra.RA_ERR_INVALID_ARG
    assert ra.ra_merge(None, None, None, None, 0, 8, ra.RA_BF16, None) == ra.RA_OK  # empty
    assert ra.ra_stripe(p, p, 1, 10, 3, 16, 0, None) == ra.RA_ERR_INVALID_ARG  # S % N
    assert ra.ra_stripe(p, p, 1, 8, 2, 6, 0, None) == ra.RA_ERR_INVALID_ARG   # row_bytes % 4
    assert ra.ra_stripe(p, ctypes.c_void_p(16 * 1024 + 64), 1, 8, 2, 16, 0, None) == \
        ra.RA_ERR_INVALID_ARG  # overlapping buffers


def test_plan_errors(lib):
    n = ctypes.c_int64()
    T = ra.ra_plan_tile
    assert T(256, 2, 1, 0, 128, 0, 0, None, 0, None) == ra.RA_ERR_INVALID_ARG
    assert T(256, 2, 1, 2, 96, 0, 0, None, 0, ctypes.byref(n)) == ra.RA_ERR_INVALID_ARG
    assert T(256, 2, 1, 0, 128, 2, 0, None, 0, ctypes.byref(n)) == ra.RA_ERR_INVALID_ARG
    assert T(256, 2, 1, 0, 128, 0, 1, None, 0, ctypes.byref(n)) == ra.RA_ERR_INVALID_ARG
    assert T(256, 2, 1, 0, 128, 1, 0, None, 0, ctypes.byref(n)) == ra.RA_OK
    assert n.value == 2  # shard 1 of 2, contiguous causal: shard 0 full, own diagonal
    buf = (ctypes.c_int32 * 4)()
    assert T(256, 2, 1, 0, 128, 1, 0, buf, 1, ctypes.byref(n)) == ra.RA_ERR_CAPACITY
    assert n.value == 2
    # the whole schedule
    assert ra.ra_plan(256, 2, 1, 0, 128, None, 0, None) == ra.RA_ERR_INVALID_ARG
    assert ra.ra_plan(256, 2, 1, 2, 96, None, 0, ctypes.byref(n)) == ra.RA_ERR_INVALID_ARG
    assert ra.ra_plan(255, 2, 1, 0, 128, None, 0, ctypes.byref(n)) == ra.RA_ERR_INVALID_ARG
    assert ra.ra_plan(256, 2, 1, 0, 128, None, 0, ctypes.byref(n)) == ra.RA_OK
    assert n.value == 3  # shard 0: its diagonal; shard 1: shard 0 full and its diagonal
    buf = (ctypes.c_int32 * 12)()
    assert ra.ra_plan(256, 2, 1, 0, 128, buf, 2, ctypes.byref(n)) == ra.RA_ERR_CAPACITY
    assert n.value == 3


@pytest.mark.parametrize("causal,striped", [(False, False), (True, False), (True, True),
                                            (True, 2)])
@pytest.mark.parametrize("S,N,T", [(512, 4, 32), (768, 3, 64), (256, 1, 128), (1024, 8, 16),
                                   (96, 6, 2)])
def test_plan_equals_bruteforce_schedule(lib, causal, striped, S, N, T):
    """Bit-exact: the library's closed-form fold list == oracle brute force."""
    ref = oracle.fold_schedule(S, N, causal, striped, T, T)
    by_tile = {}
    for (i, qt, s, j, kt, kind) in ref:
        by_tile.setdefault((i, qt), []).append((s, j, kt, kind))
    nt = -(-(S // N) // T)
    for i in range(N):
        for qt in range(nt):
            assert ra.plan(S, N, causal, striped, i, qt, tile=T) == by_tile.get((i, qt), []), \
                (i, qt)


@pytest.mark.parametrize("causal,striped", [(False, False), (True, False), (True, True),
                                            (True, 2)])
@pytest.mark.parametrize("S,N,T", [(512, 4, 32), (600, 3, 60), (256, 1, 128), (7 * 44, 7, 22)])
def test_whole_schedule_equals_bruteforce_schedule(lib, causal, striped, S, N, T):
    """Bit-exact: ra_plan's ordered work list == the oracle's brute-force
    schedule, entry by entry (shards, tiles, ring steps, key tiles, kinds)."""
    if striped == 2 and (S // N) % (2 * T):
        pytest.skip("zigzag chunks must be whole tiles")
    want = [tuple(int(x) for x in e) for e in oracle.fold_schedule(S, N, causal, striped, T, T)]
    assert ra.plan_schedule(S, N, causal, striped, tile=T) == want


@pytest.mark.parametrize("causal,striped", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("S,N,T", [(600, 3, 64), (130, 1, 16), (7 * 44, 7, 8)])
def test_plan_with_a_partial_last_tile(lib, causal, striped, S, N, T):
    """Shards whose size is not a multiple of the tile: ceil(Sb/T) tiles, the
    last partial; the planner still equals the brute-force schedule."""
    ref = oracle.fold_schedule(S, N, causal, striped, T, T)
    by_tile = {}
    for (i, qt, s, j, kt, kind) in ref:
        by_tile.setdefault((i, qt), []).append((s, j, kt, kind))
    nt = -(-(S // N) // T)
    assert (S // N) % T
    for i in range(N):
        for qt in range(nt):
            assert ra.plan(S, N, causal, striped, i, qt, tile=T) == by_tile.get((i, qt), []), \
                (i, qt)


def test_backward_host_validation(lib):
    """ra_backward refuses bad arguments on the host (no device needed)."""
    n = ctypes.c_int64()
    assert lib.ra_backward_workspace(2, 4, 1000, 128, ctypes.byref(n)) == ra.RA_OK
    assert n.value == 32000  # delta: 4 bytes for each of 2*4*1000 rows, already 256-aligned
    assert lib.ra_backward_workspace(1, 1, 10, 8, ctypes.byref(n)) == ra.RA_OK and n.value == 256
    assert lib.ra_backward_workspace(-1, 4, 1000, 128, ctypes.byref(n)) == ra.RA_ERR_INVALID_ARG
    assert lib.ra_backward_workspace(1, 0, 1000, 128, ctypes.byref(n)) == ra.RA_ERR_INVALID_ARG
    assert lib.ra_backward_workspace(0, 4, 1000, 128, ctypes.byref(n)) == ra.RA_OK and n.value == 0
    assert lib.ra_backward_workspace(1, 1, 10, 8, None) == ra.RA_ERR_INVALID_ARG
    p = ctypes.c_void_p(16 * 1024)  # never dereferenced: validation fails first

    def call(D=64, ws=1 << 30, nulls=(), kernel=ra.RA_KERNEL_AUTO, S=256):
        a = [p] * 10
        for i in nulls:
            a[i] = None
        return ra.ra_backward_ex(*a, ws, 1, 2, 1, S, D, 2, 1, 1, 0.0, ra.RA_BF16, kernel, None)

    assert call(nulls=(4,)) == ra.RA_ERR_INVALID_ARG      # lse
    assert call(nulls=(9,)) == ra.RA_ERR_INVALID_ARG      # workspace
    assert call(nulls=(6,)) == ra.RA_ERR_INVALID_ARG      # dq
    assert call(D=192) == ra.RA_ERR_UNSUPPORTED
    assert call(ws=100) == ra.RA_ERR_CAPACITY
    assert call(kernel=9) == ra.RA_ERR_INVALID_ARG
    assert call(S=255) == ra.RA_ERR_INVALID_ARG           # S % N


@pytest.mark.parametrize("causal,striped", [(False, False), (True, False), (True, True),
                                            (True, 2)])
@pytest.mark.parametrize("S,N,T", [(512, 4, 32), (768, 3, 64), (256, 1, 128), (1024, 8, 16),
                                   (600, 3, 64), (130, 1, 16)])
def test_plan_backward_equals_transposed_bruteforce(lib, causal, striped, S, N, T):
    """Bit-exact: the dk/dv visiting order of every key tile is the oracle's
    brute-force schedule read by key tile: query shards ascending (the block
    goes round the ring entering at device 0, reaching shard i at step
    s = (i - j) mod N), then query tiles ascending."""
    if striped == 2 and (S // N) % (2 * T):
        pytest.skip("zigzag needs whole-tile chunks")
    ref = oracle.fold_schedule(S, N, causal, striped, T, T)
    by_key = {}
    for (i, qt, s, j, kt, kind) in ref:
        assert (i - j) % N == s
        by_key.setdefault((j, kt), []).append((s, i, qt, kind))
    nt = -(-(S // N) // T)
    for j in range(N):
        for kt in range(nt):
            want = sorted(by_key.get((j, kt), []), key=lambda e: (e[1], e[2]))
            assert ra.plan_backward(S, N, causal, striped, j, kt, tile=T) == want, (j, kt)


def test_empty_problems_are_noops_without_a_device(lib):
    """B == 0 or S == 0: nothing to read or write.  The attention entry points
    return RA_OK before any CUDA call (this test runs without a GPU), accept
    NULL buffers, and still reject invalid non-size arguments; the self tests
    and the fold log, which need a kernel, reject an empty problem."""
    nul = None
    for B, S in ((0, 256), (1, 0), (0, 0)):
        assert ra.ra_forward(nul, nul, nul, nul, nul, B, 2, 1, S, 128, 2, 1, 1, 0.0, ra.RA_BF16,
                             None) == ra.RA_OK
        assert ra.ra_forward_ex(nul, nul, nul, nul, nul, B, 2, 1, S, 64, 2, 0, 2, 0.0, ra.RA_F32,
                                ra.RA_KERNEL_TC, None) == ra.RA_OK
        assert ra.ra_forward_noalloc(nul, nul, nul, nul, nul, B, 2, 1, S, 128, 2, 1, 1, 0.0,
                                     None) == ra.RA_OK
        assert ra.ra_forward_host(nul, nul, nul, nul, nul, nul, nul, nul, nul, nul, B, 2, 1, S,
                                  128, 2, 1, 1, 0.0, ra.RA_BF16, None) == ra.RA_OK
        assert ra.ra_backward(*([nul] * 10), 0, B, 2, 1, S, 128, 2, 1, 1, 0.0, ra.RA_BF16,
                              None) == ra.RA_OK
        assert ra.ra_watchdog_selftest(nul, nul, nul, nul, nul, B, 2, 1, S, 128, 2, 1, 1, 0.0,
                                       1 << 20, None) == ra.RA_ERR_INVALID_ARG
        assert ra.ra_watchdog_selftest_backward(*([nul] * 10), 0, B, 2, 1, S, 128, 2, 1, 1, 0.0,
                                                1 << 20, 0, None) == ra.RA_ERR_INVALID_ARG
    # the other arguments are still checked on an empty problem
    assert ra.ra_forward(nul, nul, nul, nul, nul, 0, 3, 2, 256, 128, 2, 1, 1, 0.0, ra.RA_BF16,
                         None) == ra.RA_ERR_INVALID_ARG   # Hq % Hkv
    assert ra.ra_forward(nul, nul, nul, nul, nul, 0, 2, 1, 255, 128, 2, 1, 1, 0.0, ra.RA_BF16,
                         None) == ra.RA_ERR_INVALID_ARG   # S % N
    assert ra.ra_forward(nul, nul, nul, nul, nul, 1, 2, 1, 0, 512, 2, 1, 1, 0.0, ra.RA_BF16,
                         None) == ra.RA_ERR_UNSUPPORTED   # D > 256
    assert ra.ra_forward(nul, nul, nul, nul, nul, 1, 2, 1, 0, 128, 2, 1, 1, 0.0, 9,
                         None) == ra.RA_ERR_INVALID_ARG   # dtype
    assert ra.ra_backward(*([nul] * 10), 0, 0, 2, 1, 256, 192, 2, 1, 1, 0.0, ra.RA_BF16,
                          None) == ra.RA_ERR_UNSUPPORTED  # backward D > 128
    # a non-empty problem still needs its buffers
    assert ra.ra_forward(nul, nul, nul, nul, nul, 1, 2, 1, 256, 128, 2, 1, 1, 0.0, ra.RA_BF16,
                         None) == ra.RA_ERR_INVALID_ARG


def test_size_limits_are_rejected_before_any_device_work(lib):
    """Problems beyond a kernel's envelope (int32 TMA row coordinates, 65535
    grid rows) are refused on the host, before any CUDA call: this test runs
    without a GPU and passes placeholder pointers that are never touched."""
    p = ctypes.c_void_p(16 * 1024)
    fwd = lambda B, Hq, Hkv, S, D, N, kernel: ra.ra_forward_ex(
        p, p, p, p, None, B, Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16, kernel, None)
    # B*Hq*S = 2^31 rows: past the tensor-core kernel's int32 row coordinates
    assert fwd(1, 1 << 14, 1, 1 << 17, 128, 16, ra.RA_KERNEL_TC) == ra.RA_ERR_UNSUPPORTED
    # ... and B*Hq = 65536 query heads: past the SIMT kernel's grid, so no kernel fits
    assert fwd(1, 1 << 16, 1, 1 << 15, 128, 8, ra.RA_KERNEL_AUTO) == ra.RA_ERR_UNSUPPORTED
    # N = 65536 ring devices: past the SIMT kernel's grid
    assert fwd(1, 1, 1, 1 << 16, 128, 1 << 16, ra.RA_KERNEL_SIMT) == ra.RA_ERR_UNSUPPORTED
    # D = 256 is SIMT-only; the tensor-core kernel refuses it
    assert fwd(1, 2, 1, 256, 256, 2, ra.RA_KERNEL_TC) == ra.RA_ERR_UNSUPPORTED
    bwd = lambda B, Hq, Hkv, S, D, N, kernel: ra.ra_backward_ex(
        *([p] * 10), 1 << 40, B, Hq, Hkv, S, D, N, 1, 1, 0.0, ra.RA_BF16, kernel, None)
    assert bwd(1, 1 << 14, 1, 1 << 17, 128, 16, ra.RA_KERNEL_TC) == ra.RA_ERR_UNSUPPORTED
    assert bwd(1, 1 << 16, 1, 1 << 15, 128, 8, ra.RA_KERNEL_AUTO) == ra.RA_ERR_UNSUPPORTED
    assert bwd(1, 2, 1, 256, 32, 2, ra.RA_KERNEL_TC) == ra.RA_ERR_UNSUPPORTED  # D = 32


def test_ring_step_host_validation(lib):
    """ra_ring_step refuses bad arguments on the host, before any CUDA call."""
    p = ctypes.c_void_p(16 * 1024)  # never dereferenced: validation fails first
    odd = ctypes.c_void_p(16 * 1024 + 8)

    def call(q=p, st_o=p, st_l=p, out=p, lse=p, B=1, Hq=2, Hkv=1, Sb=256, D=128, N=4, i=1,
             j=0, layout=1, flags=0):
        return ra.ra_ring_step(q, p, p, st_o, st_l, out, lse, B, Hq, Hkv, Sb, D, N, i, j, 1,
                               layout, 0.0, flags, None)

    F, L = ra.RA_STEP_FIRST, ra.RA_STEP_LAST
    assert call(i=4) == ra.RA_ERR_INVALID_ARG            # shard outside the ring
    assert call(j=-1) == ra.RA_ERR_INVALID_ARG
    assert call(Hq=3, Hkv=2) == ra.RA_ERR_INVALID_ARG    # Hq % Hkv
    assert call(flags=4) == ra.RA_ERR_INVALID_ARG        # unknown flag
    assert call(layout=3) == ra.RA_ERR_INVALID_ARG
    assert call(layout=2, Sb=255) == ra.RA_ERR_INVALID_ARG
    assert call(q=None) == ra.RA_ERR_INVALID_ARG
    assert call(st_o=None) == ra.RA_ERR_INVALID_ARG      # the state is read and written
    assert call(st_l=None, flags=F) == ra.RA_ERR_INVALID_ARG
    assert call(out=None, flags=L) == ra.RA_ERR_INVALID_ARG
    assert call(st_o=odd) == ra.RA_ERR_ALIGN
    assert call(lse=odd, flags=L) == ra.RA_ERR_ALIGN
    assert call(D=96) == ra.RA_ERR_UNSUPPORTED           # tensor-core head dimensions only
    assert call(layout=2, Sb=384) == ra.RA_ERR_UNSUPPORTED  # zigzag chunks must be whole tiles
    assert call(B=0) == ra.RA_OK                         # empty: nothing to do
    assert call(Sb=0, q=None) == ra.RA_OK


def test_ring_step_backward_host_validation(lib):
    """ra_ring_step_backward refuses bad arguments on the host, before any
    CUDA call."""
    p = ctypes.c_void_p(16 * 1024)  # never dereferenced: validation fails first
    odd = ctypes.c_void_p(16 * 1024 + 8)

    def call(q=p, out=p, lse=p, dout=p, delta=p, dqs=p, dks=p, dvs=p, dq=p, dk=p, dv=p, B=1,
             Hq=2, Hkv=1, Sb=256, D=128, N=4, i=1, j=0, layout=1, flags=0):
        return ra.ra_ring_step_backward(q, p, p, out, lse, dout, delta, dqs, dks, dvs, dq, dk,
                                        dv, B, Hq, Hkv, Sb, D, N, i, j, 1, layout, 0.0, flags,
                                        None)

    F, L = ra.RA_STEP_FIRST, ra.RA_STEP_LAST
    assert call(i=4) == ra.RA_ERR_INVALID_ARG            # shard outside the ring
    assert call(j=-1) == ra.RA_ERR_INVALID_ARG
    assert call(Hq=3, Hkv=2) == ra.RA_ERR_INVALID_ARG    # Hq % Hkv
    assert call(flags=4) == ra.RA_ERR_INVALID_ARG        # unknown flag
    assert call(layout=3) == ra.RA_ERR_INVALID_ARG
    assert call(delta=None) == ra.RA_ERR_INVALID_ARG     # delta is always needed
    assert call(out=None, flags=F) == ra.RA_ERR_INVALID_ARG  # the first step forms delta
    assert call(dks=None) == ra.RA_ERR_INVALID_ARG       # the block's state is read and written
    assert call(dq=None, flags=L) == ra.RA_ERR_INVALID_ARG
    assert call(dqs=odd) == ra.RA_ERR_ALIGN
    assert call(D=96) == ra.RA_ERR_UNSUPPORTED           # tensor-core head dimensions only
    assert call(layout=2, Sb=384) == ra.RA_ERR_UNSUPPORTED
    assert call(B=0) == ra.RA_OK                         # empty: nothing to do
    # out, the states and the outputs may be NULL where the flags do not use them
    assert call(out=None, dq=None, dk=None, dv=None, D=96) == ra.RA_ERR_UNSUPPORTED
    assert call(dqs=None, dks=None, dvs=None, flags=F | L, D=96) == ra.RA_ERR_UNSUPPORTED

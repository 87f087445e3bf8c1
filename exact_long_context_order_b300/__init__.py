"""Ring attention (exact blockwise self-attention over N virtual ring devices)
on one B300, as a C-ABI shared library with a thin ctypes binding.

The functions named ``ra_*`` mirror ``include/ra.h`` one to one: plain
integers and pointers in, an RA_* status out; they only marshal arguments.
``forward``, ``backward``, ``merge``, ``stripe`` and ``plan`` are conveniences over them
for torch CUDA tensors (PyTorch is used only for device memory and streams);
every step of the computation runs in the library's CUDA kernels.

If ``libra.so`` has not been built, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libra.so")

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_ALIGN = 0, 1, 2, 3
RA_ERR_CUDA, RA_ERR_TIMEOUT, RA_ERR_BOUNDS, RA_ERR_CAPACITY = 4, 5, 6, 7
RA_BF16, RA_F32 = 0, 1
RA_KERNEL_AUTO, RA_KERNEL_TC, RA_KERNEL_SIMT = 0, 1, 2
RA_FOLD_FULL, RA_FOLD_INCL, RA_FOLD_STRICT = 0, 1, 2
RA_LAYOUT_CONTIGUOUS, RA_LAYOUT_STRIPED, RA_LAYOUT_ZIGZAG = 0, 1, 2
RA_STEP_FIRST, RA_STEP_LAST = 1, 2

_c = ctypes
_vp, _i32, _i64, _f32 = _c.c_void_p, _c.c_int, _c.c_int64, _c.c_float
_SIGNATURES = {
    "ra_forward": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _i32, _i32, _i32,
                    _f32, _i32, _vp], _i32),
    "ra_forward_ex": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _i32, _i32, _i32,
                       _f32, _i32, _i32, _vp], _i32),
    "ra_forward_host": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                         _i64, _i32, _i32, _i32, _i32, _f32, _i32, _vp], _i32),
    "ra_merge": ([_vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp], _i32),
    "ra_ring_step": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _i32,
                      _i32, _i32, _i32, _i32, _f32, _i32, _vp], _i32),
    "ra_ring_step_backward": ([_vp] * 13 + [_i32, _i32, _i32, _i64, _i32, _i32, _i32, _i32,
                                           _i32, _i32, _f32, _i32, _vp], _i32),
    "ra_stripe": ([_vp, _vp, _i64, _i64, _i32, _i64, _i32, _vp], _i32),
    "ra_relayout": ([_vp, _vp, _i64, _i64, _i32, _i64, _i32, _i32, _vp], _i32),
    "ra_ulysses_exchange": ([_vp, _vp, _i32, _i32, _i64, _i32, _i64, _i32, _vp], _i32),
    "ra_plan": ([_i64, _i32, _i32, _i32, _i32, _vp, _i64, _c.POINTER(_i64)], _i32),
    "ra_plan_tile": ([_i64, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _i64, _c.POINTER(_i64)],
                     _i32),
    "ra_plan_backward": ([_i64, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _i64, _c.POINTER(_i64)],
                         _i32),
    "ra_fold_log": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _i32, _i32, _i32,
                     _f32, _vp, _vp, _i32, _vp], _i32),
    "ra_forward_noalloc": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                            _i32, _f32, _vp], _i32),
    "ra_watchdog_selftest": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                              _i32, _f32, _i64, _vp], _i32),
    "ra_backward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
                     _i64, _i32, _i32, _i32, _i32, _f32, _i32, _vp], _i32),
    "ra_backward_ex": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32,
                        _i32, _i64, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp], _i32),
    "ra_backward_workspace": ([_i32, _i32, _i64, _i32, _c.POINTER(_i64)], _i32),
    "ra_watchdog_selftest_backward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                       _i32, _i32, _i32, _i64, _i32, _i32, _i32, _i32, _f32,
                                       _i64, _i32, _vp], _i32),
    "ra_check": ([_vp], _i32),
    "ra_strerror": ([_i32], _c.c_char_p),
    "ra_tile_config": ([_c.POINTER(_i32), _c.POINTER(_i32)], _i32),
    "ra_version": ([], _i32),
}

_lib = None


class RAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ra_strerror(code)} (status {code})")


def lib():
    """The loaded libra.so (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m exact_long_context_order_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


# ------------------------------------------------------------ raw C ABI
def ra_forward(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale, dtype, stream):
    return lib().ra_forward(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale,
                            dtype, stream)


def ra_forward_ex(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale, dtype, kernel,
                  stream):
    return lib().ra_forward_ex(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale,
                               dtype, kernel, stream)


def ra_forward_host(q_h, k_h, v_h, out_h, lse_h, q_d, k_d, v_d, out_d, lse_d, B, Hq, Hkv, S, D,
                    N, causal, striped, scale, dtype, stream):
    """ra_forward on host buffers: H2D copies, the forward and D2H copies, all
    enqueued on `stream` (host pointers, device staging pointers)."""
    return lib().ra_forward_host(q_h, k_h, v_h, out_h, lse_h, q_d, k_d, v_d, out_d, lse_d, B, Hq,
                                 Hkv, S, D, N, causal, striped, scale, dtype, stream)


def ra_merge(out_a, lse_a, out_b, lse_b, rows, D, dtype, stream):
    return lib().ra_merge(out_a, lse_a, out_b, lse_b, rows, D, dtype, stream)


def ra_ring_step(q, k, v, state_o, state_lse, out, lse, B, Hq, Hkv, Sb, D, N, i, j, causal,
                 layout, scale, flags, stream):
    return lib().ra_ring_step(q, k, v, state_o, state_lse, out, lse, B, Hq, Hkv, Sb, D, N, i, j,
                              causal, layout, scale, flags, stream)


def ra_ring_step_backward(q, k, v, out, lse, dout, delta, dq_state, dk_state, dv_state, dq, dk,
                          dv, B, Hq, Hkv, Sb, D, N, i, j, causal, layout, scale, flags, stream):
    return lib().ra_ring_step_backward(q, k, v, out, lse, dout, delta, dq_state, dk_state,
                                       dv_state, dq, dk, dv, B, Hq, Hkv, Sb, D, N, i, j, causal,
                                       layout, scale, flags, stream)


def ra_stripe(src, dst, BH, S, N, row_bytes, inverse, stream):
    return lib().ra_stripe(src, dst, BH, S, N, row_bytes, inverse, stream)


def ra_relayout(src, dst, BH, S, N, row_bytes, layout, inverse, stream):
    return lib().ra_relayout(src, dst, BH, S, N, row_bytes, layout, inverse, stream)


def ra_ulysses_exchange(src, dst, B, H, S, N, row_bytes, inverse, stream):
    return lib().ra_ulysses_exchange(src, dst, B, H, S, N, row_bytes, inverse, stream)


def ra_plan(S, N, causal, striped, tile, items, cap, n_items):
    return lib().ra_plan(S, N, causal, striped, tile, items, cap, n_items)


def ra_plan_tile(S, N, causal, striped, tile, i, qt, items, cap, n_items):
    return lib().ra_plan_tile(S, N, causal, striped, tile, i, qt, items, cap, n_items)


def ra_plan_backward(S, N, causal, striped, tile, j, kt, items, cap, n_items):
    return lib().ra_plan_backward(S, N, causal, striped, tile, j, kt, items, cap, n_items)


def ra_fold_log(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale, log, counts,
                max_entries, stream):
    return lib().ra_fold_log(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale, log,
                             counts, max_entries, stream)


def ra_forward_noalloc(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale, stream):
    """ra_forward for callers that must not allocate device memory (bf16,
    tensor-core shapes only; scratch in a static device array shared by all
    calls, so calls that overlap on the GPU race)."""
    return lib().ra_forward_noalloc(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped,
                                    scale, stream)


def ra_watchdog_selftest(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale,
                         timeout_cycles, stream):
    return lib().ra_watchdog_selftest(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped,
                                      scale, timeout_cycles, stream)


def ra_backward(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, S,
                D, N, causal, striped, scale, dtype, stream):
    return lib().ra_backward(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B,
                             Hq, Hkv, S, D, N, causal, striped, scale, dtype, stream)


def ra_backward_ex(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv,
                   S, D, N, causal, striped, scale, dtype, kernel, stream):
    return lib().ra_backward_ex(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes,
                                B, Hq, Hkv, S, D, N, causal, striped, scale, dtype, kernel, stream)


def ra_backward_workspace(B, Hq, S, D):
    """Returns (status, bytes)."""
    n = _i64()
    rc = lib().ra_backward_workspace(B, Hq, S, D, ctypes.byref(n))
    return rc, n.value


def ra_watchdog_selftest_backward(q, k, v, out, lse, dout, dq, dk, dv, workspace,
                                  workspace_bytes, B, Hq, Hkv, S, D, N, causal, striped, scale,
                                  timeout_cycles, which, stream):
    return lib().ra_watchdog_selftest_backward(q, k, v, out, lse, dout, dq, dk, dv, workspace,
                                               workspace_bytes, B, Hq, Hkv, S, D, N, causal,
                                               striped, scale, timeout_cycles, which, stream)


def ra_check(stream):
    return lib().ra_check(stream)


def ra_strerror(code: int) -> str:
    return lib().ra_strerror(code).decode()


def ra_tile_config():
    tq, tk = _i32(), _i32()
    lib().ra_tile_config(ctypes.byref(tq), ctypes.byref(tk))
    return tq.value, tk.value


def ra_version() -> int:
    return lib().ra_version()


# ------------------------------------------------------------ torch helpers
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != RA_OK:
        raise RAError(rc, where)


_KERNELS = {"auto": RA_KERNEL_AUTO, "tc": RA_KERNEL_TC, "simt": RA_KERNEL_SIMT}


def forward(q, k, v, N: int, causal: bool = False, striped: bool = False, scale=None, out=None,
            lse=None, want_lse: bool = True, kernel: str = "auto", stream=None):
    """Ring attention over shard-major torch CUDA tensors.

    q [B, Hq, S, D], k and v [B, Hkv, S, D], all bf16 or all float32,
    contiguous, on the current device.  ``striped`` is the layout: False/0
    contiguous, True/1 striped, 2 zigzag.  Returns (out, lse): out like q, lse
    [B, Hq, S] float32 (None when want_lse is False and lse is None).
    """
    import torch
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    if q.dtype == torch.bfloat16:
        dtype = RA_BF16
    elif q.dtype == torch.float32:
        dtype = RA_F32
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    for t in (k, v):
        if t.dtype != q.dtype or t.shape != (B, Hkv, S, D) or not t.is_contiguous():
            raise ValueError("k and v must be contiguous [B, Hkv, S, D] of q's dtype")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    rc = ra_forward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D, N,
                       int(causal), int(striped), float(scale or 0.0), dtype, _KERNELS[kernel],
                       _stream_handle(stream))
    _check(rc, "ra_forward")
    return out, lse


def ring_step(q, k, v, N: int, i: int, j: int, state_o=None, state_lse=None, out=None, lse=None,
              first: bool = False, last: bool = False, causal: bool = False, layout=0,
              scale=None, stream=None):
    """One ring step over torch CUDA tensors: query shard i (q [B, Hq, Sb, D]
    bf16) folds key/value block j (k, v [B, Hkv, Sb, D]) into its running
    state (state_o float32 like q, state_lse float32 [B, Hq, Sb]).  With
    ``last`` the result goes to out (bf16, allocated when None) and lse
    instead.  Returns (state_o, state_lse, out, lse)."""
    import torch
    B, Hq, Sb, D = q.shape
    Hkv = k.shape[1]
    if q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("ring_step takes bf16 q, k, v")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k and v must be contiguous")
    if k.shape != (B, Hkv, Sb, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Sb, D] with q's Sb and D")
    if not (first and last):
        if state_o is None:
            state_o = torch.empty((B, Hq, Sb, D), dtype=torch.float32, device=q.device)
        if state_lse is None:
            state_lse = torch.empty((B, Hq, Sb), dtype=torch.float32, device=q.device)
    if last:
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, Hq, Sb), dtype=torch.float32, device=q.device)
    flags = (RA_STEP_FIRST if first else 0) | (RA_STEP_LAST if last else 0)
    rc = ra_ring_step(_ptr(q), _ptr(k), _ptr(v), _ptr(state_o), _ptr(state_lse), _ptr(out),
                      _ptr(lse), B, Hq, Hkv, Sb, D, N, i, j, int(causal), int(layout),
                      float(scale or 0.0), flags, _stream_handle(stream))
    _check(rc, "ra_ring_step")
    return state_o, state_lse, out, lse


def ring_step_backward(q, k, v, out, lse, dout, N: int, i: int, j: int, delta=None,
                       dq_state=None, dk_state=None, dv_state=None, first: bool = False,
                       last: bool = False, causal: bool = False, layout=0, scale=None,
                       stream=None):
    """One backward ring step over torch CUDA tensors (ra_ring_step_backward):
    query shard i (q, out, dout [B, Hq, Sb, D] bf16, lse float32) against
    block j (k, v [B, Hkv, Sb, D]).  delta (float32 [B, Hq, Sb]) is computed
    on the first step and must be passed back on the later ones, as must the
    shard's dq_state and the block's dk_state / dv_state (float32, allocated
    when None).  Returns (delta, dq_state, dk_state, dv_state, dq, dk, dv);
    dq, dk, dv (bf16) are set on the last step only."""
    import torch
    B, Hq, Sb, D = q.shape
    Hkv = k.shape[1]
    for t in (q, k, v, out, dout):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k, v, out and dout must be contiguous bf16")
    if k.shape != (B, Hkv, Sb, D) or v.shape != k.shape or dout.shape != q.shape:
        raise ValueError("k and v must be [B, Hkv, Sb, D], dout like q")
    f32 = dict(dtype=torch.float32, device=q.device)
    if delta is None:
        delta = torch.empty((B, Hq, Sb), **f32)
    if not (first and last):
        dq_state = torch.empty((B, Hq, Sb, D), **f32) if dq_state is None else dq_state
        dk_state = torch.empty((B, Hkv, Sb, D), **f32) if dk_state is None else dk_state
        dv_state = torch.empty((B, Hkv, Sb, D), **f32) if dv_state is None else dv_state
    dq = dk = dv = None
    if last:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flags = (RA_STEP_FIRST if first else 0) | (RA_STEP_LAST if last else 0)
    rc = ra_ring_step_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                               _ptr(delta), _ptr(dq_state), _ptr(dk_state), _ptr(dv_state),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sb, D, N, i, j,
                               int(causal), int(layout), float(scale or 0.0), flags,
                               _stream_handle(stream))
    _check(rc, "ra_ring_step_backward")
    return delta, dq_state, dk_state, dv_state, dq, dk, dv


def backward(q, k, v, out, lse, dout, N: int, causal: bool = False, striped: bool = False,
             scale=None, kernel: str = "auto", workspace=None, stream=None, dq=None, dk=None,
             dv=None):
    """Gradients (dq, dk, dv) of ``forward`` over shard-major torch CUDA tensors.

    q, k, v, out and lse are the forward's inputs and outputs, dout = dL/dout
    (like out).  The workspace (a uint8 CUDA tensor of at least
    ra_backward_workspace bytes) is allocated here when not given, and so are
    dq (like q), dk and dv (like k) when not given (contiguous, q's dtype).
    """
    import torch
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    dtype = {torch.bfloat16: RA_BF16, torch.float32: RA_F32}.get(q.dtype)
    if dtype is None:
        raise TypeError(f"unsupported dtype {q.dtype}")
    for t in (k, v):
        if t.dtype != q.dtype or t.shape != (B, Hkv, S, D) or not t.is_contiguous():
            raise ValueError("k and v must be contiguous [B, Hkv, S, D] of q's dtype")
    for t in (q, out, dout):
        if t.dtype != q.dtype or t.shape != (B, Hq, S, D) or not t.is_contiguous():
            raise ValueError("q, out and dout must be contiguous [B, Hq, S, D] of one dtype")
    if lse is None or lse.dtype != torch.float32 or lse.shape != (B, Hq, S):
        raise ValueError("lse must be the forward's float32 [B, Hq, S]")
    rc, need = ra_backward_workspace(B, Hq, S, D)
    _check(rc, "ra_backward_workspace")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, like in ((dq, q), (dk, k), (dv, v)):
        if t.dtype != q.dtype or t.shape != like.shape or not t.is_contiguous():
            raise ValueError("dq must be like q, dk and dv like k (contiguous, q's dtype)")
    rc = ra_backward_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                        _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, Hq, Hkv, S, D,
                        N, int(causal), int(striped), float(scale or 0.0), dtype,
                        _KERNELS[kernel], _stream_handle(stream))
    _check(rc, "ra_backward")
    return dq, dk, dv


def fold_log(q, k, v, N: int, causal: bool, striped: bool, scale=None, stream=None):
    """Runs the logging variant of the tensor-core kernel.

    Returns (out, lse, log, counts): log is int32 [tiles, N*Sb/128, 4] with
    (s, j, kt, kind) per live fold of each query tile, tiles indexed
    ((b*Hq + h)*N + i)*(Sb/128) + qt; counts int32 [tiles].
    """
    import torch
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    nt = (S // N + 127) // 128  # a shard's last tile may be partial
    tiles = B * Hq * N * nt
    max_entries = N * nt
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    log = torch.full((tiles, max_entries, 4), -1, dtype=torch.int32, device=q.device)
    counts = torch.full((tiles,), -1, dtype=torch.int32, device=q.device)
    rc = ra_fold_log(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D, N,
                     int(causal), int(striped), float(scale or 0.0), _ptr(log), _ptr(counts),
                     max_entries, _stream_handle(stream))
    _check(rc, "ra_fold_log")
    return out, lse, log, counts


def merge(out_a, lse_a, out_b, lse_b, stream=None):
    """In place: (out_a, lse_a) <- merge of the two partials (torch CUDA tensors)."""
    import torch
    D = out_a.shape[-1]
    rows = out_a.numel() // D
    dtype = RA_BF16 if out_a.dtype == torch.bfloat16 else RA_F32
    rc = ra_merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), rows, D, dtype,
                  _stream_handle(stream))
    _check(rc, "ra_merge")
    return out_a, lse_a


def stripe(x, N: int, inverse: bool = False, out=None, stream=None):
    """Token order <-> striped shard-major order along dim -2 of [..., S, D]."""
    import torch
    S = x.shape[-2]
    row_bytes = x.shape[-1] * x.element_size()
    BH = x.numel() // (S * x.shape[-1])
    if out is None:
        out = torch.empty_like(x)
    rc = ra_stripe(_ptr(x), _ptr(out), BH, S, N, row_bytes, int(inverse), _stream_handle(stream))
    _check(rc, "ra_stripe")
    return out


def relayout(x, N: int, layout: int, inverse: bool = False, out=None, stream=None):
    """Token order <-> shard-major layout (RA_LAYOUT_*) along dim -2 of [..., S, D]."""
    import torch
    S = x.shape[-2]
    row_bytes = x.shape[-1] * x.element_size()
    BH = x.numel() // (S * x.shape[-1])
    if out is None:
        out = torch.empty_like(x)
    rc = ra_relayout(_ptr(x), _ptr(out), BH, S, N, row_bytes, int(layout), int(inverse),
                     _stream_handle(stream))
    _check(rc, "ra_relayout")
    return out


def ulysses_exchange(x, N: int, inverse: bool = False, out=None, stream=None):
    """Sequence-sharded [N, B, H, S/N, D] <-> head-sharded [N, B, H/N, S, D]."""
    import torch
    if not inverse:
        n, B, H, Sb, D = x.shape
        shape = (N, B, H // N, N * Sb, D)
        S = N * Sb
    else:
        n, B, Hl, S, D = x.shape
        shape = (N, B, Hl * N, S // N, D)
        H = Hl * N
    if out is None:
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    rc = ra_ulysses_exchange(_ptr(x), _ptr(out), B, H, S, N, D * x.element_size(), int(inverse),
                             _stream_handle(stream))
    _check(rc, "ra_ulysses_exchange")
    return out


def plan(S: int, N: int, causal: bool, striped: bool, i: int, qt: int, tile: int = 128):
    """Host-side fold list of query tile (i, qt): list of (s, j, kt, kind)."""
    n = _i64()
    _check(ra_plan_tile(S, N, int(causal), int(striped), tile, i, qt, None, 0, ctypes.byref(n)),
           "ra_plan_tile")
    buf = (ctypes.c_int32 * (4 * max(1, n.value)))()
    _check(ra_plan_tile(S, N, int(causal), int(striped), tile, i, qt, buf, n.value,
                        ctypes.byref(n)), "ra_plan_tile")
    return [tuple(buf[4 * e:4 * e + 4]) for e in range(n.value)]


def plan_schedule(S: int, N: int, causal: bool, striped, tile: int = 128):
    """The whole fold schedule: list of (i, qt, s, j, kt, kind) in order."""
    n = _i64()
    _check(ra_plan(S, N, int(causal), int(striped), tile, None, 0, ctypes.byref(n)), "ra_plan")
    buf = (ctypes.c_int32 * (6 * max(1, n.value)))()
    _check(ra_plan(S, N, int(causal), int(striped), tile, buf, n.value, ctypes.byref(n)),
           "ra_plan")
    return [tuple(buf[6 * e:6 * e + 6]) for e in range(n.value)]


def plan_backward(S: int, N: int, causal: bool, striped, j: int, kt: int, tile: int = 128):
    """The dk/dv visiting order of key tile kt of shard j as [(s, i, qt, kind)]."""
    n = _i64()
    _check(ra_plan_backward(S, N, int(causal), int(striped), tile, j, kt, None, 0,
                            ctypes.byref(n)), "ra_plan_backward")
    buf = (_i32 * (4 * max(n.value, 1)))()
    _check(ra_plan_backward(S, N, int(causal), int(striped), tile, j, kt, buf, n.value,
                            ctypes.byref(n)), "ra_plan_backward")
    return [tuple(buf[4 * e:4 * e + 4]) for e in range(n.value)]


def check(stream=None):
    """Synchronise and raise if a kernel recorded a device-side failure."""
    _check(ra_check(_stream_handle(stream)), "ra_check")


def attention(q, k, v, N: int, causal: bool = False, striped=False, scale=None):
    """Ring attention with autograd: ``forward`` in the forward pass and
    ``backward`` (dq, dk, dv from the saved q, k, v, out and lse) in the
    backward pass.  Tensors as for ``forward``; returns out (like q).  For
    training, the way the method is used (1M-token training on the pages)."""
    return _AttentionFn.apply(q, k, v, N, causal, striped, scale)


def _autograd_function():
    import torch

    class AttentionFn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, N, causal, striped, scale):
            q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
            out, lse = forward(q, k, v, N, causal=causal, striped=striped, scale=scale)
            ctx.save_for_backward(q, k, v, out, lse)
            ctx.cfg = (N, causal, striped, scale)
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            N, causal, striped, scale = ctx.cfg
            dq, dk, dv = backward(q, k, v, out, lse, dout.contiguous(), N, causal=causal,
                                  striped=striped, scale=scale)
            return dq, dk, dv, None, None, None, None

    return AttentionFn


class _LazyFn:
    """Builds the autograd Function on first use (importing the package does
    not import torch)."""
    fn = None

    @classmethod
    def apply(cls, *args):
        if cls.fn is None:
            cls.fn = _autograd_function()
        return cls.fn.apply(*args)


_AttentionFn = _LazyFn

"""Seeded synthetic inputs for the ring-attention workloads.

This package is the one piece shared by the CPU oracle side (tests, the CPU
baseline) and the GPU side (tests, bench, smoke).  It holds no attention
arithmetic: it maps (seed, tensor id, element index) to a standard-normal
sample with a counter-based generator (Philox-4x32-10 + Box-Muller, see
``ragen.c``), so any element subset of any tensor can be regenerated
independently.

Two implementations of the same definition live here:

* ``libragen.so`` (C, OpenMP) -- fast, used for real inputs;
* ``philox4x32_10_np`` / ``normal_f32_numpy`` -- a NumPy twin used only to
  check the C build bit for bit.

bf16 tensors are returned as raw ``uint16`` words (NumPy has no bfloat16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .workloads import WORKLOADS, Workload, TENSOR_Q, TENSOR_K, TENSOR_V, TENSOR_DO  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ragen.c")
_LIB_PATH = os.path.join(_HERE, "libragen.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libragen.so`` in place (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
             "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, u64, u32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32
        vp = ctypes.c_void_p
        lib.ragen_philox4x32_10.argtypes = [vp, vp]
        lib.ragen_philox4x32_10.restype = None
        lib.ragen_normal_f32.argtypes = [u64, u32, i64, i64, vp]
        lib.ragen_normal_f32.restype = None
        lib.ragen_normal_bf16.argtypes = [u64, u32, i64, i64, vp]
        lib.ragen_normal_bf16.restype = None
        lib.ragen_normal_bf16_rows.argtypes = [u64, u32, vp, i64, i64, vp]
        lib.ragen_normal_bf16_rows.restype = None
        _lib = lib
    return _lib


def philox4x32_10(ctr, key) -> np.ndarray:
    """One Philox-4x32-10 block (C build)."""
    c = np.array(ctr, dtype=np.uint32).copy()
    k = np.array(key, dtype=np.uint32).copy()
    _load().ragen_philox4x32_10(c.ctypes.data, k.ctypes.data)
    return c


def normal_f32(seed: int, tensor_id: int, n: int, start: int = 0, out=None) -> np.ndarray:
    """Elements [start, start+n) of tensor (seed, tensor_id) as float32."""
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _load().ragen_normal_f32(seed, tensor_id, start, n, out.ctypes.data)
    return out


def normal_bf16(seed: int, tensor_id: int, n: int, start: int = 0, out=None) -> np.ndarray:
    """Elements [start, start+n) of tensor (seed, tensor_id) as bf16 words (uint16).

    ``out`` may be any writable C-contiguous uint16 buffer of n elements, for
    example a NumPy view of pinned host memory.
    """
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    _load().ragen_normal_bf16(seed, tensor_id, start, n, out.ctypes.data)
    return out


def normal_bf16_rows(seed: int, tensor_id: int, rows, row_len: int) -> np.ndarray:
    """Rows ``rows`` (each ``row_len`` consecutive elements) of a bf16 tensor."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, row_len), dtype=np.uint16)
    _load().ragen_normal_bf16_rows(seed, tensor_id, rows.ctypes.data, rows.size,
                                   row_len, out.ctypes.data)
    return out


# ---------------------------------------------------------------- NumPy twin
_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = np.uint32(0x9E3779B9), np.uint32(0xBB67AE85)


def philox4x32_10_np(ctr: np.ndarray, key) -> np.ndarray:
    """Vectorised Philox-4x32-10: ctr is [n, 4] uint32, key is (k0, k1)."""
    c = np.array(ctr, dtype=np.uint32, copy=True).reshape(-1, 4)
    k0, k1 = np.uint32(key[0]), np.uint32(key[1])
    mask = np.uint64(0xFFFFFFFF)
    with np.errstate(over="ignore"):
        for _ in range(10):
            p0 = _M0 * c[:, 0].astype(np.uint64)
            p1 = _M1 * c[:, 2].astype(np.uint64)
            hi0 = (p0 >> np.uint64(32)).astype(np.uint32)
            lo0 = (p0 & mask).astype(np.uint32)
            hi1 = (p1 >> np.uint64(32)).astype(np.uint32)
            lo1 = (p1 & mask).astype(np.uint32)
            n0 = hi1 ^ c[:, 1] ^ k0
            n2 = hi0 ^ c[:, 3] ^ k1
            c = np.stack([n0, lo1, n2, lo0], axis=1)
            k0 = np.uint32((int(k0) + int(_W0)) & 0xFFFFFFFF)
            k1 = np.uint32((int(k1) + int(_W1)) & 0xFFFFFFFF)
    return c


def normal_f32_numpy(seed: int, tensor_id: int, n: int, start: int = 0) -> np.ndarray:
    """NumPy twin of ``normal_f32`` (same definition, independent code)."""
    b0, b1 = start // 4, (start + n - 1) // 4
    blk = np.arange(b0, b1 + 1, dtype=np.uint64)
    ctr = np.zeros((blk.size, 4), dtype=np.uint32)
    ctr[:, 0] = (blk & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    ctr[:, 1] = (blk >> np.uint64(32)).astype(np.uint32)
    w = philox4x32_10_np(ctr, (seed & 0xFFFFFFFF, tensor_id))
    u1 = (w[:, 0::2].astype(np.float64) + 1.0) / 4294967296.0
    u2 = w[:, 1::2].astype(np.float64) / 4294967296.0
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * np.pi * u2
    z = np.empty((blk.size, 4), dtype=np.float64)
    z[:, 0::2] = r * np.cos(th)
    z[:, 1::2] = r * np.sin(th)
    z = z.astype(np.float32).reshape(-1)
    off = start - b0 * 4
    return z[off:off + n]


def f32_to_bf16_bits_numpy(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest even), returned as uint16 words."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)

"""Seeded synthetic inputs for the MaxSim operator (input preparation only).

Thin ctypes wrapper over ``gen.c``. Nothing here computes any part of the
operator: it only draws token embeddings, lengths, masks, INT8 quantised
embeddings and upstream gradients, so the CUDA path and the CPU oracle can be
fed identical bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libmaxsim_datagen.so")
_lock = threading.Lock()
_lib = None

# tensor ids: each tensor of a workload draws from its own family of streams
TID_Q, TID_D, TID_LEN_D, TID_QMASK, TID_DMASK, TID_GRAD, TID_LEN_Q = 1, 2, 3, 4, 5, 6, 7
TID_PAIR_D = 8  # document index of each (query, document) pair
TID_CLOUD_P, TID_CLOUD_Q, TID_CLOUD_GRAD = 9, 10, 11  # Chamfer point clouds and upstream gradient

DTYPE_CODES = {"f16": 0, "bf16": 1, "f64": 2, "f32": 3}


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, i32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.dg_gaussian_rows.argtypes = [u64, u64, i64, i64, i64, ctypes.c_int, ctypes.c_int, vp]
            lib.dg_int8_rows.argtypes = [u64, u64, i64, i64, i64, vp, vp]
            lib.dg_uniform_int.argtypes = [u64, u64, i64, i32, i32, vp]
            lib.dg_normal_f32.argtypes = [u64, u64, i64, vp]
            lib.dg_mask_drop_tail.argtypes = [u64, u64, i64, i64, i32, vp]
            lib.dg_mask_random_subset.argtypes = [u64, u64, i64, i64, i32, vp]
            for f in (lib.dg_gaussian_rows, lib.dg_int8_rows, lib.dg_uniform_int, lib.dg_normal_f32,
                      lib.dg_mask_drop_tail, lib.dg_mask_random_subset):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def gaussian_rows(seed: int, tensor_id: int, nrows: int, dim: int, dtype: str = "f16",
                  row0: int = 0, normalize: bool = True, out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+nrows) of a seeded Gaussian [*, dim] tensor.

    f16 / bf16 come back as raw uint16 bit patterns; f64 / f32 as floats.
    Row r always holds the same values whatever subset is generated.
    """
    np_dtype = {"f16": np.uint16, "bf16": np.uint16, "f64": np.float64, "f32": np.float32}[dtype]
    if out is None:
        out = np.empty((nrows, dim), dtype=np_dtype)
    assert out.dtype == np_dtype and out.size == nrows * dim
    rc = _load().dg_gaussian_rows(seed, tensor_id, row0, nrows, dim, int(normalize), DTYPE_CODES[dtype], _ptr(out))
    if rc:
        raise ValueError("dg_gaussian_rows rejected its arguments")
    return out


def int8_rows(seed: int, tensor_id: int, nrows: int, dim: int, row0: int = 0):
    """Per-token symmetric INT8 quantisation of l2-normalised Gaussian rows.

    Returns (q int8 [nrows, dim], scale float32 [nrows]).
    """
    q = np.empty((nrows, dim), dtype=np.int8)
    s = np.empty((nrows,), dtype=np.float32)
    if _load().dg_int8_rows(seed, tensor_id, row0, nrows, dim, _ptr(q), _ptr(s)):
        raise ValueError("dg_int8_rows rejected its arguments")
    return q, s


def uniform_int(seed: int, tensor_id: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.int32)
    if _load().dg_uniform_int(seed, tensor_id, n, lo, hi, _ptr(out)):
        raise ValueError("dg_uniform_int rejected its arguments")
    return out


def normal_f32(seed: int, tensor_id: int, n: int) -> np.ndarray:
    out = np.empty((n,), dtype=np.float32)
    if _load().dg_normal_f32(seed, tensor_id, n, _ptr(out)):
        raise ValueError("dg_normal_f32 rejected its arguments")
    return out


def mask_drop_tail(seed: int, tensor_id: int, n: int, L: int, kmax: int) -> np.ndarray:
    out = np.empty((n, L), dtype=np.uint8)
    if _load().dg_mask_drop_tail(seed, tensor_id, n, L, kmax, _ptr(out)):
        raise ValueError("dg_mask_drop_tail rejected its arguments")
    return out


def mask_random_subset(seed: int, tensor_id: int, n: int, L: int, kmax: int) -> np.ndarray:
    out = np.empty((n, L), dtype=np.uint8)
    if _load().dg_mask_random_subset(seed, tensor_id, n, L, kmax, _ptr(out)):
        raise ValueError("dg_mask_random_subset rejected its arguments")
    return out


def f16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """binary16 bit patterns -> float64 via numpy's own half type."""
    return bits.view(np.float16).astype(np.float64)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (bf16 is the top half of binary32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bits_to_float(bits: np.ndarray, dtype: str) -> np.ndarray:
    return f16_bits_to_float(bits) if dtype == "f16" else bf16_bits_to_float(bits)


def float_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exactly representable values -> storage bits (used for hand-built inputs)."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f16":
        h = x.astype(np.float16)
        assert np.array_equal(h.astype(np.float64), x), "value not exact in binary16"
        return h.view(np.uint16)
    f = x.astype(np.float32)
    b = f.view(np.uint32)
    assert np.array_equal(((b >> 16) << 16).view(np.float32).astype(np.float64), x), "value not exact in bfloat16"
    return (b >> 16).astype(np.uint16)

"""CPU fp64 oracle for attention over a paged KV cache (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It loads ``liboracle.so`` built from
``pa_oracle.c`` (plain C, fp64, OpenMP) and shares no code with the CUDA
library.  ``brute`` holds an independent NumPy restatement on contiguous K/V
used to pin the oracle.

Arrays cross the boundary as NumPy: bf16 tensors as their uint16 bit patterns,
FP8 (e4m3) pools as their uint8 codes, integer metadata as int32, results as
float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def load(path: Optional[str] = None):
    """Load (building first if missing or stale) and declare the C entry points."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        if _needs_build():
            build()
        path = _LIB_PATH
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_kv_block_bytes.restype = ctypes.c_size_t
    lib.oracle_kv_block_bytes.argtypes = [i, i, i, i]
    lib.oracle_cache_write.restype = i
    lib.oracle_cache_write.argtypes = [P, i, i, i, i, P, P, P, i]
    lib.oracle_gather.restype = i
    lib.oracle_gather.argtypes = [P, P, P, i, i, i, i, P, i]
    lib.oracle_attention.restype = i
    lib.oracle_attention.argtypes = [P, P, P, i, P, i, i, i, i, i, P, i, P, ctypes.c_double,
                                     P, i, i]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
    lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.oracle_cache_write_fp8.restype = i
    lib.oracle_cache_write_fp8.argtypes = [P, i, i, i, i, P, P, P, i, ctypes.c_float,
                                           ctypes.c_float]
    lib.oracle_attention_fp8.restype = i
    lib.oracle_attention_fp8.argtypes = [P, P, P, i, P, ctypes.c_double, ctypes.c_double, i, i,
                                         i, i, i, P, i, P, ctypes.c_double, P, i, i]
    lib.oracle_max_threads.restype = i
    lib.oracle_max_threads.argtypes = []
    if path == _LIB_PATH:
        _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """bf16 torch tensor (any device) or uint16 array -> contiguous uint16 array."""
    if hasattr(a, "dtype") and not isinstance(a, np.ndarray):
        import torch
        t = a.detach().to("cpu").contiguous()
        assert t.dtype == torch.bfloat16, t.dtype
        return t.view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16
    return a


def _u8(a) -> np.ndarray:
    """uint8 torch tensor (any device) or uint8 array -> contiguous uint8 array."""
    if hasattr(a, "dtype") and not isinstance(a, np.ndarray):
        t = a.detach().to("cpu").contiguous()
        return t.numpy().view(np.uint8)
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8
    return a


def _i32(a) -> np.ndarray:
    if hasattr(a, "dtype") and not isinstance(a, np.ndarray):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def kv_block_bytes(block_size: int, num_kv_heads: int, head_size: int,
                   dtype_bytes: int = 2, lib=None) -> int:
    """Bytes in one KV block: 2 * block_size * num_kv_heads * head_size * dtype_bytes."""
    return int((lib or load()).oracle_kv_block_bytes(block_size, num_kv_heads, head_size,
                                                     dtype_bytes))


def cache_write(kv_cache, k_new, v_new, slot_mapping, lib=None, inplace: bool = False) -> np.ndarray:
    """Return the pool (uint16 bits) with the new rows written.

    By default the input is copied first; with ``inplace=True`` ``kv_cache`` must
    already be a contiguous uint16 array and is written directly.
    """
    if inplace:
        assert isinstance(kv_cache, np.ndarray) and kv_cache.dtype == np.uint16
        assert kv_cache.flags["C_CONTIGUOUS"]
        pool = kv_cache
    else:
        pool = _u16(kv_cache).copy()
    NB, two, Hkv, bs, D = pool.shape
    assert two == 2
    kn, vn, sm = _u16(k_new), _u16(v_new), _i32(slot_mapping)
    N = sm.shape[0]
    assert kn.shape == (N, Hkv, D) and vn.shape == (N, Hkv, D)
    rc = (lib or load()).oracle_cache_write(_ptr(pool), NB, bs, Hkv, D, _ptr(kn), _ptr(vn),
                                            _ptr(sm), N)
    if rc != 0:
        raise ValueError("oracle_cache_write: slot outside the pool")
    return pool


def gather(kv_cache, block_table_row, length: int, lib=None):
    """K, V of one sequence in logical order, float64 [length, Hkv, D]."""
    pool = _u16(kv_cache)
    NB, _, Hkv, bs, D = pool.shape
    row = _i32(block_table_row)
    K = np.empty((max(length, 0), Hkv, D), dtype=np.float64)
    V = np.empty_like(K)
    rc = (lib or load()).oracle_gather(_ptr(K), _ptr(V), _ptr(pool), NB, bs, Hkv, D,
                                       _ptr(row), length)
    if rc != 0:
        raise ValueError("oracle_gather: block id outside the pool")
    return K, V


def attention(q, cu_q_lens, kv_cache, block_tables, seq_lens, num_heads: int, scale: float,
              rows=None, threads: int = 0, lib=None) -> np.ndarray:
    """fp64 attention of every (or the listed) query row; see ``oracle_attention``.

    Returns float64 [n_rows, num_heads, head_size].
    """
    pool = _u16(kv_cache)
    NB, _, Hkv, bs, D = pool.shape
    qq = _u16(q)
    cu = _i32(cu_q_lens)
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    B = sl.shape[0]
    assert cu.shape[0] == B + 1
    assert qq.shape[1:] == (num_heads, D), (qq.shape, num_heads, D)
    if bt.ndim == 1:
        bt = bt.reshape(B, -1)
    MB = bt.shape[1] if bt.size else 1
    if bt.size == 0:
        bt = np.full((B, 1), -1, dtype=np.int32)
    if rows is None:
        n = int(cu[-1])
        rows_arr = None
    else:
        rows_arr = _i32(rows)
        n = rows_arr.shape[0]
    out = np.zeros((n, num_heads, D), dtype=np.float64)
    rc = (lib or load()).oracle_attention(
        _ptr(out), _ptr(qq), _ptr(cu), B, _ptr(pool), NB, bs, num_heads, Hkv, D, _ptr(bt), MB,
        _ptr(sl), float(scale), _ptr(rows_arr) if rows_arr is not None else None,
        n if rows_arr is not None else 0, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention failed ({rc})")
    return out


def e4m3_to_double(code: int, lib=None) -> float:
    """Value of one OCP FP8 E4M3 code (NaN for the NaN codes)."""
    return float((lib or load()).oracle_e4m3_to_double(int(code)))


def e4m3_from_float(x: float, lib=None) -> int:
    """Nearest e4m3 code to the binary32 value x (ties to even, saturating at 448)."""
    return int((lib or load()).oracle_e4m3_from_float(float(np.float32(x))))


def cache_write_fp8(kv_cache, k_new, v_new, slot_mapping, k_scale: float, v_scale: float,
                    lib=None) -> np.ndarray:
    """Return a copy of the FP8 pool (uint8 codes) with the new bf16 rows quantised in."""
    pool = _u8(kv_cache).copy()
    NB, two, Hkv, bs, D = pool.shape
    assert two == 2
    kn, vn, sm = _u16(k_new), _u16(v_new), _i32(slot_mapping)
    N = sm.shape[0]
    assert kn.shape == (N, Hkv, D) and vn.shape == (N, Hkv, D)
    rc = (lib or load()).oracle_cache_write_fp8(_ptr(pool), NB, bs, Hkv, D, _ptr(kn), _ptr(vn),
                                                _ptr(sm), N, float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError("oracle_cache_write_fp8: slot outside the pool")
    return pool


def attention_fp8(q, cu_q_lens, kv_cache, k_scale: float, v_scale: float, block_tables,
                  seq_lens, num_heads: int, scale: float, rows=None, threads: int = 0,
                  lib=None) -> np.ndarray:
    """``attention`` over an FP8 pool (codes times k_scale / v_scale)."""
    pool = _u8(kv_cache)
    NB, _, Hkv, bs, D = pool.shape
    qq = _u16(q)
    cu = _i32(cu_q_lens)
    bt = _i32(block_tables)
    sl = _i32(seq_lens)
    B = sl.shape[0]
    assert cu.shape[0] == B + 1
    assert qq.shape[1:] == (num_heads, D), (qq.shape, num_heads, D)
    if bt.ndim == 1:
        bt = bt.reshape(B, -1)
    MB = bt.shape[1] if bt.size else 1
    if bt.size == 0:
        bt = np.full((B, 1), -1, dtype=np.int32)
    if rows is None:
        n = int(cu[-1])
        rows_arr = None
    else:
        rows_arr = _i32(rows)
        n = rows_arr.shape[0]
    out = np.zeros((n, num_heads, D), dtype=np.float64)
    rc = (lib or load()).oracle_attention_fp8(
        _ptr(out), _ptr(qq), _ptr(cu), B, _ptr(pool), float(k_scale), float(v_scale), NB, bs,
        num_heads, Hkv, D, _ptr(bt), MB, _ptr(sl), float(scale),
        _ptr(rows_arr) if rows_arr is not None else None, n if rows_arr is not None else 0,
        int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_fp8 failed ({rc})")
    return out


def max_threads(lib=None) -> int:
    return int((lib or load()).oracle_max_threads())

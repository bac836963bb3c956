"""Thin ctypes binding of libpagedattn (the C ABI in ``include/pa.h``).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  Functions keep the C names; tensors are PyTorch CUDA tensors
whose data pointers are passed through, and the stream defaults to PyTorch's
current stream.  If the library is missing this module raises on first use:
there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import struct
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedattn.so")

STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
          4: "PA_ERR_OOB", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_WORKSPACE",
          7: "PA_ERR_PRECONDITION"}

# Every symbol include/pa.h declares.
EXPORTS = ("pa_status_string", "pa_kv_block_bytes", "pa_kv_block_bytes_dtype", "pa_cache_write",
           "pa_cache_write_fp8", "pa_decode_fp8", "pa_prefill_chunk_fp8",
           "pa_decode_workspace_bytes", "pa_decode", "pa_decode_noalloc",
           "pa_decode_cascade_workspace_bytes", "pa_decode_cascade_kernels", "pa_decode_cascade",
           "pa_decode_cascade_fp8",
           "pa_prefill_chunk",
           "pa_attention_varlen_workspace_bytes", "pa_attention_varlen",
           "pa_attention_varlen_fp8", "pa_varlen_args_bytes", "pa_attention_varlen_packed",
           "pa_error_check")

# pa_varlen_args as laid out on a 64-bit little-endian target: out, q, k_new,
# v_new, slot_mapping, cu_q_lens, kv_cache, block_tables, seq_lens, workspace,
# workspace_bytes, stream; num_seqs, num_prefills, num_prefill_tokens,
# max_prefill_q_len, num_blocks, block_size, num_heads, num_kv_heads, head_size,
# max_blocks_per_seq, max_seq_len, kv8; scale, k_scale, v_scale.
VARLEN_ARGS = struct.Struct("<12Q12i3f")
_BF16, _I32, _U8 = torch.bfloat16, torch.int32, torch.uint8
_tls = threading.local()  # one packed-argument buffer per thread


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


_lib = None


def lib(path: Optional[str] = None):
    """Load libpagedattn.so and declare its entry points (raises if absent)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} not found: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(p)
    P, i, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_status_string.argtypes = [i]
    L.pa_kv_block_bytes.restype = sz
    L.pa_kv_block_bytes.argtypes = [i, i, i]
    L.pa_kv_block_bytes_dtype.restype = sz
    L.pa_kv_block_bytes_dtype.argtypes = [i, i, i, i]
    L.pa_cache_write_fp8.restype = i
    L.pa_cache_write_fp8.argtypes = [P, i, i, i, i, P, P, i64, P, i, ctypes.c_float,
                                     ctypes.c_float, P]
    L.pa_decode_fp8.restype = i
    L.pa_decode_fp8.argtypes = [P, P, P, i, i, i, i, i, P, i, P, i, i, ctypes.c_float,
                                ctypes.c_float, ctypes.c_float, P, sz, P]
    L.pa_prefill_chunk_fp8.restype = i
    L.pa_prefill_chunk_fp8.argtypes = [P, P, P, i, i, P, i, i, i, i, i, P, i, P, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_float, P]
    L.pa_cache_write.restype = i
    L.pa_cache_write.argtypes = [P, i, i, i, i, P, P, i64, P, i, P]
    L.pa_decode_workspace_bytes.restype = sz
    L.pa_decode_workspace_bytes.argtypes = [i, i, i, i]
    L.pa_decode.restype = i
    L.pa_decode.argtypes = [P, P, P, i, i, i, i, i, P, i, P, i, i, ctypes.c_float, P, sz, P]
    L.pa_decode_noalloc.restype = i
    L.pa_decode_noalloc.argtypes = [P, P, P, i, i, i, i, i, P, i, P, i, i, ctypes.c_float, P]
    L.pa_decode_cascade_workspace_bytes.restype = sz
    L.pa_decode_cascade_workspace_bytes.argtypes = [i, i, i, i, i]
    L.pa_decode_cascade_kernels.restype = i
    L.pa_decode_cascade_kernels.argtypes = [i, i, i, i, i, i, i, i]
    L.pa_decode_cascade.restype = i
    L.pa_decode_cascade.argtypes = [P, P, P, i, i, i, i, i, P, i, P, i, i, i, ctypes.c_float, P,
                                    sz, P]
    L.pa_decode_cascade_fp8.restype = i
    L.pa_decode_cascade_fp8.argtypes = [P, P, P, i, i, i, i, i, P, i, P, i, i, i, ctypes.c_float,
                                        ctypes.c_float, ctypes.c_float, P, sz, P]
    L.pa_prefill_chunk.restype = i
    L.pa_prefill_chunk.argtypes = [P, P, P, i, i, P, i, i, i, i, i, P, i, P, ctypes.c_float, P]
    L.pa_attention_varlen_workspace_bytes.restype = sz
    L.pa_attention_varlen_workspace_bytes.argtypes = [i, i, i, i, i]
    L.pa_attention_varlen.restype = i
    L.pa_attention_varlen.argtypes = [P, P, P, P, P, P, i, i, i, i, P, i, i, i, i, i, P, i, P, i,
                                      ctypes.c_float, P, sz, P]
    L.pa_attention_varlen_fp8.restype = i
    L.pa_attention_varlen_fp8.argtypes = [P, P, P, P, P, P, i, i, i, i, P, i, i, i, i, i, P, i, P,
                                          i, ctypes.c_float, ctypes.c_float, ctypes.c_float, P,
                                          sz, P]
    L.pa_varlen_args_bytes.restype = sz
    L.pa_varlen_args_bytes.argtypes = []
    L.pa_attention_varlen_packed.restype = i
    L.pa_attention_varlen_packed.argtypes = [P]
    if L.pa_varlen_args_bytes() < VARLEN_ARGS.size:
        raise RuntimeError("pa_varlen_args is smaller than this binding's layout")
    L.pa_error_check.restype = i
    L.pa_error_check.argtypes = [P]
    if path is None:
        _lib = L
    return L


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    try:
        return stream.cuda_stream  # torch.cuda.Stream
    except AttributeError:
        return int(stream)


def _check(status: int, where: str):
    if status != 0:
        raise PaError(status, where)


def _need(t: torch.Tensor, name: str, dtype, dims: Optional[int] = None):
    try:  # the common case in one expression (torch dtypes are singletons)
        if (t.is_cuda and t.dtype is dtype and (dims is None or t.dim() == dims)
                and t.is_contiguous() and isinstance(t, torch.Tensor)):
            return
    except AttributeError:
        pass
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _pool_geom(kv_cache: torch.Tensor):
    _need(kv_cache, "kv_cache", torch.bfloat16, 5)
    NB, two, Hkv, bs, D = kv_cache.shape
    if two != 2:
        raise ValueError("kv_cache must be [num_blocks, 2, num_kv_heads, block_size, head_size]")
    return NB, bs, Hkv, D


def pa_kv_block_bytes(block_size: int, num_kv_heads: int, head_size: int) -> int:
    return int(lib().pa_kv_block_bytes(block_size, num_kv_heads, head_size))


def pa_cache_write(kv_cache: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   slot_mapping: torch.Tensor, stream=None) -> None:
    """Scatter k_new/v_new [N, Hkv, D] rows into kv_cache at slot_mapping [N]."""
    try:  # every tensor at once; on failure the per-argument checks name the culprit
        ks = kv_cache.shape
        ok = (len(ks) == 5 and ks[1] == 2
              and kv_cache.dtype is _BF16 and kv_cache.is_cuda and kv_cache.is_contiguous()
              and k_new.dtype is _BF16 and k_new.is_cuda and k_new.is_contiguous()
              and v_new.dtype is _BF16 and v_new.is_cuda and v_new.is_contiguous()
              and slot_mapping.dtype is _I32 and slot_mapping.is_cuda
              and slot_mapping.dim() == 1 and slot_mapping.is_contiguous())
    except (AttributeError, TypeError):
        ok = False
    if not ok:
        _pool_geom(kv_cache)
        _need(k_new, "k_new", torch.bfloat16, 3)
        _need(v_new, "v_new", torch.bfloat16, 3)
        _need(slot_mapping, "slot_mapping", torch.int32, 1)
        ks = kv_cache.shape
    NB, _, Hkv, bs, D = ks
    N = slot_mapping.shape[0]
    rows = (N, Hkv, D)
    if k_new.shape != rows or v_new.shape != rows:
        raise ValueError("k_new/v_new must be [num_tokens, num_kv_heads, head_size]")
    L = _lib if _lib is not None else lib()
    _check(L.pa_cache_write(kv_cache.data_ptr(), NB, bs, Hkv, D, k_new.data_ptr(),
                            v_new.data_ptr(), Hkv * D, slot_mapping.data_ptr(), N,
                            _stream(stream)), "pa_cache_write")


def _pool8_geom(kv_cache: torch.Tensor):
    _need(kv_cache, "kv_cache", torch.uint8, 5)
    NB, two, Hkv, bs, D = kv_cache.shape
    if two != 2:
        raise ValueError("kv_cache must be [num_blocks, 2, num_kv_heads, block_size, head_size]")
    return NB, bs, Hkv, D


def pa_kv_block_bytes_dtype(block_size: int, num_kv_heads: int, head_size: int,
                            dtype_num_bytes: int) -> int:
    return int(lib().pa_kv_block_bytes_dtype(block_size, num_kv_heads, head_size,
                                             dtype_num_bytes))


def pa_cache_write_fp8(kv_cache: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       slot_mapping: torch.Tensor, k_scale: float, v_scale: float,
                       stream=None) -> None:
    """Quantise bf16 k_new/v_new [N, Hkv, D] into an FP8 (uint8 e4m3 codes) pool."""
    NB, bs, Hkv, D = _pool8_geom(kv_cache)
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    N = slot_mapping.shape[0]
    if k_new.shape != (N, Hkv, D) or v_new.shape != (N, Hkv, D):
        raise ValueError("k_new/v_new must be [num_tokens, num_kv_heads, head_size]")
    _check(lib().pa_cache_write_fp8(kv_cache.data_ptr(), NB, bs, Hkv, D, k_new.data_ptr(),
                                    v_new.data_ptr(), Hkv * D, slot_mapping.data_ptr(), N,
                                    float(k_scale), float(v_scale), _stream(stream)),
           "pa_cache_write_fp8")


def pa_decode_fp8(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                  block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                  scale: float, k_scale: float, v_scale: float, workspace: torch.Tensor,
                  stream=None) -> None:
    """Decode attention over an FP8 pool (uint8 e4m3 codes times k_scale / v_scale)."""
    NB, bs, Hkv, D = _pool8_geom(kv_cache)
    _need(q, "q", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(workspace, "workspace", torch.uint8, 1)
    B, Hq, Dq = q.shape
    if Dq != D or out.shape != q.shape or seq_lens.shape[0] != B or block_tables.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    _check(lib().pa_decode_fp8(out.data_ptr(), q.data_ptr(), kv_cache.data_ptr(), NB, bs, Hq,
                               Hkv, D, block_tables.data_ptr(), block_tables.shape[1],
                               seq_lens.data_ptr(), B, int(max_seq_len), float(scale),
                               float(k_scale), float(v_scale), workspace.data_ptr(),
                               workspace.numel(), _stream(stream)), "pa_decode_fp8")


def pa_prefill_chunk_fp8(out: torch.Tensor, q: torch.Tensor, cu_q_lens: torch.Tensor,
                         max_q_len: int, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                         seq_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float,
                         stream=None) -> None:
    """Chunked prefill over an FP8 pool (uint8 e4m3 codes times k_scale / v_scale)."""
    NB, bs, Hkv, D = _pool8_geom(kv_cache)
    _need(q, "q", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 3)
    _need(cu_q_lens, "cu_q_lens", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    n = seq_lens.shape[0]
    Hq = q.shape[1]
    if q.shape[2] != D or out.shape != q.shape or cu_q_lens.shape[0] != n + 1 or \
            block_tables.shape[0] != n:
        raise ValueError("inconsistent prefill shapes")
    _check(lib().pa_prefill_chunk_fp8(out.data_ptr(), q.data_ptr(), cu_q_lens.data_ptr(), n,
                                      int(max_q_len), kv_cache.data_ptr(), NB, bs, Hq, Hkv, D,
                                      block_tables.data_ptr(), block_tables.shape[1],
                                      seq_lens.data_ptr(), float(scale), float(k_scale),
                                      float(v_scale), _stream(stream)), "pa_prefill_chunk_fp8")


def pa_decode_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int,
                              head_size: int) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_size))


def pa_decode(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
              block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
              scale: float, workspace: torch.Tensor, stream=None) -> None:
    """Decode attention: q/out [B, Hq, D], block_tables [B, MB], seq_lens [B]."""
    try:  # every tensor at once; on failure the per-argument checks name the culprit
        ks, qs, bts = kv_cache.shape, q.shape, block_tables.shape
        ok = (len(ks) == 5 and ks[1] == 2 and len(qs) == 3 and len(bts) == 2
              and kv_cache.dtype is _BF16 and kv_cache.is_cuda and kv_cache.is_contiguous()
              and q.dtype is _BF16 and q.is_cuda and q.is_contiguous()
              and out.dtype is _BF16 and out.is_cuda and out.is_contiguous()
              and block_tables.dtype is _I32 and block_tables.is_cuda
              and block_tables.is_contiguous()
              and seq_lens.dtype is _I32 and seq_lens.is_cuda and seq_lens.dim() == 1
              and seq_lens.is_contiguous()
              and workspace.dtype is _U8 and workspace.is_cuda and workspace.dim() == 1
              and workspace.is_contiguous())
    except (AttributeError, TypeError):
        ok = False
    if not ok:
        _pool_geom(kv_cache)
        _need(q, "q", torch.bfloat16, 3)
        _need(out, "out", torch.bfloat16, 3)
        _need(block_tables, "block_tables", torch.int32, 2)
        _need(seq_lens, "seq_lens", torch.int32, 1)
        _need(workspace, "workspace", torch.uint8, 1)
        ks, qs, bts = kv_cache.shape, q.shape, block_tables.shape
    NB, _, Hkv, bs, D = ks
    B, Hq, Dq = qs
    if Dq != D or out.shape != qs or seq_lens.shape[0] != B or bts[0] != B:
        raise ValueError("inconsistent decode shapes")
    L = _lib if _lib is not None else lib()
    _check(L.pa_decode(out.data_ptr(), q.data_ptr(), kv_cache.data_ptr(), NB, bs, Hq, Hkv, D,
                       block_tables.data_ptr(), bts[1], seq_lens.data_ptr(), B,
                       int(max_seq_len), float(scale), workspace.data_ptr(), workspace.numel(),
                       _stream(stream)), "pa_decode")


def pa_decode_noalloc(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                      scale: float, stream=None) -> None:
    """pa_decode with the library's built-in scratch instead of a workspace tensor."""
    NB, bs, Hkv, D = _pool_geom(kv_cache)
    _need(q, "q", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, Dq = q.shape
    if Dq != D or out.shape != q.shape or seq_lens.shape[0] != B or block_tables.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    _check(lib().pa_decode_noalloc(out.data_ptr(), q.data_ptr(), kv_cache.data_ptr(), NB, bs, Hq,
                                   Hkv, D, block_tables.data_ptr(), block_tables.shape[1],
                                   seq_lens.data_ptr(), B, int(max_seq_len), float(scale),
                                   _stream(stream)), "pa_decode_noalloc")


def pa_decode_cascade_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int,
                                      head_size: int, shared_len: int) -> int:
    return int(lib().pa_decode_cascade_workspace_bytes(num_seqs, num_heads, num_kv_heads,
                                                       head_size, shared_len))


def pa_decode_cascade_kernels(num_seqs: int, num_heads: int, num_kv_heads: int, head_size: int,
                              block_size: int, max_seq_len: int, shared_len: int,
                              fp8: bool = False) -> int:
    """Kernels one pa_decode_cascade (fp8: pa_decode_cascade_fp8) call launches."""
    return int(lib().pa_decode_cascade_kernels(num_seqs, num_heads, num_kv_heads, head_size,
                                               block_size, max_seq_len, shared_len, int(fp8)))


def pa_decode_cascade(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                      shared_len: int, scale: float, workspace: torch.Tensor,
                      stream=None, kv_scales=None) -> None:
    """pa_decode for a batch whose first shared_len tokens sit in the same blocks.

    A uint8 (FP8 e4m3) pool goes to pa_decode_cascade_fp8 with
    kv_scales = (k_scale, v_scale)."""
    if kv_cache.dtype == torch.uint8:
        if kv_scales is None:
            raise ValueError("an FP8 pool needs kv_scales=(k_scale, v_scale)")
        return pa_decode_cascade_fp8(out, q, kv_cache, block_tables, seq_lens, max_seq_len,
                                     shared_len, scale, kv_scales[0], kv_scales[1], workspace,
                                     stream)
    NB, bs, Hkv, D = _pool_geom(kv_cache)
    _need(q, "q", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(workspace, "workspace", torch.uint8, 1)
    B, Hq, Dq = q.shape
    if Dq != D or out.shape != q.shape or seq_lens.shape[0] != B or block_tables.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    _check(lib().pa_decode_cascade(out.data_ptr(), q.data_ptr(), kv_cache.data_ptr(), NB, bs, Hq,
                                   Hkv, D, block_tables.data_ptr(), block_tables.shape[1],
                                   seq_lens.data_ptr(), B, int(max_seq_len), int(shared_len),
                                   float(scale), workspace.data_ptr(), workspace.numel(),
                                   _stream(stream)), "pa_decode_cascade")


def pa_decode_cascade_fp8(out: torch.Tensor, q: torch.Tensor, kv_cache: torch.Tensor,
                          block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                          shared_len: int, scale: float, k_scale: float, v_scale: float,
                          workspace: torch.Tensor, stream=None) -> None:
    """pa_decode_cascade over an FP8 pool (uint8 e4m3 codes times k_scale / v_scale)."""
    NB, bs, Hkv, D = _pool8_geom(kv_cache)
    _need(q, "q", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(workspace, "workspace", torch.uint8, 1)
    B, Hq, Dq = q.shape
    if Dq != D or out.shape != q.shape or seq_lens.shape[0] != B or block_tables.shape[0] != B:
        raise ValueError("inconsistent decode shapes")
    _check(lib().pa_decode_cascade_fp8(out.data_ptr(), q.data_ptr(), kv_cache.data_ptr(), NB, bs,
                                       Hq, Hkv, D, block_tables.data_ptr(),
                                       block_tables.shape[1], seq_lens.data_ptr(), B,
                                       int(max_seq_len), int(shared_len), float(scale),
                                       float(k_scale), float(v_scale), workspace.data_ptr(),
                                       workspace.numel(), _stream(stream)),
           "pa_decode_cascade_fp8")


def pa_prefill_chunk(out: torch.Tensor, q: torch.Tensor, cu_q_lens: torch.Tensor,
                     max_q_len: int, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                     seq_lens: torch.Tensor, scale: float, stream=None) -> None:
    """Chunked-prefill attention: q/out [sum q_len, Hq, D], cu_q_lens [n+1]."""
    NB, bs, Hkv, D = _pool_geom(kv_cache)
    _need(q, "q", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 3)
    _need(cu_q_lens, "cu_q_lens", torch.int32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    n = seq_lens.shape[0]
    Hq = q.shape[1]
    if q.shape[2] != D or out.shape != q.shape or cu_q_lens.shape[0] != n + 1 or \
            block_tables.shape[0] != n:
        raise ValueError("inconsistent prefill shapes")
    _check(lib().pa_prefill_chunk(out.data_ptr(), q.data_ptr(), cu_q_lens.data_ptr(), n,
                                  int(max_q_len), kv_cache.data_ptr(), NB, bs, Hq, Hkv, D,
                                  block_tables.data_ptr(), block_tables.shape[1],
                                  seq_lens.data_ptr(), float(scale), _stream(stream)),
           "pa_prefill_chunk")


def pa_attention_varlen_workspace_bytes(num_seqs: int, num_prefills: int, num_heads: int,
                                        num_kv_heads: int, head_size: int) -> int:
    return int(lib().pa_attention_varlen_workspace_bytes(num_seqs, num_prefills, num_heads,
                                                         num_kv_heads, head_size))


def pa_attention_varlen(out: torch.Tensor, q: torch.Tensor, k_new: Optional[torch.Tensor],
                        v_new: Optional[torch.Tensor], slot_mapping: Optional[torch.Tensor],
                        cu_q_lens: torch.Tensor, num_prefills: int, num_prefill_tokens: int,
                        max_prefill_q_len: int, kv_cache: torch.Tensor,
                        block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                        scale: float, workspace: torch.Tensor, stream=None,
                        kv_scales: Optional[tuple] = None) -> None:
    """One step over a flattened mixed batch (chunks first, then decode tokens):
    optional cache write, chunked prefill, decode.  A uint8 kv_cache is an FP8
    (e4m3) pool and needs kv_scales = (k_scale, v_scale)."""
    fp8 = kv_cache.dtype is _U8
    if fp8 and kv_scales is None:
        raise ValueError("an FP8 pool needs kv_scales=(k_scale, v_scale)")
    # Every tensor's device, dtype, rank and contiguity in one expression (this
    # call runs once per step of a serving loop); any failure re-runs the
    # argument-by-argument checks, which name the offending tensor.
    try:
        ks, qs, bts = kv_cache.shape, q.shape, block_tables.shape
        ok = (len(ks) == 5 and ks[1] == 2 and len(qs) == 3 and len(bts) == 2
              and kv_cache.is_cuda and kv_cache.is_contiguous()
              and q.dtype is _BF16 and q.is_cuda and q.is_contiguous()
              and out.dtype is _BF16 and out.is_cuda and out.is_contiguous()
              and cu_q_lens.dtype is _I32 and cu_q_lens.is_cuda and cu_q_lens.dim() == 1
              and cu_q_lens.is_contiguous()
              and block_tables.dtype is _I32 and block_tables.is_cuda
              and block_tables.is_contiguous()
              and seq_lens.dtype is _I32 and seq_lens.is_cuda and seq_lens.dim() == 1
              and seq_lens.is_contiguous()
              and workspace.dtype is _U8 and workspace.is_cuda and workspace.dim() == 1
              and workspace.is_contiguous()
              and (fp8 or kv_cache.dtype is _BF16))
    except (AttributeError, TypeError):
        ok = False
    if not ok:
        (_pool8_geom if fp8 else _pool_geom)(kv_cache)
        _need(q, "q", torch.bfloat16, 3)
        _need(out, "out", torch.bfloat16, 3)
        _need(cu_q_lens, "cu_q_lens", torch.int32, 1)
        _need(block_tables, "block_tables", torch.int32, 2)
        _need(seq_lens, "seq_lens", torch.int32, 1)
        _need(workspace, "workspace", torch.uint8, 1)
        ks, qs, bts = kv_cache.shape, q.shape, block_tables.shape
    NB, _, Hkv, bs, D = ks
    B = seq_lens.shape[0]
    rows, Hq, Dq = qs
    if Dq != D or out.shape != qs or bts[0] != B or \
            rows != num_prefill_tokens + B - num_prefills:
        raise ValueError("inconsistent varlen shapes")
    kp = vp = sp = 0
    if slot_mapping is not None:
        try:
            ok = (k_new.dtype is _BF16 and k_new.is_cuda and k_new.is_contiguous()
                  and v_new.dtype is _BF16 and v_new.is_cuda and v_new.is_contiguous()
                  and slot_mapping.dtype is _I32 and slot_mapping.is_cuda
                  and slot_mapping.is_contiguous())
        except (AttributeError, TypeError):
            ok = False
        if not ok:
            _need(k_new, "k_new", torch.bfloat16, 3)
            _need(v_new, "v_new", torch.bfloat16, 3)
            _need(slot_mapping, "slot_mapping", torch.int32, 1)
        kv_rows = (rows, Hkv, D)
        if k_new.shape != kv_rows or v_new.shape != kv_rows or slot_mapping.shape != (rows,):
            raise ValueError("k_new/v_new [rows, num_kv_heads, head_size] and slot_mapping "
                             "[rows]: one row per query row")
        kp, vp, sp = k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr()
    L = _lib if _lib is not None else lib()
    try:
        buf, addr = _tls.varlen
    except AttributeError:
        buf = ctypes.create_string_buffer(L.pa_varlen_args_bytes())
        addr = ctypes.addressof(buf)
        _tls.varlen = (buf, addr)
    if fp8:
        ks, vs = float(kv_scales[0]), float(kv_scales[1])
    else:
        ks = vs = 1.0
    # One struct and one foreign call: per-argument conversion would cost more
    # than the call itself.
    VARLEN_ARGS.pack_into(
        buf, 0, out.data_ptr(), q.data_ptr(), kp, vp, sp, cu_q_lens.data_ptr(),
        kv_cache.data_ptr(), block_tables.data_ptr(), seq_lens.data_ptr(), workspace.data_ptr(),
        workspace.numel(), _stream(stream) or 0, B, int(num_prefills), int(num_prefill_tokens),
        int(max_prefill_q_len), NB, bs, Hq, Hkv, D, bts[1], int(max_seq_len), fp8,
        float(scale), ks, vs)
    st = L.pa_attention_varlen_packed(addr)
    if st:
        raise PaError(st, "pa_attention_varlen_fp8" if fp8 else "pa_attention_varlen")


def pa_error_check(stream=None) -> None:
    """Synchronise the stream and raise if a kernel flagged bad device data."""
    _check(lib().pa_error_check(_stream(stream)), "pa_error_check")

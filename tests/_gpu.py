"""GPU-test helpers: run a PagedBatch through the C ABI and through the oracle."""

from __future__ import annotations

from typing import Optional

import numpy as np
import torch

import oracle
from paged_kv_cache_287_gb300 import binding

MAX_ABS = 1e-2   # bf16 attention outputs vs the fp64 oracle (max abs error)
MEAN_ABS = 1e-3  # ... and mean abs error


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def workspace_for(b, num_seqs: Optional[int] = None) -> torch.Tensor:
    n = b.num_seqs if num_seqs is None else num_seqs
    nbytes = binding.pa_decode_workspace_bytes(n, b.num_heads, b.num_kv_heads, b.head_size)
    return torch.empty(nbytes, dtype=torch.uint8, device=b.kv_cache.device)


def gpu_write(b) -> None:
    binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping)


def gpu_decode(b, lo: int = 0, hi: Optional[int] = None) -> torch.Tensor:
    """Decode sequences lo..hi-1 (each has exactly one query row)."""
    hi = b.num_seqs if hi is None else hi
    r0 = int(b.cu_q_lens[lo])
    q = b.q[r0:r0 + (hi - lo)]
    out = torch.full_like(q, float("nan"))
    lens = b.seq_lens[lo:hi]
    binding.pa_decode(out, q, b.kv_cache, b.block_tables[lo:hi], lens,
                      int(lens.max()) if hi > lo else 0, b.scale, workspace_for(b, hi - lo))
    return out


def gpu_prefill(b, lo: int = 0, hi: Optional[int] = None) -> torch.Tensor:
    hi = b.num_seqs if hi is None else hi
    r0, r1 = int(b.cu_q_lens[lo]), int(b.cu_q_lens[hi])
    q = b.q[r0:r1]
    out = torch.full_like(q, float("nan"))
    cu = (b.cu_q_lens[lo:hi + 1] - r0).contiguous()
    binding.pa_prefill_chunk(out, q, cu, int(b.q_lens[lo:hi].max()), b.kv_cache,
                             b.block_tables[lo:hi], b.seq_lens[lo:hi], b.scale)
    return out


def oracle_pool(b) -> np.ndarray:
    """The pool after the oracle's own cache write (bits), from the pre-write pool."""
    return oracle.cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping)


def oracle_rows(b, pool_bits: np.ndarray, rows=None) -> np.ndarray:
    return oracle.attention(b.q, b.cu_q_lens, pool_bits, b.block_tables, b.seq_lens,
                            b.num_heads, b.scale, rows=rows)


# (what, max |d|, mean |d|, that largest |d| in bf16 ulps of the rounded oracle
# value where it occurs, max and mean |d| against the bf16-rounded oracle) of
# every compare() in this process, reported at the end of the test session.
ULP_LOG: list = []


def bf16_ulps(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """|got - bf16(want)| in units in the last place of bf16(want) (2^(e-7) for a
    value in [2^e, 2^(e+1)); the smallest normal's ulp for zero)."""
    w = torch.from_numpy(np.ascontiguousarray(want)).to(torch.bfloat16).double().numpy()
    aw = np.abs(w)
    e = np.floor(np.log2(np.where(aw > 0, aw, 2.0 ** -126)))
    ulp = np.exp2(np.maximum(e, -126.0) - 7.0)
    return np.abs(got - w) / ulp


def compare(got: torch.Tensor, want: np.ndarray, what: str = ""):
    g = got.detach().float().cpu().double().numpy()
    assert g.shape == want.shape, (g.shape, want.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    d = np.abs(g - want)
    mx, mean = float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0
    i = int(np.argmax(d)) if d.size else 0
    ulps = float(bf16_ulps(g.reshape(-1)[i:i + 1], want.reshape(-1)[i:i + 1])[0]) if d.size else 0.0
    # The same against the oracle rounded to bf16 (RNE), as the kernels round
    # their outputs: what is left is the kernels' own arithmetic.
    wr = torch.from_numpy(np.ascontiguousarray(want)).to(torch.bfloat16).double().numpy()
    dr = np.abs(g - wr)
    rmx, rmean = (float(dr.max()), float(dr.mean())) if dr.size else (0.0, 0.0)
    ULP_LOG.append((what, mx, mean, ulps, rmx, rmean))
    note = " (within one bf16 ulp of the rounded oracle there: output rounding)" if ulps <= 1 else ""
    assert mx <= MAX_ABS and mean <= MEAN_ABS, \
        f"{what}: max|d| {mx:.3e} mean|d| {mean:.3e}, {ulps:.1f} bf16 ulps{note}"
    return mx, mean

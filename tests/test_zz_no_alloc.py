"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (an engine whose KV-cache pool already holds nearly all of HBM, a
host program that only receives device pointers, a decode loop that cannot
afford an allocation that may synchronise the device) get the same decode with
scratch from a fixed array inside the library.  These tests call it through the
C ABI and check it against pa_decode with a caller-provided workspace, bit for
bit, on two calls in a row, since every call reuses the same array.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import make_batch, make_config
from tests._gpu import bits, gpu_write, workspace_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")


def _noalloc(b, out):
    L = binding.lib()
    NB, _, Hkv, bs, D = b.kv_cache.shape
    return L.pa_decode_noalloc(out.data_ptr(), b.q.data_ptr(), b.kv_cache.data_ptr(), NB, bs,
                               b.num_heads, Hkv, D, b.block_tables.data_ptr(),
                               b.block_tables.shape[1], b.seq_lens.data_ptr(), b.num_seqs,
                               b.max_seq_len, ctypes.c_float(b.scale),
                               torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("workload", ["small", 2])
def test_noalloc_matches_workspace_decode_twice(workload):
    if workload == "small":
        b = make_batch(name="na", seq_lens=[700, 1, 33, 2048, 95], q_lens=[1] * 5, num_heads=32,
                       num_kv_heads=8, head_size=128, block_size=16, scale=128 ** -0.5, seed=31,
                       device=DEV)
    else:
        b = make_config(workload, device=DEV)
    gpu_write(b)
    ref = torch.empty_like(b.q)
    binding.pa_decode(ref, b.q, b.kv_cache, b.block_tables, b.seq_lens, b.max_seq_len, b.scale,
                      workspace_for(b))
    torch.cuda.synchronize()
    ref_bits = bits(ref)
    for _ in range(2):
        out = torch.full_like(b.q, float("nan"))
        assert _noalloc(b, out) == 0
        binding.pa_error_check()
        # The same kernel, the same split of the contexts over the grid, the same
        # inputs: only the scratch differs, so the outputs agree bit for bit (a
        # scratch region carved one record off would not).
        assert np.array_equal(bits(out), ref_bits), "pa_decode_noalloc differs from pa_decode"


def test_noalloc_holds_the_largest_batch_pa_decode_accepts():
    """The largest batch of head size 128 that pa_decode's tables hold (15 091
    sequences, group 4): its workspace fits the 16 MiB scratch on this GPU, and the
    call runs and agrees bit for bit with pa_decode."""
    L = binding.lib()
    B = 15091
    assert L.pa_decode_workspace_bytes(B, 4, 1, 128) <= 16 << 20
    g = torch.Generator().manual_seed(33)
    lens = torch.randint(1, 40, (B,), generator=g).tolist()
    b = make_batch(name="nmax", seq_lens=lens, q_lens=[1] * B, num_heads=4, num_kv_heads=1,
                   head_size=128, block_size=16, scale=128 ** -0.5, seed=34, device=DEV)
    gpu_write(b)
    ref = torch.empty_like(b.q)
    binding.pa_decode(ref, b.q, b.kv_cache, b.block_tables, b.seq_lens, b.max_seq_len, b.scale,
                      workspace_for(b))
    out = torch.full_like(b.q, float("nan"))
    assert _noalloc(b, out) == 0
    binding.pa_error_check()
    assert np.array_equal(bits(out), bits(ref))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    L = binding.lib()
    huge = 5_000_000   # the split-state table alone exceeds the 16 MiB scratch
    assert L.pa_decode_workspace_bytes(huge, 32, 8, 128) > 16 << 20
    status = L.pa_decode_noalloc(1 << 20, 1 << 20, 1 << 20, 10, 16, 32, 8, 128, 1 << 20, 4,
                                 1 << 20, huge, 64, ctypes.c_float(0.1), None)
    assert binding.STATUS[status] == "PA_ERR_UNSUPPORTED"

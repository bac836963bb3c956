"""Bitwise invariance of every attention entry point under a permutation of the
physical blocks.

Blocks are only the index from a sequence's tokens to their K/V ("Inside vLLM:
Anatomy of a High-Throughput LLM Inference System", §Engine core): where a
block sits in the pool must not change a single bit of any output.  Each test
builds one batch, a second batch with the same logical content whose blocks are
re-placed by a random permutation of the pool (tables and slots follow), runs
the same call on both, and compares the outputs bit for bit.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import (FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of,
                                                make_batch)
from tests._gpu import bits

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")
SCALES = (FP8_K_SCALE, FP8_V_SCALE)


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.pa_error_check()
    yield
    binding.pa_error_check()


def pair(seed: int, perm_seed: int, **kw):
    """The batch and a copy of it whose physical blocks are permuted."""
    a = make_batch(seed=seed, device=DEV, **kw)
    b = make_batch(seed=seed, device=DEV, **kw)
    bs = b.block_size
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(perm_seed))
    perm = perm.to(DEV)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(b.num_blocks, device=DEV)
    b.kv_cache = b.kv_cache[inv].contiguous()        # block i of a is block perm[i] of b
    b.block_tables = torch.where(b.block_tables >= 0, perm[b.block_tables.long()].int(),
                                 b.block_tables)
    b.slot_mapping = torch.where(b.slot_mapping >= 0,
                                 (perm[(b.slot_mapping // bs).long()] * bs +
                                  b.slot_mapping % bs).int(), b.slot_mapping)
    assert not torch.equal(a.block_tables, b.block_tables)
    return a, b


def pool_of(b, fp8: bool):
    """Write the batch's new rows into its pool (bf16 or FP8) and return the pool."""
    if fp8:
        pool = fp8_pool_of(b)
        binding.pa_cache_write_fp8(pool, b.k_new, b.v_new, b.slot_mapping, *SCALES)
        return pool
    binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping)
    return b.kv_cache


def same_bits(x: torch.Tensor, y: torch.Tensor) -> bool:
    return np.array_equal(bits(x), bits(y))


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill_is_invariant_to_block_placement_bitwise(fp8):
    kw = dict(name="ip", seq_lens=[700, 129, 2100, 64], q_lens=[300, 129, 65, 64],
              num_heads=32, num_kv_heads=8, head_size=128, block_size=16, scale=128 ** -0.5)
    outs = []
    for b in pair(41, 5, **kw):
        pool = pool_of(b, fp8)
        out = torch.full_like(b.q, float("nan"))
        if fp8:
            binding.pa_prefill_chunk_fp8(out, b.q, b.cu_q_lens, int(b.q_lens.max()), pool,
                                         b.block_tables, b.seq_lens, b.scale, *SCALES)
        else:
            binding.pa_prefill_chunk(out, b.q, b.cu_q_lens, int(b.q_lens.max()), pool,
                                     b.block_tables, b.seq_lens, b.scale)
        binding.pa_error_check()
        outs.append(out)
    assert same_bits(*outs)


@pytest.mark.parametrize("suffix", ["short", "long"])
@pytest.mark.parametrize("fp8", [False, True])
def test_cascade_is_invariant_to_block_placement_bitwise(fp8, suffix):
    """Both paths: short own suffixes (prefix pass first) and long ones (the prefix
    pass beside the own tokens' decode in one launch)."""
    g = torch.Generator().manual_seed(43)
    pb = 16 if suffix == "short" else 32
    own = [16, 1, 7, 16, 3, 12, 9] if suffix == "short" else \
        torch.randint(1, 4097, (48,), generator=g).tolist()
    kw = dict(name="ic", seq_lens=[pb * 16 + x for x in own], q_lens=[1] * len(own),
              num_heads=32, num_kv_heads=8, head_size=128, block_size=16, scale=128 ** -0.5,
              shared_prefix_blocks=pb)
    outs = []
    for b in pair(44, 6, **kw):
        pool = pool_of(b, fp8)
        out = torch.full_like(b.q, float("nan"))
        ws = torch.empty(binding.pa_decode_cascade_workspace_bytes(
            b.num_seqs, b.num_heads, b.num_kv_heads, b.head_size, pb * 16), dtype=torch.uint8,
            device=DEV)
        binding.pa_decode_cascade(out, b.q, pool, b.block_tables, b.seq_lens, b.max_seq_len,
                                  pb * 16, b.scale, ws, kv_scales=SCALES if fp8 else None)
        binding.pa_error_check()
        outs.append(out)
    assert same_bits(*outs)


@pytest.mark.parametrize("fp8", [False, True])
def test_varlen_step_is_invariant_to_block_placement_bitwise(fp8):
    """The whole step (cache write, chunks and decode tokens in one launch)."""
    g = torch.Generator().manual_seed(45)
    dec = torch.randint(200, 3000, (40,), generator=g).tolist()
    kw = dict(name="iv", seq_lens=[900, 513] + dec, q_lens=[256, 513] + [1] * 40,
              num_heads=32, num_kv_heads=8, head_size=128, block_size=16, scale=128 ** -0.5)
    outs = []
    for b in pair(46, 7, **kw):
        pool = fp8_pool_of(b) if fp8 else b.kv_cache
        out = torch.full_like(b.q, float("nan"))
        ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
            b.num_seqs, 2, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8,
            device=DEV)
        binding.pa_attention_varlen(out, b.q, b.k_new, b.v_new, b.slot_mapping,
                                    b.cu_q_lens[:3].contiguous(), 2, int(b.cu_q_lens[2]),
                                    int(b.q_lens[:2].max()), pool, b.block_tables, b.seq_lens,
                                    int(b.seq_lens[2:].max()), b.scale, ws,
                                    kv_scales=SCALES if fp8 else None)
        binding.pa_error_check()
        outs.append(out)
    assert same_bits(*outs)

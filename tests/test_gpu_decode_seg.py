"""Decode of small batches in one launch: a CTA per (sequence, KV head).

When every (sequence, KV head) pair of a batch gets an SM of its own and
max_seq_len is at most 12 tiles of 16 tokens, pa_decode runs one kernel: the
pair's CTA splits its tiles over its warps and merges them in place, instead of
the split kernel and its merge kernel.  The outputs must meet the oracle bar of
every other decode (1e-2 max, 1e-3 mean absolute error against fp64), empty
sequences give zero rows, and the result is bitwise independent of where the
blocks sit in the pool.
"""

from __future__ import annotations

import pytest
import torch

import oracle
from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import (FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of,
                                                make_batch, make_config)
from tests._gpu import compare, gpu_decode, gpu_write, oracle_pool, oracle_rows, workspace_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")
SMS = torch.cuda.get_device_properties(DEV).multi_processor_count


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.pa_error_check()
    yield
    binding.pa_error_check()


def kernels(b, max_len=None, kv8=0):
    return binding.lib().pa_decode_cascade_kernels(
        b.num_seqs, b.num_heads, b.num_kv_heads, b.head_size, b.block_size,
        b.max_seq_len if max_len is None else max_len, 0, kv8)


SEG_SHAPES = [
    # seq_lens, Hq, Hkv, D, bs
    ([192, 1, 0, 17, 160, 33, 16, 191], 32, 8, 128, 16),   # 12 tiles at most, an empty one
    ([35, 74, 41, 42], 32, 4, 64, 16),                      # TinyLlama heads
    ([190, 7, 96, 0, 129], 16, 4, 128, 8),                  # block 8: two blocks per tile
    ([100, 3, 64], 48, 8, 64, 32),                          # group 6, block 32
    ([16] * 19, 64, 8, 128, 16),                            # 152 pairs, one tile each
    ([5], 8, 1, 128, 16),                                   # one pair, one tile
]


@pytest.mark.parametrize("case", range(len(SEG_SHAPES)))
def test_seg_cta_decode_matches_oracle(case):
    lens, Hq, Hkv, D, bs = SEG_SHAPES[case]
    b = make_batch(name=f"sc{case}", seq_lens=lens, q_lens=[1] * len(lens), num_heads=Hq,
                   num_kv_heads=Hkv, head_size=D, block_size=bs, scale=D ** -0.5,
                   seed=400 + case, device=DEV)
    if len(lens) * Hkv <= SMS:
        assert kernels(b) == 1
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_decode(b)
    binding.pa_error_check()
    compare(out, oracle_rows(b, pool), f"one-launch decode case {case}")
    for s, L in enumerate(lens):
        if L == 0:
            assert (out[s] == 0).all()


def test_one_tile_past_the_limit_takes_the_split_path():
    """193 tokens is 13 tiles: the split kernel and its merge, same results."""
    b = make_batch(name="sc13", seq_lens=[193, 40, 176], q_lens=[1] * 3, num_heads=32,
                   num_kv_heads=8, head_size=128, block_size=16, scale=0.09, seed=410,
                   device=DEV)
    assert kernels(b) == 2
    assert kernels(b, max_len=192) == 1
    pool = oracle_pool(b)
    gpu_write(b)
    compare(gpu_decode(b), oracle_rows(b, pool), "13-tile decode")


def test_tiny_workload_is_one_launch_and_matches_oracle():
    b = make_config(1, device=DEV)
    assert kernels(b) == 1
    pool = oracle_pool(b)
    gpu_write(b)
    o1, o2 = gpu_decode(b), gpu_decode(b)
    compare(o1, oracle_rows(b, pool), "tiny workload, one launch")
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("fp8", [False, True])
def test_seg_cta_decode_is_invariant_to_block_placement_bitwise(fp8):
    lens = [192, 77, 1, 130, 0, 45]
    kw = dict(name="scp", seq_lens=lens, q_lens=[1] * len(lens), num_heads=32, num_kv_heads=8,
              head_size=128, block_size=16, scale=128 ** -0.5, device=DEV)
    a = make_batch(seed=411, **kw)
    b = make_batch(seed=411, **kw)
    assert kernels(a, kv8=int(fp8)) == 1
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(412)).to(DEV)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(b.num_blocks, device=DEV)
    b.kv_cache = b.kv_cache[inv].contiguous()
    b.block_tables = torch.where(b.block_tables >= 0, perm[b.block_tables.long()].int(),
                                 b.block_tables)
    sm = b.slot_mapping.long()
    b.slot_mapping = torch.where(sm >= 0, perm[(sm // 16).clamp(min=0)] * 16 + sm % 16,
                                 sm).int()  # padding rows (-1) stay padding
    outs = []
    for x in (a, b):
        if fp8:
            pool8 = fp8_pool_of(x)
            binding.pa_cache_write_fp8(pool8, x.k_new, x.v_new, x.slot_mapping, FP8_K_SCALE,
                                       FP8_V_SCALE)
            out = torch.full_like(x.q, float("nan"))
            binding.pa_decode_fp8(out, x.q, pool8, x.block_tables, x.seq_lens, x.max_seq_len,
                                  x.scale, FP8_K_SCALE, FP8_V_SCALE, workspace_for(x))
        else:
            gpu_write(x)
            out = gpu_decode(x)
        outs.append(out)
    binding.pa_error_check()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_seg_cta_fp8_decode_matches_oracle():
    b = make_batch(name="sc8", seq_lens=[192, 1, 0, 100, 31], q_lens=[1] * 5, num_heads=64,
                   num_kv_heads=8, head_size=128, block_size=16, scale=128 ** -0.5, seed=413,
                   device=DEV)
    assert kernels(b, kv8=1) == 1
    pool8 = fp8_pool_of(b)
    codes = oracle.cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE,
                                   FP8_V_SCALE)
    binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE,
                               FP8_V_SCALE)
    out = torch.full_like(b.q, float("nan"))
    binding.pa_decode_fp8(out, b.q, pool8, b.block_tables, b.seq_lens, b.max_seq_len, b.scale,
                          FP8_K_SCALE, FP8_V_SCALE, workspace_for(b))
    binding.pa_error_check()
    want = oracle.attention_fp8(b.q, b.cu_q_lens, codes, FP8_K_SCALE, FP8_V_SCALE,
                                b.block_tables, b.seq_lens, b.num_heads, b.scale)
    compare(out, want, "one-launch fp8 decode")
    assert (out[2] == 0).all()

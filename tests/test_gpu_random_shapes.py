"""Seeded random-shape parity sweep over every attention entry point.

Each case draws a group size (1..8), head size (64 or 128), block size (8, 16,
32), a batch size and lengths that include the awkward ones (1, multiples of the
block and tile sizes and their neighbours), builds the batch with the shared
seeded generators and compares the CUDA path with the oracle.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import (FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of,
                                                make_batch)
from tests._gpu import (bits, compare, gpu_decode, gpu_prefill, gpu_write, oracle_pool,
                        oracle_rows)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")
AWKWARD = [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.pa_error_check()
    yield
    binding.pa_error_check()


def _shape(seed: int):
    g = np.random.default_rng(seed)
    hkv = int(g.choice([1, 2, 4, 8]))
    group = int(g.integers(1, 9))
    D = int(g.choice([64, 128]))
    bs = int(g.choice([8, 16, 32]))
    return g, hkv, group, D, bs


def _lens(g, n, hi):
    out = []
    for _ in range(n):
        out.append(int(g.choice(AWKWARD)) if g.random() < 0.5 else int(g.integers(1, hi)))
    return out


@pytest.mark.parametrize("seed", range(12))
def test_random_decode(seed):
    g, hkv, group, D, bs = _shape(1000 + seed)
    B = int(g.integers(1, 40))
    lens = _lens(g, B, 1500)
    b = make_batch(name=f"rd{seed}", seq_lens=lens, q_lens=[1] * B, num_heads=hkv * group,
                   num_kv_heads=hkv, head_size=D, block_size=bs, scale=float(D) ** -0.5,
                   seed=2000 + seed, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    assert np.array_equal(bits(b.kv_cache), pool)
    compare(gpu_decode(b), oracle_rows(b, pool), f"random decode {seed}: G{group} D{D} bs{bs}")


@pytest.mark.parametrize("seed", range(10))
def test_random_prefill(seed):
    g, hkv, group, D, bs = _shape(3000 + seed)
    n = int(g.integers(1, 5))
    qls = [int(x) for x in g.choice(AWKWARD[:-3] + [300, 513], n)]
    lens = [q + int(g.integers(0, 700)) for q in qls]
    b = make_batch(name=f"rp{seed}", seq_lens=lens, q_lens=qls, num_heads=hkv * group,
                   num_kv_heads=hkv, head_size=D, block_size=bs, scale=float(D) ** -0.5,
                   seed=4000 + seed, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    compare(gpu_prefill(b), oracle_rows(b, pool), f"random prefill {seed}: G{group} D{D} bs{bs}")


@pytest.mark.parametrize("seed", range(8))
def test_random_varlen(seed):
    g, hkv, group, D, bs = _shape(5000 + seed)
    n_pre, n_dec = int(g.integers(1, 4)), int(g.integers(1, 30))
    qls = [int(x) for x in g.choice([2, 16, 33, 128, 200], n_pre)] + [1] * n_dec
    lens = [q + int(g.integers(0, 600)) for q in qls[:n_pre]] + _lens(g, n_dec, 1200)
    b = make_batch(name=f"rv{seed}", seq_lens=lens, q_lens=qls, num_heads=hkv * group,
                   num_kv_heads=hkv, head_size=D, block_size=bs, scale=float(D) ** -0.5,
                   seed=6000 + seed, device=DEV)
    pool = oracle_pool(b)
    out = torch.full_like(b.q, float("nan"))
    ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, n_pre, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8,
        device=DEV)
    binding.pa_attention_varlen(out, b.q, b.k_new, b.v_new, b.slot_mapping,
                                b.cu_q_lens[:n_pre + 1].contiguous(), n_pre,
                                int(b.cu_q_lens[n_pre]), max(qls[:n_pre]), b.kv_cache,
                                b.block_tables, b.seq_lens, int(b.seq_lens[n_pre:].max()),
                                b.scale, ws)
    binding.pa_error_check()
    assert np.array_equal(bits(b.kv_cache), pool)
    compare(out, oracle_rows(b, pool), f"random varlen {seed}: G{group} D{D} bs{bs}")


@pytest.mark.parametrize("seed", range(6))
def test_random_cascade(seed):
    g, hkv, group, D, bs = _shape(7000 + seed)
    pb = int(g.integers(1, 40)) * (32 // bs) if bs < 16 else int(g.integers(1, 40))
    if (pb * bs) % 16:
        pb += 1
    B = int(g.integers(1, 50))
    lens = [pb * bs + int(x) for x in g.integers(1, 400, B)]
    b = make_batch(name=f"rc{seed}", seq_lens=lens, q_lens=[1] * B, num_heads=hkv * group,
                   num_kv_heads=hkv, head_size=D, block_size=bs, scale=float(D) ** -0.5,
                   seed=8000 + seed, shared_prefix_blocks=pb, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = torch.full_like(b.q, float("nan"))
    ws = torch.empty(binding.pa_decode_cascade_workspace_bytes(
        B, b.num_heads, b.num_kv_heads, D, pb * bs), dtype=torch.uint8, device=DEV)
    binding.pa_decode_cascade(out, b.q, b.kv_cache, b.block_tables, b.seq_lens, max(lens),
                              pb * bs, b.scale, ws)
    binding.pa_error_check()
    compare(out, oracle_rows(b, pool), f"random cascade {seed}: G{group} D{D} bs{bs} P{pb * bs}")


@pytest.mark.parametrize("seed", range(6))
def test_random_fp8_decode(seed):
    g, hkv, group, _, bs = _shape(9000 + seed)
    B = int(g.integers(1, 40))
    lens = _lens(g, B, 1500)
    b = make_batch(name=f"rf{seed}", seq_lens=lens, q_lens=[1] * B, num_heads=hkv * group,
                   num_kv_heads=hkv, head_size=128, block_size=bs, scale=128 ** -0.5,
                   seed=10000 + seed, device=DEV)
    pool8 = fp8_pool_of(b)
    codes = oracle.cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE,
                                   FP8_V_SCALE)
    binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE, FP8_V_SCALE)
    out = torch.full_like(b.q, float("nan"))
    ws = torch.empty(binding.pa_decode_workspace_bytes(B, b.num_heads, hkv, 128),
                     dtype=torch.uint8, device=DEV)
    binding.pa_decode_fp8(out, b.q, pool8, b.block_tables, b.seq_lens, max(lens), b.scale,
                          FP8_K_SCALE, FP8_V_SCALE, ws)
    binding.pa_error_check()
    assert np.array_equal(pool8.cpu().numpy(), codes)
    want = oracle.attention_fp8(b.q, b.cu_q_lens, codes, FP8_K_SCALE, FP8_V_SCALE,
                                b.block_tables, b.seq_lens, b.num_heads, b.scale)
    compare(out, want, f"random fp8 decode {seed}: G{group} bs{bs}")

"""Parity of the FP8 (e4m3) KV-cache path with the CPU fp64 oracle.

The FP8 cache write must match the oracle's quantisation bit for bit over the
whole pool; FP8 decode must lie within the same 1e-2 max / 1e-3 mean absolute
error of the oracle's fp64 attention over the dequantised pool as bf16 decode.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import (FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of,
                                                make_batch, make_config)
from tests._gpu import compare, workspace_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.pa_error_check()
    yield
    binding.pa_error_check()


def _write(b, pool8, ks, vs):
    want = oracle.cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, ks, vs)
    binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, ks, vs)
    binding.pa_error_check()
    return want


def _decode(b, pool8, ks, vs):
    out = torch.full_like(b.q, float("nan"))
    binding.pa_decode_fp8(out, b.q, pool8, b.block_tables, b.seq_lens, b.max_seq_len, b.scale,
                          ks, vs, workspace_for(b))
    binding.pa_error_check()
    return out


def _oracle(b, pool_codes, ks, vs, rows=None):
    return oracle.attention_fp8(b.q, b.cu_q_lens, pool_codes, ks, vs, b.block_tables,
                                b.seq_lens, b.num_heads, b.scale, rows=rows)


WRITE_SHAPES = [
    # seq_lens, q_lens, Hkv, D, bs
    ([40, 7, 90], [5, 1, 33], 2, 64, 8),
    ([33, 64, 1], [33, 3, 1], 8, 128, 16),
    ([300], [100], 4, 128, 32),
]


@pytest.mark.parametrize("case", range(len(WRITE_SHAPES)))
def test_fp8_cache_write_bit_exact(case):
    lens, qls, Hkv, D, bs = WRITE_SHAPES[case]
    b = make_batch(name=f"w8{case}", seq_lens=lens, q_lens=qls, num_heads=Hkv, num_kv_heads=Hkv,
                   head_size=D, block_size=bs, scale=0.1, seed=800 + case, device=DEV)
    pool8 = fp8_pool_of(b)
    b.slot_mapping[1] = -1  # a padding row is skipped
    want = _write(b, pool8, 0.05, 0.0123)
    assert np.array_equal(pool8.cpu().numpy(), want)


def test_fp8_cache_write_saturates_rounds_ties_and_keeps_signs():
    b = make_batch(name="w8s", seq_lens=[16], q_lens=[16], num_heads=2, num_kv_heads=2,
                   head_size=64, block_size=16, scale=0.1, seed=810, device=DEV)
    pool8 = fp8_pool_of(b)
    # Every bf16 magnitude class: huge (saturates), exact codes, ties, tiny (to +-0).
    g = torch.Generator().manual_seed(3)
    e = torch.randint(-40, 40, b.k_new.shape, generator=g).float()
    x = torch.sign(torch.randn(b.k_new.shape, generator=g)) * torch.exp2(e) * \
        (1 + torch.randint(0, 16, b.k_new.shape, generator=g).float() / 16)
    b.k_new.copy_(x.to(torch.bfloat16).to(DEV))
    b.v_new.copy_((-x).to(torch.bfloat16).to(DEV))
    want = _write(b, pool8, 1.0, 0.5)
    assert np.array_equal(pool8.cpu().numpy(), want)


@pytest.mark.parametrize("ks,vs", [
    (2.0 ** -100, 2.0 ** 100),  # powers of two: the write multiplies by 1 / scale
    (2.0 ** 126, 2.0 ** -126),  # reciprocals at the ends of the normal range
    (2.0 ** 127, 0.75),         # 2^-127 is subnormal, 0.75 no power of two: division
    (0.25, 3.0),
])
def test_fp8_cache_write_bit_exact_over_the_whole_exponent_range(ks, vs):
    """x / scale, rounded to e4m3, for bf16 inputs of every binary32 exponent;
    a power-of-two scale takes the multiply by its exact reciprocal, which must
    give the same codes as the division."""
    b = make_batch(name="w8e", seq_lens=[64], q_lens=[64], num_heads=4, num_kv_heads=4,
                   head_size=128, block_size=16, scale=0.1, seed=811, device=DEV)
    pool8 = fp8_pool_of(b)
    g = torch.Generator().manual_seed(5)
    e = torch.randint(-133, 128, b.k_new.shape, generator=g).float()
    x = torch.sign(torch.randn(b.k_new.shape, generator=g)) * torch.exp2(e) * \
        (1 + torch.randint(0, 16, b.k_new.shape, generator=g).float() / 16)
    x = x.clamp(-3.0e38, 3.0e38)
    b.k_new.copy_(x.to(torch.bfloat16).to(DEV))
    b.v_new.copy_(x.flip(0).to(torch.bfloat16).to(DEV))
    want = _write(b, pool8, ks, vs)
    assert np.array_equal(pool8.cpu().numpy(), want)


DECODE_SHAPES = [
    # seq_lens, Hq, Hkv, bs
    ([1, 15, 16, 17, 31, 32, 33, 100], 8, 8, 16),      # group 1
    ([5, 64, 200, 1], 8, 4, 16),                       # group 2
    ([129, 77, 3, 256, 40], 16, 4, 8),                 # group 4, block 8
    ([300, 2, 63, 97], 64, 8, 32),                     # group 8, block 32
    ([513, 1000, 17], 24, 8, 16),                      # group 3
]


@pytest.mark.parametrize("case", range(len(DECODE_SHAPES)))
def test_fp8_decode_small_shapes(case):
    lens, Hq, Hkv, bs = DECODE_SHAPES[case]
    b = make_batch(name=f"d8{case}", seq_lens=lens, q_lens=[1] * len(lens), num_heads=Hq,
                   num_kv_heads=Hkv, head_size=128, block_size=bs, scale=128 ** -0.5,
                   seed=820 + case, device=DEV)
    pool8 = fp8_pool_of(b)
    codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    compare(_decode(b, pool8, FP8_K_SCALE, FP8_V_SCALE),
            _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE), f"fp8 decode case {case}")


@pytest.mark.parametrize("ks,vs", [(0.25, 0.003), (0.0123, 0.9)])
def test_fp8_decode_other_scales(ks, vs):
    b = make_batch(name="d8s", seq_lens=[400, 90, 1, 777], q_lens=[1] * 4, num_heads=32,
                   num_kv_heads=8, head_size=128, block_size=16, scale=-0.07, seed=830,
                   device=DEV)
    pool8 = fp8_pool_of(b, ks, vs)
    codes = _write(b, pool8, ks, vs)
    compare(_decode(b, pool8, ks, vs), _oracle(b, codes, ks, vs), f"fp8 decode scales {ks} {vs}")


def test_fp8_decode_empty_sequences_give_zeros():
    b = make_batch(name="d8e", seq_lens=[0, 20, 0, 5], q_lens=[1] * 4, num_heads=8,
                   num_kv_heads=2, head_size=128, block_size=16, scale=0.1, seed=840,
                   device=DEV)
    pool8 = fp8_pool_of(b)
    codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    out = _decode(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    compare(out, _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE), "fp8 decode, empty sequences")
    assert (out[0] == 0).all() and (out[2] == 0).all()


def test_fp8_decode_large_queries_stay_in_range():
    """Queries far outside f16 range are scaled per head by a power of two."""
    b = make_batch(name="d8q", seq_lens=[50, 300], q_lens=[1, 1], num_heads=16, num_kv_heads=4,
                   head_size=128, block_size=16, scale=1e-6, seed=850, q_scale=1e6,
                   device=DEV)
    pool8 = fp8_pool_of(b)
    codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    compare(_decode(b, pool8, FP8_K_SCALE, FP8_V_SCALE),
            _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE), "fp8 decode, large queries")


def test_fp8_decode_workload_full_size():
    b = make_config(2, device=DEV)
    pool8 = fp8_pool_of(b)
    codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    assert np.array_equal(pool8.cpu().numpy(), codes), "fp8 cache write"
    out = _decode(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    rows = np.arange(0, b.num_seqs, 5, dtype=np.int32)
    compare(out[torch.as_tensor(rows, device=DEV).long()],
            _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE, rows), "fp8 workload 2 (sampled)")


def test_fp8_decode_rejects_head_size_64():
    b = make_batch(name="d8r", seq_lens=[10], q_lens=[1], num_heads=4, num_kv_heads=4,
                   head_size=64, block_size=16, scale=0.1, seed=860, device=DEV)
    pool8 = fp8_pool_of(b)
    with pytest.raises(binding.PaError) as e:
        _decode(b, pool8, 1.0, 1.0)
    assert e.value.status == 2


PREFILL_SHAPES = [
    # seq_lens, q_lens, Hq, Hkv, bs
    ([300, 40, 513], [129, 40, 200], 32, 8, 16),   # group 4, several tiles, ragged
    ([150, 260], [70, 129], 8, 8, 8),              # group 1, block 8
    ([2000, 700], [1024, 333], 64, 8, 32),         # group 8, block 32, long
    ([37, 5], [37, 1], 24, 8, 16),                 # group 3, tiny chunks
]


@pytest.mark.parametrize("case", range(len(PREFILL_SHAPES)))
def test_fp8_prefill_small_shapes(case):
    lens, qls, Hq, Hkv, bs = PREFILL_SHAPES[case]
    b = make_batch(name=f"p8{case}", seq_lens=lens, q_lens=qls, num_heads=Hq, num_kv_heads=Hkv,
                   head_size=128, block_size=bs, scale=128 ** -0.5, seed=870 + case, device=DEV)
    pool8 = fp8_pool_of(b)
    codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    out = torch.full_like(b.q, float("nan"))
    binding.pa_prefill_chunk_fp8(out, b.q, b.cu_q_lens, max(qls), pool8, b.block_tables,
                                 b.seq_lens, b.scale, FP8_K_SCALE, FP8_V_SCALE)
    binding.pa_error_check()
    compare(out, _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE), f"fp8 prefill case {case}")


def test_fp8_prefill_more_chunks_than_the_ranking_holds_and_one_long_chunk():
    """300 short ragged chunks (past the 256 the kernel ranks by context), then
    one 3000-token chunk after 1000 cached tokens, from an FP8 pool."""
    g = np.random.default_rng(83)
    qls = [int(x) for x in g.integers(2, 25, 300)]
    lens = [q + int(c) for q, c in zip(qls, g.integers(0, 200, 300))]
    for name, lens, qls, seed, rows in (
            ("p8many", lens, qls, 84, None),
            ("p8one", [4000, 70], [3000, 70], 85,
             [0, 1, 63, 64, 127, 128, 1000, 2047, 2048, 2944, 2999, 3000, 3069])):
        b = make_batch(name=name, seq_lens=lens, q_lens=qls, num_heads=16, num_kv_heads=4,
                       head_size=128, block_size=16, scale=128 ** -0.5, seed=seed, device=DEV)
        pool8 = fp8_pool_of(b)
        codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
        out = torch.full_like(b.q, float("nan"))
        binding.pa_prefill_chunk_fp8(out, b.q, b.cu_q_lens, max(qls), pool8, b.block_tables,
                                     b.seq_lens, b.scale, FP8_K_SCALE, FP8_V_SCALE)
        binding.pa_error_check()
        got = out if rows is None else out[rows]
        compare(got, _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE, rows=rows), f"fp8 prefill {name}")


def test_fp8_prefill_long_context_and_empty_chunk():
    """The FP8 prefill (conversion warp in the loop) over a 40 000-token cached
    context, with an empty chunk between two others."""
    lens, qls = [40300, 5000, 3000], [300, 0, 257]
    b = make_batch(name="p8long", seq_lens=lens, q_lens=qls, num_heads=32, num_kv_heads=8,
                   head_size=128, block_size=16, scale=128 ** -0.5, seed=32, device=DEV)
    pool8 = fp8_pool_of(b)
    codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    out = torch.full_like(b.q, float("nan"))
    binding.pa_prefill_chunk_fp8(out, b.q, b.cu_q_lens, max(qls), pool8, b.block_tables,
                                 b.seq_lens, b.scale, FP8_K_SCALE, FP8_V_SCALE)
    binding.pa_error_check()
    rows = [0, 1, 31, 32, 63, 64, 150, 299, 300, 301, 430, 556]
    compare(out[rows], _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE, rows=rows),
            "fp8 long-context prefill")


@pytest.mark.parametrize("scale", [-0.1, 0.0])
def test_fp8_prefill_negative_and_zero_scale_and_other_kv_scales(scale):
    b = make_batch(name="p8s", seq_lens=[400, 90], q_lens=[200, 90], num_heads=16,
                   num_kv_heads=4, head_size=128, block_size=16, scale=scale, seed=880,
                   q_scale=300.0, device=DEV)
    ks, vs = 0.2, 0.0045
    pool8 = fp8_pool_of(b, ks, vs)
    codes = _write(b, pool8, ks, vs)
    out = torch.full_like(b.q, float("nan"))
    binding.pa_prefill_chunk_fp8(out, b.q, b.cu_q_lens, 200, pool8, b.block_tables, b.seq_lens,
                                 b.scale, ks, vs)
    binding.pa_error_check()
    compare(out, _oracle(b, codes, ks, vs), f"fp8 prefill, scale {scale}")


def test_fp8_prefill_mixed_workload_chunks():
    b = make_config(4, device=DEV)
    pool8 = fp8_pool_of(b)
    codes = _write(b, pool8, FP8_K_SCALE, FP8_V_SCALE)
    q = b.q[:4096]
    out = torch.full_like(q, float("nan"))
    binding.pa_prefill_chunk_fp8(out, q, b.cu_q_lens[:9].contiguous(), 512, pool8,
                                 b.block_tables[:8], b.seq_lens[:8], b.scale, FP8_K_SCALE,
                                 FP8_V_SCALE)
    binding.pa_error_check()
    rows = np.arange(0, 4096, 41, dtype=np.int32)
    compare(out[torch.as_tensor(rows, device=DEV).long()],
            _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE, rows), "fp8 prefill, mixed workload")


def _varlen_fp8(b, n_pre, ks, vs):
    out = torch.full_like(b.q, float("nan"))
    ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, n_pre, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8,
        device=DEV)
    binding.pa_attention_varlen(out, b.q, b.k_new, b.v_new, b.slot_mapping,
                                b.cu_q_lens[:n_pre + 1].contiguous(), n_pre,
                                int(b.cu_q_lens[n_pre]), int(b.q_lens[:n_pre].max()), pool8_of[0],
                                b.block_tables, b.seq_lens, int(b.seq_lens[n_pre:].max()),
                                b.scale, ws, kv_scales=(ks, vs))
    binding.pa_error_check()
    return out


pool8_of = [None]


@pytest.mark.parametrize("shape", [
    ([300, 40, 513, 90, 17, 1], [129, 40, 200, 1, 1, 1], 32, 8, 16),
    ([64, 700, 33, 2000], [64, 1, 1, 1], 64, 8, 32),
])
def test_fp8_varlen_one_launch(shape):
    lens, qls, Hq, Hkv, bs = shape
    b = make_batch(name="v8", seq_lens=lens, q_lens=qls, num_heads=Hq, num_kv_heads=Hkv,
                   head_size=128, block_size=bs, scale=128 ** -0.5, seed=890 + len(lens),
                   device=DEV)
    n_pre = sum(1 for q in qls if q > 1)
    pool8_of[0] = fp8_pool_of(b)
    codes = oracle.cache_write_fp8(pool8_of[0], b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE,
                                   FP8_V_SCALE)
    out = _varlen_fp8(b, n_pre, FP8_K_SCALE, FP8_V_SCALE)
    assert np.array_equal(pool8_of[0].cpu().numpy(), codes), "fp8 cache write"
    compare(out, _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE), f"fp8 varlen {lens}")


def test_fp8_varlen_mixed_workload():
    b = make_config(4, device=DEV)
    pool8_of[0] = fp8_pool_of(b)
    codes = oracle.cache_write_fp8(pool8_of[0], b.k_new, b.v_new, b.slot_mapping, FP8_K_SCALE,
                                   FP8_V_SCALE)
    out = _varlen_fp8(b, 8, FP8_K_SCALE, FP8_V_SCALE)
    assert np.array_equal(pool8_of[0].cpu().numpy(), codes), "fp8 cache write"
    pre = torch.empty_like(b.q[:4096])
    binding.pa_prefill_chunk_fp8(pre, b.q[:4096], b.cu_q_lens[:9].contiguous(), 512,
                                 pool8_of[0], b.block_tables[:8], b.seq_lens[:8], b.scale,
                                 FP8_K_SCALE, FP8_V_SCALE)
    assert torch.equal(pre.view(torch.int16), out[:4096].view(torch.int16)), "chunk rows"
    rows = np.concatenate([np.arange(0, 4096, 97), np.arange(4096, 4344)]).astype(np.int32)
    compare(out[torch.as_tensor(rows, device=DEV).long()],
            _oracle(b, codes, FP8_K_SCALE, FP8_V_SCALE, rows), "fp8 mixed workload, one launch")

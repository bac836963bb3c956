"""Parity of the CUDA path (through the C ABI) with the CPU fp64 oracle.

Cache writes must match bit for bit over the whole pool; attention outputs must
lie within 1e-2 max abs and 1e-3 mean abs error of the oracle's unrounded fp64
result.  Small shapes span several tiles with ragged tails; the five numbered
workloads run at full size in the launch configuration the benchmark times.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import make_batch, make_config
from tests._gpu import (bits, compare, gpu_decode, gpu_prefill, gpu_write, oracle_pool,
                        oracle_rows, workspace_for)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.pa_error_check()
    yield
    binding.pa_error_check()


# ----------------------------------------------------------------- cache write

def test_cache_write_decode_slots_bit_exact():
    b = make_config(1, device=DEV)
    want = oracle_pool(b)
    gpu_write(b)
    assert np.array_equal(bits(b.kv_cache), want)


def test_cache_write_scatter_to_free_slots_bit_exact():
    """Four rows to slots drawn from every slot no live token uses; the other
    slots of the pool stay untouched, bit for bit."""
    b = make_config(1, device=DEV)
    NB, _, Hkv, bs, D = b.kv_cache.shape
    used = set()
    for s in range(b.num_seqs):
        for t in range(int(b.seq_lens[s])):
            used.add(int(b.block_tables[s, t // bs]) * bs + t % bs)
    free = sorted(set(range(NB * bs)) - used)
    g = torch.Generator().manual_seed(2871)
    pick = [free[i] for i in torch.randperm(len(free), generator=g)[:4].tolist()]
    b.slot_mapping = torch.tensor(pick, dtype=torch.int32, device=DEV)
    want = oracle_pool(b)
    gpu_write(b)
    assert np.array_equal(bits(b.kv_cache), want)


def test_cache_write_mixed_config_and_padding():
    b = make_batch(name="w", seq_lens=[40, 77, 9], q_lens=[40, 13, 1], num_heads=4,
                   num_kv_heads=4, head_size=64, block_size=8, scale=0.125, seed=5, device=DEV)
    b.slot_mapping[3] = -1    # a padding row is skipped
    want = oracle_pool(b)
    gpu_write(b)
    assert np.array_equal(bits(b.kv_cache), want)


def test_cache_write_out_of_pool_slot_is_flagged_and_skipped():
    b = make_config(1, device=DEV)
    b.slot_mapping[0] = b.num_blocks * b.block_size + 5
    keep = b.slot_mapping.clone()
    b.slot_mapping[0] = -1
    want = oracle_pool(b)
    b.slot_mapping = keep
    gpu_write(b)
    with pytest.raises(binding.PaError) as e:
        binding.pa_error_check()
    assert e.value.status == 4
    assert np.array_equal(bits(b.kv_cache), want)


# ----------------------------------------------------------------- decode

DECODE_SHAPES = [
    # seq_lens, Hq, Hkv, D, bs
    ([1, 15, 16, 17, 31, 32, 33, 100], 8, 8, 128, 16),      # group 1
    ([5, 64, 200, 1], 8, 4, 64, 16),                        # group 2
    ([129, 77, 3, 256, 40], 16, 4, 128, 8),                 # group 4, block 8
    ([300, 2, 63, 97], 32, 4, 64, 32),                      # group 8, block 32
    ([513, 1000, 17], 24, 8, 128, 16),                      # group 3
    ([1], 8, 1, 128, 16),
]


@pytest.mark.parametrize("case", range(len(DECODE_SHAPES)))
def test_decode_small_shapes(case):
    lens, Hq, Hkv, D, bs = DECODE_SHAPES[case]
    b = make_batch(name=f"d{case}", seq_lens=lens, q_lens=[1] * len(lens), num_heads=Hq,
                   num_kv_heads=Hkv, head_size=D, block_size=bs, scale=D ** -0.5,
                   seed=100 + case, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_decode(b)
    compare(out, oracle_rows(b, pool), f"decode case {case}")


def test_decode_empty_sequence_gives_zeros():
    b = make_batch(name="e", seq_lens=[0, 20, 0, 5], q_lens=[1, 1, 1, 1], num_heads=8,
                   num_kv_heads=2, head_size=128, block_size=16, scale=0.1, seed=9, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_decode(b)
    compare(out, oracle_rows(b, pool), "decode with empty sequences")
    assert (out[0] == 0).all() and (out[2] == 0).all()


def test_decode_is_invariant_to_block_placement_bitwise():
    lens = [700, 33, 1500, 64]
    kw = dict(name="p", seq_lens=lens, q_lens=[1] * 4, num_heads=32, num_kv_heads=8,
              head_size=128, block_size=16, scale=128 ** -0.5, device=DEV)
    a = make_batch(seed=11, **kw)
    b = make_batch(seed=11, **kw)
    # Same logical content, different physical placement: re-place b's blocks.
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(3)).to(DEV)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(b.num_blocks, device=DEV)
    b.kv_cache = b.kv_cache[inv].contiguous()
    b.block_tables = torch.where(b.block_tables >= 0, perm[b.block_tables.long()].int(),
                                 b.block_tables)
    b.slot_mapping = (perm[(b.slot_mapping // 16).long()] * 16 + b.slot_mapping % 16).int()
    gpu_write(a)
    gpu_write(b)
    oa, ob = gpu_decode(a), gpu_decode(b)
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))


def test_decode_is_deterministic():
    b = make_config(1, device=DEV)
    gpu_write(b)
    o1, o2 = gpu_decode(b), gpu_decode(b)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_decode_out_of_pool_block_is_flagged_not_faulted():
    b = make_batch(name="oob", seq_lens=[40, 20], q_lens=[1, 1], num_heads=8, num_kv_heads=2,
                   head_size=64, block_size=16, scale=0.1, seed=4, device=DEV)
    gpu_write(b)
    b.block_tables[0, 1] = b.num_blocks + 1000
    gpu_decode(b)
    with pytest.raises(binding.PaError) as e:
        binding.pa_error_check()
    assert e.value.status == 4


def test_decode_leaves_neighbouring_memory_untouched():
    b = make_batch(name="g", seq_lens=[90, 3, 260], q_lens=[1, 1, 1], num_heads=16,
                   num_kv_heads=2, head_size=128, block_size=16, scale=0.09, seed=6, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    guard = 4096
    buf = torch.full((guard * 2 + b.q.numel(),), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[guard:guard + b.q.numel()].view_as(b.q)
    binding.pa_decode(out, b.q, b.kv_cache, b.block_tables, b.seq_lens, b.max_seq_len, b.scale,
                      workspace_for(b))
    assert (buf[:guard] == 7.0).all() and (buf[guard + b.q.numel():] == 7.0).all()
    compare(out, oracle_rows(b, pool), "decode with guard bands")


# ----------------------------------------------------------------- chunked prefill

PREFILL_SHAPES = [
    # seq_lens (context + chunk), q_lens, Hq, Hkv, D, bs
    ([37, 100], [37, 20], 8, 2, 128, 16),          # no context / context + ragged chunk
    ([300, 65, 129], [1, 64, 129], 32, 8, 128, 16),
    ([200, 90], [70, 90], 8, 8, 64, 8),            # group 1, block 8
    ([500, 33], [160, 17], 16, 2, 128, 32),        # group 8, block 32
    ([260], [130], 24, 8, 64, 16),                 # group 3
]


@pytest.mark.parametrize("case", range(len(PREFILL_SHAPES)))
def test_prefill_small_shapes(case):
    lens, qls, Hq, Hkv, D, bs = PREFILL_SHAPES[case]
    b = make_batch(name=f"p{case}", seq_lens=lens, q_lens=qls, num_heads=Hq, num_kv_heads=Hkv,
                   head_size=D, block_size=bs, scale=D ** -0.5, seed=200 + case, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_prefill(b)
    compare(out, oracle_rows(b, pool), f"prefill case {case}")


def test_prefill_of_single_token_chunks_matches_decode():
    lens = [50, 17, 300]
    b = make_batch(name="pd", seq_lens=lens, q_lens=[1, 1, 1], num_heads=16, num_kv_heads=4,
                   head_size=128, block_size=16, scale=0.088, seed=12, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    compare(gpu_prefill(b), oracle_rows(b, pool), "prefill q_len 1")
    compare(gpu_decode(b), oracle_rows(b, pool), "decode")


def test_prefill_more_chunks_than_the_ranking_holds():
    """300 chunks: more than the kernel ranks by cached context (256), so the
    CTAs take chunks in index order; short ragged chunks, some without context."""
    g = np.random.default_rng(77)
    qls = [int(x) for x in g.integers(2, 25, 300)]
    lens = [q + int(c) for q, c in zip(qls, g.integers(0, 200, 300))]
    b = make_batch(name="p300", seq_lens=lens, q_lens=qls, num_heads=8, num_kv_heads=2,
                   head_size=128, block_size=16, scale=128 ** -0.5, seed=78, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    compare(gpu_prefill(b), oracle_rows(b, pool), "prefill, 300 chunks")


def test_prefill_one_long_chunk():
    """One 3000-token chunk after 1000 cached tokens (47 query-tile pairs, the
    last ragged; the latest rows see 4000 keys); rows sampled across tiles."""
    b = make_batch(name="pl1", seq_lens=[4000, 70], q_lens=[3000, 70], num_heads=32,
                   num_kv_heads=8, head_size=128, block_size=16, scale=128 ** -0.5, seed=81,
                   device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_prefill(b)
    rows = [0, 1, 63, 64, 127, 128, 1000, 1999, 2047, 2048, 2943, 2944, 2998, 2999, 3000, 3069]
    compare(out[rows], oracle_rows(b, pool, rows=rows), "prefill, one 3000-token chunk")


def test_prefill_long_context_and_empty_chunk():
    """A chunk after a 40 000-token cached context (316 K/V tiles through each
    query tile's hand-over chain), an empty chunk between two others, and a
    ragged last chunk; rows sampled across tile and chunk boundaries."""
    lens, qls = [40300, 5000, 3000], [300, 0, 257]
    b = make_batch(name="plong", seq_lens=lens, q_lens=qls, num_heads=32, num_kv_heads=8,
                   head_size=128, block_size=16, scale=128 ** -0.5, seed=31, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_prefill(b)
    rows = [0, 1, 31, 32, 63, 64, 150, 298, 299, 300, 301, 332, 430, 555, 556]
    compare(out[rows], oracle_rows(b, pool, rows=rows), "long-context prefill")


# ----------------------------------------------------------------- full-size workloads

def _sample_rows(b, per_chunk: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    rows = []
    cu = b.cu_q_lens.tolist()
    for s in range(b.num_seqs):
        n = cu[s + 1] - cu[s]
        if n <= per_chunk:
            rows += list(range(cu[s], cu[s + 1]))
        else:
            pick = set(torch.randperm(n, generator=g)[:per_chunk - 2].tolist()) | {0, n - 1}
            rows += sorted(cu[s] + i for i in pick)
    return np.array(rows, dtype=np.int32)


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_decode_workload_full_size(n):
    b = make_config(n, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    assert np.array_equal(bits(b.kv_cache), pool), "cache write"
    out = gpu_decode(b)
    binding.pa_error_check()
    compare(out, oracle_rows(b, pool), f"workload {n}")


def test_mixed_workload_full_size():
    b = make_config(4, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    assert np.array_equal(bits(b.kv_cache), pool), "cache write"
    pre = gpu_prefill(b, 0, 8)
    dec = gpu_decode(b, 8, b.num_seqs)
    binding.pa_error_check()
    rows = _sample_rows(b, 40, seed=4)
    pre_rows = rows[rows < 4096]
    compare(pre[torch.as_tensor(pre_rows, device=DEV).long()], oracle_rows(b, pool, pre_rows),
            "mixed: prefill chunks (sampled rows)")
    compare(dec, oracle_rows(b, pool, np.arange(4096, 4344, dtype=np.int32)), "mixed: decode")


@pytest.mark.parametrize("scale", [-0.125, 0.0])
def test_negative_and_zero_softmax_scale(scale):
    """The scale is a free parameter: a negative one flips which keys win, zero
    gives the mean of the visible values."""
    b = make_batch(name="sc", seq_lens=[150, 40, 260], q_lens=[70, 1, 129], num_heads=16,
                   num_kv_heads=4, head_size=128, block_size=16, scale=scale, seed=77,
                   device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    compare(gpu_prefill(b), oracle_rows(b, pool), f"prefill, scale {scale}")
    d = make_batch(name="scd", seq_lens=[150, 40, 260], q_lens=[1, 1, 1], num_heads=16,
                   num_kv_heads=4, head_size=64, block_size=16, scale=scale, seed=78, device=DEV)
    pool = oracle_pool(d)
    gpu_write(d)
    compare(gpu_decode(d), oracle_rows(d, pool), f"decode, scale {scale}")


def test_decode_at_the_largest_batch_the_tables_hold():
    """15 091 sequences (group 4, head size 128) fill the kernel's per-CTA length and
    prefix tables; one more is refused on the host before anything is launched."""
    B = 15091
    g = torch.Generator().manual_seed(31)
    lens = torch.randint(1, 40, (B,), generator=g).tolist()
    b = make_batch(name="maxb", seq_lens=lens, q_lens=[1] * B, num_heads=4, num_kv_heads=1,
                   head_size=128, block_size=16, scale=128 ** -0.5, seed=32, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_decode(b)
    binding.pa_error_check()
    rows = np.arange(0, B, 37, dtype=np.int32)
    compare(out[torch.as_tensor(rows, device=DEV).long()], oracle_rows(b, pool, rows),
            "decode, largest batch (sampled rows)")
    over = torch.cat([b.seq_lens, b.seq_lens[:1]])
    tables = torch.cat([b.block_tables, b.block_tables[:1]])
    q = torch.cat([b.q, b.q[:1]])
    with pytest.raises(binding.PaError) as e:
        binding.pa_decode(torch.empty_like(q), q, b.kv_cache, tables, over, int(over.max()),
                          b.scale, workspace_for(b, B + 1))
    assert e.value.status == 2

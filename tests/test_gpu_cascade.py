"""Parity of the shared-prefix (cascade) decode with the CPU fp64 oracle.

The oracle knows nothing of the cascade: it gathers each sequence's whole
context through its own block table and applies the plain definition, so these
tests check that attending the shared blocks once for the batch and merging
with each sequence's own tokens gives ordinary decode attention.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import (FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of,
                                                make_batch, make_config)
from tests._gpu import bits, compare, gpu_decode, gpu_write, oracle_pool, oracle_rows

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.pa_error_check()
    yield
    binding.pa_error_check()


def gpu_cascade(b, shared_len: int, seq_lens=None) -> torch.Tensor:
    lens = b.seq_lens if seq_lens is None else seq_lens
    out = torch.full_like(b.q, float("nan"))
    nbytes = binding.pa_decode_cascade_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads,
                                                       b.head_size, shared_len)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    binding.pa_decode_cascade(out, b.q, b.kv_cache, b.block_tables, lens, int(lens.max()),
                              shared_len, b.scale, ws)
    return out


CASCADE_SHAPES = [
    # num_seqs, prefix blocks, suffix range, Hq, Hkv, D, bs
    (40, 20, (1, 300), 64, 8, 128, 16),     # group 8: two prefix CTAs, 3 key tiles, ragged
    (7, 9, (1, 40), 8, 8, 128, 16),         # group 1, one short key tile
    (50, 34, (5, 150), 16, 4, 64, 8),       # group 4, block 8, 272 shared tokens
    (33, 8, (1, 100), 24, 8, 128, 32),      # group 3, block 32, 256 shared tokens
    (130, 40, (64, 400), 32, 8, 128, 16),   # many splits over 640 shared tokens
]


@pytest.mark.parametrize("case", range(len(CASCADE_SHAPES)))
def test_cascade_small_shapes(case):
    B, pb, (lo, hi), Hq, Hkv, D, bs = CASCADE_SHAPES[case]
    g = torch.Generator().manual_seed(500 + case)
    suffix = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    lens = [pb * bs + x for x in suffix]
    b = make_batch(name=f"c{case}", seq_lens=lens, q_lens=[1] * B, num_heads=Hq,
                   num_kv_heads=Hkv, head_size=D, block_size=bs, scale=D ** -0.5,
                   seed=600 + case, shared_prefix_blocks=pb, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_cascade(b, pb * bs)
    binding.pa_error_check()
    compare(out, oracle_rows(b, pool), f"cascade case {case}")


def test_cascade_with_sequences_that_have_no_own_tokens():
    """A sequence whose length equals the shared length attends to the prefix only."""
    pb, bs = 12, 16
    b = make_batch(name="cz", seq_lens=[pb * bs + x for x in (5, 70, 1, 33, 9)],
                   q_lens=[1] * 5, num_heads=32, num_kv_heads=8, head_size=128, block_size=bs,
                   scale=128 ** -0.5, seed=71, shared_prefix_blocks=pb, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    lens = b.seq_lens.clone()
    lens[0] = pb * bs
    lens[3] = pb * bs
    out = gpu_cascade(b, pb * bs, lens)
    binding.pa_error_check()
    want = oracle_rows(type(b)(**{**b.__dict__, "seq_lens": lens}), pool)
    compare(out, want, "cascade, empty suffixes")


def test_cascade_without_shared_tokens_is_plain_decode_bitwise():
    b = make_batch(name="c0", seq_lens=[33, 200, 17, 90], q_lens=[1] * 4, num_heads=32,
                   num_kv_heads=8, head_size=128, block_size=16, scale=0.09, seed=72,
                   device=DEV)
    gpu_write(b)
    assert np.array_equal(bits(gpu_cascade(b, 0)), bits(gpu_decode(b)))


def test_cascade_matches_decode_and_is_deterministic():
    b = make_batch(name="cd", seq_lens=[512 + x for x in (100, 3, 250, 64, 1, 77)],
                   q_lens=[1] * 6, num_heads=64, num_kv_heads=8, head_size=128, block_size=16,
                   scale=128 ** -0.5, seed=73, shared_prefix_blocks=32, device=DEV)
    gpu_write(b)
    c1 = gpu_cascade(b, 512)
    c2 = gpu_cascade(b, 512)
    assert np.array_equal(bits(c1), bits(c2))
    d = gpu_decode(b)
    assert (c1.float() - d.float()).abs().max().item() <= 1e-2


def test_cascade_prefix_workload_full_size():
    b = make_config(5, device=DEV)
    pool = oracle_pool(b)
    gpu_write(b)
    out = gpu_cascade(b, b.shared_prefix_blocks * b.block_size)
    binding.pa_error_check()
    compare(out, oracle_rows(b, pool), "prefix-shared workload, cascade")


@pytest.mark.parametrize("fp8", [False, True])
def test_cascade_segments_finished_whole(fp8):
    """Own suffixes of at most 16 tokens: one tile per (sequence, KV head), one tile
    per warp of the small grid, so every segment is finished whole by one warp and
    reaches the output only through its segment record and the merge kernel's fold
    of the prefix partials; two sequences have no own tokens at all."""
    pb, bs = 16, 16
    suffix = [16, 1, 7, 16, 3, 12, 9]
    b = make_batch(name=f"cw{int(fp8)}", seq_lens=[pb * bs + x for x in suffix],
                   q_lens=[1] * len(suffix), num_heads=32, num_kv_heads=8, head_size=128,
                   block_size=bs, scale=128 ** -0.5, seed=75 + fp8, shared_prefix_blocks=pb,
                   device=DEV)
    lens = b.seq_lens.clone()
    lens[2] = pb * bs
    lens[5] = pb * bs
    if fp8:
        out, want, _ = _fp8_case(b, pb * bs, seq_lens=lens)
    else:
        pool = oracle_pool(b)
        gpu_write(b)
        out = gpu_cascade(b, pb * bs, lens)
        binding.pa_error_check()
        want = oracle_rows(type(b)(**{**b.__dict__, "seq_lens": lens}), pool)
    compare(out, want, f"cascade, whole segments{' (FP8)' if fp8 else ''}")


@pytest.mark.parametrize("fp8", [False, True])
def test_cascade_long_own_suffixes(fp8):
    """A short shared prefix and long own suffixes: the shape that runs the prefix
    pass beside the own tokens' decode in one launch (the full prefix-sharing
    workload does too)."""
    pb, bs = 32, 16
    g = torch.Generator().manual_seed(90 + fp8)
    suffix = torch.randint(1, 4097, (48,), generator=g).tolist()
    b = make_batch(name=f"cl{int(fp8)}", seq_lens=[pb * bs + x for x in suffix],
                   q_lens=[1] * len(suffix), num_heads=32, num_kv_heads=8, head_size=128,
                   block_size=bs, scale=128 ** -0.5, seed=91 + fp8, shared_prefix_blocks=pb,
                   device=DEV)
    if fp8:
        out, want, _ = _fp8_case(b, pb * bs)
    else:
        pool = oracle_pool(b)
        gpu_write(b)
        out = gpu_cascade(b, pb * bs)
        binding.pa_error_check()
        want = oracle_rows(b, pool)
    compare(out, want, f"cascade, long own suffixes{' (FP8)' if fp8 else ''}")


def test_cascade_rejects_unaligned_shared_length():
    b = make_batch(name="cu", seq_lens=[40, 50], q_lens=[1, 1], num_heads=8, num_kv_heads=8,
                   head_size=64, block_size=8, scale=0.1, seed=74, shared_prefix_blocks=3,
                   device=DEV)
    with pytest.raises(binding.PaError) as e:
        gpu_cascade(b, 24)  # three blocks of 8: not a multiple of 16
    assert e.value.status == 2


# ----------------------------------------------------------------- FP8 pool

def _fp8_case(b, shared_len, ks=FP8_K_SCALE, vs=FP8_V_SCALE, seq_lens=None):
    """Quantise the batch's K/V into an FP8 pool (the new rows by the CUDA write,
    checked bit-exact against the oracle's), run the FP8 cascade and return it
    with the oracle's plain FP8 decode of the same codes."""
    pool8 = fp8_pool_of(b, ks, vs)
    codes = oracle.cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, ks, vs)
    binding.pa_cache_write_fp8(pool8, b.k_new, b.v_new, b.slot_mapping, ks, vs)
    binding.pa_error_check()
    assert np.array_equal(pool8.cpu().numpy(), codes)
    lens = b.seq_lens if seq_lens is None else seq_lens
    out = torch.full_like(b.q, float("nan"))
    ws = torch.empty(binding.pa_decode_cascade_workspace_bytes(
        b.num_seqs, b.num_heads, b.num_kv_heads, b.head_size, shared_len), dtype=torch.uint8,
        device=DEV)
    binding.pa_decode_cascade(out, b.q, pool8, b.block_tables, lens, int(lens.max()),
                              shared_len, b.scale, ws, kv_scales=(ks, vs))
    binding.pa_error_check()
    want = oracle.attention_fp8(b.q, b.cu_q_lens, codes, ks, vs, b.block_tables, lens,
                                b.num_heads, b.scale)
    return out, want, pool8


@pytest.mark.parametrize("case", [0, 1, 3, 4])
def test_fp8_cascade_small_shapes(case):
    B, pb, (lo, hi), Hq, Hkv, D, bs = CASCADE_SHAPES[case]  # head size 128 cases
    g = torch.Generator().manual_seed(700 + case)
    suffix = torch.randint(lo, hi + 1, (B,), generator=g).tolist()
    lens = [pb * bs + x for x in suffix]
    b = make_batch(name=f"c8{case}", seq_lens=lens, q_lens=[1] * B, num_heads=Hq,
                   num_kv_heads=Hkv, head_size=D, block_size=bs, scale=D ** -0.5,
                   seed=800 + case, shared_prefix_blocks=pb, device=DEV)
    out, want, _ = _fp8_case(b, pb * bs)
    compare(out, want, f"fp8 cascade case {case}")


def test_fp8_cascade_other_scales_and_empty_suffixes():
    pb, bs = 12, 16
    b = make_batch(name="c8z", seq_lens=[pb * bs + x for x in (5, 70, 1, 33, 9)],
                   q_lens=[1] * 5, num_heads=32, num_kv_heads=8, head_size=128, block_size=bs,
                   scale=-0.07, seed=81, shared_prefix_blocks=pb, device=DEV)
    lens = b.seq_lens.clone()
    lens[1] = pb * bs
    out, want, _ = _fp8_case(b, pb * bs, ks=0.2, vs=0.0045, seq_lens=lens)
    compare(out, want, "fp8 cascade, other scales, empty suffixes")


def test_fp8_cascade_matches_fp8_decode():
    b = make_batch(name="c8d", seq_lens=[512 + x for x in (100, 3, 250, 64, 1, 77)],
                   q_lens=[1] * 6, num_heads=64, num_kv_heads=8, head_size=128, block_size=16,
                   scale=128 ** -0.5, seed=83, shared_prefix_blocks=32, device=DEV)
    out, _, pool8 = _fp8_case(b, 512)
    d = torch.full_like(b.q, float("nan"))
    ws = torch.empty(binding.pa_decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads,
                                                       b.head_size), dtype=torch.uint8,
                     device=DEV)
    binding.pa_decode_fp8(d, b.q, pool8, b.block_tables, b.seq_lens, int(b.seq_lens.max()),
                          b.scale, FP8_K_SCALE, FP8_V_SCALE, ws)
    binding.pa_error_check()
    assert (out.float() - d.float()).abs().max().item() <= 1e-2


def test_fp8_cascade_prefix_workload_full_size():
    b = make_config(5, device=DEV)
    out, want, _ = _fp8_case(b, b.shared_prefix_blocks * b.block_size)
    compare(out, want, "prefix-shared workload, FP8 cascade")


@pytest.mark.parametrize("shape", ["whole", "one_launch"])
@pytest.mark.parametrize("fp8", [False, True])
def test_cascade_flags_a_diverging_shared_table(shape, fp8):
    """The shared blocks are read through sequence 0's table; a sequence whose
    shared entries name another block breaks the stated precondition.  The
    kernels compare the entries and pa_error_check reports PA_ERR_PRECONDITION
    (no fault: the other block is a valid pool block)."""
    pb, bs = (16, 16) if shape == "whole" else (32, 16)
    suffix = [16, 1, 7, 16, 3, 12, 9] if shape == "whole" else \
        torch.randint(1, 4097, (48,), generator=torch.Generator().manual_seed(95)).tolist()
    b = make_batch(name=f"cp{shape}{int(fp8)}", seq_lens=[pb * bs + x for x in suffix],
                   q_lens=[1] * len(suffix), num_heads=32, num_kv_heads=8, head_size=128,
                   block_size=bs, scale=128 ** -0.5, seed=96 + fp8, shared_prefix_blocks=pb,
                   device=DEV)
    s = len(suffix) - 2
    b.block_tables[s, pb // 2] = b.block_tables[s, pb]   # one of its own blocks instead
    pool = fp8_pool_of(b) if fp8 else b.kv_cache
    out = torch.empty_like(b.q)
    ws = torch.empty(binding.pa_decode_cascade_workspace_bytes(
        b.num_seqs, b.num_heads, b.num_kv_heads, b.head_size, pb * bs), dtype=torch.uint8,
        device=DEV)
    binding.pa_decode_cascade(out, b.q, pool, b.block_tables, b.seq_lens, b.max_seq_len,
                              pb * bs, b.scale, ws,
                              kv_scales=(FP8_K_SCALE, FP8_V_SCALE) if fp8 else None)
    with pytest.raises(binding.PaError) as e:
        binding.pa_error_check()
    assert binding.STATUS[e.value.status] == "PA_ERR_PRECONDITION"
    # The same call on the intact tables reports nothing.
    b.block_tables[s, pb // 2] = b.block_tables[0, pb // 2]
    binding.pa_decode_cascade(out, b.q, pool, b.block_tables, b.seq_lens, b.max_seq_len,
                              pb * bs, b.scale, ws,
                              kv_scales=(FP8_K_SCALE, FP8_V_SCALE) if fp8 else None)
    binding.pa_error_check()


@pytest.mark.parametrize("fp8", [False, True])
def test_cascade_where_the_prefix_pass_arrives_last(fp8):
    """One long own suffix makes the host run the prefix pass beside the own
    tokens' decode in one launch; the other 63 sequences own 1-16 tokens, which
    the decode finishes within microseconds, long before the prefix pass over
    2048 shared tokens ends.  The merge kernel, a programmatic dependent of that
    launch, then merges every segment (the long sequence's, split over many
    decode warps, included): deterministic and equal to the oracle."""
    pb, bs = 128, 16
    g = torch.Generator().manual_seed(97)
    suffix = [8192] + torch.randint(1, 17, (63,), generator=g).tolist()
    b = make_batch(name=f"cpl{int(fp8)}", seq_lens=[pb * bs + x for x in suffix],
                   q_lens=[1] * len(suffix), num_heads=32, num_kv_heads=8, head_size=128,
                   block_size=bs, scale=128 ** -0.5, seed=98 + fp8, shared_prefix_blocks=pb,
                   device=DEV)
    if fp8:
        out, want, pool8 = _fp8_case(b, pb * bs)
        again = torch.full_like(b.q, float("nan"))
        ws = torch.empty(binding.pa_decode_cascade_workspace_bytes(
            b.num_seqs, b.num_heads, b.num_kv_heads, b.head_size, pb * bs), dtype=torch.uint8,
            device=DEV)
        binding.pa_decode_cascade(again, b.q, pool8, b.block_tables, b.seq_lens, b.max_seq_len,
                                  pb * bs, b.scale, ws, kv_scales=(FP8_K_SCALE, FP8_V_SCALE))
        binding.pa_error_check()
    else:
        pool = oracle_pool(b)
        gpu_write(b)
        out = gpu_cascade(b, pb * bs)
        again = gpu_cascade(b, pb * bs)
        binding.pa_error_check()
        want = oracle_rows(b, pool)
    assert np.array_equal(bits(out), bits(again))
    compare(out, want, f"cascade, prefix pass last{' (FP8)' if fp8 else ''}")


@pytest.mark.parametrize("fp8", [False, True])
def test_cascade_with_the_prefix_keys_split_in_the_one_launch(fp8):
    """A 4096-token shared prefix and own suffixes of up to 1024 tokens (2048 from
    an FP8 pool, whose decode streams half the bytes), Llama-3-70B heads: the host
    balances the long prefix pass against the own tokens' decode by splitting the
    prefix keys over two CTAs per row group in the one launch, so every segment
    merges two prefix partials with its decode pieces."""
    pb, bs = 256, 16
    g = torch.Generator().manual_seed(99)
    suffix = torch.randint(64, 2049 if fp8 else 1025, (128,), generator=g).tolist()
    b = make_batch(name=f"cs{int(fp8)}", seq_lens=[pb * bs + x for x in suffix],
                   q_lens=[1] * len(suffix), num_heads=64, num_kv_heads=8, head_size=128,
                   block_size=bs, scale=128 ** -0.5, seed=100 + fp8, shared_prefix_blocks=pb,
                   device=DEV)
    assert binding.lib().pa_decode_cascade_kernels(b.num_seqs, 64, 8, 128, bs, b.max_seq_len,
                                                   pb * bs, int(fp8)) == 2
    if fp8:
        out, want, _ = _fp8_case(b, pb * bs)
    else:
        pool = oracle_pool(b)
        gpu_write(b)
        out = gpu_cascade(b, pb * bs)
        binding.pa_error_check()
        want = oracle_rows(b, pool)
    compare(out, want, f"cascade, split prefix keys{' (FP8)' if fp8 else ''}")

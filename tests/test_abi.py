"""The C ABI library loads, exports every declared symbol, and rejects bad host
arguments before touching the GPU (no compute calls; runs without a GPU)."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

from paged_kv_cache_287_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from paged_kv_cache_287_gb300 import build
        build.build()
    return binding.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    return set(re.findall(r"^\S[^;(]*?\b(pa_[a-z_0-9]+)\s*\(", src, re.M))


def test_header_and_binding_agree():
    assert _declared() == set(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_block_bytes_formula(lib):
    assert lib.pa_kv_block_bytes(16, 4, 64) == 16384
    assert lib.pa_kv_block_bytes(16, 8, 128) == 65536
    assert lib.pa_kv_block_bytes(0, 8, 128) == 0


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert lib.pa_status_string(code).decode() == name


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every call below fails host checks


def test_cache_write_host_checks(lib):
    ok = (FAKE, 10, 16, 8, 128, FAKE, FAKE, 8 * 128, FAKE, 4, None)
    assert lib.pa_cache_write(None, *ok[1:]) == 1                      # null pool
    assert lib.pa_cache_write(FAKE + 2, *ok[1:]) == 1                  # misaligned pool
    assert lib.pa_cache_write(FAKE, 10, 16, 8, 96, *ok[5:]) == 2       # head_size 96
    assert lib.pa_cache_write(FAKE, 10, 12, 8, 128, *ok[5:]) == 2      # block_size 12
    assert lib.pa_cache_write(*ok[:7], 100, *ok[8:]) == 1              # row stride too small
    assert lib.pa_cache_write(*ok[:9], -1, None) == 1                  # negative count
    assert lib.pa_cache_write(*ok[:9], 0, None) == 0                   # empty: no-op


def test_decode_host_checks(lib):
    args = [FAKE, FAKE, FAKE, 10, 16, 32, 8, 128, FAKE, 4, FAKE, 3, 64, 0.1, FAKE, 1 << 30, None]
    bad = list(args)
    bad[6] = 5                                  # 32 heads over 5 kv heads
    assert lib.pa_decode(*bad) == 1
    bad = list(args)
    bad[5], bad[6] = 64, 4                      # group 16 unsupported
    assert lib.pa_decode(*bad) == 2
    bad = list(args)
    bad[13] = float("nan")
    assert lib.pa_decode(*bad) == 1
    bad = list(args)
    bad[12] = 4 * 16 + 1                        # max_seq_len beyond the table
    assert lib.pa_decode(*bad) == 1
    bad = list(args)
    bad[11] = 0                                 # no sequences: no-op
    assert lib.pa_decode(*bad) == 0


def test_prefill_host_checks(lib):
    args = [FAKE, FAKE, FAKE, 2, 64, FAKE, 10, 16, 32, 8, 128, FAKE, 4, FAKE, 0.1, None]
    bad = list(args)
    bad[10] = 256
    assert lib.pa_prefill_chunk(*bad) == 2
    bad = list(args)
    bad[1] = FAKE + 8                           # misaligned q
    assert lib.pa_prefill_chunk(*bad) == 1
    bad = list(args)
    bad[4] = 0                                  # empty: no-op
    assert lib.pa_prefill_chunk(*bad) == 0


def test_cascade_host_checks(lib):
    args = [FAKE, FAKE, FAKE, 10, 16, 32, 8, 128, FAKE, 4, FAKE, 3, 64, 32, 0.1, FAKE, 1 << 30,
            None]
    bad = list(args)
    bad[13] = 65                                # shared_len beyond max_seq_len
    assert lib.pa_decode_cascade(*bad) == 1
    bad = list(args)
    bad[13] = 8                                 # not a multiple of 16
    assert lib.pa_decode_cascade(*bad) == 2
    bad = list(args)
    bad[13] = -16
    assert lib.pa_decode_cascade(*bad) == 1
    bad = list(args)
    bad[11] = 0                                 # no sequences: no-op
    assert lib.pa_decode_cascade(*bad) == 0
    assert lib.pa_decode_cascade_workspace_bytes(0, 32, 8, 128, 64) == 0
    # The FP8 form: the same checks, plus head size 128 only and positive scales.
    a8 = args[:15] + [0.5, 0.25] + args[15:]
    bad = list(a8)
    bad[13] = 8
    assert lib.pa_decode_cascade_fp8(*bad) == 2
    bad = list(a8)
    bad[7] = 64                                 # head_size 64 is bf16-only
    assert lib.pa_decode_cascade_fp8(*bad) == 2
    bad = list(a8)
    bad[16] = 0.0                               # v_scale must be > 0
    assert lib.pa_decode_cascade_fp8(*bad) == 1
    bad = list(a8)
    bad[15] = float("inf")                      # k_scale must be finite
    assert lib.pa_decode_cascade_fp8(*bad) == 1
    bad = list(a8)
    bad[11] = 0                                 # no sequences: no-op
    assert lib.pa_decode_cascade_fp8(*bad) == 0


def test_cascade_kernel_count_query(lib):
    q = lib.pa_decode_cascade_kernels
    assert q(0, 32, 8, 128, 16, 64, 32, 0) == 0            # no sequences: nothing launched
    # No shared tokens: pa_decode, one launch when every (sequence, KV head) gets an
    # SM and is at most 12 tiles long (one tile per warp), else split + merge.
    assert q(1, 8, 1, 128, 16, 192, 0, 0) == 1             # one segment of 12 tiles
    assert q(1, 8, 1, 128, 16, 193, 0, 0) == 2             # 13 tiles
    assert q(5, 32, 8, 128, 16, 4096, 0, 0) == 2
    assert q(5, 32, 8, 128, 16, 64, 0, 0) in (1, 2)        # 40 segments: the SM count decides
    assert q(5, 32, 8, 128, 16, 64, 32, 0) in (2, 3)       # depends on the device's SMs
    assert q(5, 32, 8, 128, 16, 64, 32, 1) in (2, 3)       # FP8 pool: the same choice
    assert q(5, 32, 8, 128, 16, 64, 65, 0) == -1           # shared_len beyond max_seq_len
    assert q(5, 30, 8, 128, 16, 64, 32, 0) == -1           # heads not a multiple
    assert q(5, 32, 8, 96, 16, 64, 32, 0) == -1            # head size
    assert q(5, 32, 8, 128, 12, 64, 32, 0) == -1           # block size
    assert q(-1, 32, 8, 128, 16, 64, 32, 0) == -1


def test_fp8_host_checks(lib):
    wr = [FAKE, 10, 16, 8, 128, FAKE, FAKE, 8 * 128, FAKE, 4, 0.5, 0.25, None]
    bad = list(wr)
    bad[10] = 0.0                               # k_scale must be > 0
    assert lib.pa_cache_write_fp8(*bad) == 1
    bad = list(wr)
    bad[11] = float("nan")
    assert lib.pa_cache_write_fp8(*bad) == 1
    bad = list(wr)
    bad[9] = 0                                  # empty: no-op
    assert lib.pa_cache_write_fp8(*bad) == 0
    dec = [FAKE, FAKE, FAKE, 10, 16, 32, 8, 128, FAKE, 4, FAKE, 3, 64, 0.1, 0.5, 0.5, FAKE,
           1 << 30, None]
    bad = list(dec)
    bad[7] = 64                                 # head_size 64 is bf16-only
    assert lib.pa_decode_fp8(*bad) == 2
    bad = list(dec)
    bad[15] = -1.0                              # v_scale must be > 0
    assert lib.pa_decode_fp8(*bad) == 1
    bad = list(dec)
    bad[11] = 0                                 # no sequences: no-op
    assert lib.pa_decode_fp8(*bad) == 0
    assert lib.pa_kv_block_bytes_dtype(16, 8, 128, 1) == 32768
    assert lib.pa_kv_block_bytes_dtype(16, 8, 128, 2) == lib.pa_kv_block_bytes(16, 8, 128)


def test_varlen_host_checks(lib):
    args = [FAKE, FAKE, None, None, None, FAKE, 4, 2, 100, 64, FAKE, 10, 16, 32, 8, 128, FAKE, 4,
            FAKE, 64, 0.1, FAKE, 1 << 30, None]
    bad = list(args)
    bad[7] = 5                                  # more chunk sequences than sequences
    assert lib.pa_attention_varlen(*bad) == 1
    bad = list(args)
    bad[8] = 1                                  # fewer chunk rows than chunk sequences
    assert lib.pa_attention_varlen(*bad) == 1
    bad = list(args)
    bad[7], bad[8] = 0, 3                       # chunk rows without chunk sequences
    assert lib.pa_attention_varlen(*bad) == 1
    bad = list(args)
    bad[6] = 0                                  # empty batch: no-op
    bad[7] = bad[8] = 0
    assert lib.pa_attention_varlen(*bad) == 0
    assert lib.pa_attention_varlen_workspace_bytes(4, 5, 32, 8, 128) == 0


def test_varlen_checks_everything_before_enqueueing(lib):
    """A fault in the attention arguments is caught before the step's cache write
    is enqueued: with valid write arguments and a misaligned cu_q_lens, the call
    returns PA_ERR_INVALID_ARG (it would be PA_ERR_CUDA here, with no GPU, had the
    write been launched first)."""
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, 4, 2, 100, 64, FAKE, 10, 16, 32, 8, 128,
            FAKE, 4, FAKE, 64, 0.1, FAKE, 1 << 30, None]
    assert lib.pa_attention_varlen(*args) == 1
    a8 = args[:21] + [0.5, 0.5] + args[21:]
    assert lib.pa_attention_varlen_fp8(*a8) == 1
    bad = list(args)
    bad[5] = FAKE
    bad[21] = FAKE + 64                         # workspace not 256-byte aligned
    assert lib.pa_attention_varlen(*bad) == 6


def _packed(lib, args, kv8=0, k_scale=1.0, v_scale=1.0):
    """pa_attention_varlen's argument list (as in the tests above) through
    pa_attention_varlen_packed."""
    (out, q, kn, vn, sm, cu, B, npf, npt, mq, kv, NB, bs, Hq, Hkv, D, bt, mb, sl, ml, scale, ws,
     wsb, stream) = args
    buf = ctypes.create_string_buffer(lib.pa_varlen_args_bytes())
    binding.VARLEN_ARGS.pack_into(buf, 0, out or 0, q or 0, kn or 0, vn or 0, sm or 0, cu or 0,
                                  kv or 0, bt or 0, sl or 0, ws or 0, wsb, stream or 0, B, npf,
                                  npt, mq, NB, bs, Hq, Hkv, D, mb, ml, kv8, scale, k_scale,
                                  v_scale)
    return lib.pa_attention_varlen_packed(ctypes.addressof(buf))


def test_packed_varlen_layout_and_host_checks(lib):
    """The packed struct's layout (12 eight-byte fields, 12 int32, 3 float) and
    the same statuses as the unpacked calls, each decided by a different field."""
    assert lib.pa_varlen_args_bytes() == 160 and binding.VARLEN_ARGS.size == 156
    assert lib.pa_attention_varlen_packed(None) == 1
    args = [FAKE, FAKE, None, None, None, FAKE, 4, 2, 100, 64, FAKE, 10, 16, 32, 8, 128, FAKE, 4,
            FAKE, 64, 0.1, FAKE, 1 << 30, None]
    for i, v in ((7, 5), (8, 1)):               # num_prefills > num_seqs; too few chunk rows
        bad = list(args)
        bad[i] = v
        assert _packed(lib, bad) == lib.pa_attention_varlen(*bad) == 1
    bad = list(args)
    bad[6] = bad[7] = bad[8] = 0                # empty batch: no-op
    assert _packed(lib, bad) == 0
    w = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, 4, 2, 100, 64, FAKE, 10, 16, 32, 8, 128, FAKE, 4,
         FAKE, 64, 0.1, FAKE, 1 << 30, None]
    assert _packed(lib, w) == 1                 # misaligned cu_q_lens
    assert _packed(lib, w, kv8=1, k_scale=0.5, v_scale=0.5) == 1
    bad = list(w)
    bad[5] = FAKE
    bad[21] = FAKE + 64                         # workspace not 256-byte aligned
    assert _packed(lib, bad) == lib.pa_attention_varlen(*bad) == 6
    small = list(w)
    small[5] = FAKE
    small[22] = 1                               # workspace too small: all else valid
    assert _packed(lib, small) == lib.pa_attention_varlen(*small) == 6
    assert _packed(lib, small, kv8=1, k_scale=0.5, v_scale=0.5) == 6
    assert _packed(lib, small, kv8=1, k_scale=0.0, v_scale=0.5) == 1   # scales must be > 0
    assert _packed(lib, small, kv8=1, k_scale=0.5, v_scale=-1.0) == 1
    bad = list(small)
    bad[15] = 64                                # FP8 pool: head size 128 only
    assert _packed(lib, bad, kv8=1, k_scale=0.5, v_scale=0.5) == 2
    assert _packed(lib, bad) == 6               # a bf16 pool takes head size 64


def test_varlen_binding_checks_its_tensors_before_the_call(lib):
    """The binding's one-expression check of every tensor falls back to the
    argument-by-argument checks, which name the tensor at fault (here: host
    tensors, so no call reaches the library)."""
    import torch
    from paged_kv_cache_287_gb300.workloads import make_config
    b = make_config(1, device="cpu")
    ws = torch.empty(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="kv_cache must be a CUDA tensor"):
        binding.pa_attention_varlen(torch.empty_like(b.q), b.q, b.k_new, b.v_new,
                                    b.slot_mapping, b.cu_q_lens[:1].contiguous(), 0, 0, 0,
                                    b.kv_cache, b.block_tables, b.seq_lens, 80, b.scale, ws)
    with pytest.raises(ValueError, match="kv_scales"):
        binding.pa_attention_varlen(torch.empty_like(b.q), b.q, None, None, None,
                                    b.cu_q_lens[:1].contiguous(), 0, 0, 0,
                                    b.kv_cache.view(torch.uint8)[..., :64], b.block_tables,
                                    b.seq_lens, 80, b.scale, ws)

"""The unified call over a flattened mixed batch (pa_attention_varlen): the
step's cache write, its prefill chunks and its decode tokens in one call,
checked against the oracle's write and attention of the same flattened batch."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import make_batch, make_config
from tests._gpu import (bits, compare, gpu_decode, gpu_prefill, gpu_write, oracle_pool,
                        oracle_rows)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _clean_errors():
    binding.pa_error_check()
    yield
    binding.pa_error_check()


def varlen(b, num_prefills: int, write: bool = True) -> torch.Tensor:
    out = torch.full_like(b.q, float("nan"))
    npt = int(b.cu_q_lens[num_prefills])
    max_q = int(b.q_lens[:num_prefills].max()) if num_prefills else 0
    dec_lens = b.seq_lens[num_prefills:]
    max_len = int(dec_lens.max()) if dec_lens.numel() else 0
    ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, num_prefills, b.num_heads, b.num_kv_heads, b.head_size) or 1,
        dtype=torch.uint8, device=DEV)
    binding.pa_attention_varlen(out, b.q, b.k_new if write else None,
                                b.v_new if write else None, b.slot_mapping if write else None,
                                b.cu_q_lens[:num_prefills + 1].contiguous(), num_prefills, npt,
                                max_q, b.kv_cache, b.block_tables, b.seq_lens, max_len, b.scale,
                                ws)
    binding.pa_error_check()
    return out


@pytest.mark.parametrize("shape", [
    # seq_lens, q_lens (chunks first), Hq, Hkv, D, bs
    ([300, 40, 513, 90, 17, 1], [129, 40, 200, 1, 1, 1], 32, 8, 128, 16),
    ([64, 700, 33], [64, 1, 1], 16, 4, 64, 8),
    ([150, 260], [70, 129], 8, 2, 128, 32),      # chunks only
    ([5, 99, 1000], [1, 1, 1], 24, 8, 128, 16),  # decode tokens only
])
def test_varlen_small_batches(shape):
    lens, qls, Hq, Hkv, D, bs = shape
    b = make_batch(name="v", seq_lens=lens, q_lens=qls, num_heads=Hq, num_kv_heads=Hkv,
                   head_size=D, block_size=bs, scale=D ** -0.5, seed=900 + len(lens),
                   device=DEV)
    n_pre = sum(1 for q in qls if q > 1) if any(q > 1 for q in qls) else 0
    pool = oracle_pool(b)
    out = varlen(b, n_pre)
    assert np.array_equal(bits(b.kv_cache), pool), "cache write"
    compare(out, oracle_rows(b, pool), f"varlen {lens}")


def test_varlen_more_chunks_than_the_ranking_holds():
    """270 prefill chunks (more than the 256 the kernel ranks by context) and 10
    decode tokens in one call."""
    g = np.random.default_rng(79)
    qls = [int(x) for x in g.integers(2, 20, 270)] + [1] * 10
    lens = [q + int(c) for q, c in zip(qls, g.integers(0, 300, 280))]
    b = make_batch(name="v280", seq_lens=lens, q_lens=qls, num_heads=16, num_kv_heads=4,
                   head_size=128, block_size=16, scale=128 ** -0.5, seed=80, device=DEV)
    pool = oracle_pool(b)
    out = varlen(b, 270)
    assert np.array_equal(bits(b.kv_cache), pool), "cache write"
    compare(out, oracle_rows(b, pool), "varlen, 270 chunks + 10 decode tokens")


def test_varlen_mixed_workload_one_launch():
    """Chunks and decode tokens in one launch: the chunk rows equal the separate
    prefill call bit for bit (same kernel body), the decode rows match the oracle
    (their context split differs from the separate call's), and the call is
    deterministic."""
    b = make_config(4, device=DEV)
    pool = oracle_pool(b)
    out = varlen(b, 8)
    assert np.array_equal(bits(b.kv_cache), pool), "cache write"
    again = varlen(b, 8)
    assert np.array_equal(bits(out), bits(again)), "deterministic"
    pre = gpu_prefill(b, 0, 8)
    assert np.array_equal(bits(out[:4096]), bits(pre))
    dec = gpu_decode(b, 8, b.num_seqs)
    assert (out[4096:].float() - dec.float()).abs().max().item() <= 1e-2
    rows = np.concatenate([np.arange(0, 4096, 97), np.arange(4096, 4344)]).astype(np.int32)
    compare(out[torch.as_tensor(rows, device=DEV).long()], oracle_rows(b, pool, rows),
            "mixed workload, unified call (sampled chunk rows, every decode row)")


def test_varlen_split_from_the_write_launch_equals_its_own_launch():
    """With a cache write in the call, the split of the mixed launch's SMs is
    computed by one extra block of the write's launch; without one, by a launch
    of its own.  Both compute the same split (256-thread blocks at 8 KV heads of
    128), so the rows are equal bit for bit."""
    a = make_config(4, device=DEV)
    b = make_config(4, device=DEV)
    out_a = varlen(a, 8)
    gpu_write(b)
    out_b = varlen(b, 8, write=False)
    assert np.array_equal(bits(a.kv_cache), bits(b.kv_cache)), "same pool"
    assert np.array_equal(bits(out_a), bits(out_b))


@pytest.mark.parametrize("num_seqs", [4, 300])
def test_varlen_decode_reads_the_tokens_its_call_just_wrote(num_seqs):
    """Decode tokens only: the decode starts as a programmatic dependent of the
    cache write and must read the pool only after that write completes.  With
    one token per sequence the softmax has a single key, so each query head's
    row is exactly its KV head's new V row; fresh V rows every call show a stale
    read at once.  4 sequences: one CTA per (sequence, KV head); 300: the split
    kernel and its merge kernel."""
    b = make_batch(name=f"vw{num_seqs}", seq_lens=[1] * num_seqs, q_lens=[1] * num_seqs,
                   num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                   scale=128 ** -0.5, seed=990 + num_seqs, device=DEV)
    G = b.num_heads // b.num_kv_heads
    g = torch.Generator(device="cpu").manual_seed(num_seqs)
    for it in range(12):
        b.k_new.copy_(torch.randn(b.k_new.shape, generator=g).to(torch.bfloat16))
        b.v_new.copy_(torch.randn(b.v_new.shape, generator=g).to(torch.bfloat16))
        out = varlen(b, 0)
        want = b.v_new.repeat_interleave(G, dim=1)  # [N, Hq, D]
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), f"call {it}"


@pytest.mark.parametrize("n_dec", [1, 31, 600])
def test_varlen_one_launch_decode_counts(n_dec):
    """From one decode sequence (one decode CTA busy) to many."""
    g = torch.Generator().manual_seed(n_dec)
    dec = torch.randint(1, 3000, (n_dec,), generator=g).tolist()
    lens = [700, 1300] + dec
    qls = [300, 57] + [1] * n_dec
    b = make_batch(name=f"vd{n_dec}", seq_lens=lens, q_lens=qls, num_heads=32, num_kv_heads=8,
                   head_size=128, block_size=16, scale=128 ** -0.5, seed=960 + n_dec,
                   device=DEV)
    pool = oracle_pool(b)
    out = varlen(b, 2)
    rows = np.concatenate([np.arange(0, 357, 11), 357 + np.arange(0, n_dec, max(1, n_dec // 60))])
    rows = rows.astype(np.int32)
    compare(out[torch.as_tensor(rows, device=DEV).long()], oracle_rows(b, pool, rows),
            f"one launch, {n_dec} decode sequences")


@pytest.mark.parametrize("n_dec", [3, 240])
def test_varlen_one_launch_group_8(n_dec):
    """Eight query heads per KV head at head size 128: the decode role's twelve
    two-stage rings do not fit the launch's shared memory, so it runs eleven
    warps; the step is still one attention launch (the plan in the workspace is
    written) and matches the oracle."""
    g = torch.Generator().manual_seed(70 + n_dec)
    dec = torch.randint(1, 2500, (n_dec,), generator=g).tolist()
    lens = [900, 260] + dec
    qls = [256, 129] + [1] * n_dec
    b = make_batch(name=f"vg8_{n_dec}", seq_lens=lens, q_lens=qls, num_heads=64,
                   num_kv_heads=8, head_size=128, block_size=16, scale=128 ** -0.5,
                   seed=970 + n_dec, device=DEV)
    pool = oracle_pool(b)
    nb = binding.pa_attention_varlen_workspace_bytes(b.num_seqs, 2, 64, 8, 128)
    ws = torch.full((nb,), 255, dtype=torch.uint8, device=DEV)  # plan slots read -1
    out = torch.full_like(b.q, float("nan"))
    npt = int(b.cu_q_lens[2])
    binding.pa_attention_varlen(out, b.q, b.k_new, b.v_new, b.slot_mapping,
                                b.cu_q_lens[:3].contiguous(), 2, npt, 256, b.kv_cache,
                                b.block_tables, b.seq_lens, max(dec), b.scale, ws)
    binding.pa_error_check()
    plan = ws[nb - 256:nb - 248].view(torch.int32).tolist()
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert 1 <= plan[0] < sms and plan[1] == 11 * plan[0], plan
    assert np.array_equal(bits(b.kv_cache), pool)
    rows = np.concatenate([np.arange(0, npt, 7), npt + np.arange(0, n_dec, max(1, n_dec // 50))])
    rows = rows.astype(np.int32)
    compare(out[torch.as_tensor(rows, device=DEV).long()], oracle_rows(b, pool, rows),
            f"one launch, group 8, {n_dec} decode sequences")


def test_varlen_without_slot_mapping_writes_nothing():
    b = make_batch(name="vn", seq_lens=[40, 20], q_lens=[8, 1], num_heads=8, num_kv_heads=2,
                   head_size=128, block_size=16, scale=0.1, seed=950, device=DEV)
    binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping)
    before = bits(b.kv_cache).copy()
    b.k_new.fill_(7.0)
    varlen(b, 1, write=False)
    assert np.array_equal(bits(b.kv_cache), before)


@pytest.mark.parametrize("fp8", [False, True])
def test_varlen_host_fault_leaves_the_pool_untouched(fp8):
    """Every host check runs before the step's cache write is enqueued: with valid
    write arguments and a misaligned cu_q_lens pointer, the call returns
    PA_ERR_INVALID_ARG and the pool keeps every byte it had."""
    import ctypes
    b = make_batch(name="vs", seq_lens=[300, 40, 513, 90], q_lens=[129, 40, 1, 1],
                   num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
                   scale=128 ** -0.5, seed=977, device=DEV)
    pool = torch.full((b.num_blocks, 2, 8, 16, 128), 0x5A, dtype=torch.uint8, device=DEV) \
        if fp8 else torch.full_like(b.kv_cache, 3.25)
    before = pool.clone()
    out = torch.zeros_like(b.q)
    cu = b.cu_q_lens[:3].contiguous()
    ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, 2, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8, device=DEV)
    L = binding.lib()
    args = [out.data_ptr(), b.q.data_ptr(), b.k_new.data_ptr(), b.v_new.data_ptr(),
            b.slot_mapping.data_ptr(), cu.data_ptr() + 2, b.num_seqs, 2, int(b.cu_q_lens[2]),
            129, pool.data_ptr(), b.num_blocks, 16, 32, 8, 128, b.block_tables.data_ptr(),
            b.block_tables.shape[1], b.seq_lens.data_ptr(), int(b.seq_lens.max()),
            ctypes.c_float(b.scale)]
    tail = [ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream]
    if fp8:
        status = L.pa_attention_varlen_fp8(*args, ctypes.c_float(1 / 64), ctypes.c_float(1 / 64),
                                           *tail)
    else:
        status = L.pa_attention_varlen(*args, *tail)
    torch.cuda.synchronize()
    assert binding.STATUS[status] == "PA_ERR_INVALID_ARG"
    assert torch.equal(pool.view(torch.uint8), before.view(torch.uint8))


@pytest.mark.parametrize("fp8", [False, True])
def test_unpacked_and_packed_entry_points_agree_bitwise(fp8):
    """pa_attention_varlen(_fp8) with its 24 (26) arguments and
    pa_attention_varlen_packed (which the binding calls) run the same step: the
    same pool bytes and the same output bits, chunks and decode tokens in one
    launch."""
    import ctypes
    from paged_kv_cache_287_gb300.workloads import FP8_K_SCALE, FP8_V_SCALE, fp8_pool_of
    lens, qls = [300, 40, 513, 90, 17, 1], [129, 40, 1, 1, 1, 1]
    kw = dict(name="vpk", seq_lens=lens, q_lens=qls, num_heads=32, num_kv_heads=8,
              head_size=128, block_size=16, scale=128 ** -0.5, seed=981, device=DEV)
    outs, pools = [], []
    for packed in (False, True):
        b = make_batch(**kw)
        pool = fp8_pool_of(b) if fp8 else b.kv_cache
        cu = b.cu_q_lens[:3].contiguous()
        npt = int(b.cu_q_lens[2])
        max_dec = int(b.seq_lens[2:].max())
        ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
            b.num_seqs, 2, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8,
            device=DEV)
        out = torch.full_like(b.q, float("nan"))
        if packed:
            kv = {"kv_scales": (FP8_K_SCALE, FP8_V_SCALE)} if fp8 else {}
            binding.pa_attention_varlen(out, b.q, b.k_new, b.v_new, b.slot_mapping, cu, 2, npt,
                                        129, pool, b.block_tables, b.seq_lens, max_dec,
                                        b.scale, ws, **kv)
        else:
            L = binding.lib()
            args = [out.data_ptr(), b.q.data_ptr(), b.k_new.data_ptr(), b.v_new.data_ptr(),
                    b.slot_mapping.data_ptr(), cu.data_ptr(), b.num_seqs, 2, npt, 129,
                    pool.data_ptr(), b.num_blocks, 16, 32, 8, 128, b.block_tables.data_ptr(),
                    b.block_tables.shape[1], b.seq_lens.data_ptr(), max_dec,
                    ctypes.c_float(b.scale)]
            tail = [ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream]
            if fp8:
                st = L.pa_attention_varlen_fp8(*args, ctypes.c_float(FP8_K_SCALE),
                                               ctypes.c_float(FP8_V_SCALE), *tail)
            else:
                st = L.pa_attention_varlen(*args, *tail)
            assert st == 0
        binding.pa_error_check()
        outs.append(out)
        pools.append(pool)
    assert torch.equal(pools[0].view(torch.uint8), pools[1].view(torch.uint8))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_varlen_binding_names_the_tensor_at_fault():
    """Wrong shapes, dtypes or layouts raise ValueError before any launch."""
    b = make_batch(name="vbad", seq_lens=[40, 20], q_lens=[8, 1], num_heads=8, num_kv_heads=2,
                   head_size=128, block_size=16, scale=0.1, seed=951, device=DEV)
    ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(2, 1, 8, 2, 128),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty_like(b.q)
    cu = b.cu_q_lens[:2].contiguous()

    def call(**kw):
        a = dict(out=out, q=b.q, k_new=b.k_new, v_new=b.v_new, slot_mapping=b.slot_mapping)
        a.update(kw)
        binding.pa_attention_varlen(a["out"], a["q"], a["k_new"], a["v_new"], a["slot_mapping"],
                                    cu, 1, 8, 8, b.kv_cache, b.block_tables, b.seq_lens, 20,
                                    b.scale, ws)

    with pytest.raises(ValueError, match="one row per query row"):
        call(k_new=b.k_new[:-1])
    with pytest.raises(ValueError, match="slot_mapping must be torch.int32"):
        call(slot_mapping=b.slot_mapping.long())
    with pytest.raises(ValueError, match="q must be contiguous"):
        call(q=b.q.transpose(0, 1).contiguous().transpose(0, 1))
    with pytest.raises(ValueError, match="inconsistent varlen shapes"):
        call(out=out[:-1])
    binding.pa_error_check()

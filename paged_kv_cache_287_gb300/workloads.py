"""Seeded synthetic inputs for attention over a paged KV cache.

This module only draws random numbers and lays out who owns which block. It
holds none of the attention or cache-write arithmetic; both the CUDA path and
the CPU oracle consume what it returns.

Shapes follow "Inside vLLM: Anatomy of a High-Throughput LLM Inference System"
(§Engine core: a pool of free KV blocks that a sequence reaches through its
block table; §Block size: blocks of ``block_size`` tokens, 16 by default, bf16
at 2 bytes; §Generate function: the forward pass sees the whole batch as one
flattened token sequence).

Conventions shared by both sides (the pages leave them open):

* ``kv_cache`` is bf16 ``[num_blocks, 2, num_kv_heads, block_size, head_size]``:
  index 0 of the second axis holds K, index 1 holds V, so one physical block is
  one contiguous run of ``2*block_size*num_kv_heads*head_size*2`` bytes.
* Sequence ``s`` owns ``seq_lens[s]`` tokens, in logical order, in the blocks
  ``block_tables[s, 0..ceil(seq_lens[s]/block_size)-1]``; unused table entries
  are -1.
* Each sequence has ``q_len`` new tokens at positions
  ``seq_lens[s]-q_len .. seq_lens[s]-1``.  Their K/V (``k_new``/``v_new``, one
  row per query row) are not yet in the pool; ``slot_mapping`` gives each new
  row's slot ``block*block_size + offset``.  Decode is the case ``q_len = 1``.
* Every pool element that no live token owns, including the slots of the new
  tokens before they are written, holds NaN, so a read of stale data shows.

Values are N(0,1) drawn in fp32 and rounded to bf16 (round to nearest even).
Metadata (lengths, placement) always comes from a CPU generator, so it is the
same on every machine; the large value tensors may be drawn on a CUDA device
for speed, in which case they differ from a CPU draw but are still seeded.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

__all__ = ["PagedBatch", "make_batch", "make_config", "config_spec", "sample_of_config",
           "CONFIG_NAMES", "config_seed"]

CONFIG_NAMES = {
    1: "tiny-decode-tinyllama-b4",
    2: "llama3-8b-decode-b256",
    3: "long-skewed-decode-b32",
    4: "mixed-prefill8x512-decode248",
    5: "prefix-shared-decode-llama3-70b-b128",
}


def config_seed(n: int) -> int:
    """Seed of numbered workload ``n`` (287 + n)."""
    return 287 + n


@dataclass
class PagedBatch:
    """One flattened batch over a paged KV cache (all tensors on one device)."""

    name: str
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    scale: float
    kv_cache: torch.Tensor      # bf16 [num_blocks, 2, Hkv, bs, D]; new slots not yet written
    block_tables: torch.Tensor  # int32 [B, max_blocks_per_seq], -1 padded
    seq_lens: torch.Tensor      # int32 [B], tokens including the new ones
    q_lens: torch.Tensor        # int32 [B], new tokens (= query rows) per sequence
    cu_q_lens: torch.Tensor     # int32 [B+1], prefix sum of q_lens
    q: torch.Tensor             # bf16 [sum(q_lens), Hq, D]
    k_new: torch.Tensor         # bf16 [sum(q_lens), Hkv, D]
    v_new: torch.Tensor         # bf16 [sum(q_lens), Hkv, D]
    slot_mapping: torch.Tensor  # int32 [sum(q_lens)]
    shared_prefix_blocks: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.num_seqs else 0

    def to(self, device) -> "PagedBatch":
        kw = {}
        for k, v in self.__dict__.items():
            kw[k] = v.to(device) if isinstance(v, torch.Tensor) else v
        return PagedBatch(**kw)


def _randn_bf16(shape, gen: torch.Generator, device, scale: float = 1.0,
                chunk: int = 1 << 26) -> torch.Tensor:
    """N(0,1)*scale drawn in fp32 and rounded to bf16, in chunks to bound memory."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        x = torch.randn(hi - lo, generator=gen, dtype=torch.float32, device=device)
        if scale != 1.0:
            x.mul_(scale)
        out[lo:hi] = x.to(torch.bfloat16)
    return out.view(*shape)


def make_batch(*, name: str, seq_lens: Sequence[int], q_lens: Sequence[int],
               num_heads: int, num_kv_heads: int, head_size: int, block_size: int,
               scale: float, seed: int, num_blocks: Optional[int] = None,
               free_fraction: float = 0.10, q_scale: float = 1.0,
               shared_prefix_blocks: int = 0, max_blocks_per_seq: Optional[int] = None,
               device="cpu", poison: bool = True) -> PagedBatch:
    """Build a batch whose sequences own random physical blocks of one pool.

    ``shared_prefix_blocks`` > 0 makes every sequence's table start with the
    same physical blocks (a shared prompt prefix); each sequence then needs
    ``seq_lens[s] > shared_prefix_blocks*block_size``.
    """
    B = len(seq_lens)
    assert len(q_lens) == B
    bs = block_size
    lens = [int(x) for x in seq_lens]
    qls = [int(x) for x in q_lens]
    for L, ql in zip(lens, qls):
        assert 0 <= ql <= L or (ql == 1 and L == 0), (L, ql)
    meta = torch.Generator(device="cpu").manual_seed(seed)
    nblk = [-(-L // bs) for L in lens]
    if shared_prefix_blocks:
        for L in lens:
            assert L > shared_prefix_blocks * bs
        own = [n - shared_prefix_blocks for n in nblk]
        live = shared_prefix_blocks + sum(own)
    else:
        own = nblk
        live = sum(own)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(live * (1.0 + free_fraction)))
    assert num_blocks >= live, (num_blocks, live)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max([1] + nblk)
    perm = torch.randperm(num_blocks, generator=meta).tolist()
    tables = torch.full((B, max_blocks_per_seq), -1, dtype=torch.int32)
    cursor = 0
    prefix_ids: List[int] = []
    if shared_prefix_blocks:
        prefix_ids = perm[:shared_prefix_blocks]
        cursor = shared_prefix_blocks
    for s in range(B):
        ids = list(prefix_ids) + perm[cursor:cursor + own[s]]
        cursor += own[s]
        if ids:
            tables[s, :len(ids)] = torch.tensor(ids, dtype=torch.int32)

    # Slots of the new tokens, in query-row order.
    slots: List[int] = []
    for s in range(B):
        for pos in range(lens[s] - qls[s], lens[s]):
            if pos < 0:
                # decode row of an empty sequence: nothing to write
                slots.append(-1)
                continue
            slots.append(int(tables[s, pos // bs]) * bs + pos % bs)
    cu = [0]
    for ql in qls:
        cu.append(cu[-1] + ql)
    total_q = cu[-1]

    dev = torch.device(device)
    vgen = torch.Generator(device=dev).manual_seed(seed + 1_000_003)
    Hq, Hkv, D = num_heads, num_kv_heads, head_size
    kv_cache = _randn_bf16((num_blocks, 2, Hkv, bs, D), vgen, dev)
    q = _randn_bf16((total_q, Hq, D), vgen, dev, scale=q_scale)
    k_new = _randn_bf16((total_q, Hkv, D), vgen, dev)
    v_new = _randn_bf16((total_q, Hkv, D), vgen, dev)

    if poison:
        nan = float("nan")
        used = torch.zeros(num_blocks, dtype=torch.bool)
        for s in range(B):
            n = nblk[s]
            if n:
                used[tables[s, :n].long()] = True
            if n and lens[s] % bs:
                # tail of the last block beyond the sequence end
                kv_cache[int(tables[s, n - 1]), :, :, lens[s] % bs:, :] = nan
        free_ids = (~used).nonzero().flatten()
        if free_ids.numel():
            kv_cache[free_ids.to(dev)] = nan
        for sl in slots:
            if sl >= 0:
                kv_cache[sl // bs, :, :, sl % bs, :] = nan

    lens_t = torch.tensor(lens, dtype=torch.int32)
    return PagedBatch(
        name=name, num_heads=Hq, num_kv_heads=Hkv, head_size=D, block_size=bs,
        num_blocks=num_blocks, scale=float(scale), kv_cache=kv_cache,
        block_tables=tables.to(dev), seq_lens=lens_t.to(dev),
        q_lens=torch.tensor(qls, dtype=torch.int32).to(dev),
        cu_q_lens=torch.tensor(cu, dtype=torch.int32).to(dev),
        q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.tensor(slots, dtype=torch.int32).to(dev),
        shared_prefix_blocks=shared_prefix_blocks)


def _uniform_int(gen: torch.Generator, lo: int, hi: int, n: int) -> List[int]:
    """n integers uniform on [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def config_spec(n: int, seed: Optional[int] = None) -> dict:
    """Keyword arguments of ``make_batch`` for numbered workload ``n``.

    1 tiny decode: TinyLlama-1.1B heads (32 q / 4 kv / 64), 4 sequences,
      lengths U{1..128}, a 64-block pool, scale 1/8.
    2 Llama-3-8B decode: 32 q / 8 kv / 128, 256 sequences, lengths U{512..4096}.
    3 long skewed decode: 32 sequences, lengths floor(exp(U[ln 1024, ln 131072])),
      Q drawn N(0,1)*2.
    4 mixed batch: 8 prefill chunks of 512 tokens after a cached context
      U{0..8192}, then 248 decode sequences with lengths U{256..4096}.
    5 prefix-shared decode: Llama-3-70B per-layer heads (64 q / 8 kv / 128),
      128 sequences sharing 128 physical blocks (2048 tokens), then own
      suffixes of U{64..1024} tokens.
    All use block_size 16; configs 2-5 use scale 1/sqrt(128) and a pool 10%
    larger than the live blocks.  Every sequence's newest token(s) are the
    ones written through ``slot_mapping`` in the same step.
    """
    seed = config_seed(n) if seed is None else seed
    g = torch.Generator(device="cpu").manual_seed(seed)
    llama = dict(num_kv_heads=8, head_size=128, block_size=16, scale=1.0 / math.sqrt(128))
    if n == 1:
        lens = _uniform_int(g, 1, 128, 4)
        return dict(name=CONFIG_NAMES[1], seq_lens=lens, q_lens=[1] * 4, num_heads=32,
                    num_kv_heads=4, head_size=64, block_size=16, scale=1.0 / 8, num_blocks=64,
                    max_blocks_per_seq=8, seed=seed)
    if n == 2:
        lens = _uniform_int(g, 512, 4096, 256)
        return dict(name=CONFIG_NAMES[2], seq_lens=lens, q_lens=[1] * 256, num_heads=32,
                    max_blocks_per_seq=256, seed=seed, **llama)
    if n == 3:
        u = torch.rand(32, generator=g, dtype=torch.float64)
        lo, hi = math.log(1024), math.log(131072)
        lens = [int(math.floor(math.exp(lo + (hi - lo) * float(x)))) for x in u]
        return dict(name=CONFIG_NAMES[3], seq_lens=lens, q_lens=[1] * 32, num_heads=32,
                    q_scale=2.0, max_blocks_per_seq=8192, seed=seed, **llama)
    if n == 4:
        ctx = _uniform_int(g, 0, 8192, 8)
        dec = _uniform_int(g, 256, 4096, 248)
        return dict(name=CONFIG_NAMES[4], seq_lens=[c + 512 for c in ctx] + dec,
                    q_lens=[512] * 8 + [1] * 248, num_heads=32, max_blocks_per_seq=544,
                    seed=seed, **llama)
    if n == 5:
        suffix = _uniform_int(g, 64, 1024, 128)
        return dict(name=CONFIG_NAMES[5], seq_lens=[2048 + x for x in suffix],
                    q_lens=[1] * 128, num_heads=64, shared_prefix_blocks=128,
                    max_blocks_per_seq=192, seed=seed, **llama)
    raise ValueError(f"unknown workload {n}")


def make_config(n: int, device="cpu", seed: Optional[int] = None, poison: bool = True) -> PagedBatch:
    """Numbered workload ``n`` (see ``config_spec``) with its values drawn on ``device``."""
    return make_batch(device=device, poison=poison, **config_spec(n, seed))


def sample_of_config(n: int, first: int, device="cpu", seed: Optional[int] = None) -> PagedBatch:
    """The first ``first`` sequences of workload ``n``, with a pool of their own.

    Same shapes, lengths and value distribution as the full workload; used where
    a bounded sample of the workload is wanted (CPU timings).
    """
    spec = config_spec(n, seed)
    spec["seq_lens"] = spec["seq_lens"][:first]
    spec["q_lens"] = spec["q_lens"][:first]
    spec.pop("num_blocks", None)
    spec["name"] = f"{spec['name']}[:{first}]"
    return make_batch(device=device, **spec)


# Per-tensor scales of the FP8 (e4m3) pools built below: N(0,1) values divided by
# 1/64 stay far inside the format's +-448 range, using most of its exponents.
FP8_K_SCALE = 1.0 / 64
FP8_V_SCALE = 1.0 / 64


def fp8_pool_of(b: PagedBatch, k_scale: float = FP8_K_SCALE,
                v_scale: float = FP8_V_SCALE) -> torch.Tensor:
    """The batch's pool as an FP8 pool: uint8 OCP e4m3 codes of value / scale, in the
    same layout, drawn through PyTorch's float8_e4m3fn cast of the values clamped
    to +-448 (input data only; NaN poison stays NaN).  The new tokens' slots still hold NaN codes, to be written
    by the FP8 cache write."""
    out = torch.empty(b.kv_cache.shape, dtype=torch.uint8, device=b.kv_cache.device)
    for side, sc in ((0, k_scale), (1, v_scale)):
        for lo in range(0, b.num_blocks, 4096):
            hi = min(b.num_blocks, lo + 4096)
            x = (b.kv_cache[lo:hi, side].float() / sc).clamp(-448.0, 448.0)  # NaN stays NaN
            out[lo:hi, side] = x.to(torch.float8_e4m3fn).view(torch.uint8)
    return out

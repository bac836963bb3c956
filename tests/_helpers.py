"""Test-side helpers: build paged pools from contiguous per-sequence K/V.

The placement here is written directly against the pool's axes
``[block, K|V, kv_head, offset, dim]`` with Python loops, independently of the
oracle's C gather and of the CUDA kernels, so that comparing either against a
contiguous computation checks their indexing.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch


@dataclass
class Contig:
    """A batch stored contiguously: per-sequence K/V plus flattened queries."""

    Ks: List[torch.Tensor]       # bf16 [L_s, Hkv, D]
    Vs: List[torch.Tensor]
    q: torch.Tensor              # bf16 [sum q_len, Hq, D]
    q_lens: List[int]
    scale: float

    @property
    def seq_lens(self) -> List[int]:
        return [int(k.shape[0]) for k in self.Ks]

    @property
    def cu_q_lens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    def positions(self, s: int) -> np.ndarray:
        L, ql = self.seq_lens[s], self.q_lens[s]
        return np.arange(L - ql, L)


def random_contig(seed: int, seq_lens: Sequence[int], q_lens: Sequence[int], Hq: int, Hkv: int,
                  D: int, scale: Optional[float] = None, q_mult: float = 1.0) -> Contig:
    g = torch.Generator().manual_seed(seed)
    Ks = [torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16) for L in seq_lens]
    Vs = [torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16) for L in seq_lens]
    q = (torch.randn(sum(q_lens), Hq, D, generator=g) * q_mult).to(torch.bfloat16)
    return Contig(Ks, Vs, q, list(q_lens), 1.0 / math.sqrt(D) if scale is None else scale)


def page(c: Contig, block_size: int, seed: int = 0, extra_blocks: int = 3,
         fill=float("nan")):
    """Scatter c into a randomly placed pool.

    Returns (kv_cache bf16 [NB,2,Hkv,bs,D], block_tables int32 [B,MB]).
    Unowned slots hold ``fill``.
    """
    Hkv, D = c.Ks[0].shape[1], c.Ks[0].shape[2]
    bs = block_size
    need = [-(-L // bs) for L in c.seq_lens]
    NB = sum(need) + extra_blocks
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(seed)).tolist()
    MB = max([1] + need)
    tables = torch.full((len(need), MB), -1, dtype=torch.int32)
    pool = torch.full((NB, 2, Hkv, bs, D), fill, dtype=torch.bfloat16)
    cur = 0
    for s, n in enumerate(need):
        ids = perm[cur:cur + n]
        cur += n
        if ids:
            tables[s, :n] = torch.tensor(ids, dtype=torch.int32)
        for t in range(c.seq_lens[s]):
            blk = ids[t // bs]
            pool[blk, 0, :, t % bs, :] = c.Ks[s][t]
            pool[blk, 1, :, t % bs, :] = c.Vs[s][t]
    return pool, tables


def brute_reference(c: Contig) -> np.ndarray:
    """Contiguous NumPy attention for every query row of c (float64)."""
    from oracle.brute import attention_contiguous
    outs = []
    cu = c.cu_q_lens
    for s in range(len(c.Ks)):
        qs = c.q[cu[s]:cu[s + 1]].double().numpy()
        if qs.shape[0] == 0:
            continue
        K = c.Ks[s].double().numpy()
        V = c.Vs[s].double().numpy()
        outs.append(attention_contiguous(qs, K, V, c.positions(s), c.scale))
    return np.concatenate(outs, axis=0)


def oracle_on(c: Contig, block_size: int, seed: int = 0, lib=None, rows=None) -> np.ndarray:
    import oracle
    pool, tables = page(c, block_size, seed)
    return oracle.attention(c.q, c.cu_q_lens, pool, tables, np.array(c.seq_lens, np.int32),
                            c.q.shape[1], c.scale, rows=rows, lib=lib)

"""CUDA-graph capture of the decode step (cache write -> decode).

The post notes that the engine captures CUDA graphs of its forward pass so a
replay skips per-kernel launch overhead ("Inside vLLM: Anatomy of a
High-Throughput LLM Inference System", §Worker procedures, Initialize KV
cache).  The C ABI calls only enqueue work on the caller's stream, so a step
made of them can be captured and replayed; a replay must give exactly the
eager result.
"""

from __future__ import annotations

import pytest
import torch

from paged_kv_cache_287_gb300 import binding
from paged_kv_cache_287_gb300.workloads import make_config
from tests._gpu import compare, oracle_pool, oracle_rows, workspace_for

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda:0")


@pytest.mark.parametrize("n", [1, 2])
def test_graph_replay_of_write_and_decode_matches_eager(n):
    b = make_config(n, device=DEV)
    pool = oracle_pool(b)
    ws = workspace_for(b)
    eager = torch.empty_like(b.q)
    out = torch.empty_like(b.q)
    max_len = b.max_seq_len

    def step(dst):
        binding.pa_cache_write(b.kv_cache, b.k_new, b.v_new, b.slot_mapping)
        binding.pa_decode(dst, b.q, b.kv_cache, b.block_tables, b.seq_lens, max_len, b.scale, ws)

    step(eager)                      # also warms up (attributes, tensor-map encoder)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(out)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    binding.pa_error_check()
    compare(out, oracle_rows(b, pool), f"graph replay, workload {n}")


@pytest.mark.parametrize("n", [1, 2, 4])
def test_graph_replay_of_the_varlen_step_matches_eager(n):
    """The one-call step, captured: decode tokens only (1, 2: the decode starts
    as a programmatic dependent of the write, a dependency the capture keeps) and
    the mixed batch (4: the write's extra block chooses the split read by the
    attention launch)."""
    b = make_config(n, device=DEV)
    n_pre = int((b.q_lens > 1).sum())
    npt = int(b.cu_q_lens[n_pre])
    max_q = int(b.q_lens[:n_pre].max()) if n_pre else 0
    max_dec = int(b.seq_lens[n_pre:].max())
    cu = b.cu_q_lens[:n_pre + 1].contiguous()
    ws = torch.empty(binding.pa_attention_varlen_workspace_bytes(
        b.num_seqs, n_pre, b.num_heads, b.num_kv_heads, b.head_size), dtype=torch.uint8,
        device=DEV)
    eager = torch.empty_like(b.q)
    out = torch.empty_like(b.q)

    def step(dst):
        binding.pa_attention_varlen(dst, b.q, b.k_new, b.v_new, b.slot_mapping, cu, n_pre, npt,
                                    max_q, b.kv_cache, b.block_tables, b.seq_lens, max_dec,
                                    b.scale, ws)

    step(eager)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(out)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    binding.pa_error_check()

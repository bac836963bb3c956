"""Pins for the CPU fp64 oracle (no GPU).

Each pin ties the oracle to something other than itself: the block-byte
formula printed in "Inside vLLM: Anatomy of a High-Throughput LLM Inference
System" (§Block size), closed forms solved by hand, an independent contiguous
NumPy computation, PyTorch's own scaled-dot-product attention in float64,
exact invariances (physical placement, block size), and special cases with
known answers.  ``test_planted_mistakes_are_caught`` compiles altered copies
of the oracle and checks that the pins reject each one.
"""

from __future__ import annotations

import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from tests._helpers import Contig, brute_reference, oracle_on, page, random_contig

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
# Altered oracle copies are compiled in a git-ignored folder inside the repository.
MUT_DIR = os.path.join(os.path.dirname(oracle.__file__), "_build")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- block bytes

def test_block_bytes_match_printed_formula(oracle_lib):
    rows = _golden_rows("block_geometry.txt")
    assert len(rows) >= 5
    for bs, hkv, d, nbytes, expect in rows:
        got = oracle.kv_block_bytes(int(bs), int(hkv), int(d), int(nbytes), lib=oracle_lib)
        assert got == int(expect), (bs, hkv, d, nbytes)


@pytest.mark.parametrize("bs,hkv,d", [(16, 4, 64), (16, 8, 128), (8, 2, 32), (32, 1, 16)])
def test_block_bytes_equal_pool_block_stride(oracle_lib, bs, hkv, d):
    """One physical block of the pool layout spans exactly the formula's bytes."""
    pool = torch.zeros(3, 2, hkv, bs, d, dtype=torch.bfloat16)
    stride_bytes = pool.stride(0) * pool.element_size()
    assert stride_bytes == oracle.kv_block_bytes(bs, hkv, d, 2, lib=oracle_lib)


# ---------------------------------------------------------------- cache write / gather

def _scatter_case(seed=5, NB=6, bs=4, Hkv=2, D=8, N=5):
    g = torch.Generator().manual_seed(seed)
    pool = torch.randn(NB, 2, Hkv, bs, D, generator=g).to(torch.bfloat16)
    kn = torch.randn(N, Hkv, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(N, Hkv, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:N].to(torch.int32)
    slots[1] = -1  # padding row
    return pool, kn, vn, slots


def test_cache_write_places_bits_and_leaves_rest(oracle_lib):
    pool, kn, vn, slots = _scatter_case()
    NB, _, Hkv, bs, D = pool.shape
    out = oracle.cache_write(pool, kn, vn, slots, lib=oracle_lib)
    expect = pool.view(torch.int16).numpy().view(np.uint16).copy()
    kb = kn.view(torch.int16).numpy().view(np.uint16)
    vb = vn.view(torch.int16).numpy().view(np.uint16)
    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        expect[s // bs, 0, :, s % bs, :] = kb[i]
        expect[s // bs, 1, :, s % bs, :] = vb[i]
    assert np.array_equal(out, expect)
    # the padding row's data appears nowhere it was not already
    changed = (out != pool.view(torch.int16).numpy().view(np.uint16))
    assert changed.sum() <= 2 * Hkv * D * (len(slots) - 1)


def test_cache_write_rejects_slot_outside_pool(oracle_lib):
    pool, kn, vn, slots = _scatter_case()
    slots[0] = pool.shape[0] * pool.shape[3]
    with pytest.raises(ValueError):
        oracle.cache_write(pool, kn, vn, slots, lib=oracle_lib)


def test_write_then_gather_round_trip(oracle_lib):
    """Writing a sequence token by token through its table, then gathering, returns it."""
    c = random_contig(11, [23], [1], 2, 2, 8)
    bs = 4
    _, tables = page(c, bs, seed=3)
    NB = int(tables.max()) + 2
    pool = torch.full((NB, 2, 2, bs, 8), float("nan"), dtype=torch.bfloat16)
    row = tables[0].tolist()
    slots = torch.tensor([row[t // bs] * bs + t % bs for t in range(23)], dtype=torch.int32)
    pool_bits = oracle.cache_write(pool, c.Ks[0], c.Vs[0], slots, lib=oracle_lib)
    K, V = oracle.gather(pool_bits, tables[0], 23, lib=oracle_lib)
    assert np.array_equal(K, c.Ks[0].double().numpy())
    assert np.array_equal(V, c.Vs[0].double().numpy())


# ---------------------------------------------------------------- attention pins

CASES = [
    # seed, seq_lens, q_lens, Hq, Hkv, D, bs
    (1, [1, 7, 40], [1, 1, 1], 4, 1, 8, 4),
    (2, [17, 33, 5, 9], [1, 1, 1, 1], 8, 2, 16, 8),
    (3, [12, 30], [5, 12], 4, 4, 8, 2),       # chunked prefill: q_len > 1, context before
    (4, [16, 1, 32], [16, 1, 8], 8, 1, 4, 16),
    (5, [39], [39], 2, 2, 16, 1),             # whole prompt as one chunk
]


@pytest.mark.parametrize("case", CASES)
def test_oracle_matches_contiguous_bruteforce(oracle_lib, case):
    seed, lens, qls, Hq, Hkv, D, bs = case
    c = random_contig(seed, lens, qls, Hq, Hkv, D)
    got = oracle_on(c, bs, seed=seed, lib=oracle_lib)
    want = brute_reference(c)
    assert got.shape == want.shape
    assert np.max(np.abs(got - want)) < 1e-12


@pytest.mark.parametrize("case", CASES)
def test_oracle_matches_torch_sdpa_float64(oracle_lib, case):
    """PyTorch's attention (float64, explicit causal mask, its own GQA grouping)."""
    if "enable_gqa" not in torch.nn.functional.scaled_dot_product_attention.__doc__:
        pytest.skip("torch without enable_gqa")
    seed, lens, qls, Hq, Hkv, D, bs = case
    c = random_contig(seed, lens, qls, Hq, Hkv, D)
    got = oracle_on(c, bs, seed=seed, lib=oracle_lib)
    cu = c.cu_q_lens
    parts = []
    for s, L in enumerate(lens):
        q = c.q[cu[s]:cu[s + 1]].double().permute(1, 0, 2)     # [Hq, n, D]
        k = c.Ks[s].double().permute(1, 0, 2)                  # [Hkv, L, D]
        v = c.Vs[s].double().permute(1, 0, 2)
        pos = torch.as_tensor(c.positions(s))
        mask = torch.arange(L)[None, :] <= pos[:, None]         # [n, L]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=mask, scale=c.scale, enable_gqa=True)
        parts.append(o.permute(1, 0, 2).numpy())
    want = np.concatenate(parts, axis=0)
    assert np.max(np.abs(got - want)) < 1e-12


def test_placement_invariance_is_exact(oracle_lib):
    c = random_contig(21, [37, 64, 3], [1, 4, 1], 8, 2, 16)
    a = oracle_on(c, 8, seed=1, lib=oracle_lib)
    b = oracle_on(c, 8, seed=99, lib=oracle_lib)
    assert np.array_equal(a, b)


def test_block_size_invariance_is_exact(oracle_lib):
    c = random_contig(22, [45, 16, 33], [1, 16, 3], 4, 2, 8)
    outs = [oracle_on(c, bs, seed=bs, lib=oracle_lib) for bs in (1, 2, 8, 16, 32)]
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def test_weights_are_a_distribution(oracle_lib):
    """With one-hot value rows the output is the weight vector: >= 0, sums to 1,
    and is zero on keys beyond the query's position."""
    L, D = 24, 32
    c = random_contig(31, [L], [6], 4, 2, D, q_mult=3.0)
    eye = torch.zeros(L, 2, D, dtype=torch.bfloat16)
    for j in range(L):
        eye[j, :, j] = 1.0
    c.Vs = [eye]
    out = oracle_on(c, 4, lib=oracle_lib)
    pos = c.positions(0)
    for r in range(out.shape[0]):
        for h in range(4):
            w = out[r, h]
            assert abs(w.sum() - 1.0) < 1e-12
            assert (w >= 0).all()
            assert (w[pos[r] + 1:] == 0).all()
            assert (w[:pos[r] + 1] > 0).all()


def test_constant_values_return_that_value(oracle_lib):
    c = random_contig(41, [29, 7], [3, 1], 4, 1, 8, q_mult=4.0)
    row = torch.randn(1, 1, 8).to(torch.bfloat16)
    c.Vs = [row.expand(29, 1, 8).clone(), row.expand(7, 1, 8).clone()]
    out = oracle_on(c, 4, lib=oracle_lib)
    assert np.max(np.abs(out - row.double().numpy()[0, 0])) < 1e-12


def test_single_token_returns_its_value_exactly(oracle_lib):
    c = random_contig(51, [1, 1, 1], [1, 1, 1], 4, 2, 16)
    out = oracle_on(c, 16, lib=oracle_lib)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(out[s, h], c.Vs[s][0, h // 2].double().numpy())


@pytest.mark.parametrize("zero", ["q", "scale"])
def test_uniform_scores_average_the_visible_values(oracle_lib, zero):
    c = random_contig(61, [13, 20], [1, 4], 4, 2, 8)
    if zero == "q":
        c.q = torch.zeros_like(c.q)
    else:
        c.scale = 0.0
    out = oracle_on(c, 4, lib=oracle_lib)
    cu = c.cu_q_lens
    for s in range(2):
        V = c.Vs[s].double().numpy()
        for i, p in enumerate(c.positions(s)):
            want = V[:p + 1].mean(axis=0)                      # [Hkv, D]
            for h in range(4):
                assert np.max(np.abs(out[cu[s] + i, h] - want[h // 2])) < 1e-12


def test_dominant_key_selects_its_value(oracle_lib):
    c = random_contig(71, [30], [1], 2, 1, 16, scale=1.0)
    j = 17
    K = c.Ks[0].clone()
    K[j, 0] = (c.q[0, 0].float() * 8).to(torch.bfloat16)       # q.k_j >> q.k_i
    K[:, 0] = torch.where(torch.arange(30)[:, None] == j, K[:, 0], K[:, 0] * 0.01)
    c.Ks = [K]
    c.q[0, 1] = c.q[0, 0]
    out = oracle_on(c, 8, lib=oracle_lib)
    for h in range(2):
        assert np.max(np.abs(out[0, h] - c.Vs[0][j, 0].double().numpy())) < 1e-12


def test_chunk_rows_equal_decode_at_each_position(oracle_lib):
    """Row i of a chunk after context c equals a decode step with seq_len c+i+1."""
    ctx, ql = 19, 7
    c = random_contig(81, [ctx + ql], [ql], 4, 2, 8)
    chunk = oracle_on(c, 4, lib=oracle_lib)
    for i in range(ql):
        L = ctx + i + 1
        d = Contig([c.Ks[0][:L]], [c.Vs[0][:L]], c.q[i:i + 1], [1], c.scale)
        assert np.array_equal(oracle_on(d, 4, lib=oracle_lib)[0], chunk[i])


def test_future_tokens_do_not_leak(oracle_lib):
    ctx, ql = 10, 6
    c = random_contig(91, [ctx + ql], [ql], 2, 1, 8)
    a = oracle_on(c, 4, lib=oracle_lib)
    K, V = c.Ks[0].clone(), c.Vs[0].clone()
    K[ctx + 3:] = 100.0
    V[ctx + 3:] = -100.0
    c.Ks, c.Vs = [K], [V]
    b = oracle_on(c, 4, lib=oracle_lib)
    # rows 0..2 sit at positions ctx..ctx+2 and never see the altered tokens
    assert np.array_equal(a[:3], b[:3])
    for r in range(3, ql):
        assert not np.array_equal(a[r], b[r])


def test_empty_sequence_decodes_to_zeros(oracle_lib):
    c = random_contig(95, [0, 5], [1, 1], 2, 1, 8)
    pool, tables = page(c, 4)
    out = oracle.attention(c.q, c.cu_q_lens, pool, tables, np.array([0, 5], np.int32), 2,
                           c.scale, lib=oracle_lib)
    assert np.array_equal(out[0], np.zeros((2, 8)))
    assert np.isfinite(out[1]).all()


def test_closed_forms(oracle_lib):
    vals = {r[0]: (float(r[1]), float(r[2])) for r in _golden_rows("closed_forms.txt")}
    cases = {
        "A": ([1, 0], [[1, 0], [0, 0]], [[1, 0], [0, 1]]),
        "B": ([1, 1], [[0, 0], [1, 0], [0, 1]], [[2, 0], [0, 2], [2, 2]]),
        "C": ([0.5, -0.5], [[2, 2]], [[3, -1]]),
    }
    for name, (q, k, v) in cases.items():
        L = len(k)
        c = Contig([torch.tensor(k, dtype=torch.bfloat16).view(L, 1, 2)],
                   [torch.tensor(v, dtype=torch.bfloat16).view(L, 1, 2)],
                   torch.tensor(q, dtype=torch.bfloat16).view(1, 1, 2), [1], 1.0)
        out = oracle_on(c, 2, lib=oracle_lib)[0, 0]
        assert np.max(np.abs(out - np.array(vals[name]))) < 1e-15, name


def test_row_subset_matches_full(oracle_lib):
    c = random_contig(99, [20, 31, 8], [5, 1, 8], 4, 2, 8)
    full = oracle_on(c, 4, lib=oracle_lib)
    rows = np.array([13, 0, 5, 7], dtype=np.int32)
    sub = oracle_on(c, 4, lib=oracle_lib, rows=rows)
    assert np.array_equal(sub, full[rows])


# ---------------------------------------------------------------- planted mistakes

def _pins_pass(lib) -> bool:
    """A compact battery of the pins above, run against a given oracle build."""
    try:
        for case in CASES[:4]:
            seed, lens, qls, Hq, Hkv, D, bs = case
            c = random_contig(seed, lens, qls, Hq, Hkv, D)
            if np.max(np.abs(oracle_on(c, bs, seed=seed, lib=lib) - brute_reference(c))) > 1e-12:
                return False
        pool, kn, vn, slots = _scatter_case()
        out = oracle.cache_write(pool, kn, vn, slots, lib=lib)
        _, _, _, bs, _ = pool.shape
        kb = kn.view(torch.int16).numpy().view(np.uint16)
        for i, s in enumerate(slots.tolist()):
            if s >= 0 and not np.array_equal(out[s // bs, 0, :, s % bs, :], kb[i]):
                return False
        return True
    except Exception:
        return False


MUTATIONS = {
    "gqa_modulo": ("pos, h / group,", "pos, h % num_kv_heads,"),
    "causal_off_by_one": ("const int pos = context + (r - r0);",
                          "const int pos = context + (r - r0) - 1;"),
    "scale_dropped": ("x[j] = scale * dot;", "x[j] = dot;"),
    "k_read_from_v": ("K[dst] = pool_value(kv_cache, kv_fp8,\n"
                      "                                                pool_index(block, 0,",
                      "K[dst] = pool_value(kv_cache, kv_fp8,\n"
                      "                                                pool_index(block, 1,"),
    "no_normalisation": ("out[d] /= denom;", "out[d] /= 1.0;"),
    "offset_and_head_swapped": (
        "((((size_t)block * 2 + (size_t)kv) * (size_t)num_kv_heads + (size_t)head) *\n"
        "                (size_t)block_size + (size_t)offset)",
        "((((size_t)block * 2 + (size_t)kv) * (size_t)block_size + (size_t)offset) *\n"
        "                (size_t)num_kv_heads + (size_t)head)"),
    "write_offset_wrong": ("int offset = (int)(slot % block_size);",
                           "int offset = (int)((slot / block_size) % block_size);"),
    "exp_sign_flipped": ("double w = exp(x[j] - m);", "double w = exp(m - x[j]);"),
}


def test_unmodified_oracle_passes_battery(oracle_lib):
    assert _pins_pass(oracle_lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    os.makedirs(MUT_DIR, exist_ok=True)
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    with tempfile.TemporaryDirectory(prefix="_mut_", dir=MUT_DIR) as d:
        p = os.path.join(d, "mut.c")
        with open(p, "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(d, "libmut.so")
        oracle.build(src=p, out=so)
        lib = oracle.load(so)
        assert not _pins_pass(lib), f"planted mistake {name} survived the pins"

"""Pins for the oracle's FP8 (OCP E4M3, "e4m3fn") KV-cache functions (no GPU).

The codec is pinned by PyTorch's own float8_e4m3fn type (every code's value,
and the encoding of in-range values), by values fixed by the format's
definition (largest finite 448, smallest normal 2^-6, smallest subnormal
2^-9), by round trips, ties and saturation.  FP8 attention is pinned to the
already pinned bf16 attention: with power-of-two scales every dequantised
element is exactly a bf16 value, so the two must agree bit for bit.  Altered
copies of the oracle (planted mistakes) must each fail one of these pins.
"""

from __future__ import annotations

import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle

MUT_DIR = os.path.join(os.path.dirname(oracle.__file__), "_build")


def _torch_codes(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


# ---------------------------------------------------------------- codec

def test_e4m3_table_matches_torch(oracle_lib):
    want = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c, lib=oracle_lib) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_e4m3_values_fixed_by_the_format(oracle_lib):
    v = lambda c: oracle.e4m3_to_double(c, lib=oracle_lib)
    assert v(0x00) == 0.0 and np.signbit(v(0x80))
    assert v(0x01) == 2.0 ** -9                 # smallest subnormal
    assert v(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert v(0x08) == 2.0 ** -6                 # smallest normal
    assert v(0x38) == 1.0 and v(0x39) == 1.125
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    finite = [v(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(finite, finite[1:]))   # codes order by value


def test_e4m3_encode_round_trips_every_code(oracle_lib):
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_from_float(oracle.e4m3_to_double(c, lib=oracle_lib),
                                      lib=oracle_lib) == c, hex(c)


def test_e4m3_encode_ties_to_even_and_saturates(oracle_lib):
    enc = lambda x: oracle.e4m3_from_float(x, lib=oracle_lib)
    v = lambda c: oracle.e4m3_to_double(c, lib=oracle_lib)
    for c in range(0x7E):
        mid = 0.5 * (v(c) + v(c + 1))
        even = c if c % 2 == 0 else c + 1
        assert enc(mid) == even and enc(-mid) == 0x80 | even, hex(c)
        gap = v(c + 1) - v(c)
        assert enc(mid - gap / 8) == c and enc(mid + gap / 8) == c + 1
    assert enc(448.0) == 0x7E and enc(449.0) == 0x7E and enc(1e30) == 0x7E
    assert enc(-500.0) == 0xFE and enc(float("-inf")) == 0xFE
    assert enc(float("nan")) == 0x7F
    assert enc(2.0 ** -10) == 0x00 and enc(-(2.0 ** -10)) == 0x80
    assert enc(2.0 ** -10 * 1.01) == 0x01 and enc(1e-30) == 0x00 and enc(-0.0) == 0x80


def test_e4m3_encode_matches_torch_in_range(oracle_lib):
    g = np.random.default_rng(7)
    x = (g.standard_normal(4000) * np.exp2(g.integers(-12, 9, 4000))).astype(np.float32)
    x = x[np.abs(x) < 464]
    got = np.array([oracle.e4m3_from_float(float(t), lib=oracle_lib) for t in x], dtype=np.uint8)
    want = _torch_codes(x)
    bad = got != want
    assert not bad.any(), list(zip(x[bad][:5], got[bad][:5], want[bad][:5]))


# ---------------------------------------------------------------- cache write

def _fp8_case(seed=3, NB=7, bs=4, Hkv=2, D=8, N=6):
    g = torch.Generator().manual_seed(seed)
    pool = torch.randint(0, 0x7E, (NB, 2, Hkv, bs, D), generator=g, dtype=torch.uint8)
    k = (torch.randn(N, Hkv, D, generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn(N, Hkv, D, generator=g) * 0.2).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:N].to(torch.int32)
    slots[2] = -1
    return pool, k, v, slots


def test_cache_write_fp8_quantises_with_the_tensor_scales(oracle_lib):
    pool, k, v, slots = _fp8_case()
    ks, vs = 0.0625, 0.0078125 * 3
    got = oracle.cache_write_fp8(pool, k, v, slots, ks, vs, lib=oracle_lib)
    NB, _, Hkv, bs, D = pool.shape
    want = pool.numpy().copy()
    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        kq = (k[i].float() / torch.tensor(ks, dtype=torch.float32)).numpy()
        vq = (v[i].float() / torch.tensor(vs, dtype=torch.float32)).numpy()
        want[s // bs, 0, :, s % bs, :] = _torch_codes(kq)
        want[s // bs, 1, :, s % bs, :] = _torch_codes(vq)
    assert np.array_equal(got, want)


def test_cache_write_fp8_rejects_slot_outside_pool(oracle_lib):
    pool, k, v, slots = _fp8_case()
    slots[0] = pool.shape[0] * pool.shape[3]
    with pytest.raises(ValueError):
        oracle.cache_write_fp8(pool, k, v, slots, 1.0, 1.0, lib=oracle_lib)


# ---------------------------------------------------------------- attention

def _attention_pair(lib, seed=11, ks=0.25, vs=4.0):
    g = torch.Generator().manual_seed(seed)
    B, Hq, Hkv, D, bs = 3, 8, 2, 16, 4
    lens = [9, 1, 14]
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + 2
    perm = torch.randperm(NB, generator=g)
    tables = torch.full((B, max(nblk)), -1, dtype=torch.int32)
    c = 0
    for s in range(B):
        tables[s, :nblk[s]] = perm[c:c + nblk[s]].to(torch.int32)
        c += nblk[s]
    codes = torch.randint(0, 0x7E, (NB, 2, Hkv, bs, D), generator=g, dtype=torch.uint8)
    sign = torch.randint(0, 2, codes.shape, generator=g, dtype=torch.uint8) * 0x80
    codes = codes | sign
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64)
    vals[:, 0] *= ks
    vals[:, 1] *= vs
    pool16 = vals.to(torch.bfloat16)
    assert torch.equal(pool16.to(torch.float64), vals)     # exactly representable
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    cu = torch.arange(B + 1, dtype=torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32)
    a8 = oracle.attention_fp8(q, cu, codes, ks, vs, tables, sl, Hq, 0.3, lib=lib)
    a16 = oracle.attention(q, cu, pool16, tables, sl, Hq, 0.3, lib=lib)
    return a8, a16


def test_attention_fp8_equals_bf16_attention_on_the_dequantised_pool(oracle_lib):
    a8, a16 = _attention_pair(oracle_lib)
    assert np.array_equal(a8, a16)


# ---------------------------------------------------------------- planted mistakes

FP8_MUTATIONS = {
    "exponent_bias": ("ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 9)"),
    "subnormal_scale": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "ties_to_odd": ("c = (lo & 1) == 0 ? lo : lo + 1;", "c = (lo & 1) == 1 ? lo : lo + 1;"),
    "saturate_low": ("if (a >= 448.0)", "if (a >= 240.0)"),
    "sign_dropped": ("return sign | (uint8_t)c;", "return (uint8_t)c;"),
    "v_uses_k_scale": ("oracle_e4m3_from_float(v / v_scale)", "oracle_e4m3_from_float(v / k_scale)"),
    "dequant_scale_swapped": (
        "return attention_impl(out, q, cu_q_lens, num_seqs, kv_cache, 1, k_scale, v_scale,",
        "return attention_impl(out, q, cu_q_lens, num_seqs, kv_cache, 1, v_scale, k_scale,"),
}


def _fp8_pins_pass(lib) -> bool:
    checks = [test_e4m3_table_matches_torch, test_e4m3_values_fixed_by_the_format,
              test_e4m3_encode_round_trips_every_code, test_e4m3_encode_ties_to_even_and_saturates,
              test_e4m3_encode_matches_torch_in_range,
              test_cache_write_fp8_quantises_with_the_tensor_scales,
              test_attention_fp8_equals_bf16_attention_on_the_dequantised_pool]
    for chk in checks:
        try:
            chk(lib)
        except AssertionError:
            return False
    return True


def test_unmodified_oracle_passes_fp8_battery(oracle_lib):
    assert _fp8_pins_pass(oracle_lib)


@pytest.mark.parametrize("name", sorted(FP8_MUTATIONS))
def test_fp8_planted_mistakes_are_caught(name):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    os.makedirs(MUT_DIR, exist_ok=True)
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")).read()
    old, new = FP8_MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found"
    with tempfile.TemporaryDirectory(prefix="_mut_", dir=MUT_DIR) as d:
        p = os.path.join(d, "mut.c")
        with open(p, "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(d, "libmut.so")
        oracle.build(src=p, out=so)
        lib = oracle.load(so)
        assert not _fp8_pins_pass(lib), f"planted mistake {name} survived the fp8 pins"

"""Host-side checks of the seeded input generators (no GPU)."""

import math

import torch

from paged_kv_cache_287_gb300.workloads import make_batch, make_config


def _live_mask(b):
    NB, _, Hkv, bs, D = b.kv_cache.shape
    live = torch.zeros(NB, bs, dtype=torch.bool)
    for s in range(b.num_seqs):
        L = int(b.seq_lens[s])
        for t in range(L):
            live[int(b.block_tables[s, t // bs]), t % bs] = True
    return live


def test_tiny_config_shape_and_placement():
    b = make_config(1)
    assert (b.num_heads, b.num_kv_heads, b.head_size, b.block_size) == (32, 4, 64, 16)
    assert b.num_blocks == 64 and b.kv_cache.shape == (64, 2, 4, 16, 64)
    assert b.kv_cache.dtype == torch.bfloat16
    assert b.num_seqs == 4 and b.q.shape == (4, 32, 64)
    assert all(1 <= int(L) <= 128 for L in b.seq_lens)
    assert b.scale == 1.0 / 8
    ids = []
    for s in range(4):
        n = -(-int(b.seq_lens[s]) // 16)
        row = b.block_tables[s].tolist()
        assert all(x >= 0 for x in row[:n]) and all(x == -1 for x in row[n:])
        ids += row[:n]
    assert len(ids) == len(set(ids))        # no block owned twice


def test_new_token_slots_and_poison():
    b = make_config(1)
    bs = b.block_size
    live = _live_mask(b)
    for s in range(b.num_seqs):
        L = int(b.seq_lens[s])
        slot = int(b.slot_mapping[s])
        assert slot == int(b.block_tables[s, (L - 1) // bs]) * bs + (L - 1) % bs
        # the new token's slot is not yet written
        assert torch.isnan(b.kv_cache[slot // bs, :, :, slot % bs].float()).all()
        live[slot // bs, slot % bs] = False
    vals = b.kv_cache.float().permute(0, 3, 1, 2, 4)          # [NB, bs, 2, Hkv, D]
    assert torch.isfinite(vals[live]).all()
    assert torch.isnan(vals[~live]).all()


def test_generators_are_seeded():
    a, b = make_config(1), make_config(1)
    assert torch.equal(a.kv_cache.view(torch.int16), b.kv_cache.view(torch.int16))
    assert torch.equal(a.block_tables, b.block_tables)
    c = make_config(1, seed=1234)
    assert not torch.equal(a.block_tables, c.block_tables)


def test_shared_prefix_tables():
    b = make_batch(name="t", seq_lens=[70, 90, 65], q_lens=[1, 1, 1], num_heads=8,
                   num_kv_heads=2, head_size=16, block_size=16, scale=0.25, seed=3,
                   shared_prefix_blocks=4)
    pre = b.block_tables[:, :4]
    assert (pre == pre[0]).all()
    own = []
    for s in range(3):
        n = -(-int(b.seq_lens[s]) // 16)
        own += b.block_tables[s, 4:n].tolist()
    assert len(own) == len(set(own)) and not set(own) & set(pre[0].tolist())
    assert b.num_blocks == math.ceil((4 + len(own)) * 1.1)


def test_mixed_chunk_rows_and_slots():
    b = make_batch(name="m", seq_lens=[20, 9], q_lens=[8, 1], num_heads=4, num_kv_heads=2,
                   head_size=8, block_size=4, scale=0.5, seed=9)
    assert b.cu_q_lens.tolist() == [0, 8, 9]
    assert b.q.shape == (9, 4, 8) and b.k_new.shape == (9, 2, 8)
    slots = b.slot_mapping.tolist()
    for i, pos in enumerate(range(12, 20)):
        assert slots[i] == int(b.block_tables[0, pos // 4]) * 4 + pos % 4
    assert slots[8] == int(b.block_tables[1, 8 // 4]) * 4 + 0

"""The seeded workloads follow the configurations they stand for (sizes,
formats, length distributions, pool slack, block-table structure)."""

import math

import numpy as np
import pytest

import workloads


def _used(b):
    return [b.block_tables[s, : -(-int(b.seq_lens[s]) // b.block_size)] for s in range(b.num_seqs)]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name,S,Hq,Hkv,D,B,q,kv,scale", [
    ("tiny", 4, 4, 4, 64, 16, "f16", "f16", 1 / 8),
    ("gqa_32x4k", 32, 32, 8, 128, 16, "bf16", "bf16", 1 / math.sqrt(128)),
    ("long_32k", 8, 64, 8, 128, 16, "bf16", "bf16", 1 / math.sqrt(128)),
    ("fp8_mix", 256, 32, 8, 128, 16, "bf16", "e4m3", 1 / math.sqrt(128)),
    ("int8_mix", 256, 32, 8, 128, 16, "bf16", "i8", 1 / math.sqrt(128)),
])
def test_shapes_formats_and_tables(name, S, Hq, Hkv, D, B, q, kv, scale, seed):
    b = workloads.make_batch(name, seed=seed)
    assert (b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size) == (S, Hq, Hkv, D, B)
    assert (b.q_fmt, b.kv_fmt) == (q, kv) and b.scale == pytest.approx(scale, rel=1e-12)
    used = _used(b)
    flat = np.concatenate(used)
    # every used entry is a distinct block of the pool, the rest of a row is -1
    assert len(np.unique(flat)) == len(flat) and flat.min() >= 0 and flat.max() < b.num_blocks
    for s, u in enumerate(used):
        assert np.all(b.block_tables[s, len(u):] == -1)
    # the pool holds the blocks the batch needs plus the stated slack, and the free list is the rest
    needed = len(flat)
    if name == "tiny":
        assert b.num_blocks == 64
    else:
        slack = 0.0 if name == "long_32k" else 0.10
        assert b.num_blocks == math.ceil(needed * (1 + slack))
    assert sorted(np.concatenate([flat, b.free_blocks]).tolist()) == list(range(b.num_blocks))
    # the appended token's slot is position seq_len - 1 through the table
    for s in range(S):
        T = int(b.seq_lens[s])
        assert b.new_slots[s] == b.block_tables[s, (T - 1) // B] * B + (T - 1) % B


def test_length_distributions():
    t = np.concatenate([workloads.make_batch("tiny", seed=k).seq_lens for k in range(50)])
    assert t.min() >= 2 and t.max() <= 129                  # cached ~U{1..128}, plus the appended token
    g = np.concatenate([workloads.make_batch("gqa_32x4k", seed=k).seq_lens for k in range(20)])
    assert g.min() >= 1 and g.max() <= 4096
    assert abs(g.mean() - 2048.5) < 4 * 4096 / math.sqrt(12 * len(g))   # U{1..4096}: mean 2048.5
    assert np.all(workloads.make_batch("long_32k", seed=0).seq_lens == 32768)
    f = np.concatenate([workloads.make_batch("fp8_mix", seed=k).seq_lens for k in range(8)])
    assert f.min() >= 16 and f.max() <= 8192
    # clip(round(lognormal(7, 1)), 16, 8192): median e^7 = 1097, about 2.2 % clipped at the top
    assert 950 < np.median(f) < 1250
    assert 0.005 < np.mean(f == 8192) < 0.045
    i = workloads.make_batch("int8_mix", seed=3)
    assert np.array_equal(i.seq_lens, workloads.make_batch("fp8_mix", seed=3).seq_lens)   # the same batch


def test_beam_scenario_shape():
    sc = workloads.beam_cow_scenario(0)
    assert (sc["num_beams"], sc["num_heads"], sc["num_kv_heads"], sc["head_dim"], sc["block_size"]) == \
        (6, 40, 40, 128, 16)
    assert sc["prompt_len"] == 1000 and -(-1000 // 16) == 63 and 1000 - 62 * 16 == 8   # 63 blocks, last holds 8
    assert sc["tails"].min() >= 1 and sc["tails"].max() <= 256 and len(sc["tails"]) == 6
    assert sc["prompt_k"].shape == (1000, 40, 128) and sc["q"].shape == (6, 40, 128)
    assert sorted(sc["free_order"].tolist()) == list(range(sc["num_blocks"]))

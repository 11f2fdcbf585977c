"""The bench's algorithmic byte count (the roofline's numerator) against a count
made position by position.

A decode launch must read, at minimum, the K and V rows of every attended
position (H_kv * d elements each), the block-table entry of every block that
holds one, q and out once per query, and the lengths.  Tail slots, the split
workspace and the 8-bit scales are overhead, not counted.  With a window, the
attended positions of a sequence of length T with L queries are the union over
its queries of their windows: max(0, T - L + 1 - W) .. T - 1.
"""

import numpy as np
import pytest

import bench
import workloads


def _count(batch, window, q_len):
    S, Hq, Hkv, D, B = batch.num_seqs, batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size
    b_kv, b_q = bench.FMT_BYTES[batch.kv_fmt], bench.FMT_BYTES[batch.q_fmt]
    kv = entries = 0
    for s in range(S):
        T = int(batch.seq_lens[s])
        seen = set()
        for i in range(q_len):
            qpos = T - q_len + i
            first = max(0, qpos - window + 1) if window > 0 else 0
            seen.update(range(first, qpos + 1))
        seen = {p for p in seen if 0 <= p < T}
        # a query at a negative position attends nothing; rows are still read once
        kv += len(seen) * Hkv * D * b_kv * 2
        entries += len({p // B for p in seen})
    return kv, kv + q_len * 2 * S * Hq * D * b_q + 4 * entries + 4 * S


@pytest.mark.parametrize("window,q_len", [(0, 1), (1, 1), (100, 1), (1024, 1), (0, 4), (7, 2), (64, 3)])
@pytest.mark.parametrize("name,kw", [
    ("gqa_32x4k", dict(num_seqs=6, lengths=("uniform", 1, 900))),
    ("fp8_mix", dict(num_seqs=5, lengths=("lognormal", 5.0, 1.0, 16, 700))),
    ("tiny", dict()),
])
def test_algorithmic_bytes_match_a_position_by_position_count(name, kw, window, q_len):
    b = workloads.make_batch(name, seed=3, **kw)
    b.seq_lens[0] = 1                        # a one-token sequence in every batch
    got = bench.algorithmic_bytes(b, window, q_len)
    kv, decode = _count(b, window, q_len)
    assert got["kv"] == kv
    assert got["decode"] == decode


def test_gqa_context_token_costs_4096_bytes():
    # 2 (K and V) x 8 KV heads x 128 x 2 bytes per context token of the GQA workload
    b = workloads.make_batch("gqa_32x4k", seed=0, num_seqs=3, lengths=("const", 1000))
    got = bench.algorithmic_bytes(b)
    assert got["kv"] == 3 * 1000 * 4096

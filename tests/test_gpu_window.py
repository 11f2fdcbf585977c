"""Sliding-window decode (pa_decode_ex, window > 0) against the oracle.

The query at position T-1 attends to positions max(0, T-W) .. T-1 (the
"局限性与未来工作" list of the dihengye.cn notes names sliding-window attention;
the oracle states the reading).  Windows are chosen to start inside a unit,
on unit and block boundaries, to cover the whole sequence and to be a single
row; blocks wholly before a window are marked unreadable.
"""

import numpy as np
import pytest

import workloads
from paged_cases import PA_TOL, bits_equal, run_gpu, run_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_144_gb300 as pa  # noqa: E402


def _check(batch, vals, window, partition_size=0):
    out, kc, vc, err = run_gpu(batch, vals, partition_size=partition_size, window=window)
    ref, okc, ovc = run_oracle(batch, vals, window=window)
    assert err == 0, f"device error bits {err}"
    assert bits_equal(kc, okc) and bits_equal(vc, ovc)
    assert np.all(np.isfinite(out))
    d = np.abs(out - ref).max()
    assert d <= PA_TOL, f"max abs err {d:.3e}"
    return d


@pytest.mark.parametrize("W", [1, 5, 16, 31, 32, 33, 100, 256, 1000, 5000])
@pytest.mark.parametrize("mode", [0, 256])
def test_window_gqa_bf16(W, mode):
    b = workloads.make_batch("gqa_32x4k", seed=40, num_seqs=6, lengths=("uniform", 1, 1200))
    _check(b, workloads.host_values(b, seed=40), W, partition_size=mode)


@pytest.mark.parametrize("B", [8, 16, 32, 128])
@pytest.mark.parametrize("W", [3, 40, 129])
def test_window_block_sizes_f16(B, W):
    b = workloads.make_batch("tiny", seed=41, block_size=B, num_seqs=5, lengths=("uniform", 1, 400),
                             pool=("slack", 0.1))
    _check(b, workloads.host_values(b, seed=41), W)


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("W", [7, 64, 300])
def test_window_fp8(B, W):
    b = workloads.make_batch("fp8_mix", seed=42, num_seqs=12, block_size=B)
    _check(b, workloads.host_values(b, seed=42), W)


@pytest.mark.parametrize("W", [9, 200])
def test_window_int8(W):
    b = workloads.make_batch("int8_mix", seed=46, num_seqs=10)
    _check(b, workloads.host_values(b, seed=46), W)


def test_window_long_extreme_logits():
    b = workloads.make_batch("long_32k", seed=43, num_seqs=2, lengths=("const", 5000))
    _check(b, workloads.host_values(b, seed=43, q_mult=30.0), 777)


def test_blocks_before_window_are_not_read():
    """Rows before the window hold NaN and wholly earlier table entries are -1."""
    B, W = 8, 21
    b = workloads.make_batch("tiny", seed=44, block_size=B, num_seqs=4, lengths=("uniform", 60, 200),
                             pool=("slack", 0.1))
    v = workloads.host_values(b, seed=44, nan_tails=False)
    b.block_tables = b.block_tables.copy()
    for s in range(b.num_seqs):
        T = int(b.seq_lens[s])
        lo = T - W
        for pos in range(lo):
            blk = int(b.block_tables[s][pos // B])
            v["k_cache"][blk, :, pos % B] = np.nan
            v["v_cache"][blk, :, pos % B] = np.nan
        b.block_tables[s, : lo // B] = -1
    out, _, _, err = run_gpu(b, v, window=W)
    ref, _, _ = run_oracle(b, v, window=W)
    assert err == 0, f"device error bits {err}"
    assert np.all(np.isfinite(out))
    assert np.abs(out - ref).max() <= PA_TOL


def test_window_rejects_negative():
    b = workloads.make_batch("tiny", seed=45)
    v = workloads.host_values(b, seed=45)
    with pytest.raises(pa.PagedAttnError):
        run_gpu(b, v, window=-1)

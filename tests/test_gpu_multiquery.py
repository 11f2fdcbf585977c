"""Several queries per sequence (pa_decode_ex q_len > 1) against the oracle.

Query i of a sequence of length T sits at position T-L+i and attends to the
positions up to its own (oracle.paged_multi_query_attention).  Shapes cover
L * G from 2 to 64 (query, head) rows: up to 16 rows one consumer warp per
ring, beyond that 2, 3 or 4 warps sharing each ring, 16 rows each; 16-bit and
8-bit caches, windows, both split modes and sequences shorter than their
query count.
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


def _check(batch, vals, window=0, partition_size=0):
    out, kc, vc, err = run_gpu(batch, vals, partition_size=partition_size, window=window)
    ref, okc, ovc = run_oracle(batch, vals, window=window)
    assert err == 0, f"device error bits {err}"
    assert bits_equal(kc, okc) and bits_equal(vc, ovc)
    assert out.shape == ref.shape
    assert np.all(np.isfinite(out))
    d = np.abs(out - ref).max()
    assert d <= PA_TOL, f"max abs err {d:.3e}"
    return d


@pytest.mark.parametrize("L", [2, 3, 4])
@pytest.mark.parametrize("mode", [0, 128])
def test_multi_query_gqa4_bf16(L, mode):
    b = workloads.make_batch("gqa_32x4k", seed=60, num_seqs=7, lengths=("uniform", 1, 700))
    _check(b, workloads.host_values(b, seed=60, q_len=L), partition_size=mode)


@pytest.mark.parametrize("L", [2, 5, 16])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_multi_query_mha_f16_d64(L, B):
    b = workloads.make_batch("tiny", seed=61, block_size=B, num_seqs=5, lengths=("uniform", 1, 260),
                             pool=("slack", 0.1))
    _check(b, workloads.host_values(b, seed=61, q_len=L))


@pytest.mark.parametrize("L", [1, 2])
def test_multi_query_group8(L):
    b = workloads.make_batch("long_32k", seed=62, num_seqs=2, lengths=("const", 1500))
    _check(b, workloads.host_values(b, seed=62, q_len=L, q_mult=30.0))


@pytest.mark.parametrize("kv", ["fp8_mix", "int8_mix"])
@pytest.mark.parametrize("L", [2, 4])
def test_multi_query_8bit(kv, L):
    b = workloads.make_batch(kv, seed=63, num_seqs=8, lengths=("lognormal", 6.0, 1.0, 16, 1200))
    _check(b, workloads.host_values(b, seed=63, q_len=L))


@pytest.mark.parametrize("W", [1, 5, 40])
def test_multi_query_with_window(W):
    b = workloads.make_batch("gqa_32x4k", seed=64, num_seqs=6, lengths=("uniform", 1, 500))
    _check(b, workloads.host_values(b, seed=64, q_len=3), window=W)


def test_multi_query_sequences_shorter_than_query_count():
    """T < L: queries at negative positions see nothing and give 0."""
    b = workloads.make_batch("gqa_32x4k", seed=65, num_seqs=6, lengths=("uniform", 1, 3))
    _check(b, workloads.host_values(b, seed=65, q_len=4))


@pytest.mark.parametrize("L", [3, 4, 6, 8])
@pytest.mark.parametrize("mode", [0, 256])
def test_multi_query_group8_shared_rings(L, mode):
    """G = 8: 24, 32, 48 and 64 rows (2, 2, 3 and 4 warps per ring), logits x30 for the longest."""
    b = workloads.make_batch("long_32k", seed=67, num_seqs=3, lengths=("uniform", 1, 1400))
    _check(b, workloads.host_values(b, seed=67, q_len=L, q_mult=30.0 if L == 8 else 1.0), partition_size=mode)


@pytest.mark.parametrize("L", [5, 8, 16])
def test_multi_query_gqa4_shared_rings(L):
    b = workloads.make_batch("gqa_32x4k", seed=68, num_seqs=6, lengths=("uniform", 1, 900))
    _check(b, workloads.host_values(b, seed=68, q_len=L))


@pytest.mark.parametrize("L", [17, 40, 64])
def test_multi_query_mha_shared_rings(L):
    b = workloads.make_batch("tiny", seed=69, num_seqs=5, lengths=("uniform", 1, 200), pool=("slack", 0.1))
    _check(b, workloads.host_values(b, seed=69, q_len=L))


@pytest.mark.parametrize("kv", ["fp8_mix", "int8_mix"])
@pytest.mark.parametrize("L", [8, 16])
def test_multi_query_8bit_shared_rings(kv, L):
    b = workloads.make_batch(kv, seed=70, num_seqs=6, lengths=("lognormal", 6.0, 1.0, 16, 1000))
    _check(b, workloads.host_values(b, seed=70, q_len=L))


@pytest.mark.parametrize("W", [1, 33])
def test_multi_query_shared_rings_with_window(W):
    b = workloads.make_batch("long_32k", seed=71, num_seqs=4, lengths=("uniform", 1, 600))
    _check(b, workloads.host_values(b, seed=71, q_len=5), window=W)


def test_multi_query_shared_rings_short_sequences():
    """T < L with 4 warps per ring: queries at negative positions give 0."""
    b = workloads.make_batch("long_32k", seed=72, num_seqs=5, lengths=("uniform", 1, 6))
    _check(b, workloads.host_values(b, seed=72, q_len=8))


def test_multi_query_rejects_too_many_rows():
    b = workloads.make_batch("gqa_32x4k", seed=66, num_seqs=2, lengths=("uniform", 5, 9))
    with pytest.raises(pa.PagedAttnError):
        run_gpu(b, workloads.host_values(b, seed=66, q_len=17))   # 17 * G(4) = 68 rows > 64


@pytest.mark.parametrize("name,L", [("gqa_32x4k", 4), ("gqa_32x4k", 8), ("long_32k", 4), ("int8_mix", 4)])
def test_multi_query_many_fragments_per_ring(name, L):
    """Several hundred short sequences: every ring crosses many segments, so the
    ring's query buffer is refilled at each of its fragments (one warp per ring
    at 16 rows, two at 32)."""
    b = workloads.make_batch(name, seed=73, num_seqs=400, lengths=("uniform", 1, 120))
    _check(b, workloads.host_values(b, seed=73, q_len=L))

"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (an allocator-free serving loop, a plugin handed only its
input and output buffers, a process whose device memory pool belongs to
another framework) cannot pass pa_decode a workspace.  pa_decode_noalloc
uses a fixed array the library keeps in device memory instead.  These tests
call it through the C ABI and compare it with pa_decode on a caller-owned
workspace, twice in a row (the array keeps the previous call's contents).
This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

import workloads
from paged_cases import PA_TOL, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_144_gb300 as pa  # noqa: E402
from paged_kv_cache_144_gb300 import _lib  # noqa: E402


def _device_case(name, seed, **kw):
    b = workloads.make_batch(name, seed=seed, **kw)
    v = workloads.host_values(b, seed=seed, nan_tails=False)   # every slot holds a finite value
    dev = "cuda"
    t = dict(q=to_torch(v["q"], b.q_fmt, dev), k=to_torch(v["k_cache"], b.kv_fmt, dev),
             v=to_torch(v["v_cache"], b.kv_fmt, dev), tables=torch.from_numpy(b.block_tables).to(dev),
             lens=torch.from_numpy(b.seq_lens).to(dev))
    return b, t


def _noalloc_raw(b, t, out, partition_size=0):
    """Call the C entry point directly (argument marshalling only)."""
    q = t["q"]
    return _lib.pa_decode_noalloc(
        ctypes.c_void_p(out.data_ptr()), _lib.PA_F32, ctypes.c_void_p(q.data_ptr()), pa.dtype_code(q), q.stride(0),
        ctypes.c_void_p(t["k"].data_ptr()), ctypes.c_void_p(t["v"].data_ptr()), pa.dtype_code(t["k"]),
        t["k"].shape[0], None, None, ctypes.c_void_p(t["tables"].data_ptr()), b.max_blocks_per_seq,
        ctypes.c_void_p(t["lens"].data_ptr()), b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim,
        float(b.scale), b.block_size, partition_size,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name,kw", [
    ("gqa_32x4k", dict(num_seqs=8, lengths=("uniform", 1, 900))),
    ("long_32k", dict(num_seqs=2, lengths=("const", 2500))),
    ("tiny", {}),
])
def test_noalloc_matches_workspace_decode_twice(name, kw):
    b, t = _device_case(name, 21, **kw)
    ref = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device="cuda")
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                  b.max_blocks_per_seq, 0, pa.dtype_code(t["k"]))
    assert n <= pa.pa_decode_noalloc_capacity()
    ws = pa.new_workspace(n, "cuda")
    pa.decode(ref, t["q"], t["k"], t["v"], t["tables"], t["lens"], b.num_kv_heads, b.scale, b.block_size,
              workspace=ws)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_raw(b, t, out) == pa.PA_OK
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        d = (out - ref).abs().max().item()
        assert d <= PA_TOL, d


def test_noalloc_fixed_partitions_and_rejection():
    b, t = _device_case("gqa_32x4k", 22, num_seqs=4, lengths=("uniform", 100, 700))
    ref = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device="cuda")
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                  b.max_blocks_per_seq, 64, pa.dtype_code(t["k"]))
    pa.decode(ref, t["q"], t["k"], t["v"], t["tables"], t["lens"], b.num_kv_heads, b.scale, b.block_size,
              partition_size=64, workspace=pa.new_workspace(n, "cuda"))
    out = torch.empty_like(ref)
    assert _noalloc_raw(b, t, out, partition_size=64) == pa.PA_OK
    torch.cuda.synchronize()
    assert (out - ref).abs().max().item() <= PA_TOL
    # a batch whose fixed partitions need more records than the array holds is refused on the host
    big_tables = torch.zeros((16384, 512), dtype=torch.int32, device="cuda")
    big_lens = torch.ones(16384, dtype=torch.int32, device="cuda")
    q = torch.zeros((16384, 32, 128), dtype=torch.bfloat16, device="cuda")
    out_big = torch.empty((16384, 32, 128), dtype=torch.float32, device="cuda")
    st = _lib.pa_decode_noalloc(
        ctypes.c_void_p(out_big.data_ptr()), _lib.PA_F32, ctypes.c_void_p(q.data_ptr()), _lib.PA_BF16, 32 * 128,
        ctypes.c_void_p(t["k"].data_ptr()), ctypes.c_void_p(t["v"].data_ptr()), _lib.PA_BF16, t["k"].shape[0],
        None, None, ctypes.c_void_p(big_tables.data_ptr()), 512, ctypes.c_void_p(big_lens.data_ptr()),
        16384, 32, 8, 128, 0.1, 16, 16, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_ERR_WORKSPACE
    assert "more than the fixed" in _lib.load().pa_last_error_detail().decode()

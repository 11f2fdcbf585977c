"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (an allocator-free serving loop, a plugin handed only its
input and output buffers, a process whose device memory pool belongs to
another framework) cannot pass pa_decode a workspace.  pa_decode_noalloc
uses a fixed array the library keeps in device memory instead.  These tests
call it through the C ABI and require the same bits as pa_decode on a
caller-owned workspace (the same kernel, launched the same way), twice in a
row (the array keeps the previous call's contents), and agreement with the
oracle within the attention tolerance.  This file is collected last on
purpose.
"""

import ctypes

import numpy as np
import pytest

import oracle
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
    if b.kv_fmt == "e4m3":
        # the pool holds the oracle's quantisation of bf16 rows in every slot
        rng = np.random.default_rng(seed)
        for c in ("k_cache", "v_cache"):
            src = workloads.bf16_bits_from_f32(rng.standard_normal(v[c].shape, dtype=np.float32))
            v[c] = oracle.e4m3_encode_f32(oracle.bf16_bits_to_f64(src).astype(np.float32) * np.float32(40.0))
        v["k_scale"] = v["v_scale"] = np.full(b.num_kv_heads, 1.0 / 40.0, dtype=np.float32)
    t = dict(q=to_torch(v["q"], b.q_fmt, dev), k=to_torch(v["k_cache"], b.kv_fmt, dev),
             v=to_torch(v["v_cache"], b.kv_fmt, dev), tables=torch.from_numpy(b.block_tables).to(dev),
             lens=torch.from_numpy(b.seq_lens).to(dev), ks=None, vs=None)
    if b.kv_fmt == "e4m3":
        t["ks"] = torch.from_numpy(v["k_scale"]).to(dev)
        t["vs"] = torch.from_numpy(v["v_scale"]).to(dev)
    ref = oracle.paged_decode_attention(v["q"], v["k_cache"], v["v_cache"], b.block_tables, b.seq_lens, b.scale,
                                        b.block_size, q_fmt=b.q_fmt, kv_fmt=b.kv_fmt, k_scale=v.get("k_scale"),
                                        v_scale=v.get("v_scale"))
    return b, t, ref


def _vp(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _noalloc_raw(b, t, out, partition_size=0, kv_dtype=None):
    """Call the C entry point directly (argument marshalling only)."""
    q = t["q"]
    return _lib.pa_decode_noalloc(
        _vp(out), _lib.PA_F32, _vp(q), pa.dtype_code(q), q.stride(0),
        _vp(t["k"]), _vp(t["v"]), pa.dtype_code(t["k"]) if kv_dtype is None else kv_dtype,
        t["k"].shape[0], _vp(t["ks"]), _vp(t["vs"]), _vp(t["tables"]), b.max_blocks_per_seq,
        _vp(t["lens"]), b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim,
        float(b.scale), b.block_size, partition_size,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name,kw", [
    ("gqa_32x4k", dict(num_seqs=8, lengths=("uniform", 1, 900))),
    ("long_32k", dict(num_seqs=2, lengths=("const", 2500))),
    ("fp8_mix", dict(num_seqs=6, lengths=("lognormal", 6.0, 1.0, 16, 1500))),
    ("tiny", {}),
])
def test_noalloc_matches_workspace_decode_twice(name, kw):
    b, t, oref = _device_case(name, 21, **kw)
    ref = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device="cuda")
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                  b.max_blocks_per_seq, 0, pa.dtype_code(t["k"]))
    assert n <= pa.pa_decode_noalloc_capacity()
    ws = pa.new_workspace(n, "cuda")
    pa.decode(ref, t["q"], t["k"], t["v"], t["tables"], t["lens"], b.num_kv_heads, b.scale, b.block_size,
              k_scale=t["ks"], v_scale=t["vs"], workspace=ws)
    torch.cuda.synchronize()
    assert np.max(np.abs(ref.cpu().numpy().astype(np.float64) - oref)) <= PA_TOL
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_raw(b, t, out) == pa.PA_OK
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert torch.equal(out, ref)             # same kernel, same launch: the same bits


def test_noalloc_fixed_partitions_and_rejection():
    b, t, oref = _device_case("gqa_32x4k", 22, num_seqs=4, lengths=("uniform", 100, 700))
    ref = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device="cuda")
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                  b.max_blocks_per_seq, 64, pa.dtype_code(t["k"]))
    pa.decode(ref, t["q"], t["k"], t["v"], t["tables"], t["lens"], b.num_kv_heads, b.scale, b.block_size,
              partition_size=64, workspace=pa.new_workspace(n, "cuda"))
    out = torch.empty_like(ref)
    assert _noalloc_raw(b, t, out, partition_size=64) == pa.PA_OK
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert np.max(np.abs(out.cpu().numpy().astype(np.float64) - oref)) <= PA_TOL
    # rejected on the host, before anything is enqueued: INT8 caches (no zero-point arguments), a NULL output
    assert _noalloc_raw(b, t, out, kv_dtype=_lib.PA_INT8) == pa.PA_ERR_UNSUPPORTED
    t_null = dict(t, tables=None)
    assert _noalloc_raw(b, t_null, out) == pa.PA_ERR_NULL
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

"""Fused append + decode (pa_decode_ex with k_new / v_new) against the oracle.

One launch writes every sequence's newest rows into their cache slots and
attends over them; the result must equal the cache write followed by the
decode (oracle.paged_append_decode): cache bytes bit-exact, attention within
2e-3.  The stale slot holds NaN beforehand (16-bit caches), so a kernel that
attends the old row instead of the new one fails.
"""

import numpy as np
import pytest

import oracle
import workloads
from paged_cases import PA_TOL, bits_equal, to_numpy, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_144_gb300 as pa  # noqa: E402


def _run(batch, vals, *, window=0, partition_size=0, device="cuda"):
    kv, B = batch.kv_fmt, batch.block_size
    quant = kv in ("e4m3", "i8")
    src_fmt = "bf16" if quant else kv
    q = to_torch(vals["q"], batch.q_fmt, device)
    kc = to_torch(vals["k_cache"], kv, device)
    vc = to_torch(vals["v_cache"], kv, device)
    okc, ovc = vals["k_cache"], vals["v_cache"]
    ks = vs = kis = vis = kz = vz = None
    zkw = {}
    if quant:
        ks, vs = (torch.from_numpy(vals[n]).to(device) for n in ("k_scale", "v_scale"))
        kis, vis = (torch.from_numpy(vals[n]).to(device) for n in ("k_inv_scale", "v_inv_scale"))
        if kv == "i8":
            kz, vz = (torch.from_numpy(vals[n]).to(device) for n in ("k_zero_point", "v_zero_point"))
            zkw = dict(k_zero_point=vals["k_zero_point"], v_zero_point=vals["v_zero_point"])
        pa.reshape_and_cache(to_torch(vals["k_src"], "bf16", device), to_torch(vals["v_src"], "bf16", device),
                             kc, vc, torch.from_numpy(vals["src_slots"]).to(device), B, k_inv_scale=kis,
                             v_inv_scale=vis, k_zero_point=kz, v_zero_point=vz)
        okc, ovc = oracle.reshape_and_cache(vals["k_src"], vals["v_src"], okc, ovc, vals["src_slots"], B,
                                            src_fmt="bf16", kv_fmt=kv, k_inv_scale=vals["k_inv_scale"],
                                            v_inv_scale=vals["v_inv_scale"], **zkw)
    tables = torch.from_numpy(batch.block_tables).to(device)
    lens = torch.from_numpy(batch.seq_lens).to(device)
    out = torch.empty((batch.num_seqs, batch.num_heads, batch.head_dim), dtype=torch.float32, device=device)
    n = pa.decode_workspace_bytes(batch.num_seqs, batch.num_heads, batch.num_kv_heads, batch.head_dim, B,
                                  batch.max_blocks_per_seq, partition_size, pa.dtype_code(kc))
    ws = pa.new_workspace(n, device) if n else None
    pa.decode(out, q, kc, vc, tables, lens, batch.num_kv_heads, batch.scale, B, k_scale=ks, v_scale=vs,
              partition_size=partition_size, workspace=ws, window=window, k_zero_point=kz, v_zero_point=vz,
              k_new=to_torch(vals["k_new"], src_fmt, device), v_new=to_torch(vals["v_new"], src_fmt, device),
              k_inv_scale=kis, v_inv_scale=vis)
    err = pa.get_device_error()
    ref, rk, rv = oracle.paged_append_decode(
        vals["q"], vals["k_new"], vals["v_new"], okc, ovc, batch.block_tables, batch.seq_lens, batch.scale, B,
        q_fmt=batch.q_fmt, src_fmt=src_fmt, kv_fmt=kv, k_scale=vals.get("k_scale"), v_scale=vals.get("v_scale"),
        k_inv_scale=vals.get("k_inv_scale"), v_inv_scale=vals.get("v_inv_scale"), window=window, **zkw)
    assert err == 0, f"device error bits {err}"
    assert bits_equal(to_numpy(kc, kv), rk), "k_cache bytes differ"
    assert bits_equal(to_numpy(vc, kv), rv), "v_cache bytes differ"
    o = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o))
    d = np.abs(o - ref).max()
    assert d <= PA_TOL, f"max abs err {d:.3e}"
    return d


@pytest.mark.parametrize("mode", [0, 128])
def test_append_gqa_bf16(mode):
    b = workloads.make_batch("gqa_32x4k", seed=50, num_seqs=9, lengths=("uniform", 1, 900))
    _run(b, workloads.host_values(b, seed=50), partition_size=mode)


@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_append_block_sizes_f16_d64(B):
    b = workloads.make_batch("tiny", seed=51, block_size=B, num_seqs=6, lengths=("uniform", 1, 300),
                             pool=("slack", 0.1))
    _run(b, workloads.host_values(b, seed=51))


@pytest.mark.parametrize("kv", ["fp8_mix", "int8_mix"])
@pytest.mark.parametrize("B", [16, 32])
def test_append_quantised_caches(kv, B):
    b = workloads.make_batch(kv, seed=52, num_seqs=10, block_size=B, lengths=("lognormal", 6.0, 1.0, 16, 1500))
    _run(b, workloads.host_values(b, seed=52))


def test_append_with_window_and_single_token_sequences():
    b = workloads.make_batch("gqa_32x4k", seed=53, num_seqs=7, lengths=("uniform", 1, 40))
    b.seq_lens = b.seq_lens.copy()
    b.seq_lens[:3] = 1
    _run(b, workloads.host_values(b, seed=53), window=17)


def test_append_long_group8():
    b = workloads.make_batch("long_32k", seed=54, num_seqs=2, lengths=("const", 2049))
    _run(b, workloads.host_values(b, seed=54))

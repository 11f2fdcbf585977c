"""The bounded-wait path of the decode kernel, exercised without any fault.

Every wait of the decode pipeline on a barrier gives up after a limit and
records PA_DEVERR_TIMEOUT instead of hanging.  Here the limit is shortened to
10 ms and the producer warp is told to issue no copy (pa_debug_set_decode_wait),
so every consumer waits on a barrier that nothing completes: the call must
return, the error bit must be set, and after the workspace is zeroed again
(as pa.h asks after a timeout) the next ordinary call must match the oracle.
"""

import time

import numpy as np
import pytest

import workloads
from paged_cases import PA_TOL, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import paged_kv_cache_144_gb300 as pa  # noqa: E402


@pytest.mark.parametrize("name,kw", [
    ("gqa_32x4k", dict(num_seqs=6, lengths=("uniform", 50, 900))),
    ("fp8_mix", dict(num_seqs=6, lengths=("lognormal", 6.0, 1.0, 16, 1500))),
])
def test_wait_limit_runs_out_then_next_call_is_exact(name, kw):
    b = workloads.make_batch(name, seed=31, **kw)
    v = workloads.host_values(b, seed=31, nan_tails=False)
    dev = "cuda"
    ks = vs = None
    if b.kv_fmt == "e4m3":
        rng = np.random.default_rng(31)
        for c in ("k_cache", "v_cache"):
            v[c] = oracle.e4m3_encode_f32(rng.standard_normal(v[c].shape).astype(np.float32) * np.float32(40.0))
        v["k_scale"] = v["v_scale"] = np.full(b.num_kv_heads, 1.0 / 40.0, dtype=np.float32)
        ks = torch.from_numpy(v["k_scale"]).to(dev)
        vs = torch.from_numpy(v["v_scale"]).to(dev)
    q = to_torch(v["q"], b.q_fmt, dev)
    kc, vc = to_torch(v["k_cache"], b.kv_fmt, dev), to_torch(v["v_cache"], b.kv_fmt, dev)
    tables, lens = torch.from_numpy(b.block_tables).to(dev), torch.from_numpy(b.seq_lens).to(dev)
    out = torch.zeros((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device=dev)
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                  b.max_blocks_per_seq, 0, pa.dtype_code(kc))
    ws = pa.new_workspace(n, dev)
    assert pa.get_device_error() == 0
    pa.pa_debug_set_decode_wait(10_000_000, True)      # 10 ms, and no copy is ever issued
    try:
        t0 = time.perf_counter()
        pa.decode(out, q, kc, vc, tables, lens, b.num_kv_heads, b.scale, b.block_size, k_scale=ks, v_scale=vs,
                  workspace=ws)
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
    finally:
        pa.pa_debug_set_decode_wait(0, False)           # the default limit, copies issued again
    err = pa.get_device_error()
    assert err & pa.PA_DEVERR_TIMEOUT, f"error bits {err}"
    assert waited < 1.0, f"the call took {waited:.3f} s: the short limit was not applied"
    ws.zero_()
    out.zero_()
    pa.decode(out, q, kc, vc, tables, lens, b.num_kv_heads, b.scale, b.block_size, k_scale=ks, v_scale=vs,
              workspace=ws)
    assert pa.get_device_error() == 0
    ref = oracle.paged_decode_attention(v["q"], v["k_cache"], v["v_cache"], b.block_tables, b.seq_lens, b.scale,
                                        b.block_size, q_fmt=b.q_fmt, kv_fmt=b.kv_fmt, k_scale=v.get("k_scale"),
                                        v_scale=v.get("v_scale"))
    assert np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)) <= PA_TOL

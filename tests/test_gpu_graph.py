"""A serving step recorded as a CUDA graph (pa.StepGraph) and replayed gives the same bytes as the step
issued call by call: the cache write of the new tokens and the decode, with programmatic dependent launch,
inputs staged from pinned host memory and the output copied back; and the result matches the oracle."""

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


@pytest.mark.parametrize("pdl", [True, False])
def test_recorded_step_replays_the_eager_step(pdl):
    b = workloads.make_batch("gqa_32x4k", seed=41, num_seqs=9, lengths=("uniform", 1, 800))
    v = workloads.host_values(b, seed=41)
    dev = "cuda"
    B = b.block_size
    kc0, vc0 = to_torch(v["k_cache"], b.kv_fmt, dev), to_torch(v["v_cache"], b.kv_fmt, dev)
    tables = torch.from_numpy(b.block_tables).to(dev)
    lens = torch.from_numpy(b.seq_lens).to(dev)
    slots = torch.from_numpy(b.new_slots).to(dev)
    h_q = to_torch(v["q"], b.q_fmt, "cpu").pin_memory()
    h_k, h_v = to_torch(v["k_new"], b.kv_fmt, "cpu").pin_memory(), to_torch(v["v_new"], b.kv_fmt, "cpu").pin_memory()
    d_q, d_k, d_v = torch.empty_like(h_q, device=dev), torch.empty_like(h_k, device=dev), torch.empty_like(h_v, device=dev)
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, B, b.max_blocks_per_seq, 0,
                                  pa.dtype_code(kc0))
    ws = pa.new_workspace(n, dev)
    out = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device=dev)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def step(kc, vc):
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        pa.reshape_and_cache(d_k, d_v, kc, vc, slots, B, pdl=pdl)
        pa.decode(out, d_q, kc, vc, tables, lens, b.num_kv_heads, b.scale, B, workspace=ws, pdl=pdl)
        h_out.copy_(out, non_blocking=True)

    kc1, vc1 = kc0.clone(), vc0.clone()
    step(kc1, vc1)
    torch.cuda.synchronize()
    eager = h_out.clone()
    kc2, vc2 = kc0.clone(), vc0.clone()
    g = pa.StepGraph(lambda: step(kc2, vc2))
    for _ in range(3):
        h_out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(h_out, eager)
    # byte comparison: unused slots of the pool hold NaN
    assert torch.equal(kc1.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc1.view(torch.int16), vc2.view(torch.int16))
    assert pa.get_device_error() == 0
    okc, ovc = oracle.reshape_and_cache(v["k_new"], v["v_new"], v["k_cache"], v["v_cache"], b.new_slots, B,
                                        src_fmt=b.kv_fmt, kv_fmt=b.kv_fmt)
    ref = oracle.paged_decode_attention(v["q"], okc, ovc, b.block_tables, b.seq_lens, b.scale, B, q_fmt=b.q_fmt,
                                        kv_fmt=b.kv_fmt)
    assert np.max(np.abs(eager.numpy().astype(np.float64) - ref)) <= PA_TOL

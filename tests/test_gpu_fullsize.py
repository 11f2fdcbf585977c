"""Full-size workloads in the launch configuration bench.py times (balanced
split with workspace); outputs sampled per (sequence, head) and checked
against the oracle computed one by one from host copies of the used blocks."""

import numpy as np
import pytest

import oracle
import workloads
from paged_cases import PA_TOL, bits_equal, to_numpy

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_144_gb300 as pa  # noqa: E402


def _samples(batch, n, rng):
    S, Hq = batch.num_seqs, batch.num_heads
    order = np.argsort(batch.seq_lens)
    seqs = [int(order[0]), int(order[-1])] + [int(x) for x in rng.integers(0, S, size=n - 2)]
    return [(s, int(rng.integers(0, Hq))) for s in seqs]


def _run_full(name, seed, *, q_mult=1.0, n_samples=12, **overrides):
    dev = "cuda"
    b = workloads.make_batch(name, seed=seed, **overrides)
    vals = workloads.device_values(b, seed, dev, q_mult=q_mult)
    B, Hkv, D = b.block_size, b.num_kv_heads, b.head_dim
    kc, vc = vals["k_cache"], vals["v_cache"]
    quant = b.kv_fmt in ("e4m3", "i8")
    ks = vs = kis = vis = None
    kz, vz = vals.get("k_zero_point"), vals.get("v_zero_point")
    if quant:
        ks, vs, kis, vis = vals["k_scale"], vals["v_scale"], vals["k_inv_scale"], vals["v_inv_scale"]
        pa.reshape_and_cache(vals["k_src"], vals["v_src"], kc, vc, vals["src_slots"], B,
                             k_inv_scale=kis, v_inv_scale=vis, k_zero_point=kz, v_zero_point=vz)
    pa.reshape_and_cache(vals["k_new"], vals["v_new"], kc, vc, torch.from_numpy(b.new_slots).to(dev), B,
                         k_inv_scale=kis, v_inv_scale=vis, k_zero_point=kz, v_zero_point=vz)
    tables = torch.from_numpy(b.block_tables).to(dev)
    lens = torch.from_numpy(b.seq_lens).to(dev)
    out = torch.empty((b.num_seqs, b.num_heads, D), dtype=torch.float32, device=dev)
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, Hkv, D, B, b.max_blocks_per_seq, 0,
                                  pa.dtype_code(kc))
    ws = pa.new_workspace(n, dev)
    pa.decode(out, vals["q"], kc, vc, tables, lens, Hkv, b.scale, B, k_scale=ks, v_scale=vs, workspace=ws,
              k_zero_point=kz, v_zero_point=vz)
    assert pa.get_device_error() == 0
    out_h = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(out_h))
    q_h = to_numpy(vals["q"], b.q_fmt)
    rng = np.random.default_rng(seed + 99)
    src_off = np.concatenate([[0], np.cumsum(b.seq_lens.astype(np.int64) - 1)])
    worst = 0.0
    for s, h in _samples(b, n_samples, rng):
        T = int(b.seq_lens[s])
        nb = -(-T // B)
        blocks = torch.from_numpy(b.block_tables[s, :nb].astype(np.int64)).to(dev)
        gk = to_numpy(kc.index_select(0, blocks), b.kv_fmt)
        gv = to_numpy(vc.index_select(0, blocks), b.kv_fmt)
        local_tables = np.arange(nb, dtype=np.int32)[None, :]
        if quant:
            # the sequence's bytes must equal the oracle's quantisation of its bf16 rows
            zkw = {}
            if b.kv_fmt == "i8":
                zkw = dict(k_zero_point=kz.cpu().numpy(), v_zero_point=vz.cpu().numpy())
            rows = slice(int(src_off[s]), int(src_off[s + 1]))
            kr = np.concatenate([to_numpy(vals["k_src"][rows], "bf16"), to_numpy(vals["k_new"][s:s + 1], "bf16")])
            vr = np.concatenate([to_numpy(vals["v_src"][rows], "bf16"), to_numpy(vals["v_new"][s:s + 1], "bf16")])
            zero = np.zeros_like(gk)
            ok, ov = oracle.reshape_and_cache(kr, vr, zero, zero, np.arange(T), B, src_fmt="bf16", kv_fmt=b.kv_fmt,
                                              k_inv_scale=kis.cpu().numpy(), v_inv_scale=vis.cpu().numpy(), **zkw)
            assert bits_equal(gk, ok) and bits_equal(gv, ov), f"{b.kv_fmt} cache bytes of sequence {s}"
            ref = oracle.paged_decode_attention_one(q_h[s:s + 1], ok, ov, local_tables, np.array([T]), b.scale, B,
                                                    0, h, q_fmt=b.q_fmt, kv_fmt=b.kv_fmt, k_scale=ks.cpu().numpy(),
                                                    v_scale=vs.cpu().numpy(), num_kv_heads=Hkv, **zkw)
        else:
            # the appended row landed in its slot
            kvh = h // b.group
            slot = int(b.new_slots[s])
            assert bits_equal(gk[(T - 1) // B, kvh, (T - 1) % B], to_numpy(vals["k_new"][s, kvh], b.kv_fmt))
            ref = oracle.paged_decode_attention_one(q_h[s:s + 1], gk, gv, local_tables, np.array([T]), b.scale, B,
                                                    0, h, q_fmt=b.q_fmt, kv_fmt=b.kv_fmt, num_kv_heads=Hkv)
            assert slot // B == b.block_tables[s, (T - 1) // B]
        err = float(np.max(np.abs(out_h[s, h] - ref)))
        worst = max(worst, err)
        assert err <= PA_TOL, f"(s={s}, h={h}) err {err:.3e}"
    return worst


def test_gqa_32x4k_full():
    _run_full("gqa_32x4k", 0, n_samples=16)


@pytest.mark.parametrize("q_mult", [1.0, 30.0])
def test_long_32k_full(q_mult):
    _run_full("long_32k", 0, q_mult=q_mult, n_samples=8)


@pytest.mark.parametrize("B", [16, 32])
def test_fp8_mix_full(B):
    _run_full("fp8_mix", 0, block_size=B, n_samples=10)


def test_int8_mix_full():
    _run_full("int8_mix", 0, n_samples=10)

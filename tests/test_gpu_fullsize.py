"""Full-size workloads in the launch configuration bench.py times (balanced
split with workspace): every output of every (sequence, query head) is
compared with the oracle, computed sequence by sequence from host copies of
the blocks that sequence uses.  The cache write of each sequence's newest
token (and, for 8-bit caches, the quantising write of every row) is checked
byte for byte on the same host copies."""

import numpy as np
import pytest

import workloads
from paged_cases import check_sequence, oracle_pool, to_numpy

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_144_gb300 as pa  # noqa: E402


def _run_full(name, seed, *, q_mult=1.0, **overrides):
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
    qkw, quant_rows = {}, None
    if quant:
        qkw = dict(k_scale=ks.cpu().numpy(), v_scale=vs.cpu().numpy())
        if b.kv_fmt == "i8":
            qkw.update(k_zero_point=kz.cpu().numpy(), v_zero_point=vz.cpu().numpy())
        quant_rows = (to_numpy(vals["k_src"], "bf16"), to_numpy(vals["v_src"], "bf16"),
                      np.concatenate([[0], np.cumsum(b.seq_lens.astype(np.int64) - 1)]),
                      kis.cpu().numpy(), vis.cpu().numpy())
        k_new, v_new = to_numpy(vals["k_new"], "bf16"), to_numpy(vals["v_new"], "bf16")
    else:
        k_new, v_new = to_numpy(vals["k_new"], b.kv_fmt), to_numpy(vals["v_new"], b.kv_fmt)
    meta = dict(B=B, scale=b.scale, q_fmt=b.q_fmt, kv_fmt=b.kv_fmt, qkw=qkw)

    def items():
        # host copies of one sequence at a time: the blocks it uses, its query rows, its written rows
        for s in range(b.num_seqs):
            T = int(b.seq_lens[s])
            nb = -(-T // B)
            blocks = torch.from_numpy(b.block_tables[s, :nb].astype(np.int64)).to(dev)
            gk = to_numpy(kc.index_select(0, blocks), b.kv_fmt)
            gv = to_numpy(vc.index_select(0, blocks), b.kv_fmt)
            item = dict(meta, s=s, T=T, gk=gk, gv=gv, q=q_h[s:s + 1], out=out_h[s], k_new=k_new[s], v_new=v_new[s],
                        new_slot=int(b.new_slots[s]), table=b.block_tables[s, :nb].copy())
            if quant:
                k_src, v_src, off, kis_h, vis_h = quant_rows
                rows = slice(int(off[s]), int(off[s + 1]))
                item.update(k_rows=k_src[rows], v_rows=v_src[rows], k_inv_scale=kis_h, v_inv_scale=vis_h)
            yield item

    worst = 0.0
    for s, err, msg in oracle_pool().imap(check_sequence, items(), chunksize=1):
        assert msg is None, f"sequence {s}: {msg}"
        worst = max(worst, err)
    return worst


def test_gqa_32x4k_full():
    _run_full("gqa_32x4k", 0)


@pytest.mark.parametrize("q_mult", [1.0, 30.0])
def test_long_32k_full(q_mult):
    _run_full("long_32k", 0, q_mult=q_mult)


@pytest.mark.parametrize("B", [16, 32])
def test_fp8_mix_full(B):
    _run_full("fp8_mix", 0, block_size=B)


def test_int8_mix_full():
    _run_full("int8_mix", 0)

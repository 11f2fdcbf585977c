"""Programmatic dependent launch (pa_decode_ex option pdl) against the oracle
and against the ordinary launch.

With pdl on, the decode's set-up runs while the kernel launched just before
it on the stream is still running.  The cases put right before it a kernel
that writes what the decode reads afterwards:
  * a cache write of every attended row into pools that hold NaN everywhere,
    so a decode that read the cache before that write had finished would
    return NaN (or values off by far more than the tolerance);
  * a decode on the same workspace, whose split counters the earlier decode
    resets only at its very end.
The decode itself is deterministic (fixed merge order), so the pdl and the
ordinary launch must give the same bits.
"""

import numpy as np
import pytest

import oracle
import workloads
from paged_cases import PA_TOL, bits_equal, run_gpu, run_oracle, to_numpy, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_144_gb300 as pa  # noqa: E402

NAN16 = {"f16": np.uint16(0x7E00), "bf16": np.uint16(0x7FC0)}

CASES = [
    ("tiny", dict(), 0),
    ("gqa_32x4k", dict(num_seqs=8, lengths=("uniform", 1, 1500)), 0),
    ("gqa_32x4k", dict(num_seqs=8, lengths=("uniform", 1, 1500)), 512),
    ("long_32k", dict(num_seqs=2, lengths=("const", 4000)), 0),
]


def _all_rows(batch, kc, vc):
    """Every attended row of the (oracle) caches as [N, H_kv, d] sources, with their slots."""
    B = batch.block_size
    blk, off = [], []
    for s in range(batch.num_seqs):
        pos = np.arange(int(batch.seq_lens[s]))
        blk.append(batch.block_tables[s][pos // B])
        off.append(pos % B)
    blk, off = np.concatenate(blk), np.concatenate(off)
    slots = (blk.astype(np.int64) * B + off).astype(np.int64)
    return kc[blk, :, off, :], vc[blk, :, off, :], slots


def _setup(name, kw, seed=11):
    b = workloads.make_batch(name, seed=seed, **kw)
    vals = workloads.host_values(b, seed=seed)
    ref, okc, ovc = run_oracle(b, vals)
    return b, vals, ref, okc, ovc


def _decode(b, q, kc, vc, tables, lens, ws, partition_size, pdl):
    out = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device="cuda")
    pa.decode(out, q, kc, vc, tables, lens, b.num_kv_heads, b.scale, b.block_size, partition_size=partition_size,
              workspace=ws, pdl=pdl)
    return out


@pytest.mark.parametrize("name,kw,partition_size", CASES)
def test_pdl_decode_after_a_cache_write_of_every_row(name, kw, partition_size):
    b, vals, ref, okc, ovc = _setup(name, kw)
    kv = b.kv_fmt
    ksrc, vsrc, slots = _all_rows(b, okc, ovc)
    nan_pool = np.full(okc.shape, NAN16[kv], dtype=np.uint16)
    kc = to_torch(nan_pool.view(np.float16) if kv == "f16" else nan_pool, kv, "cuda")
    vc = to_torch(nan_pool.view(np.float16) if kv == "f16" else nan_pool, kv, "cuda")
    q = to_torch(vals["q"], b.q_fmt, "cuda")
    tables = torch.from_numpy(b.block_tables).cuda()
    lens = torch.from_numpy(b.seq_lens).cuda()
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                  b.max_blocks_per_seq, partition_size, pa.dtype_code(kc))
    ws = pa.new_workspace(n, "cuda") if n else None
    torch.cuda.synchronize()
    # the write and the decode right after it, on one stream, nothing between them
    pa.reshape_and_cache(to_torch(ksrc, kv, "cuda"), to_torch(vsrc, kv, "cuda"), kc, vc,
                         torch.from_numpy(slots).cuda(), b.block_size)
    out_pdl = _decode(b, q, kc, vc, tables, lens, ws, partition_size, True)
    out_ord = _decode(b, q, kc, vc, tables, lens, ws, partition_size, False)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    o = out_pdl.cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all()
    assert np.max(np.abs(o - ref)) <= PA_TOL
    assert bits_equal(out_pdl.cpu().numpy(), out_ord.cpu().numpy())
    # the written slots hold the oracle's bytes
    kg = to_numpy(kc, kv)
    blk, off = slots // b.block_size, slots % b.block_size
    assert bits_equal(kg[blk, :, off, :], np.ascontiguousarray(okc[blk, :, off, :]))


@pytest.mark.parametrize("name,kw,partition_size", CASES[1:])
def test_pdl_back_to_back_decodes_on_one_workspace(name, kw, partition_size):
    b, vals, ref, okc, ovc = _setup(name, kw, seed=12)
    kv = b.kv_fmt
    kc, vc = to_torch(okc, kv, "cuda"), to_torch(ovc, kv, "cuda")
    q = to_torch(vals["q"], b.q_fmt, "cuda")
    tables = torch.from_numpy(b.block_tables).cuda()
    lens = torch.from_numpy(b.seq_lens).cuda()
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                  b.max_blocks_per_seq, partition_size, pa.dtype_code(kc))
    assert n > 0, "the case must split segments"
    ws = pa.new_workspace(n, "cuda")
    torch.cuda.synchronize()
    outs = [_decode(b, q, kc, vc, tables, lens, ws, partition_size, True) for _ in range(5)]
    first = _decode(b, q, kc, vc, tables, lens, ws, partition_size, False)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    o = first.cpu().numpy()
    assert np.max(np.abs(o.astype(np.float64) - ref)) <= PA_TOL
    for x in outs:
        assert bits_equal(x.cpu().numpy(), o)


@pytest.mark.parametrize("name,kw", [
    ("fp8_mix", dict(num_seqs=8, lengths=("lognormal", 6.0, 1.0, 16, 1500))),
    ("int8_mix", dict(num_seqs=8, lengths=("lognormal", 6.0, 1.0, 16, 1500))),
])
def test_pdl_decode_after_quantising_cache_writes(name, kw):
    b = workloads.make_batch(name, seed=13, **kw)
    vals = workloads.host_values(b, seed=13)
    ref, okc, ovc = run_oracle(b, vals)
    out, kc, vc, err = run_gpu(b, vals, pdl=True)
    out0, _, _, _ = run_gpu(b, vals, pdl=False)
    assert err == 0
    assert bits_equal(kc, okc) and bits_equal(vc, ovc)
    assert np.max(np.abs(out - ref)) <= PA_TOL
    assert bits_equal(out, out0)


def test_pdl_fused_append_after_a_decode():
    b, vals, _, _, _ = _setup("gqa_32x4k", dict(num_seqs=6, lengths=("uniform", 1, 1200)), seed=14)
    kv, B = b.kv_fmt, b.block_size
    q = to_torch(vals["q"], b.q_fmt, "cuda")
    tables = torch.from_numpy(b.block_tables).cuda()
    lens = torch.from_numpy(b.seq_lens).cuda()
    res = []
    for pdl in (True, False):
        kc, vc = to_torch(vals["k_cache"], kv, "cuda"), to_torch(vals["v_cache"], kv, "cuda")
        n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, B,
                                      b.max_blocks_per_seq, 0, pa.dtype_code(kc))
        ws = pa.new_workspace(n, "cuda") if n else None
        torch.cuda.synchronize()
        warm = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=torch.float32, device="cuda")
        pa.decode(warm, q, kc, vc, tables, lens, b.num_kv_heads, b.scale, B, workspace=ws)  # before the new rows
        out = torch.empty_like(warm)
        pa.decode(out, q, kc, vc, tables, lens, b.num_kv_heads, b.scale, B, workspace=ws,
                  k_new=to_torch(vals["k_new"], kv, "cuda"), v_new=to_torch(vals["v_new"], kv, "cuda"), pdl=pdl)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        res.append((out.cpu().numpy(), to_numpy(kc, kv), to_numpy(vc, kv)))
    ref, rk, rv = oracle.paged_append_decode(vals["q"], vals["k_new"], vals["v_new"], vals["k_cache"], vals["v_cache"],
                                             b.block_tables, b.seq_lens, b.scale, B, q_fmt=b.q_fmt, src_fmt=kv,
                                             kv_fmt=kv)
    (o1, k1, v1), (o0, k0, v0) = res
    assert bits_equal(k1, rk) and bits_equal(v1, rv)
    assert np.max(np.abs(o1.astype(np.float64) - ref)) <= PA_TOL
    assert bits_equal(o1, o0) and bits_equal(k1, k0) and bits_equal(v1, v0)


def _scaled_rows(rows, fmt, factor):
    """rows (16-bit storage) times a power of two, exactly, in the same storage."""
    t = torch.from_numpy(np.ascontiguousarray(rows).view(np.int16 if fmt == "bf16" else np.float16))
    t = t.view(torch.bfloat16) if fmt == "bf16" else t
    out = (t.float() * factor).to(t.dtype)
    return out.view(torch.int16).numpy().view(np.uint16) if fmt == "bf16" else out.numpy()


@pytest.mark.parametrize("name,kw", [CASES[1][:2], CASES[3][:2]])
def test_pdl_cache_write_waits_for_the_decode_before_it(name, kw):
    """A cache write launched with pdl right after a decode rewrites every row that decode reads (with
    values of another scale); the decode must still see the old rows, the cache must end with the new."""
    b, vals, ref, okc, ovc = _setup(name, kw, seed=15)
    kv, B = b.kv_fmt, b.block_size
    ksrc, vsrc, slots = _all_rows(b, okc, ovc)
    knew, vnew = _scaled_rows(ksrc, kv, -4.0), _scaled_rows(vsrc, kv, 8.0)
    kc, vc = to_torch(okc, kv, "cuda"), to_torch(ovc, kv, "cuda")
    q = to_torch(vals["q"], b.q_fmt, "cuda")
    tables = torch.from_numpy(b.block_tables).cuda()
    lens = torch.from_numpy(b.seq_lens).cuda()
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, B, b.max_blocks_per_seq, 0,
                                  pa.dtype_code(kc))
    ws = pa.new_workspace(n, "cuda") if n else None
    kn, vn, sl = to_torch(knew, kv, "cuda"), to_torch(vnew, kv, "cuda"), torch.from_numpy(slots).cuda()
    torch.cuda.synchronize()
    out = _decode(b, q, kc, vc, tables, lens, ws, 0, True)
    pa.reshape_and_cache(kn, vn, kc, vc, sl, B, pdl=True)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)) <= PA_TOL
    rk, rv = oracle.reshape_and_cache(knew, vnew, okc, ovc, slots, B, src_fmt=kv, kv_fmt=kv)
    assert bits_equal(to_numpy(kc, kv), rk) and bits_equal(to_numpy(vc, kv), rv)


@pytest.mark.parametrize("name,kw", [CASES[0][:2], CASES[1][:2]])
def test_pdl_chain_of_write_and_decode_steps(name, kw):
    """Steps of (cache write of every row, pdl) -> (decode, pdl) on one stream and one workspace, each step
    with rows of another scale: every decode sees its own step's rows and none of the next step's."""
    b, vals, _, okc, ovc = _setup(name, kw, seed=16)
    kv, B = b.kv_fmt, b.block_size
    ksrc, vsrc, slots = _all_rows(b, okc, ovc)
    kc, vc = to_torch(okc, kv, "cuda"), to_torch(ovc, kv, "cuda")
    q = to_torch(vals["q"], b.q_fmt, "cuda")
    tables = torch.from_numpy(b.block_tables).cuda()
    lens = torch.from_numpy(b.seq_lens).cuda()
    n = pa.decode_workspace_bytes(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, B, b.max_blocks_per_seq, 0,
                                  pa.dtype_code(kc))
    ws = pa.new_workspace(n, "cuda") if n else None
    sl = torch.from_numpy(slots).cuda()
    factors = [(0.5, 2.0), (-1.0, 0.25), (2.0, -1.0), (0.25, 4.0)]
    rows = [(_scaled_rows(ksrc, kv, fk), _scaled_rows(vsrc, kv, fv)) for fk, fv in factors]
    dev_rows = [(to_torch(a, kv, "cuda"), to_torch(c, kv, "cuda")) for a, c in rows]
    torch.cuda.synchronize()
    outs = []
    for kn, vn in dev_rows:
        pa.reshape_and_cache(kn, vn, kc, vc, sl, B, pdl=True)
        outs.append(_decode(b, q, kc, vc, tables, lens, ws, 0, True))
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    for (knew, vnew), o in zip(rows, outs):
        rk, rv = oracle.reshape_and_cache(knew, vnew, okc, ovc, slots, B, src_fmt=kv, kv_fmt=kv)
        ref = oracle.paged_decode_attention(vals["q"], rk, rv, b.block_tables, b.seq_lens, b.scale, B,
                                            q_fmt=b.q_fmt, kv_fmt=kv)
        assert np.max(np.abs(o.cpu().numpy().astype(np.float64) - ref)) <= PA_TOL
    assert bits_equal(to_numpy(kc, kv), rk) and bits_equal(to_numpy(vc, kv), rv)


@pytest.mark.parametrize("name,kw,partition_size,window", [
    ("gqa_32x4k", dict(num_seqs=8, lengths=("uniform", 1, 1500)), 0, 0),
    ("gqa_32x4k", dict(num_seqs=8, lengths=("uniform", 1, 1500)), 512, 0),
    ("gqa_32x4k", dict(num_seqs=8, lengths=("uniform", 1, 1500)), 0, 100),
    ("gqa_32x4k", dict(num_seqs=40, lengths=("uniform", 1, 3)), 0, 0),
    ("long_32k", dict(num_seqs=2, lengths=("const", 4000)), 0, 0),
    ("fp8_mix", dict(num_seqs=8, lengths=("lognormal", 6.0, 1.0, 16, 1500)), 0, 0),
    ("int8_mix", dict(num_seqs=8, lengths=("lognormal", 6.0, 1.0, 16, 1500)), 0, 0),
])
def test_early_kv_decode_after_the_steps_cache_write(name, kw, partition_size, window):
    """The step as a serving loop issues it: the cache write of each sequence's newest row, then the decode
    with pdl and early_kv, which copies the other rows before that write has finished.  Before the write the
    newest rows' slots hold NaN (16-bit caches), so a decode that copied one of them early would not match;
    sequences of 1-3 tokens have no unit without their newest row."""
    b = workloads.make_batch(name, seed=16, **kw)
    vals = workloads.host_values(b, seed=16)
    if b.kv_fmt in NAN16:
        blk, off = b.new_slots // b.block_size, b.new_slots % b.block_size
        for c in ("k_cache", "v_cache"):
            raw = vals[c].view(np.uint16)
            raw[blk, :, off, :] = NAN16[b.kv_fmt]
    ref, okc, ovc = run_oracle(b, vals, window=window)
    out, kc, vc, err = run_gpu(b, vals, partition_size=partition_size, window=window, pdl=True, early_kv=True)
    out0, _, _, err0 = run_gpu(b, vals, partition_size=partition_size, window=window, pdl=False)
    assert err == 0 and err0 == 0
    assert bits_equal(kc, okc) and bits_equal(vc, ovc)
    assert np.isfinite(out).all()
    assert np.max(np.abs(out - ref)) <= PA_TOL
    assert bits_equal(out, out0)

"""Helpers shared by the GPU tests, smoke() and bench: run one decode case on
the CUDA path (through the C ABI) and on the oracle, from the same inputs."""

from __future__ import annotations

import numpy as np

import oracle
import workloads

TORCH_DT = {"f16": "float16", "bf16": "bfloat16", "e4m3": "uint8", "i8": "int8", "f32": "float32"}
PA_TOL = 2e-3          # max-abs error bound for attention outputs (fp32 out)


def to_torch(x: np.ndarray, fmt: str, device):
    import torch
    if fmt == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    if fmt == "e4m3":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8)).to(device)
    if fmt == "i8":
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int8)).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def to_numpy(t, fmt: str) -> np.ndarray:
    import torch
    t = t.detach().cpu()
    if fmt == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def out_tolerance(ref: np.ndarray, out_fmt: str) -> np.ndarray:
    """2e-3 plus half an ulp of the reference in the output type."""
    if out_fmt == "f32":
        return np.full(ref.shape, PA_TOL)
    if out_fmt == "f16":
        spacing = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    else:  # bf16: 8 significant bits
        e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126)))
        spacing = 2.0 ** (e - 7)
    return PA_TOL + 0.5 * spacing


def run_gpu(batch, vals, *, out_fmt="f32", partition_size=0, workspace="auto", device="cuda", window=0, pdl=False,
            early_kv=False):
    """Fill the cache (8-bit caches: quantising writes), append the new token, decode.

    q of shape [S, L, H_q, d] (L > 1) decodes L queries per sequence (pa_decode_ex q_len).
    Returns (out float64 numpy, k_cache numpy, v_cache numpy, device error bits).
    """
    import torch
    import paged_kv_cache_144_gb300 as pa

    kv = batch.kv_fmt
    B = batch.block_size
    q = to_torch(vals["q"], batch.q_fmt, device)
    kc = to_torch(vals["k_cache"], kv, device)
    vc = to_torch(vals["v_cache"], kv, device)
    quant = kv in ("e4m3", "i8")
    src_fmt = "bf16" if quant else kv   # 8-bit caches are written from bf16 rows
    ks = vs = kis = vis = kz = vz = None
    if quant:
        ks = torch.from_numpy(vals["k_scale"]).to(device)
        vs = torch.from_numpy(vals["v_scale"]).to(device)
        kis = torch.from_numpy(vals["k_inv_scale"]).to(device)
        vis = torch.from_numpy(vals["v_inv_scale"]).to(device)
        if kv == "i8":
            kz = torch.from_numpy(vals["k_zero_point"]).to(device)
            vz = torch.from_numpy(vals["v_zero_point"]).to(device)
        slots = torch.from_numpy(vals["src_slots"]).to(device)
        pa.reshape_and_cache(to_torch(vals["k_src"], "bf16", device), to_torch(vals["v_src"], "bf16", device),
                             kc, vc, slots, B, k_inv_scale=kis, v_inv_scale=vis, k_zero_point=kz, v_zero_point=vz)
    new_slots = torch.from_numpy(batch.new_slots).to(device)
    pa.reshape_and_cache(to_torch(vals["k_new"], src_fmt, device), to_torch(vals["v_new"], src_fmt, device),
                         kc, vc, new_slots, B, k_inv_scale=kis, v_inv_scale=vis, k_zero_point=kz, v_zero_point=vz)
    tables = torch.from_numpy(batch.block_tables).to(device)
    lens = torch.from_numpy(batch.seq_lens).to(device)
    q_len = vals["q"].shape[1] if vals["q"].ndim == 4 else 1
    oshape = (batch.num_seqs, batch.num_heads, batch.head_dim) if q_len == 1 else \
        (batch.num_seqs, q_len, batch.num_heads, batch.head_dim)
    out = torch.empty(oshape, dtype=getattr(torch, TORCH_DT[out_fmt]), device=device)
    ws = None
    if workspace == "auto":
        n = pa.decode_workspace_bytes(batch.num_seqs, batch.num_heads, batch.num_kv_heads, batch.head_dim, B,
                                      batch.max_blocks_per_seq, partition_size, pa.dtype_code(kc), q_len=q_len)
        ws = pa.new_workspace(n, device) if n else None
    pa.decode(out, q, kc, vc, tables, lens, batch.num_kv_heads, batch.scale, B, k_scale=ks, v_scale=vs,
              partition_size=partition_size, workspace=ws, window=window, k_zero_point=kz, v_zero_point=vz, pdl=pdl,
              early_kv=early_kv)
    err = pa.get_device_error()
    return (out.float().cpu().numpy().astype(np.float64), to_numpy(kc, kv), to_numpy(vc, kv), err)


def run_oracle(batch, vals, window=0):
    """Oracle caches after the same writes, and the oracle attention output."""
    kv = batch.kv_fmt
    B = batch.block_size
    kc, vc = vals["k_cache"], vals["v_cache"]
    quant = kv in ("e4m3", "i8")
    src_fmt = "bf16" if quant else kv
    kis = vals.get("k_inv_scale")
    vis = vals.get("v_inv_scale")
    kz, vz = vals.get("k_zero_point"), vals.get("v_zero_point")
    if quant:
        kc, vc = oracle.reshape_and_cache(vals["k_src"], vals["v_src"], kc, vc, vals["src_slots"], B,
                                          src_fmt="bf16", kv_fmt=kv, k_inv_scale=kis, v_inv_scale=vis,
                                          k_zero_point=kz, v_zero_point=vz)
    kc, vc = oracle.reshape_and_cache(vals["k_new"], vals["v_new"], kc, vc, batch.new_slots, B,
                                      src_fmt=src_fmt, kv_fmt=kv, k_inv_scale=kis, v_inv_scale=vis,
                                      k_zero_point=kz, v_zero_point=vz)
    fn = oracle.paged_multi_query_attention if vals["q"].ndim == 4 else oracle.paged_decode_attention
    ref = fn(vals["q"], kc, vc, batch.block_tables, batch.seq_lens, batch.scale, B, q_fmt=batch.q_fmt, kv_fmt=kv,
             k_scale=vals.get("k_scale"), v_scale=vals.get("v_scale"), window=window, k_zero_point=kz,
             v_zero_point=vz)
    return ref, kc, vc


def bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def check_sequence(item):
    """One sequence of a full-size run against the oracle (runs in an oracle worker process).

    8-bit caches: the sequence's cache bytes must equal the oracle's quantisation of its bf16 rows (the
    cached ones and the appended one); 16-bit caches: the appended rows must sit in their slot.  Then every
    query head's output is compared with the oracle's attention over the sequence's blocks.
    Returns (s, max abs error, None) or (s, error, reason of the first failure).
    """
    s, T, B = item["s"], item["T"], item["B"]
    gk, gv = item["gk"], item["gv"]
    nb = gk.shape[0]
    kv = item["kv_fmt"]
    if kv in ("e4m3", "i8"):
        zkw = {k: item["qkw"][k] for k in ("k_zero_point", "v_zero_point") if k in item["qkw"]}
        kr = np.concatenate([item["k_rows"], item["k_new"][None]])
        vr = np.concatenate([item["v_rows"], item["v_new"][None]])
        zero = np.zeros_like(gk)
        ok, ov = oracle.reshape_and_cache(kr, vr, zero, zero, np.arange(T), B, src_fmt="bf16", kv_fmt=kv,
                                          k_inv_scale=item["k_inv_scale"], v_inv_scale=item["v_inv_scale"], **zkw)
        if not (bits_equal(gk, ok) and bits_equal(gv, ov)):
            return s, float("inf"), f"{kv} cache bytes differ from the oracle's quantisation"
        gk, gv = ok, ov
    else:
        r, p = (T - 1) // B, (T - 1) % B
        if item["new_slot"] != int(item["table"][r]) * B + p:
            return s, float("inf"), "slot of the appended token"
        if not (bits_equal(gk[r, :, p], item["k_new"]) and bits_equal(gv[r, :, p], item["v_new"])):
            return s, float("inf"), "appended rows not in their slot"
    ref = oracle.paged_decode_attention(item["q"], gk, gv, np.arange(nb, dtype=np.int32)[None, :], np.array([T]),
                                        item["scale"], B, q_fmt=item["q_fmt"], kv_fmt=kv, **item["qkw"])[0]
    err = np.abs(item["out"] - ref)
    if not np.all(err <= PA_TOL):
        bad = np.nonzero(err.max(axis=1) > PA_TOL)[0]
        return s, float(err.max()), f"heads {bad.tolist()} max abs err {err.max():.3e} > {PA_TOL}"
    return s, float(err.max()), None


_POOL = None


def oracle_pool():
    """A process pool for oracle work, started with spawn (safe after CUDA is initialised), one per session."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        import os
        os.environ.setdefault("OMP_NUM_THREADS", "1")
        n = max(1, min(16, os.cpu_count() or 1))
        _POOL = mp.get_context("spawn").Pool(processes=n)
        import atexit
        atexit.register(_POOL.terminate)
    return _POOL

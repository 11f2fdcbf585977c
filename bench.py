#!/usr/bin/env python3
"""Benchmark of the paged decode step on GB300: KV-read HBM GB/s, % of HBM peak, tokens/s.

One step = one pass of the whole hot path over one batch:
  pa_reshape_and_cache (the new token of every sequence -> its slot)
  + pa_decode (paged single-query attention over every sequence, split-K
  partials merged in-kernel).  Copy-on-write copies are issued only when a
  write hits a shared block; the batch workloads timed here share no block, so
  pa_copy_blocks is called with no pairs and launches nothing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gqa_32x4k]
  python bench.py --impl reference ...    # the float64 CPU oracle on host cores

N > 1 runs under torch.distributed.run, one rank per GPU: every rank decodes
its own batch of the same shape (weak scaling, no collective on the data
path); the timed region is bracketed by barriers and the max over ranks is
taken.  Inputs are resident in HBM before the timed region; between steps
the KV pools rotate over enough replicas that each step reads data last
touched > 4x L2 ago.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged-decode KV-read HBM GB/s & % of GB300 peak; decode attn tokens/s"
UNIT = "GB/s"
FMT_BYTES = {"f16": 2, "bf16": 2, "e4m3": 1, "i8": 1, "f32": 4}
KERNEL_SOURCES = ["pa_common.cuh", "pa_decode.cuh", "pa_decode_variants.h", "pa_decode_dispatch.cu",
                  "pa_decode_f16.cu", "pa_decode_bf16.cu", "pa_decode_fp8.cu", "pa_decode_int8.cu",
                  "pa_decode_rows16.cu", "pa_decode_append16.cu", "pa_decode_append8.cu", "pa_api.cu",
                  "pa_kernels.h"]
WORKLOAD_TEXT = {
    "tiny": "4 seqs, cached len ~U{1..128} + 1, 4 heads MHA, d 64, B 16, fp16",
    "gqa_32x4k": "32 seqs, len ~U{1..4096}, 32 q heads / 8 KV heads, d 128, B 16, bf16",
    "long_32k": "8 seqs x 32768 tokens, 64 q heads / 8 KV heads, d 128, B 16, bf16",
    "fp8_mix": "256 seqs, len=clip(round(lognormal(7,1)),16,8192), 32 q / 8 KV heads, d 128, B 16, "
               "K/V fp8-e4m3 per-head scales, bf16 q",
    "int8_mix": "256 seqs, len=clip(round(lognormal(7,1)),16,8192), 32 q / 8 KV heads, d 128, B 16, "
                "K/V INT8 per-head scale + zero point, bf16 q",
    "beam_cow": "6 beams sharing a 1000-token prompt (63 blocks, refcount 6, partial block copied on write), "
                "private tails ~U{1..256}, 40 heads MHA, d 128, B 16, fp16",
}


def _code_only(text: str) -> str:
    """C++/CUDA source without its comments and blank lines (string literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                                   # string literal: copied, escapes honoured
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).split("\n")]
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_digest(root: str = ROOT) -> str:
    """Digest of the code the decode kernel is built from (comments and blank lines excluded), which keys
    the committed ncu traffic figures: counters taken on other code are not reported."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(root, "paged_kv_cache_144_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def algorithmic_bytes(batch, window: int = 0, q_len: int = 1) -> dict:
    """Bytes a step must move at minimum (attended tokens only; tails, workspace and scales excluded).

    With a sliding window only the last `window` positions of each sequence and the
    block-table entries of the blocks holding them count.  With q_len queries per
    sequence the KV rows are still read once; q and out count q_len times.
    """
    S, Hq, Hkv, D, B = batch.num_seqs, batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size
    b_kv = FMT_BYTES[batch.kv_fmt]
    b_q = FMT_BYTES[batch.q_fmt]
    T = batch.seq_lens.astype(np.int64)
    lo = np.maximum(T - q_len + 1 - window, 0) if window > 0 else np.zeros_like(T)
    kv = int((T - lo).sum()) * Hkv * D * b_kv * 2
    blocks = int(((T + B - 1) // B - lo // B).sum())
    decode = kv + q_len * (S * Hq * D * b_q + S * Hq * D * b_q) + blocks * 4 + 4 * S
    src_b = b_q if batch.kv_fmt in ("e4m3", "i8") else b_kv
    append = S * Hkv * D * (src_b + b_kv) * 2 + 8 * S
    return {"kv": kv, "decode": decode, "append": append, "step": decode + append}


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "of measured"}
    return {"hbm_gbs": 6800.0, "source": "of fallback"}


def load_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if the kernel is unchanged."""
    p = os.path.join(ROOT, "profiles", f"decode_{workload}_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_digest") != kernel_source_digest():
        return None
    return d.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 50 ms from before the timed regions to after them.

    The sampler selects the GPU by UUID (the CUDA device index and nvidia-smi's index differ when
    CUDA_VISIBLE_DEVICES is set); if that form yields no sample it retries with the index.  start()
    returns once the first sample has been written, so that a short timed region is still covered.
    """
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid: str | None, device_index: int):
        self.proc = None
        self.fh = None
        self.out = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")
        self.selectors = [s for s in (device_uuid, str(device_index)) if s]
        self.note = None

    def _spawn(self, sel):
        cmd = ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        self.fh = open(self.out, "w")
        self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)

    def _kill(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.proc = None
        if self.fh is not None:
            self.fh.close()
            self.fh = None

    def start(self, timeout_s: float = 5.0):
        for sel in self.selectors:
            try:
                self._spawn(sel)
            except (OSError, FileNotFoundError):
                self.proc = None
                self.note = "nvidia-smi not available"
                return self
            t0 = time.time()
            while time.time() - t0 < timeout_s:
                if os.path.getsize(self.out) > 0:
                    self.note = f"nvidia-smi -i {sel}"
                    return self
                if self.proc.poll() is not None:
                    break
                time.sleep(0.02)
            self._kill()
        self.note = "nvidia-smi gave no sample"
        return self

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self._kill()
        rows = []
        with open(self.out) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        power = [num(r[3]) for r in rows]
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        pairs = [(c, w) for c, w in zip(sm, power) if c is not None]
        # samples under load: power above the midpoint of the observed range
        if pairs and all(w is not None for _, w in pairs):
            lo, hi = min(w for _, w in pairs), max(w for _, w in pairs)
            loaded = [c for c, w in pairs if w >= (lo + hi) / 2]
        else:
            loaded = [c for c, _ in pairs]
        return {"sm_mhz": float(np.median(loaded)) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "source": self.note}


# ----------------------------------------------------------------------------- CPU oracle baseline

def _oracle_segment(args):
    """Worker: oracle attention for one (sequence, KV head) segment; returns seconds."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import oracle
    q, kc, vc, T, scale, B, q_fmt, kv_fmt, ks, vs, kz, vz = args
    nb = kc.shape[0]
    t0 = time.perf_counter()
    oracle.paged_decode_attention(q, kc, vc, np.arange(nb, dtype=np.int32)[None, :], np.array([T]), scale, B,
                                  q_fmt=q_fmt, kv_fmt=kv_fmt, k_scale=ks, v_scale=vs, k_zero_point=kz,
                                  v_zero_point=vz)
    return time.perf_counter() - t0


def host_segments(batch, dev_vals, seg_ids):
    """Host copies (numpy storage) of the given (s, kvh) segments: q group + its blocks."""
    import torch
    B, G = batch.block_size, batch.group
    out = []
    q_all = dev_vals["q"]
    for (s, kvh) in seg_ids:
        T = int(batch.seq_lens[s])
        nb = -(-T // B)
        blocks = torch.from_numpy(batch.block_tables[s, :nb].astype(np.int64)).to(q_all.device)

        def host(t, fmt):
            t = t.detach().cpu()
            if fmt == "bf16":
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
        kc = host(dev_vals["k_cache"].index_select(0, blocks)[:, kvh:kvh + 1], batch.kv_fmt)
        vc = host(dev_vals["v_cache"].index_select(0, blocks)[:, kvh:kvh + 1], batch.kv_fmt)
        q = host(q_all[s:s + 1, kvh * G:(kvh + 1) * G], batch.q_fmt)
        ks = vs = kz = vz = None
        if batch.kv_fmt in ("e4m3", "i8"):
            ks = dev_vals["k_scale"][kvh:kvh + 1].cpu().numpy()
            vs = dev_vals["v_scale"][kvh:kvh + 1].cpu().numpy()
        if batch.kv_fmt == "i8":
            kz = dev_vals["k_zero_point"][kvh:kvh + 1].cpu().numpy()
            vz = dev_vals["v_zero_point"][kvh:kvh + 1].cpu().numpy()
        out.append((q, kc, vc, T, batch.scale, B, batch.q_fmt, batch.kv_fmt, ks, vs, kz, vz))
    return out


def _warm_worker(_):
    import oracle  # noqa: F401  (imports numpy + the oracle once per worker)
    return os.getpid()


def oracle_rate(batch, dev_vals, target_s: float, seed: int = 0, max_procs: int | None = None):
    """Oracle GB/s on a bounded random sample of (s, kvh) segments, all host cores (spawned pool).

    Segments are drawn in a seeded random order, cycling over the batch, until
    about target_s seconds of work per core; only the oracle's own work is
    timed (the pool is started and warmed first).
    """
    import multiprocessing as mp
    rng = np.random.default_rng(seed + 4242)
    Hkv, D = batch.num_kv_heads, batch.head_dim
    b_kv, b_q = FMT_BYTES[batch.kv_fmt], FMT_BYTES[batch.q_fmt]
    order = [(int(s), int(k)) for s in rng.permutation(batch.num_seqs) for k in rng.permutation(Hkv)]
    first = host_segments(batch, dev_vals, order[:1])[0]
    _oracle_segment(first)                      # import + warm
    t1 = max(_oracle_segment(first), 1e-5)
    per_token = t1 / max(first[3], 1)
    procs = max_procs or os.cpu_count() or 1
    budget_tokens = target_s * procs / per_token
    distinct, tok, chosen = {}, 0, []
    i = 0
    while tok < budget_tokens and i < 100000:
        sg = order[i % len(order)]
        chosen.append(sg)
        tok += int(batch.seq_lens[sg[0]])
        i += 1
    for sg in set(chosen):
        distinct[sg] = host_segments(batch, dev_vals, [sg])[0]
    args = [distinct[sg] for sg in chosen]
    nbytes = sum(a[3] * D * b_kv * 2 + 2 * batch.group * D * b_q for a in args)
    os.environ["OMP_NUM_THREADS"] = "1"
    ctx = mp.get_context("spawn")
    nproc = min(procs, len(args))
    with ctx.Pool(processes=nproc) as pool:
        pool.map(_warm_worker, range(nproc))
        t0 = time.perf_counter()
        pool.map(_oracle_segment, args, chunksize=1)
        wall = time.perf_counter() - t0
    return {"value": round(nbytes / wall / 1e9, 4), "unit": UNIT, "cores": nproc, "kind": "oracle",
            "sample": f"{len(args)} seeded-random (sequence, KV head) segments of the same batch ({len(distinct)} "
                      f"distinct, cycling), {tok} context tokens x G={batch.group} query heads, float64 numpy "
                      f"oracle, one single-threaded process per core, {wall:.1f} s"}


# ----------------------------------------------------------------------------- GPU arm

def setup_distributed():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, ws, local


def max_over_ranks(x: float, world_size: int) -> float:
    if world_size <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world_size: int) -> float:
    if world_size <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world_size: int):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e nominal bandwidth (~8 TB/s), the basis the ">= 70 %" target is stated on
MIN_TIMED_S = 1.0          # every timed loop is repeated until its repeats cover at least this long
MIN_TIME_S = [MIN_TIMED_S]  # as set by --min-time


def lead_gpu(torch, us: float = 300.0):
    """Keep the stream busy for about `us` microseconds before a timed region starts (outside it), so that the
    host has enqueued the region's first launches by the time the GPU reaches it: the region then times the
    device, not the host's latency to its first launch."""
    torch.cuda._sleep(int(us * 2.2e3))  # cycles; at most 2.07 GHz here, so at least `us`


def repeat_until(one, world: int, min_s: float | None = None):
    """Run one() (the milliseconds of one timed repeat) until the repeats cover min_s seconds (default: the
    --min-time argument, else MIN_TIMED_S).  The repeat count is fixed after the first repeat and agreed across
    ranks (max), so every rank runs the same loops."""
    if min_s is None:
        min_s = MIN_TIME_S[0]
    first = one()
    n = max(1, math.ceil(min_s * 1e3 / max(first, 1e-6)))
    n = int(max_over_ranks(float(min(n, 100000)), world))
    return [first] + [one() for _ in range(n - 1)]


def spread(times_ms, per: int) -> dict:
    a = np.asarray(times_ms, dtype=np.float64) / per
    return {"n": int(a.size), "median_ms": round(float(np.median(a)), 6), "min_ms": round(float(a.min()), 6),
            "max_ms": round(float(a.max()), 6)}


class DecodeCase:
    """One workload resident on the device: rotating KV pool replicas (> 4x L2 together), tables, lengths,
    queries, the new token's rows and slots, the output and the split workspace."""

    def __init__(self, pa, torch, dev, workload, seed, *, q_len=1, partition_size=0, replicas=0, block_size=None):
        ov = {} if block_size is None else {"block_size": block_size}
        self.batch = b = workloads.make_batch(workload, seed=seed, **ov)
        vals = workloads.device_values(b, seed, dev)
        B, Hkv, D, S, Hq = b.block_size, b.num_kv_heads, b.head_dim, b.num_seqs, b.num_heads
        self.kz, self.vz = vals.get("k_zero_point"), vals.get("v_zero_point")
        if b.kv_fmt in ("e4m3", "i8"):
            pa.reshape_and_cache(vals["k_src"], vals["v_src"], vals["k_cache"], vals["v_cache"], vals["src_slots"], B,
                                 k_inv_scale=vals["k_inv_scale"], v_inv_scale=vals["v_inv_scale"],
                                 k_zero_point=self.kz, v_zero_point=self.vz)
            del vals["k_src"], vals["v_src"]
        self.pool_bytes = 2 * vals["k_cache"].numel() * vals["k_cache"].element_size()
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.replicas = replicas or max(2, math.ceil(4 * self.l2 / self.pool_bytes) + 1)
        self.caches = [(vals["k_cache"], vals["v_cache"])] + [
            (vals["k_cache"].clone(), vals["v_cache"].clone()) for _ in range(self.replicas - 1)]
        self.tables = torch.from_numpy(b.block_tables).to(dev)
        self.lens = torch.from_numpy(b.seq_lens).to(dev)
        self.slots = torch.from_numpy(b.new_slots).to(dev)
        self.q, self.k_new, self.v_new = vals["q"], vals["k_new"], vals["v_new"]
        self.ks, self.vs = vals.get("k_scale"), vals.get("v_scale")
        self.kis, self.vis = vals.get("k_inv_scale"), vals.get("v_inv_scale")
        self.q_len, self.partition_size = q_len, partition_size
        if q_len > 1:   # the q_len newest positions are queries: [S, L, H_q, d]
            gq = torch.Generator(device=dev)
            gq.manual_seed(seed * 7 + 3)
            self.q = torch.randn((S, q_len, Hq, D), generator=gq, device=dev, dtype=torch.float32).to(self.q.dtype)
        self.out = torch.empty(self.q.shape, dtype=self.q.dtype, device=dev)
        nws = pa.decode_workspace_bytes(S, Hq, Hkv, D, B, b.max_blocks_per_seq, partition_size,
                                        pa.dtype_code(vals["k_cache"]), q_len=q_len)
        self.ws = pa.new_workspace(nws, dev) if nws else None
        self.geometry = pa.pa_decode_launch_config(S, Hq, Hkv, D, B, b.max_blocks_per_seq, partition_size,
                                                   pa.dtype_code(self.q), pa.dtype_code(vals["k_cache"]))

    def decode(self, pa, i, stream, *, window=0, pdl=False, fused=False, q=None, tables=None, lens=None,
               k_new=None, v_new=None, early_kv=False):
        kc, vc = self.caches[i % self.replicas]
        b = self.batch
        extra = {}
        if fused:
            extra = dict(k_new=self.k_new if k_new is None else k_new, v_new=self.v_new if v_new is None else v_new,
                         k_inv_scale=self.kis, v_inv_scale=self.vis)
        pa.decode(self.out, self.q if q is None else q, kc, vc, self.tables if tables is None else tables,
                  self.lens if lens is None else lens, b.num_kv_heads, b.scale, b.block_size, k_scale=self.ks,
                  v_scale=self.vs, partition_size=self.partition_size, workspace=self.ws, stream=stream,
                  window=window, k_zero_point=self.kz, v_zero_point=self.vz, pdl=pdl, early_kv=early_kv, **extra)

    def cache_write(self, pa, i, stream, *, pdl=False, k=None, v=None, slots=None):
        kc, vc = self.caches[i % self.replicas]
        pa.reshape_and_cache(self.k_new if k is None else k, self.v_new if v is None else v, kc, vc,
                             self.slots if slots is None else slots, self.batch.block_size, k_inv_scale=self.kis,
                             v_inv_scale=self.vis, k_zero_point=self.kz, v_zero_point=self.vz, stream=stream, pdl=pdl)

    def time_decode_alone(self, pa, torch, stream, K, world, *, window=0, fused=False):
        """Repeats of K decode launches, each an ordinary launch between two events on the launching stream.
        Returns the per-repeat mean launch time (ms) of every repeat."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        ctr = [0]

        def one():
            barrier(world)
            torch.cuda.synchronize()
            lead_gpu(torch)
            for i in range(K):
                ev[i][0].record(stream)
                self.decode(pa, ctr[0], stream, window=window, fused=fused)
                ev[i][1].record(stream)
                ctr[0] += 1
            torch.cuda.synchronize()
            barrier(world)
            return float(np.sum([a.elapsed_time(b_) for a, b_ in ev]))

        for i in range(3):
            self.decode(pa, i, stream, window=window, fused=fused)
        return [t / K for t in repeat_until(one, world)]


def run_ours(args):
    import torch
    import paged_kv_cache_144_gb300 as pa

    rank, world, local = setup_distributed()
    dev = torch.device("cuda", local)
    pa.load()
    c = DecodeCase(pa, torch, dev, args.workload, args.seed + 1000 * rank, q_len=args.q_len,
                   partition_size=args.partition_size, replicas=args.replicas, block_size=args.block_size)
    batch = c.batch
    B, Hkv, D, S, Hq = batch.block_size, batch.num_kv_heads, batch.head_dim, batch.num_seqs, batch.num_heads
    no_pairs = torch.empty((0, 2), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    pdl = not args.no_pdl
    early_kv = pdl and batch.kv_fmt in ("f16", "bf16")

    def step(i):
        # one step as a serving loop issues it: nothing between its launches, so the decode's set-up
        # (lengths, prefix sums, block-table prefetch) overlaps the launch before it (pdl)
        if args.fused:
            # one launch: the cache write of the new rows fused into the decode
            c.decode(pa, i, stream, window=args.window, pdl=pdl, fused=True)
            return
        c.cache_write(pa, i, stream, pdl=pdl)
        kc, vc = c.caches[i % c.replicas]
        pa.copy_blocks(kc, vc, no_pairs, stream=stream)          # no shared block is written: no launch
        # the kernel before the decode is that cache write, which writes each sequence's newest row only:
        # the decode may start copying the other rows before it has finished (early_kv; 16-bit caches:
        # with the 8-bit mixes the early copies slowed the quantising write of 256 sequences more than
        # they saved, 169.6 -> 170.9 us per step on one box)
        c.decode(pa, i, stream, window=args.window, pdl=pdl, early_kv=early_kv)

    sampler = None
    if rank == 0:
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
        except Exception:
            uuid = None
        sampler = ClockSampler(uuid, local).start()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if pa.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctr = [args.warmup]

    def step_repeat():
        # exactly K steps between two events, barrier + synchronize on both sides
        barrier(world)
        torch.cuda.synchronize()
        lead_gpu(torch)
        t_start.record(stream)
        for _ in range(K):
            step(ctr[0])
            ctr[0] += 1
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return t_start.elapsed_time(t_end)

    step_times = repeat_until(step_repeat, world)
    # second timed region: K decode launches alone, each between two events on the launching stream
    dec_times = c.time_decode_alone(pa, torch, stream, K, world, window=args.window, fused=args.fused)
    # the two headline configurations' decode kernels, timed the same way (1 GPU)
    per_config = []
    if world == 1 and not args.no_per_config:
        for wl, kw in (("long_32k", {}), ("fp8_mix", {"block_size": 16})):
            if wl == args.workload and not kw:
                continue
            pc = DecodeCase(pa, torch, dev, wl, args.seed, **kw)
            t = pc.time_decode_alone(pa, torch, stream, K, world)
            ab = algorithmic_bytes(pc.batch)["decode"]
            per_config.append((wl, pc.batch, t, ab))
            del pc
            torch.cuda.empty_cache()
    clocks = sampler.stop() if sampler else None
    err = pa.get_device_error()
    if err != 0:
        raise RuntimeError(f"device error bits {err} in the timed region")
    ms_step = max_over_ranks(float(np.median(step_times)) / K, world)
    dec_ms = max_over_ranks(float(np.median(dec_times)), world)

    # end to end through the public API: pinned host inputs -> device, step, result -> host
    e2e = None
    if not args.no_e2e:
        h_q = c.q.cpu().pin_memory()
        h_k, h_v = c.k_new.cpu().pin_memory(), c.v_new.cpu().pin_memory()
        h_slots, h_tables, h_lens = c.slots.cpu().pin_memory(), c.tables.cpu().pin_memory(), c.lens.cpu().pin_memory()
        h_out = torch.empty(c.out.shape, dtype=c.out.dtype).pin_memory()
        # The step's inputs are staged in one pinned host buffer and cross in one copy, as a serving loop
        # stages them; each tensor sits at a 256-byte aligned offset (the library wants 16-byte bases).
        parts = (h_q, h_k, h_v, h_slots, h_tables, h_lens)
        offs, h2d = [], 0
        for t in parts:
            h2d = (h2d + 255) // 256 * 256
            offs.append(h2d)
            h2d += t.numel() * t.element_size()
        h_stage = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        d_stage = torch.empty(h2d, dtype=torch.uint8, device=dev)
        views = []
        for t, o in zip(parts, offs):
            nb = t.numel() * t.element_size()
            h_stage[o:o + nb].copy_(t.reshape(-1).view(torch.uint8))
            views.append(d_stage[o:o + nb].view(t.dtype).view(t.shape))
        d_q, d_k, d_v, d_slots, d_tables, d_lens = views
        d2h = h_out.numel() * h_out.element_size()

        def e2e_body(i, pdl=pdl):
            st = torch.cuda.current_stream()
            d_stage.copy_(h_stage, non_blocking=True)
            if args.fused:
                c.decode(pa, i, st, window=args.window, pdl=pdl, fused=True, q=d_q, tables=d_tables, lens=d_lens,
                         k_new=d_k, v_new=d_v)
            else:
                # no early_kv here: a step launched on an idle GPU (after the host read of the last one)
                # has the decode's early copies reach memory ahead of the cache write's few loads and
                # delay it (GQA: 76.8 -> 79.3 us per end-to-end step, one box); back to back, the cache
                # write's CTAs already wait on the SMs and the early copies pay (50.6 -> 49.3 us)
                c.cache_write(pa, i, st, pdl=pdl, k=d_k, v=d_v, slots=d_slots)
                c.decode(pa, i, st, window=args.window, pdl=pdl, q=d_q, tables=d_tables, lens=d_lens)
            h_out.copy_(c.out, non_blocking=True)

        if args.e2e_eager:
            def e2e_step(i):
                e2e_body(i)
                stream.synchronize()
        else:
            # the step as a serving loop with fixed buffers issues it: one CUDA graph per KV pool replica,
            # recorded through the same library calls (pa.StepGraph), replayed once per step
            graphs = [pa.StepGraph(lambda r=r: e2e_body(r)) for r in range(c.replicas)]

            def e2e_step(i):
                graphs[i % c.replicas].replay()
                stream.synchronize()

        for i in range(args.warmup):
            e2e_step(i)

        def e2e_repeat():
            barrier(world)
            t0 = time.perf_counter()
            for i in range(K):
                e2e_step(i)
            dt = time.perf_counter() - t0
            barrier(world)
            return dt * 1e3

        e2e_times = repeat_until(e2e_repeat, world)
        e2e = (max_over_ranks(float(np.median(e2e_times)) / K, world), h2d, d2h, e2e_times)

    ab = algorithmic_bytes(batch, args.window, args.q_len)
    total_step_bytes = sum_over_ranks(float(ab["step"]), world)
    total_kv = sum_over_ranks(float(ab["kv"]), world)
    total_seqs = sum_over_ranks(float(S), world)
    total_ctx = sum_over_ranks(float(batch.seq_lens.sum()), world)
    peaks = load_peaks()
    value = total_step_bytes / (ms_step * 1e-3) / 1e9
    kernel_bytes = ab["step"] if args.fused else ab["decode"]   # fused: the launch also moves the new rows
    achieved = kernel_bytes / (dec_ms * 1e-3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_rate(batch, {"q": c.q, "k_cache": c.caches[0][0], "v_cache": c.caches[0][1], "k_scale": c.ks,
                                  "v_scale": c.vs}, target_s=args.cpu_seconds, seed=args.seed)
    if rank != 0:
        return
    # the committed counters were taken on the plain launch of the workload; a window, several queries or
    # the fused append change what the kernel moves, so those runs report no traffic
    plain = not args.fused and args.q_len == 1 and not args.window and args.block_size is None
    traffic = load_traffic(args.workload) if plain else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": batch.kv_fmt, "data": "synthetic (seeded N(0,1) values, random block tables)",
        "config": {
            "workload": f"{args.workload}: {WORKLOAD_TEXT.get(args.workload, '')}",
            "num_seqs": S, "num_heads": Hq, "num_kv_heads": Hkv, "head_dim": D, "block_size": B,
            "context_tokens": int(batch.seq_lens.sum()), "kv_dtype": batch.kv_fmt, "q_dtype": batch.q_fmt,
            "split": "balanced" if args.partition_size == 0 else f"fixed {args.partition_size} tokens",
            "window": args.window or None,
            "q_len": args.q_len,
            "step": ("pa_decode_ex with the new token's cache write fused (one launch)" if args.fused
                     else "reshape_and_cache(1 new token/seq) + pa_decode") +
                    ((", launched with programmatic dependent launch" if args.fused
                      else ", both launched with programmatic dependent launch" +
                           ("; the decode's early_kv option lets it copy the rows other than each sequence's "
                            "newest before the cache write ends" if early_kv else ""))
                     if pdl else ""),
            "timing": f"value: repeats of exactly K={K} steps back to back (so each step's launches overlap the one "
                      f"before through programmatic dependent launch), CUDA events on the stream, barrier + "
                      f"synchronize around each repeat, repeated until >= {MIN_TIME_S[0]:g} s, median repeat; "
                      "roofline: a second loop of decode launches alone (ordinary launches, no overlap), an event "
                      "pair around each launch, repeated the same way. The two loops differ in shape, so the "
                      "step can be shorter than the decode launch alone.",
            "l2": f"{c.replicas} rotating KV pools ({c.replicas * c.pool_bytes / 1e9:.2f} GB) > L2 "
                  f"({c.l2 / 1e6:.0f} MB): inputs larger than L2, no flush",
            "seed": args.seed,
            "launch": c.geometry,
        },
        "repeats": {"step": spread(step_times, K), "decode_alone": spread(dec_times, 1)},
        "pct_of_hbm_peak": round(100.0 * value / peaks["hbm_gbs"], 2),
        "pct_of_nominal_8tbs": round(100.0 * value / NOMINAL_HBM_GBS, 2),
        "kv_read_gbps": round(total_kv / (ms_step * 1e-3) / 1e9, 2),
        "decode_tokens_per_s": round(total_seqs * args.q_len / (ms_step * 1e-3), 1),
        "context_tokens_per_s": round(total_ctx / (ms_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel (pa_decode, one launch)",
                     "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "algorithmic_bytes_per_launch": kernel_bytes, "avg_launch_ms": round(dec_ms, 6),
                     "traffic": traffic},
        "per_config": [
            {"workload": f"{wl}: {WORKLOAD_TEXT.get(wl, '')}" + (f" (block_size {pb.block_size})" if wl == "fp8_mix" else ""),
             "avg_launch_ms": round(float(np.median(t)), 6), "repeats": spread(t, 1),
             "algorithmic_bytes": abytes,
             "achieved_gbs": round(abytes / (float(np.median(t)) * 1e-3) / 1e9, 2),
             "frac": round(abytes / (float(np.median(t)) * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
             "frac_of_nominal_8tbs": round(abytes / (float(np.median(t)) * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
             "traffic": load_traffic(wl) if pb.block_size == 16 else None}
            for wl, pb, t, abytes in per_config],
        "cpu_baseline": cpu,
        # launches of this library's kernels inside the timed regions (warm-ups excluded)
        "gpu_launches": (1 if args.fused else 2) * K * len(step_times) + K * len(dec_times) +
                        sum(K * len(t) for _, _, t, _ in per_config) +
                        (0 if e2e is None else (1 if args.fused else 2) * K * len(e2e[3])),
        "clocks": clocks,
    }
    if e2e is not None:
        e2e_ms, h2d, d2h, e2e_times = e2e
        line["e2e"] = {"value": round(total_step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_ms, 6), "repeats": spread(e2e_times, K),
                       "how": ("each step issued call by call through the Python binding" if args.e2e_eager else
                               "each step replays a CUDA graph recorded through the library's calls (pa.StepGraph): "
                               "pinned host staging buffer -> device, cache write, decode, output -> pinned host") +
                              ", then a host synchronisation; host wall clock over the steps"}
    print(json.dumps(line), flush=True)
    if args.json_out:
        with open(args.json_out, "w") as f:
            json.dump(line, f, indent=1)


def build_beam_state(pa, torch, dev, seed):
    """Shared-prompt beam state built through the library (block manager, cache write, CoW copy)."""
    sc = workloads.beam_cow_scenario(seed)
    B, P, H, D = sc["block_size"], sc["prompt_len"], sc["num_kv_heads"], sc["head_dim"]
    nbeams, NB = sc["num_beams"], sc["num_blocks"]
    bm = pa.BlockManager(NB, B, free_order=sc["free_order"])
    kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)

    def put(rows_k, rows_v, slots):
        pa.reshape_and_cache(torch.from_numpy(rows_k.view(np.float16)).to(dev),
                             torch.from_numpy(rows_v.view(np.float16)).to(dev), kc, vc,
                             torch.tensor(slots, dtype=torch.int64, device=dev), B)

    put(sc["prompt_k"], sc["prompt_v"], bm.add_sequence(0, P))
    for bb in range(1, nbeams):
        bm.fork(0, bb)
    pairs = [pp for pp in (bm.copy_on_write(bb, P // B) for bb in range(nbeams)) if pp]
    pa.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int32, device=dev))
    tail_slots = [bm.append_slot(bb)[0] for bb in range(nbeams) for _ in range(int(sc["tails"][bb]))]
    put(np.concatenate(sc["tail_k"]), np.concatenate(sc["tail_v"]), tail_slots)
    new_slots = [bm.append_slot(bb)[0] for bb in range(nbeams)]
    lens = np.array([P + int(t) + 1 for t in sc["tails"]], dtype=np.int32)
    width = max(len(bm.block_table(bb)) for bb in range(nbeams))
    tables = np.array([bm.block_table(bb, width) for bb in range(nbeams)], dtype=np.int32)
    return sc, kc, vc, tables, lens, new_slots, len(pairs)


def run_beam(args):
    """Shared-prefix decode: roofline on unique KV bytes, effective GB/s on logical bytes."""
    import torch
    import paged_kv_cache_144_gb300 as pa

    rank, world, local = setup_distributed()
    dev = torch.device("cuda", local)
    pa.load()
    sc, kc0, vc0, tables_np, lens_np, new_slots, n_pairs = build_beam_state(pa, torch, dev, args.seed + 1000 * rank)
    B, H, D, Hq, S = sc["block_size"], sc["num_kv_heads"], sc["head_dim"], sc["num_heads"], sc["num_beams"]
    # distinct (block, row) pairs the decode reads, and the rows it reads counting repeats
    rows = {(int(tables_np[s, p // B]), p % B) for s in range(S) for p in range(int(lens_np[s]))}
    unique_kv = len(rows) * H * D * 2 * 2
    logical_kv = int(lens_np.sum()) * H * D * 2 * 2
    decode_bytes = unique_kv + 2 * S * Hq * D * 2 + int(((lens_np + B - 1) // B).sum()) * 4 + 4 * S
    append_bytes = S * H * D * (2 + 2) * 2 + 8 * S
    pool_bytes = 2 * kc0.numel() * kc0.element_size()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    replicas = args.replicas or max(2, math.ceil(4 * l2 / pool_bytes) + 1)
    caches = [(kc0, vc0)] + [(kc0.clone(), vc0.clone()) for _ in range(replicas - 1)]
    tables = torch.from_numpy(tables_np).to(dev)
    lens = torch.from_numpy(lens_np).to(dev)
    slots = torch.tensor(new_slots, dtype=torch.int64, device=dev)
    k_new = torch.from_numpy(sc["new_k"].view(np.float16)).to(dev)
    v_new = torch.from_numpy(sc["new_v"].view(np.float16)).to(dev)
    q = torch.from_numpy(sc["q"].view(np.float16)).to(dev)
    out = torch.empty((S, Hq, D), dtype=q.dtype, device=dev)
    nws = pa.decode_workspace_bytes(S, Hq, H, D, B, tables_np.shape[1], args.partition_size, pa.PA_F16)
    ws = pa.new_workspace(nws, dev) if nws else None
    geometry = pa.pa_decode_launch_config(S, Hq, H, D, B, tables_np.shape[1], args.partition_size, pa.PA_F16,
                                          pa.PA_F16)
    stream = torch.cuda.current_stream()

    pdl = not args.no_pdl

    def step(i):
        kc, vc = caches[i % replicas]
        pa.reshape_and_cache(k_new, v_new, kc, vc, slots, B, stream=stream, pdl=pdl)
        pa.decode(out, q, kc, vc, tables, lens, H, sc["scale"], B, partition_size=args.partition_size,
                  workspace=ws, stream=stream, pdl=pdl)

    def decode_alone(i, ev):
        kc, vc = caches[i % replicas]
        ev[0].record(stream)
        pa.decode(out, q, kc, vc, tables, lens, H, sc["scale"], B, partition_size=args.partition_size,
                  workspace=ws, stream=stream)
        ev[1].record(stream)

    sampler = None
    if rank == 0:
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
        except Exception:
            uuid = None
        sampler = ClockSampler(uuid, local).start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if pa.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    K = args.steps
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctr = [args.warmup]

    def step_repeat():
        barrier(world)
        torch.cuda.synchronize()
        lead_gpu(torch)
        t_start.record(stream)
        for _ in range(K):
            step(ctr[0])
            ctr[0] += 1
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return t_start.elapsed_time(t_end)

    def dec_repeat():
        barrier(world)
        torch.cuda.synchronize()
        lead_gpu(torch)
        for i in range(K):
            decode_alone(ctr[0], dec_ev[i])
            ctr[0] += 1
        torch.cuda.synchronize()
        barrier(world)
        return float(np.sum([a_.elapsed_time(b_) for a_, b_ in dec_ev]))

    step_times = repeat_until(step_repeat, world)
    for i in range(3):
        decode_alone(i, dec_ev[0])
    dec_times = [t / K for t in repeat_until(dec_repeat, world)]
    clocks = sampler.stop() if sampler else None
    if pa.get_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    ms_step = max_over_ranks(float(np.median(step_times)), world) / K
    dec_ms = max_over_ranks(float(np.median(dec_times)), world)
    peaks = load_peaks()
    total_step = sum_over_ranks(float(decode_bytes + append_bytes), world)
    value = total_step / (ms_step * 1e-3) / 1e9
    achieved = decode_bytes / (dec_ms * 1e-3) / 1e9
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded N(0,1) values, shared-prompt beam state)",
        "config": {"workload": f"beam_cow: {WORKLOAD_TEXT['beam_cow']}", "num_seqs": S, "num_heads": Hq,
                   "num_kv_heads": H, "head_dim": D, "block_size": B, "context_tokens": int(lens_np.sum()),
                   "cow_pairs": n_pairs, "unique_kv_bytes": unique_kv, "logical_kv_bytes": logical_kv,
                   "step": "reshape_and_cache(1 new token/beam) + pa_decode" +
                           (", both launched with programmatic dependent launch" if pdl else ""),
                   "kernel_timing": "a second timed loop of K decode launches alone (ordinary launches), "
                                    "CUDA events around each on the launching stream",
                   "l2": f"{replicas} rotating KV pools ({replicas * pool_bytes / 1e9:.2f} GB) > L2 "
                         f"({l2 / 1e6:.0f} MB); the shared prompt is read by all beams within one launch",
                   "seed": args.seed, "launch": geometry},
        "pct_of_hbm_peak": round(100.0 * value / peaks["hbm_gbs"], 2),
        "effective_logical_kv_gbps": round(logical_kv / (dec_ms * 1e-3) / 1e9, 2),
        "decode_tokens_per_s": round(S / (ms_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel (pa_decode, one launch)",
                     "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                     "algorithmic_bytes_per_launch": decode_bytes, "bytes_basis": "unique KV rows",
                     "avg_launch_ms": round(dec_ms, 6), "traffic": load_traffic("beam_cow")},
        "repeats": {"step": spread(step_times, K), "decode_alone": spread(dec_times, 1)},
        "cpu_baseline": None,
        "gpu_launches": 2 * K * len(step_times) + K * len(dec_times),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if args.json_out:
        with open(args.json_out, "w") as f:
            json.dump(line, f, indent=1)


# ----------------------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    os.environ["OMP_NUM_THREADS"] = "1"
    import oracle
    batch = workloads.make_batch(args.workload, seed=args.seed)
    # host values for a handful of segments only (bounded): one sequence's KV head
    rng = np.random.default_rng(args.seed + 5)
    B, G, D = batch.block_size, batch.group, batch.head_dim
    s = int(rng.integers(0, batch.num_seqs))
    T_full = int(batch.seq_lens[s])
    per_step_budget = max(0.002, 120.0 / max(1, args.steps + args.warmup))
    # calibrate tokens per second of the oracle on synthetic rows of this format
    vrng = np.random.default_rng(args.seed + 6)

    def make(T):
        nb = -(-T // B)
        if batch.kv_fmt == "e4m3":
            kc = vrng.integers(0, 0x7E, size=(nb, 1, B, D)).astype(np.uint8)
            vc = vrng.integers(0, 0x7E, size=(nb, 1, B, D)).astype(np.uint8)
            sc = np.array([0.01], dtype=np.float32)
        elif batch.kv_fmt == "i8":
            kc = vrng.integers(-128, 128, size=(nb, 1, B, D)).astype(np.int8)
            vc = vrng.integers(-128, 128, size=(nb, 1, B, D)).astype(np.int8)
            sc = np.array([0.01], dtype=np.float32)
        else:
            kc = workloads.configs._normal_storage(vrng, (nb, 1, B, D), batch.kv_fmt)
            vc = workloads.configs._normal_storage(vrng, (nb, 1, B, D), batch.kv_fmt)
            sc = None
        q = workloads.configs._normal_storage(vrng, (1, G, D), batch.q_fmt)
        return q, kc, vc, np.arange(nb, dtype=np.int32)[None, :], np.array([T]), sc

    q, kc, vc, tb, ln, sc = make(min(T_full, 256))
    t0 = time.perf_counter()
    zp = np.zeros(1, dtype=np.int32) if batch.kv_fmt == "i8" else None
    oracle.paged_decode_attention(q, kc, vc, tb, ln, batch.scale, B, q_fmt=batch.q_fmt, kv_fmt=batch.kv_fmt,
                                  k_scale=sc, v_scale=sc, k_zero_point=zp, v_zero_point=zp)
    per_tok = (time.perf_counter() - t0) / int(ln[0])
    T = int(max(1, min(T_full, per_step_budget / max(per_tok, 1e-9))))
    q, kc, vc, tb, ln, sc = make(T)
    b_kv, b_q = FMT_BYTES[batch.kv_fmt], FMT_BYTES[batch.q_fmt]
    step_bytes = T * D * b_kv * 2 + 2 * G * D * b_q

    def one():
        oracle.paged_decode_attention(q, kc, vc, tb, ln, batch.scale, B, q_fmt=batch.q_fmt, kv_fmt=batch.kv_fmt,
                                      k_scale=sc, v_scale=sc, k_zero_point=zp, v_zero_point=zp)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    wall = time.perf_counter() - t0
    value = step_bytes * args.steps / wall / 1e9
    world = int(os.environ.get("WORLD_SIZE", "1"))
    sample = (f"one (sequence, KV head) segment of {T} tokens (of {T_full}) x G={G} query heads per step, "
              f"float64 numpy oracle, 1 thread" + (f"; rank 0 of {world} ran it alone" if world > 1 else ""))
    # n_gpus is the N of the launch (the driver pairs this line with the other arm's at the same N)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * wall / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT.get(args.workload, '')}"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_32x4k",
                    choices=["tiny", "gqa_32x4k", "long_32k", "fp8_mix", "int8_mix", "beam_cow"])
    ap.add_argument("--fused", action="store_true",
                    help="one launch per step: the new token's cache write fused into pa_decode_ex")
    ap.add_argument("--q-len", type=int, default=1,
                    help="queries per sequence (the q_len newest positions; speculative verification)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window decode over the last W positions (bytes counted over the window)")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--block-size", type=int, default=None, help="override the workload's block size")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the decode timing of the long_32k and fp8_mix configurations")
    ap.add_argument("--replicas", type=int, default=0, help="KV pool replicas to rotate (0 = enough for > 4x L2)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch the step's decode as an ordinary launch (no programmatic dependent launch)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-eager", action="store_true",
                    help="end-to-end steps issued call by call instead of replaying a recorded CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--min-time", type=float, default=MIN_TIMED_S,
                    help="repeat every timed loop until its repeats cover this many seconds (0: one repeat)")
    ap.add_argument("--json-out", default=None)
    args = ap.parse_args()
    MIN_TIME_S[0] = args.min_time
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.q_len > 1 and args.fused:
        ap.error("--fused appends one token per sequence (q_len 1)")
    if args.impl == "reference":
        if args.workload == "beam_cow":
            ap.error("the reference arm times the batch workloads")
        run_reference(args)
    elif args.workload == "beam_cow":
        run_beam(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

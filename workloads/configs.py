"""Seeded generators for the five decode workloads (inputs only; no method arithmetic)."""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

WORKLOADS = {
    "tiny": dict(num_seqs=4, num_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                 q_fmt="f16", kv_fmt="f16", scale=1.0 / 8.0,
                 lengths=("cached_uniform", 1, 128), pool=("fixed", 64)),
    "gqa_32x4k": dict(num_seqs=32, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      q_fmt="bf16", kv_fmt="bf16", scale=1.0 / math.sqrt(128.0),
                      lengths=("uniform", 1, 4096), pool=("slack", 0.10)),
    "long_32k": dict(num_seqs=8, num_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
                     q_fmt="bf16", kv_fmt="bf16", scale=1.0 / math.sqrt(128.0),
                     lengths=("const", 32768), pool=("slack", 0.0), partition_size=512),
    "beam_cow": dict(num_seqs=6, num_heads=40, num_kv_heads=40, head_dim=128, block_size=16,
                     q_fmt="f16", kv_fmt="f16", scale=1.0 / math.sqrt(128.0),
                     prompt_len=1000, tail_max=256),
    "fp8_mix": dict(num_seqs=256, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                    q_fmt="bf16", kv_fmt="e4m3", scale=1.0 / math.sqrt(128.0),
                    lengths=("lognormal", 7.0, 1.0, 16, 8192), pool=("slack", 0.10)),
    # the fp8_mix batch with an INT8 cache (per-head scale and zero point)
    "int8_mix": dict(num_seqs=256, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                     q_fmt="bf16", kv_fmt="i8", scale=1.0 / math.sqrt(128.0),
                     lengths=("lognormal", 7.0, 1.0, 16, 8192), pool=("slack", 0.10)),
}


@dataclass
class DecodeBatch:
    """Shapes, lengths and block tables of one decode step (no values)."""
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    q_fmt: str
    kv_fmt: str
    scale: float
    seq_lens: np.ndarray          # int32 [S]: tokens attended, including the appended one
    block_tables: np.ndarray      # int32 [S, MB]; unused entries are -1
    num_blocks: int
    new_slots: np.ndarray         # int64 [S]: slot of position seq_len-1 (the appended token)
    free_blocks: np.ndarray       # int32: pool ids that no table references
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    def cached_slots(self) -> np.ndarray:
        """Slots of positions 0..seq_len-2 of every sequence, concatenated (int64)."""
        out = []
        for s in range(self.num_seqs):
            for p in range(int(self.seq_lens[s]) - 1):
                out.append(slot_of(self.block_tables[s], p, self.block_size))
        return np.asarray(out, dtype=np.int64)


def slot_of(table_row, position: int, block_size: int) -> int:
    """Slot number of a token position through a block-table row."""
    return int(table_row[position // block_size]) * block_size + position % block_size


def _draw_lengths(spec, num_seqs: int, rng: np.random.Generator) -> np.ndarray:
    kind = spec[0]
    if kind == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=num_seqs)
    if kind == "cached_uniform":
        # cached length ~U{lo..hi}; one token is appended -> attended = cached + 1
        return rng.integers(spec[1], spec[2] + 1, size=num_seqs) + 1
    if kind == "const":
        return np.full(num_seqs, spec[1], dtype=np.int64)
    if kind == "lognormal":
        mu, sigma, lo, hi = spec[1:]
        return np.clip(np.round(rng.lognormal(mu, sigma, size=num_seqs)), lo, hi).astype(np.int64)
    raise ValueError(kind)


def _max_len(spec) -> int:
    kind = spec[0]
    if kind == "uniform":
        return spec[2]
    if kind == "cached_uniform":
        return spec[2] + 1
    if kind == "const":
        return spec[1]
    if kind == "lognormal":
        return spec[4]
    raise ValueError(kind)


def build_block_tables(seq_lens, block_size: int, rng: np.random.Generator, *,
                       pool=("slack", 0.10), max_blocks_per_seq: int | None = None):
    """Assign physical blocks from a seeded permutation of the pool.

    Blocks holding the cached tokens (positions 0..len-2) are handed out first,
    sequence by sequence; a block opened by the appended token (position len-1)
    comes afterwards from the remaining ids.  Returns (tables, num_blocks, free).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    S = len(seq_lens)
    cached_blocks = [-(-max(int(t) - 1, 0) // block_size) for t in seq_lens]
    total_blocks = [-(-int(t) // block_size) for t in seq_lens]
    needed = sum(total_blocks)
    if pool[0] == "fixed":
        nb = int(pool[1])
    else:
        nb = int(math.ceil(needed * (1.0 + pool[1])))
    if nb < needed:
        raise ValueError("pool too small")
    mb = max_blocks_per_seq if max_blocks_per_seq is not None else max(max(total_blocks), 1)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((S, mb), -1, dtype=np.int32)
    cur = 0
    for s in range(S):
        n = cached_blocks[s]
        tables[s, :n] = perm[cur:cur + n]
        cur += n
    for s in range(S):
        if total_blocks[s] > cached_blocks[s]:
            tables[s, cached_blocks[s]] = perm[cur]
            cur += 1
    return tables, nb, perm[cur:].copy()


def make_batch(name: str, seed: int = 0, **overrides) -> DecodeBatch:
    """Lengths and block tables of a named workload (seeded)."""
    if name == "beam_cow":
        raise ValueError("beam_cow is built by beam_cow_scenario()")
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    rng = np.random.default_rng(seed)
    S = cfg["num_seqs"]
    B = cfg["block_size"]
    seq_lens = _draw_lengths(cfg["lengths"], S, rng)
    mb = -(-_max_len(cfg["lengths"]) // B)
    tables, nb, free = build_block_tables(seq_lens, B, rng, pool=cfg["pool"], max_blocks_per_seq=mb)
    new_slots = np.array([slot_of(tables[s], int(seq_lens[s]) - 1, B) for s in range(S)], dtype=np.int64)
    extra = {k: v for k, v in cfg.items() if k not in (
        "num_seqs", "num_heads", "num_kv_heads", "head_dim", "block_size", "q_fmt", "kv_fmt",
        "scale", "lengths", "pool")}
    extra["seed"] = seed
    return DecodeBatch(name=name, num_seqs=S, num_heads=cfg["num_heads"],
                       num_kv_heads=cfg["num_kv_heads"], head_dim=cfg["head_dim"], block_size=B,
                       q_fmt=cfg["q_fmt"], kv_fmt=cfg["kv_fmt"], scale=float(cfg["scale"]),
                       seq_lens=seq_lens.astype(np.int32), block_tables=tables, num_blocks=nb,
                       new_slots=new_slots, free_blocks=free, extra=extra)


# ----------------------------------------------------------------------------- values

def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), rounded by torch (nearest-even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _normal_storage(rng: np.random.Generator, shape, fmt: str, mult: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if mult != 1.0:
        x = (x * np.float32(mult)).astype(np.float32)
    if fmt == "f16":
        return x.astype(np.float16)
    if fmt == "bf16":
        return bf16_bits_from_f32(x)
    raise ValueError(fmt)


def fp8_scales_from_amax(amax: np.ndarray):
    """Per-KV-head calibration: scale = amax / 448 and inv = 1 / scale, both float32."""
    amax = np.asarray(amax, dtype=np.float32)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    scale = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    return scale, inv


def int8_params_from_range(mn: np.ndarray, mx: np.ndarray):
    """Per-head INT8 calibration from the value range: scale = (max - min) / 255 (float32),
    zero point = clamp(round(-128 - min / scale), -128, 127) (int32), inv = 1 / scale (float32)."""
    mn = np.asarray(mn, dtype=np.float32)
    mx = np.asarray(mx, dtype=np.float32)
    scale = ((mx - mn) / np.float32(255.0)).astype(np.float32)
    scale = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    zp = np.clip(np.round(-128.0 - mn.astype(np.float64) / scale.astype(np.float64)), -128, 127).astype(np.int32)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    return scale, zp, inv


def _bf16_range_per_head(*arrays):
    """(min, max) per KV head (axis 1) over bf16-bit arrays [N, H_kv, d], via torch."""
    import torch
    lo = hi = None
    for a in arrays:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).float()
        a_lo, a_hi = t.amin(dim=(0, 2)), t.amax(dim=(0, 2))
        lo = a_lo if lo is None else torch.minimum(lo, a_lo)
        hi = a_hi if hi is None else torch.maximum(hi, a_hi)
    return lo.numpy().astype(np.float32), hi.numpy().astype(np.float32)


def _bf16_amax_per_head(*arrays) -> np.ndarray:
    """max |x| per KV head (axis 1) over bf16-bit arrays [N, H_kv, d], via torch."""
    import torch
    m = None
    for a in arrays:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        am = t.float().abs().amax(dim=(0, 2))
        m = am if m is None else torch.maximum(m, am)
    return m.numpy().astype(np.float32)


def host_values(batch: DecodeBatch, seed: int = 0, *, q_mult: float = 1.0, nan_tails: bool = True,
                q_len: int = 1):
    """Numpy storage arrays for a (small) batch.

    16-bit caches: every cached position gets N(0,1) values; slots that no
    sequence attends are NaN when ``nan_tails`` (to prove they are never read
    into the result).  The appended token's rows are separate draws (k_new,
    v_new) that a cache write places at ``new_slots``.
    FP8 caches: the cache starts as zero bytes; ``k_src``/``v_src`` hold the
    bf16 values of every cached position (in ``cached_slots()`` order) and
    the calibration scales; the caller quantises them into the cache.
    """
    rng = np.random.default_rng(seed + 7919)
    S, Hq, Hkv, d, B, NB = (batch.num_seqs, batch.num_heads, batch.num_kv_heads,
                            batch.head_dim, batch.block_size, batch.num_blocks)
    out = {}
    # q_len > 1: [S, q_len, H_q, d], the queries of the q_len newest positions
    out["q"] = _normal_storage(rng, (S, Hq, d) if q_len == 1 else (S, q_len, Hq, d), batch.q_fmt, q_mult)
    if batch.kv_fmt in ("f16", "bf16"):
        k = _normal_storage(rng, (NB, Hkv, B, d), batch.kv_fmt)
        v = _normal_storage(rng, (NB, Hkv, B, d), batch.kv_fmt)
        if nan_tails:
            used = np.zeros((NB, B), dtype=bool)
            for s in range(S):
                for p in range(int(batch.seq_lens[s]) - 1):
                    used[batch.block_tables[s, p // B], p % B] = True
            nan_bits = np.float16(np.nan) if batch.kv_fmt == "f16" else np.uint16(0x7FC0)
            ib, io = np.nonzero(~used)
            k[ib, :, io, :] = nan_bits
            v[ib, :, io, :] = nan_bits
        out["k_cache"], out["v_cache"] = k, v
        out["k_new"] = _normal_storage(rng, (S, Hkv, d), batch.kv_fmt)
        out["v_new"] = _normal_storage(rng, (S, Hkv, d), batch.kv_fmt)
    elif batch.kv_fmt in ("e4m3", "i8"):
        slots = batch.cached_slots()
        n = len(slots)
        ks32 = rng.standard_normal(size=(n, Hkv, d), dtype=np.float32)
        vs32 = rng.standard_normal(size=(n, Hkv, d), dtype=np.float32)
        kn32 = rng.standard_normal(size=(S, Hkv, d), dtype=np.float32)
        vn32 = rng.standard_normal(size=(S, Hkv, d), dtype=np.float32)
        kb, vb = bf16_bits_from_f32(ks32), bf16_bits_from_f32(vs32)
        knb, vnb = bf16_bits_from_f32(kn32), bf16_bits_from_f32(vn32)
        out["k_src"], out["v_src"], out["src_slots"] = kb, vb, slots
        out["k_new"], out["v_new"] = knb, vnb
        if batch.kv_fmt == "e4m3":
            out["k_scale"], out["k_inv_scale"] = fp8_scales_from_amax(_bf16_amax_per_head(kb, knb))
            out["v_scale"], out["v_inv_scale"] = fp8_scales_from_amax(_bf16_amax_per_head(vb, vnb))
        else:
            out["k_scale"], out["k_zero_point"], out["k_inv_scale"] = int8_params_from_range(*_bf16_range_per_head(kb, knb))
            out["v_scale"], out["v_zero_point"], out["v_inv_scale"] = int8_params_from_range(*_bf16_range_per_head(vb, vnb))
        cdt = np.uint8 if batch.kv_fmt == "e4m3" else np.int8
        out["k_cache"] = np.zeros((NB, Hkv, B, d), dtype=cdt)
        out["v_cache"] = np.zeros((NB, Hkv, B, d), dtype=cdt)
    else:
        raise ValueError(batch.kv_fmt)
    return out


def device_values(batch: DecodeBatch, seed: int, device, *, q_mult: float = 1.0):
    """torch tensors on ``device`` for a (large) batch, drawn by torch's device RNG.

    16-bit caches: every slot of the pool is N(0,1).  FP8: bf16 sources for all
    cached positions plus calibration scales (computed on the host from the
    per-head amax), as in ``host_values``.
    """
    import torch
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    S, Hq, Hkv, d, B, NB = (batch.num_seqs, batch.num_heads, batch.num_kv_heads,
                            batch.head_dim, batch.block_size, batch.num_blocks)

    def randn(shape, fmt, mult=1.0):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if mult != 1.0:
            x.mul_(mult)
        return x.to(dt[fmt])

    out = {"q": randn((S, Hq, d), batch.q_fmt, q_mult)}
    if batch.kv_fmt in ("f16", "bf16"):
        out["k_cache"] = randn((NB, Hkv, B, d), batch.kv_fmt)
        out["v_cache"] = randn((NB, Hkv, B, d), batch.kv_fmt)
        out["k_new"] = randn((S, Hkv, d), batch.kv_fmt)
        out["v_new"] = randn((S, Hkv, d), batch.kv_fmt)
    else:
        slots = batch.cached_slots()
        n = len(slots)
        out["k_src"] = randn((n, Hkv, d), "bf16")
        out["v_src"] = randn((n, Hkv, d), "bf16")
        out["k_new"] = randn((S, Hkv, d), "bf16")
        out["v_new"] = randn((S, Hkv, d), "bf16")
        out["src_slots"] = torch.from_numpy(slots).to(device)
        for kv in ("k", "v"):
            src, new = out[f"{kv}_src"].float(), out[f"{kv}_new"].float()
            if batch.kv_fmt == "e4m3":
                a = torch.maximum(src.abs().amax(dim=(0, 2)), new.abs().amax(dim=(0, 2)))
                sc, inv = fp8_scales_from_amax(a.cpu().numpy())
            else:
                lo = torch.minimum(src.amin(dim=(0, 2)), new.amin(dim=(0, 2)))
                hi = torch.maximum(src.amax(dim=(0, 2)), new.amax(dim=(0, 2)))
                sc, zp, inv = int8_params_from_range(lo.cpu().numpy(), hi.cpu().numpy())
                out[f"{kv}_zero_point"] = torch.from_numpy(zp).to(device)
            out[f"{kv}_scale"] = torch.from_numpy(sc).to(device)
            out[f"{kv}_inv_scale"] = torch.from_numpy(inv).to(device)
        cdt = torch.uint8 if batch.kv_fmt == "e4m3" else torch.int8
        out["k_cache"] = torch.zeros((NB, Hkv, B, d), dtype=cdt, device=device)
        out["v_cache"] = torch.zeros((NB, Hkv, B, d), dtype=cdt, device=device)
    return out


def beam_cow_scenario(seed: int = 0, *, num_blocks: int = 256):
    """Raw inputs of the shared-prompt / beam workload (decisions are the block manager's).

    Returns the prompt rows, each beam's tail rows, each beam's appended row,
    the query and the free-list order of the pool.
    """
    cfg = WORKLOADS["beam_cow"]
    rng = np.random.default_rng(seed)
    nbeams, H, d, P = cfg["num_seqs"], cfg["num_kv_heads"], cfg["head_dim"], cfg["prompt_len"]
    tails = rng.integers(1, cfg["tail_max"] + 1, size=nbeams)
    free_order = rng.permutation(num_blocks).astype(np.int32)
    vrng = np.random.default_rng(seed + 104729)
    out = dict(
        num_beams=nbeams, num_heads=cfg["num_heads"], num_kv_heads=H, head_dim=d,
        block_size=cfg["block_size"], prompt_len=P, tails=tails, num_blocks=num_blocks,
        free_order=free_order, scale=cfg["scale"], q_fmt="f16", kv_fmt="f16",
        prompt_k=_normal_storage(vrng, (P, H, d), "f16"),
        prompt_v=_normal_storage(vrng, (P, H, d), "f16"),
        tail_k=[_normal_storage(vrng, (int(t), H, d), "f16") for t in tails],
        tail_v=[_normal_storage(vrng, (int(t), H, d), "f16") for t in tails],
        new_k=_normal_storage(vrng, (nbeams, H, d), "f16"),
        new_v=_normal_storage(vrng, (nbeams, H, d), "f16"),
        q=_normal_storage(vrng, (nbeams, cfg["num_heads"], d), "f16"),
    )
    return out


def shard_sequences(num_seqs: int, rank: int, world_size: int):
    """Contiguous [start, stop) share of ``num_seqs`` sequences for ``rank``."""
    base, rem = divmod(num_seqs, world_size)
    start = rank * base + min(rank, rem)
    stop = start + base + (1 if rank < rem else 0)
    return start, stop

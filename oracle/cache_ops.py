"""Byte-level semantics of the cache write and the copy-on-write block copy.

Test infrastructure (see ``oracle/__init__``).

reshape_and_cache
    [P2] §"PagedAttention: OS仮想メモリ式の管理": blocks are handed out one at a
    time as a request's tokens accumulate, and the block table maps each
    logical token position to a physical block.  A new token's K and V are
    therefore written into the slot that its position maps to.  Reading
    (the pages give no encoding): slot = physical_block * B + (position % B),
    carried as int64; a negative slot marks a padding token that is skipped.
    The row lands at cache[slot // B, h, slot % B, :] for every KV head h.
    16-bit caches receive the source bits unchanged.  FP8-e4m3 caches receive
    e4m3_rne_satfinite(float32(x) * inv_scale[h]), the product rounded in
    IEEE float32 ([P2] §"KV量子化" for FP8 storage; codec in ``codecs``).
    INT8 caches receive clamp(rne(float32(x) * inv_scale[h]) + zero_point[h],
    -128, 127) (same section, "scale / zero point"; codec in ``codecs``).

copy_blocks
    [P1] §"Copy-on-Write（CoW）によるメモリ共有": when a sequence must write into a
    block whose reference count exceeds one, a new block is allocated and the
    old block's contents are copied into it before the write.  Each
    (src, dst) pair copies the whole physical block (every KV head, every
    slot) for both K and V.  All sources are read before any destination is
    written.

Pins: hand-made fixtures (``tests/golden/``), scatter/gather round trips and
CoW isolation (``tests/test_oracle_pins.py``).
"""

from __future__ import annotations

import numpy as np

from .codecs import e4m3_encode_f32, int8_encode_f32, storage_to_f32


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, block_size, *,
                      src_fmt="f16", kv_fmt="f16", k_inv_scale=None, v_inv_scale=None,
                      k_zero_point=None, v_zero_point=None):
    """Return new (k_cache, v_cache) with tokens' rows written to their slots.

    k, v: [N, H_kv, d] in the source storage format (float16 or bf16 bits).
    caches: [NB, H_kv, B, d] in the cache storage format.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    Hkv = k_out.shape[1]
    for n, slot in enumerate(slots):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        for src, dst, inv, zp in ((k, k_out, k_inv_scale, k_zero_point), (v, v_out, v_inv_scale, v_zero_point)):
            row = np.asarray(src[n])
            if kv_fmt in ("e4m3", "i8"):
                x = storage_to_f32(row, src_fmt)                 # [H_kv, d] float32
                inv32 = np.asarray(inv, dtype=np.float32)[:Hkv, None]
                prod = (x * inv32).astype(np.float32)            # IEEE float32 product
                if kv_fmt == "e4m3":
                    dst[blk, :, off, :] = e4m3_encode_f32(prod)
                else:
                    dst[blk, :, off, :] = int8_encode_f32(prod, np.asarray(zp, dtype=np.int64)[:Hkv, None])
            else:
                if kv_fmt != src_fmt:
                    raise ValueError("16-bit caches take source bits unchanged")
                dst[blk, :, off, :] = row
    return k_out, v_out


def copy_blocks(k_cache, v_cache, pairs):
    """Return new (k_cache, v_cache) with block dst := block src for each pair."""
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    k_src = [np.array(k_cache[s], copy=True) for s, _ in pairs]
    v_src = [np.array(v_cache[s], copy=True) for s, _ in pairs]
    for i, (_, d) in enumerate(pairs):
        k_out[d] = k_src[i]
        v_out[d] = v_src[i]
    return k_out, v_out

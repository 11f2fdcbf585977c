"""Paged single-query decode attention, written as its plain definition.

Test infrastructure (see ``oracle/__init__``).

What is computed
----------------
[P1] §"Attention計算": Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V with Q a
single row during autoregressive decoding; with the cache split into blocks
K_j, V_j of B tokens, the blockwise scores A_j = Q K_j^T / sqrt(d_k) are
concatenated over j < ceil(n/B) and one softmax over the concatenation
multiplies [V_0; V_1; ...].  [P3] §"分块 Attention 计算" gives the same
per-token weights A_ij = exp(q_i.k_j/sqrt d) / sum_t exp(q_i.k_t/sqrt d) with
o_i = sum_j A_ij v_j.  Because the paged method reaches exactly this result
([P4] §6 calls it exact attention), the oracle is that definition: gather the
sequence's rows through its block table ([P1] §"PagedAttentionのメモリ管理":
logical block j -> physical block table[j]), convert to float64, form the
scaled scores, take a max-subtracted softmax and multiply by V.

Readings where the pages are silent:
  * cache layout: separate K and V pools of shape [num_blocks, H_kv, B, d];
    token position p of a sequence lives in physical block table[p // B],
    row p % B.  The layout is invisible to results.
  * grouped-query attention ([P2] §"GQAとMQA": query heads are grouped and each
    group shares one KV head): query head h reads KV head h // (H_q / H_kv).
  * scale: the float32 value passed to the kernel, widened to float64.
  * FP8 KV ([P2] §"KV量子化"): value = float64(e4m3 code) * float64(scale[h])
    with one float32 scale per KV head, separately for K and V.
  * INT8 KV (same section: "scale / zero point"): value = (code - zp[h]) *
    float64(scale[h]), one float32 scale and one integer zero point per KV
    head, separately for K and V (codec in ``codecs``).
  * a sequence of length 0 attends to nothing; its output is defined as 0.
  * several queries per sequence (the explainer's related-work and outlook
    sections tie paged KV memory to speculative decoding, which verifies a
    few proposed tokens in one step; no formula is given): with q_len = L,
    the L newest positions T-L .. T-1 of a sequence are queries and query i
    attends to the positions up to and including its own, T-L+i (causal
    among the new tokens, all older rows visible).
  * sliding window (named as a limitation of the paged kernel in the
    "局限性与未来工作" list of the dihengye.cn notes, no definition given):
    with a window W > 0 the single query of a sequence of length T, which sits
    at position T-1, attends to positions max(0, T-W) .. T-1 only; W = 0
    means the whole sequence.

Pins: brute-force triple loop, textbook numpy attention for MHA, T=1 -> v_0,
constant keys -> mean(V), one dominant logit -> that V row, block-layout
permutation invariance, GQA reduction to MHA, online-softmax agreement
(``tests/test_oracle_pins.py``).
"""

from __future__ import annotations

import numpy as np

from .codecs import int8_decode, storage_to_f64


def dequantize_kv(cache: np.ndarray, fmt: str, scale: np.ndarray | None = None,
                  zero_point: np.ndarray | None = None) -> np.ndarray:
    """Storage cache [NB, H_kv, B, d] -> float64, applying per-KV-head scale (and zero point for i8)."""
    if fmt == "i8":
        if scale is None or zero_point is None:
            raise ValueError("i8 cache needs a per-KV-head scale and zero point")
        zp = np.asarray(zero_point, dtype=np.int64)[None, :, None, None]
        sc = np.asarray(scale, dtype=np.float32).astype(np.float64)[None, :, None, None]
        return int8_decode(cache, zp) * sc
    out = storage_to_f64(cache, fmt)
    if fmt == "e4m3":
        if scale is None:
            raise ValueError("e4m3 cache needs a per-KV-head scale")
        sc = np.asarray(scale, dtype=np.float32).astype(np.float64)
        out = out * sc[None, :, None, None]
    return out


def gather_sequence(cache_f64: np.ndarray, table_row: np.ndarray, seq_len: int,
                    block_size: int, kv_head: int) -> np.ndarray:
    """Rows 0..seq_len-1 of one sequence for one KV head, through its block table."""
    n_blocks = -(-int(seq_len) // block_size)
    if n_blocks == 0:
        return np.zeros((0, cache_f64.shape[-1]), dtype=np.float64)
    phys = np.asarray(table_row[:n_blocks], dtype=np.int64)
    rows = cache_f64[phys, kv_head, :, :]          # [n_blocks, B, d]
    rows = rows.reshape(n_blocks * block_size, -1)
    return rows[: int(seq_len)]


def dense_decode_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * K q) V for one query vector, float64, max-subtracted."""
    q = np.asarray(q, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1], dtype=np.float64)
    s = float(scale) * (K @ q)
    s = s - s.max()
    w = np.exp(s)
    w = w / w.sum()
    return w @ V


def _scale64(scale: float) -> float:
    return float(np.float32(scale))


def window_start(seq_len: int, window: int) -> int:
    """First attended position of the query at position seq_len-1 (window 0 = all)."""
    return max(0, int(seq_len) - int(window)) if window and window > 0 else 0


def paged_decode_attention_one(q, k_cache, v_cache, block_tables, seq_lens, scale,
                               block_size, s, h, *, q_fmt="f16", kv_fmt="f16",
                               k_scale=None, v_scale=None, num_kv_heads=None, window=0,
                               k_zero_point=None, v_zero_point=None):
    """Output vector out[s, h, :] only (for sampled checks on large inputs).

    ``k_cache``/``v_cache`` may be the full pool or any array indexable by the
    physical block ids that sequence ``s`` uses.
    """
    Hq = q.shape[1]
    Hkv = num_kv_heads if num_kv_heads is not None else k_cache.shape[1]
    G = Hq // Hkv
    kvh = h // G
    T = int(seq_lens[s])
    n_blocks = -(-T // block_size)
    phys = np.asarray(block_tables[s][:n_blocks], dtype=np.int64)
    kb = k_cache[phys, kvh]
    vb = v_cache[phys, kvh]
    ks = None if k_scale is None else np.asarray(k_scale)[kvh:kvh + 1]
    vs = None if v_scale is None else np.asarray(v_scale)[kvh:kvh + 1]
    kz = None if k_zero_point is None else np.asarray(k_zero_point)[kvh:kvh + 1]
    vz = None if v_zero_point is None else np.asarray(v_zero_point)[kvh:kvh + 1]
    lo = window_start(T, window)
    Kf = dequantize_kv(kb[:, None], kv_fmt, ks, kz)[:, 0].reshape(-1, kb.shape[-1])[lo:T]
    Vf = dequantize_kv(vb[:, None], kv_fmt, vs, vz)[:, 0].reshape(-1, vb.shape[-1])[lo:T]
    qv = storage_to_f64(q[s, h], q_fmt)
    return dense_decode_attention(qv, Kf, Vf, _scale64(scale))


def paged_decode_attention(q, k_cache, v_cache, block_tables, seq_lens, scale, block_size,
                           *, q_fmt="f16", kv_fmt="f16", k_scale=None, v_scale=None, window=0,
                           k_zero_point=None, v_zero_point=None):
    """out[S, H_q, d] float64 for every sequence and query head (window: see module notes)."""
    S, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    G = Hq // Hkv
    Kc = dequantize_kv(k_cache, kv_fmt, k_scale, k_zero_point)
    Vc = dequantize_kv(v_cache, kv_fmt, v_scale, v_zero_point)
    qf = storage_to_f64(q, q_fmt)
    sc = _scale64(scale)
    out = np.zeros((S, Hq, d), dtype=np.float64)
    for s in range(S):
        T = int(seq_lens[s])
        lo = window_start(T, window)
        for kvh in range(Hkv):
            K = gather_sequence(Kc, block_tables[s], T, block_size, kvh)[lo:]
            V = gather_sequence(Vc, block_tables[s], T, block_size, kvh)[lo:]
            for g in range(G):
                h = kvh * G + g
                out[s, h] = dense_decode_attention(qf[s, h], K, V, sc)
    return out


def paged_append_decode(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, scale, block_size, *,
                        q_fmt="f16", src_fmt="f16", kv_fmt="f16", k_scale=None, v_scale=None,
                        k_inv_scale=None, v_inv_scale=None, k_zero_point=None, v_zero_point=None, window=0):
    """Append + decode in one step: the rows k_new[s], v_new[s] of position seq_lens[s]-1 are written to
    the slot that position maps to through the block table (the cache write of ``cache_ops``), then every
    sequence attends over its seq_lens[s] rows (including the new one).

    [P2] §"PagedAttention: OS仮想メモリ式の管理": a new token's K and V go into the slot of its position;
    [P1] §"Attention計算": the query then attends over all cached rows.  Returns (out, k_cache, v_cache).
    """
    from .cache_ops import reshape_and_cache
    S = q.shape[0]
    slots = []
    for s in range(S):
        T = int(seq_lens[s])
        if T <= 0:
            slots.append(-1)
            continue
        p = T - 1
        slots.append(int(block_tables[s][p // block_size]) * block_size + p % block_size)
    kc, vc = reshape_and_cache(k_new, v_new, k_cache, v_cache, slots, block_size, src_fmt=src_fmt, kv_fmt=kv_fmt,
                               k_inv_scale=k_inv_scale, v_inv_scale=v_inv_scale, k_zero_point=k_zero_point,
                               v_zero_point=v_zero_point)
    out = paged_decode_attention(q, kc, vc, block_tables, seq_lens, scale, block_size, q_fmt=q_fmt, kv_fmt=kv_fmt,
                                 k_scale=k_scale, v_scale=v_scale, window=window, k_zero_point=k_zero_point,
                                 v_zero_point=v_zero_point)
    return out, kc, vc


def paged_multi_query_attention(q, k_cache, v_cache, block_tables, seq_lens, scale, block_size, *,
                                q_fmt="f16", kv_fmt="f16", k_scale=None, v_scale=None, window=0,
                                k_zero_point=None, v_zero_point=None):
    """out[S, L, H_q, d]: query i of sequence s (position T-L+i) attends to positions
    max(0, T-L+i-W+1) .. T-L+i (W = window, 0 = no lower bound).  q is [S, L, H_q, d]."""
    S, L, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    G = Hq // Hkv
    Kc = dequantize_kv(k_cache, kv_fmt, k_scale, k_zero_point)
    Vc = dequantize_kv(v_cache, kv_fmt, v_scale, v_zero_point)
    qf = storage_to_f64(q, q_fmt)
    sc = _scale64(scale)
    out = np.zeros((S, L, Hq, d), dtype=np.float64)
    for s in range(S):
        T = int(seq_lens[s])
        for kvh in range(Hkv):
            K = gather_sequence(Kc, block_tables[s], T, block_size, kvh)
            V = gather_sequence(Vc, block_tables[s], T, block_size, kvh)
            for i in range(L):
                pos = T - L + i
                if pos < 0:
                    continue            # the sequence is shorter than its query count: nothing to attend
                lo = max(0, pos - window + 1) if window and window > 0 else 0
                for g in range(G):
                    h = kvh * G + g
                    out[s, i, h] = dense_decode_attention(qf[s, i, h], K[lo:pos + 1], V[lo:pos + 1], sc)
    return out

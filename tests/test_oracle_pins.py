"""Pins for the float64 oracle: checks against things other than the oracle itself.

Each check is written as a helper that takes the function under test, so the
last block of tests can plant a mistake in a copy of the oracle (on the CPU)
and show that the same check catches it.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import online_softmax as osm
from oracle import attention as att
from oracle.codecs import e4m3_decode, e4m3_encode_f32, bf16_bits_to_f64

torch = pytest.importorskip("torch")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ accounting

def test_kv_bytes_worked_example(golden_dir):
    g = _load(golden_dir, "kv_bytes.json")
    L, H, d, b = g["num_layers"], g["num_kv_heads"], g["head_dim"], g["bytes_per_scalar"]
    assert oracle.kv_bytes_per_token(L, H, d, b) == g["bytes_per_token"] == 131072
    assert oracle.kv_bytes(L, H, d, b, [g["tokens_per_request"]]) == g["bytes_per_request"]
    assert g["bytes_per_request"] == 2 ** 29  # 0.5 GiB
    assert oracle.kv_bytes(L, H, d, b, [g["tokens_per_request"]] * g["requests"]) == g["bytes_32_requests"]
    assert oracle.kv_bytes(L, g["num_kv_heads_mha"], d, b, [g["tokens_per_request"]]) == g["bytes_per_request_mha"]
    assert g["bytes_per_request_mha"] == 2 * 2 ** 30


def test_kv_bytes_verification_record(golden_dir):
    g = _load(golden_dir, "verification_record.json")
    assert oracle.kv_bytes_per_token(32, 8, 128, 2) == g["bytes_per_token"]


def test_tail_waste_bound_exhaustive():
    for B in [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]:
        for T in range(1, 4097):
            w = oracle.tail_waste_one(T, B)
            assert 0 <= w <= B - 1
            assert (w == 0) == (T % B == 0)
            # allocated capacity is the smallest multiple of B that holds T
            assert (T + w) % B == 0 and T + w - B < T


def test_tail_waste_sum_bound():
    rng = np.random.default_rng(1)
    for B in [1, 16, 32, 100]:
        lens = rng.integers(1, 5000, size=200)
        W = oracle.tail_waste(lens, B)
        assert 0 <= W <= len(lens) * (B - 1)


def test_mean_tail_waste_exact(golden_dir):
    g = _load(golden_dir, "tail_waste.json")
    n = g["uniform_max_len"]
    for B in [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]:
        assert oracle.mean_tail_waste_uniform(B, n) == Fraction(B - 1, 2)
    # other multiples kB of the page size (equation (3))
    for B, k in [(3, 7), (16, 5), (10, 13)]:
        assert oracle.mean_tail_waste_uniform(B, k * B) == Fraction(B - 1, 2)


def test_reserve_512_mean_waste(golden_dir):
    g = _load(golden_dir, "tail_waste.json")
    assert oracle.mean_reserve_waste_uniform(g["reserve_slots"], g["uniform_max_len"]) == Fraction(511, 2)
    assert float(Fraction(511, 2)) == g["reserve_mean_waste"]


def test_two_requests_fixture(golden_dir):
    g = _load(golden_dir, "two_requests.json")
    B = g["block_size"]
    for r in g["requests"]:
        assert len(r["table"]) == -(-r["tokens"] // B)
        assert sum(r["tokens_per_block"]) == r["tokens"]
        assert oracle.tail_waste_one(r["tokens"], B) == r["tail_waste"]


# ------------------------------------------------------------------ codecs

def test_e4m3_known_values():
    assert e4m3_decode(np.array([0x7E]))[0] == 448.0            # largest finite
    assert e4m3_decode(np.array([0xFE]))[0] == -448.0
    assert e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6        # smallest normal
    assert e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9        # smallest subnormal
    assert e4m3_decode(np.array([0x07]))[0] == 7 * 2.0 ** -9    # largest subnormal
    assert e4m3_decode(np.array([0x38]))[0] == 1.0
    assert e4m3_decode(np.array([0x39]))[0] == 1.125
    assert e4m3_decode(np.array([0x00]))[0] == 0.0
    z = e4m3_decode(np.array([0x80]))[0]
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    assert np.isnan(e4m3_decode(np.array([0x7F]))[0]) and np.isnan(e4m3_decode(np.array([0xFF]))[0])
    finite = e4m3_decode(np.arange(0, 0x7F))
    assert np.all(np.diff(finite) > 0)                           # magnitudes increase with the code


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3_decode(codes)
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(ours[~both_nan]))


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(e4m3_encode_f32(vals), codes)


def check_e4m3_encode_vs_torch(encode, n=200000, seed=0):
    """Encode in-range float32 values; compare with torch's float8_e4m3fn rounding."""
    rng = np.random.default_rng(seed)
    x = np.concatenate([
        rng.standard_normal(n).astype(np.float32) * np.float32(50.0),
        (rng.standard_normal(n) * 2.0 ** -8).astype(np.float32),      # subnormal range
        rng.uniform(-448.0, 448.0, n).astype(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.count_nonzero(encode(x) != ref)


def test_e4m3_encode_vs_torch():
    assert check_e4m3_encode_vs_torch(e4m3_encode_f32) == 0


def check_e4m3_ties(encode):
    """Exact midpoints between adjacent codes must go to the even code."""
    codes = np.arange(0, 0x7E, dtype=np.int64)       # pairs (c, c+1), both finite
    lo = e4m3_decode(codes.astype(np.uint8))
    hi = e4m3_decode((codes + 1).astype(np.uint8))
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)   # midpoints exact in float32
    want = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    return np.count_nonzero(encode(mid) != want) + np.count_nonzero(encode(-mid) != (want | 0x80))


def test_e4m3_ties_to_even():
    assert check_e4m3_ties(e4m3_encode_f32) == 0
    # and just off the midpoint the nearer code wins
    assert e4m3_encode_f32(np.array([np.nextafter(np.float32(1.0625), np.float32(2))]))[0] == 0x39
    assert e4m3_encode_f32(np.array([np.nextafter(np.float32(1.0625), np.float32(0))]))[0] == 0x38


def test_e4m3_saturation_and_signed_zero():
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(e4m3_encode_f32(big) == 0x7E)
    assert np.all(e4m3_encode_f32(-big) == 0xFE)
    assert e4m3_encode_f32(np.array([-0.0], dtype=np.float32))[0] == 0x80
    assert e4m3_encode_f32(np.array([-(2.0 ** -11)], dtype=np.float32))[0] == 0x80
    assert e4m3_encode_f32(np.array([2.0 ** -10], dtype=np.float32))[0] == 0x00   # tie -> even (zero)
    assert e4m3_encode_f32(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def test_bf16_decode_vs_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 16, size=100000, dtype=np.uint32).astype(np.uint16)
    exp_field = (bits >> 7) & 0xFF
    bits = bits[exp_field != 0xFF]                       # drop inf/NaN patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf16_bits_to_f64(bits), ref)


# ------------------------------------------------------------------ attention

def _rand_qkv(rng, T, d, mult=1.0):
    q = rng.standard_normal(d) * mult
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    return q, K, V


def check_online_vs_dense(online_fn, dense_fn, seed=0):
    """Largest |online - dense| over many block sizes, lengths and logit scales."""
    rng = np.random.default_rng(seed)
    worst = 0.0
    for T in [1, 2, 5, 17, 100, 513, 1000]:
        for mult in [1.0, 30.0, 1000.0]:
            q, K, V = _rand_qkv(rng, T, 16, mult)
            ref = dense_fn(q, K, V, 0.25)
            for B in [1, 2, 3, 7, 16, 32, 512]:
                worst = max(worst, float(np.max(np.abs(online_fn(q, K, V, 0.25, B) - ref))))
    return worst


def test_online_softmax_equals_dense(golden_dir):
    rec = _load(golden_dir, "verification_record.json")
    worst = check_online_vs_dense(oracle.online_softmax_attention, oracle.dense_decode_attention)
    assert worst <= 1e-12
    # the pages' own binary64 record is of the same class (a few ulp of O(1) values)
    assert rec["largest_absolute_error"] < 1e-12


def test_merge_of_partials_equals_single_pass():
    rng = np.random.default_rng(5)
    for T in [1, 3, 64, 700]:
        q, K, V = _rand_qkv(rng, T, 8, 30.0)
        ref = oracle.dense_decode_attention(q, K, V, 0.5)
        cuts = sorted(set(rng.integers(0, T + 1, size=5).tolist()) | {0, T})
        parts = [oracle.partial_state(q, K[a:b], V[a:b], 0.5, 16) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
        assert np.max(np.abs(oracle.merge_partials(parts) - ref)) <= 1e-12
        # merging is independent of how the ranges are grouped
        if len(parts) >= 2:
            assert np.max(np.abs(oracle.merge_partials(parts[::-1]) - ref)) <= 1e-12


def _brute_force_one(q, rows_k, rows_v, scale):
    """Triple loop in plain Python floats: scores, softmax, weighted sum."""
    scores = []
    for krow in rows_k:
        acc = 0.0
        for a, b in zip(q, krow):
            acc += a * b
        scores.append(scale * acc)
    top = max(scores)
    ws = [math.exp(s - top) for s in scores]
    tot = sum(ws)
    out = [0.0] * len(rows_v[0])
    for w, vrow in zip(ws, rows_v):
        for i, x in enumerate(vrow):
            out[i] += (w / tot) * x
    return out


def _tiny_paged(rng, S, Hq, Hkv, d, B, max_len, fmt="f16"):
    lens = rng.integers(1, max_len + 1, size=S)
    nbs = [-(-int(t) // B) for t in lens]
    NB = sum(nbs) + 3
    perm = rng.permutation(NB)
    tables = np.full((S, max(nbs)), -1, dtype=np.int32)
    c = 0
    for s in range(S):
        tables[s, :nbs[s]] = perm[c:c + nbs[s]]
        c += nbs[s]
    kc = rng.standard_normal((NB, Hkv, B, d)).astype(np.float16)
    vc = rng.standard_normal((NB, Hkv, B, d)).astype(np.float16)
    q = rng.standard_normal((S, Hq, d)).astype(np.float16)
    return q, kc, vc, tables, lens.astype(np.int32)


def check_brute_force(paged_fn, seed=0):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for B in [1, 2, 16]:
        for (Hq, Hkv) in [(2, 2), (4, 2), (3, 1)]:
            q, kc, vc, tables, lens = _tiny_paged(rng, 3, Hq, Hkv, 4, B, 40)
            out = paged_fn(q, kc, vc, tables, lens, 0.7, B)
            G = Hq // Hkv
            for s in range(3):
                T = int(lens[s])
                for h in range(Hq):
                    kvh = h // G
                    rows_k, rows_v = [], []
                    for p in range(T):
                        blk = int(tables[s][p // B])
                        rows_k.append([float(x) for x in kc[blk, kvh, p % B]])
                        rows_v.append([float(x) for x in vc[blk, kvh, p % B]])
                    ref = _brute_force_one([float(x) for x in q[s, h]], rows_k, rows_v, float(np.float32(0.7)))
                    worst = max(worst, float(np.max(np.abs(np.array(ref) - out[s, h]))))
    return worst


def test_brute_force_tiny():
    assert check_brute_force(oracle.paged_decode_attention) <= 1e-12


def test_mha_textbook_scipy():
    """H_q = H_kv and one block holding the whole sequence: textbook attention."""
    from scipy.special import softmax
    rng = np.random.default_rng(11)
    S, H, d, B = 3, 2, 8, 64
    q, kc, vc, tables, lens = _tiny_paged(rng, S, H, H, d, B, 60)
    out = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.35, B)
    for s in range(S):
        T = int(lens[s])
        blk = int(tables[s][0])
        for h in range(H):
            K = kc[blk, h, :T].astype(np.float64)
            V = vc[blk, h, :T].astype(np.float64)
            w = softmax(float(np.float32(0.35)) * (K @ q[s, h].astype(np.float64)))
            assert np.max(np.abs(w @ V - out[s, h])) <= 1e-13


def test_single_token_returns_v0():
    rng = np.random.default_rng(2)
    q, kc, vc, tables, _ = _tiny_paged(rng, 2, 2, 2, 8, 16, 16)
    lens = np.array([1, 1], dtype=np.int32)
    out = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.3, 16)
    for s in range(2):
        for h in range(2):
            assert np.array_equal(out[s, h], vc[tables[s][0], h, 0].astype(np.float64))


def test_constant_keys_give_mean_of_values():
    rng = np.random.default_rng(4)
    T, d = 37, 16
    q = rng.standard_normal(d)
    K = np.tile(rng.standard_normal(d), (T, 1))
    V = rng.standard_normal((T, d))
    assert np.max(np.abs(oracle.dense_decode_attention(q, K, V, 1.0) - V.mean(axis=0))) <= 1e-14


def test_dominant_logit_selects_row():
    rng = np.random.default_rng(6)
    T, d = 50, 16
    K = rng.standard_normal((T, d)) * 0.01
    q = rng.standard_normal(d)
    K[23] = q * 100.0
    V = rng.standard_normal((T, d))
    assert np.max(np.abs(oracle.dense_decode_attention(q, K, V, 1.0) - V[23])) <= 1e-12


def test_block_layout_permutation_invariance():
    """Relabel the physical blocks: the result is bit-identical (mapping idea of paging)."""
    rng = np.random.default_rng(8)
    q, kc, vc, tables, lens = _tiny_paged(rng, 4, 4, 2, 8, 4, 30)
    out = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.5, 4)
    NB = kc.shape[0]
    pi = rng.permutation(NB)                 # old id -> new id
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    t2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode_attention(q, kc2, vc2, t2, lens, 0.5, 4)
    assert np.array_equal(out, out2)


def check_gqa_reduces_to_mha(paged_fn, seed=9):
    """GQA with group G equals MHA on a cache whose KV head h is KV head h // G."""
    rng = np.random.default_rng(seed)
    Hq, Hkv, G = 6, 2, 3
    q, kc, vc, tables, lens = _tiny_paged(rng, 3, Hq, Hkv, 8, 8, 40)
    gqa = paged_fn(q, kc, vc, tables, lens, 0.5, 8)
    kc_m = np.repeat(kc, G, axis=1)
    vc_m = np.repeat(vc, G, axis=1)
    mha = paged_fn(q, kc_m, vc_m, tables, lens, 0.5, 8)
    return float(np.max(np.abs(gqa - mha)))


def test_gqa_reduces_to_mha():
    assert check_gqa_reduces_to_mha(oracle.paged_decode_attention) == 0.0


def test_paged_one_matches_full():
    rng = np.random.default_rng(12)
    q, kc, vc, tables, lens = _tiny_paged(rng, 3, 4, 2, 8, 16, 70)
    full = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.5, 16)
    for s in range(3):
        for h in range(4):
            one = oracle.paged_decode_attention_one(q, kc, vc, tables, lens, 0.5, 16, s, h)
            assert np.array_equal(one, full[s, h])


def test_empty_sequence_gives_zero():
    rng = np.random.default_rng(13)
    q, kc, vc, tables, lens = _tiny_paged(rng, 2, 2, 2, 8, 16, 20)
    lens = np.array([0, 5], dtype=np.int32)
    out = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.5, 16)
    assert np.all(out[0] == 0.0) and np.all(np.isfinite(out[1]))


def test_fp8_dequant_applies_per_head_scale():
    codes = np.full((2, 3, 4, 2), 0x38, dtype=np.uint8)     # every value 1.0
    scale = np.array([0.5, 2.0, 3.0], dtype=np.float32)
    deq = oracle.dequantize_kv(codes, "e4m3", scale)
    for h in range(3):
        assert np.all(deq[:, h] == float(scale[h]))


# ------------------------------------------------------------------ cache ops

def test_reshape_and_cache_figure_fixture(golden_dir):
    g = _load(golden_dir, "block_table_figure.json")
    B = g["block_size"]
    table = np.array(g["logical_to_physical"], dtype=np.int32)
    NB, H, d = 10, 1, 2
    kc = np.zeros((NB, H, B, d), dtype=np.float16)
    vc = np.zeros_like(kc)
    positions = [c["position"] for c in g["checks"]]
    slots = [int(table[p // B]) * B + p % B for p in positions]
    k = np.arange(len(positions) * H * d, dtype=np.float16).reshape(len(positions), H, d) + 1
    v = -k
    k2, v2 = oracle.reshape_and_cache(k, v, kc, vc, slots, B)
    for i, c in enumerate(g["checks"]):
        assert np.array_equal(k2[c["physical_block"], 0, c["offset"]], k[i, 0])
        assert np.array_equal(v2[c["physical_block"], 0, c["offset"]], v[i, 0])
    written = np.zeros((NB, B), dtype=bool)
    for c in g["checks"]:
        written[c["physical_block"], c["offset"]] = True
    ib, io = np.nonzero(~written)
    assert np.all(k2[ib, :, io] == 0)


def test_reshape_and_cache_skips_padding_and_roundtrips():
    rng = np.random.default_rng(14)
    B, NB, H, d = 4, 6, 2, 3
    kc = rng.standard_normal((NB, H, B, d)).astype(np.float16)
    vc = rng.standard_normal((NB, H, B, d)).astype(np.float16)
    k = rng.standard_normal((5, H, d)).astype(np.float16)
    v = rng.standard_normal((5, H, d)).astype(np.float16)
    slots = np.array([7, -1, 0, 23, -5], dtype=np.int64)
    k2, v2 = oracle.reshape_and_cache(k, v, kc, vc, slots, B)
    for n, sl in enumerate(slots):
        if sl >= 0:
            assert np.array_equal(k2[sl // B, :, sl % B], k[n])
            assert np.array_equal(v2[sl // B, :, sl % B], v[n])
    mask = np.ones((NB, B), dtype=bool)
    for sl in slots[slots >= 0]:
        mask[sl // B, sl % B] = False
    ib, io = np.nonzero(mask)
    assert np.array_equal(k2[ib, :, io], kc[ib, :, io])


def test_reshape_and_cache_fp8_quantises_product():
    rng = np.random.default_rng(15)
    B, NB, H, d = 4, 3, 2, 8
    src = rng.standard_normal((3, H, d)).astype(np.float16)
    inv = np.array([3.0, 0.25], dtype=np.float32)
    kc = np.zeros((NB, H, B, d), dtype=np.uint8)
    k2, _ = oracle.reshape_and_cache(src, src, kc, kc, [1, 5, 10], B, src_fmt="f16", kv_fmt="e4m3",
                                     k_inv_scale=inv, v_inv_scale=inv)
    for n, sl in enumerate([1, 5, 10]):
        for h in range(H):
            x = src[n, h].astype(np.float32) * inv[h]
            ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(k2[sl // B, h, sl % B], ref)


def test_copy_blocks_reads_before_writes():
    rng = np.random.default_rng(16)
    kc = rng.standard_normal((4, 2, 4, 3)).astype(np.float16)
    vc = rng.standard_normal((4, 2, 4, 3)).astype(np.float16)
    k2, v2 = oracle.copy_blocks(kc, vc, [(0, 1), (1, 2)])
    assert np.array_equal(k2[1], kc[0]) and np.array_equal(k2[2], kc[1])
    assert np.array_equal(v2[1], vc[0]) and np.array_equal(v2[2], vc[1])
    assert np.array_equal(k2[0], kc[0]) and np.array_equal(k2[3], kc[3])


def test_cow_isolation_and_refcounts():
    """Three sequences share a block; each writes into it once."""
    mgr = oracle.RefcountBlockManager(free_order=[7, 3, 9, 1, 4])
    shared = mgr.allocate()                    # 7
    mgr.share(shared)
    mgr.share(shared)
    tables = {0: [shared], 1: [shared], 2: [shared]}
    assert mgr.refcount[shared] == 3
    got = [oracle.copy_on_write(tables, s, 0, mgr) for s in (0, 1, 2)]
    assert got == [3, 9, 7]                     # last holder writes in place
    assert mgr.copies == [(7, 3), (7, 9)]
    assert mgr.refcount == {7: 1, 3: 1, 9: 1}
    # bytes: copies then private writes leave every other view intact
    B, H, d = 2, 1, 2
    kc = np.zeros((10, H, B, d), dtype=np.float16)
    kc[7, 0, 0] = [1, 2]
    kc, _ = oracle.copy_blocks(kc, kc, mgr.copies)
    for s, blk in enumerate(got):
        kc[blk, 0, 1] = [10 + s, 10 + s]        # each sequence's private write
    for s in (0, 1, 2):
        b = tables[s][0]
        assert list(kc[b, 0, 0]) == [1, 2]      # shared prompt bytes still seen
        assert list(kc[b, 0, 1]) == [10 + s, 10 + s]  # only its own write


# ------------------------------------------------------------------ planted mistakes

def _dense_no_scale(q, K, V, scale):
    return oracle.dense_decode_attention(q, K, V, 1.0)


def _online_no_acc_rescale(q, K, V, scale, B):
    q = np.asarray(q, dtype=np.float64)
    m, l, acc = -math.inf, 0.0, np.zeros(V.shape[-1])
    for a in range(0, K.shape[0], B):
        s = scale * (K[a:a + B] @ q)
        mn = max(m, float(s.max()))
        al = math.exp(m - mn) if m != -math.inf else 0.0
        p = np.exp(s - mn)
        l = al * l + p.sum()
        acc = acc + p @ V[a:a + B]              # planted: accumulator not rescaled
        m = mn
    return acc / l


def _paged_wrong_group(q, kc, vc, tables, lens, scale, B, **kw):
    # planted: query head h reads KV head h % H_kv instead of h // G
    S, Hq, d = q.shape
    Hkv = kc.shape[1]
    out = np.zeros((S, Hq, d))
    for s in range(S):
        for h in range(Hq):
            K = att.gather_sequence(kc.astype(np.float64), tables[s], int(lens[s]), B, h % Hkv)
            V = att.gather_sequence(vc.astype(np.float64), tables[s], int(lens[s]), B, h % Hkv)
            out[s, h] = oracle.dense_decode_attention(q[s, h].astype(np.float64), K, V, float(np.float32(scale)))
    return out


def _paged_transposed_block(q, kc, vc, tables, lens, scale, B, **kw):
    # planted: token offset and block taken in the wrong order inside a block
    S, Hq, d = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    kc2 = kc[:, :, ::-1, :]
    vc2 = vc[:, :, ::-1, :]
    return oracle.paged_decode_attention(q, np.ascontiguousarray(kc2), np.ascontiguousarray(vc2),
                                         tables, lens, scale, B)


def _e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float32)
    out = e4m3_encode_f32(x)
    codes = np.arange(0, 0x7E)
    lo = e4m3_decode(codes.astype(np.uint8))
    hi = e4m3_decode((codes + 1).astype(np.uint8))
    mids = (lo + hi) / 2
    for i, v in enumerate(np.abs(x.astype(np.float64))):
        j = np.nonzero(mids == v)[0]
        if len(j):
            out[i] = (codes[j[0]] + 1) | (0x80 if x[i] < 0 else 0)
    return out


def test_pins_catch_planted_mistakes():
    assert check_online_vs_dense(_online_no_acc_rescale, oracle.dense_decode_attention) > 1e-3
    assert check_online_vs_dense(oracle.online_softmax_attention, _dense_no_scale) > 1e-3
    assert check_brute_force(_paged_wrong_group) > 1e-3
    assert check_brute_force(_paged_transposed_block) > 1e-3
    assert check_gqa_reduces_to_mha(_paged_wrong_group) > 1e-3
    assert check_e4m3_ties(_e4m3_ties_away) > 0


# ----------------------------------------------------------------------------- sliding window

def check_window_brute_force(paged_fn, seed=21):
    """Hand loop over positions max(0, T-W) .. T-1 for every (sequence, head)."""
    rng = np.random.default_rng(seed)
    worst = 0.0
    for B in [1, 4, 16]:
        for W in [1, 3, 17, 64]:
            q, kc, vc, tables, lens = _tiny_paged(rng, 3, 4, 2, 4, B, 40)
            out = paged_fn(q, kc, vc, tables, lens, 0.6, B, window=W)
            for s in range(3):
                T = int(lens[s])
                for h in range(4):
                    kvh = h // 2
                    rows_k, rows_v = [], []
                    for p in range(max(0, T - W), T):
                        blk = int(tables[s][p // B])
                        rows_k.append([float(x) for x in kc[blk, kvh, p % B]])
                        rows_v.append([float(x) for x in vc[blk, kvh, p % B]])
                    ref = _brute_force_one([float(x) for x in q[s, h]], rows_k, rows_v, float(np.float32(0.6)))
                    worst = max(worst, float(np.max(np.abs(np.array(ref) - out[s, h]))))
    return worst


def test_window_brute_force():
    assert check_window_brute_force(oracle.paged_decode_attention) <= 1e-12


def test_window_covering_sequence_is_full_attention():
    rng = np.random.default_rng(22)
    q, kc, vc, tables, lens = _tiny_paged(rng, 4, 4, 4, 8, 16, 60)
    full = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.4, 16)
    for W in (60, 61, 1000):
        assert np.array_equal(oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.4, 16, window=W), full)


def test_window_one_returns_newest_row():
    rng = np.random.default_rng(23)
    q, kc, vc, tables, lens = _tiny_paged(rng, 3, 2, 2, 8, 4, 30)
    out = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.4, 4, window=1)
    for s in range(3):
        p = int(lens[s]) - 1
        blk = int(tables[s][p // 4])
        for h in range(2):
            assert np.array_equal(out[s, h], vc[blk, h, p % 4].astype(np.float64))


def test_window_ignores_rows_before_it():
    """Rows before the window may hold anything (NaN here) without changing the result."""
    rng = np.random.default_rng(24)
    q, kc, vc, tables, lens = _tiny_paged(rng, 3, 4, 2, 8, 4, 40)
    lens = np.maximum(lens, 12).astype(np.int32)
    nbs = -(-lens // 4)
    NB = kc.shape[0]
    need = int(nbs.sum()) + 3
    if need > NB:
        kc = np.concatenate([kc, rng.standard_normal((need - NB,) + kc.shape[1:]).astype(np.float16)])
        vc = np.concatenate([vc, rng.standard_normal((need - NB,) + vc.shape[1:]).astype(np.float16)])
    tables = np.full((3, int(nbs.max())), -1, dtype=np.int32)
    perm = rng.permutation(kc.shape[0])
    c = 0
    for s in range(3):
        tables[s, :nbs[s]] = perm[c:c + nbs[s]]
        c += nbs[s]
    W = 7
    ref = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.5, 4, window=W)
    kc2, vc2 = kc.copy(), vc.copy()
    for s in range(3):
        for p in range(int(lens[s]) - W):
            kc2[tables[s][p // 4], :, p % 4] = np.nan
            vc2[tables[s][p // 4], :, p % 4] = np.nan
    assert np.array_equal(oracle.paged_decode_attention(q, kc2, vc2, tables, lens, 0.5, 4, window=W), ref)


def test_window_one_query_helper_matches_full():
    rng = np.random.default_rng(25)
    q, kc, vc, tables, lens = _tiny_paged(rng, 3, 4, 2, 8, 4, 40)
    full = oracle.paged_decode_attention(q, kc, vc, tables, lens, 0.5, 4, window=9)
    for s in range(3):
        for h in range(4):
            one = oracle.paged_decode_attention_one(q, kc, vc, tables, lens, 0.5, 4, s, h, window=9)
            assert np.array_equal(one, full[s, h])


def _paged_window_off_by_one(q, kc, vc, tables, lens, scale, B, window=0, **kw):
    # planted: the window keeps one row too many
    return oracle.paged_decode_attention(q, kc, vc, tables, lens, scale, B, window=window + 1 if window else 0)


def test_window_pins_catch_planted_mistake():
    assert check_window_brute_force(_paged_window_off_by_one) > 1e-3


# ----------------------------------------------------------------------------- INT8 KV (scale + zero point)

def test_int8_known_values():
    enc = oracle.int8_encode_f32
    assert enc(np.array([2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5], np.float32), 0).tolist() == [2, 4, -2, -4, 0, 0, 2]
    assert enc(np.array([1000.0, -1000.0, np.inf, -np.inf, np.nan], np.float32), 0).tolist() == \
        [127, -128, 127, -128, 127]
    assert enc(np.array([120.0, -140.0, 117.0, -138.0], np.float32), 10).tolist() == [127, -128, 127, -128]
    assert enc(np.array([0.0, 1.0, -1.0], np.float32), -7).tolist() == [-7, -6, -8]


def test_int8_roundtrip_all_codes():
    codes = np.arange(-128, 128).astype(np.int8)
    for zp in (-128, -37, 0, 5, 127):
        vals = oracle.int8_decode(codes, zp)
        assert np.array_equal(vals, codes.astype(np.float64) - zp)
        assert np.array_equal(oracle.int8_encode_f32(vals.astype(np.float32), zp), codes)


def check_int8_vs_torch(encode, n=50000, seed=31):
    """torch.quantize_per_tensor with scale 1: clamp(nearbyint(x) + zp)."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(n) * 60).astype(np.float32)
    x[: n // 10] = np.round(x[: n // 10]) + 0.5          # exact ties
    bad = 0
    for zp in (-20, 0, 33):
        ref = torch.quantize_per_tensor(torch.from_numpy(x), 1.0, zp, torch.qint8).int_repr().numpy()
        bad += int(np.sum(encode(x, zp) != ref))
    return bad


def test_int8_encode_vs_torch():
    assert check_int8_vs_torch(oracle.int8_encode_f32) == 0


def test_int8_dequant_applies_per_head_scale_and_zero_point():
    codes = np.full((2, 3, 4, 2), 10, dtype=np.int8)
    scale = np.array([0.5, 2.0, 0.125], dtype=np.float32)
    zp = np.array([0, 12, -6], dtype=np.int32)
    deq = oracle.dequantize_kv(codes, "i8", scale, zp)
    for h, want in enumerate([5.0, -4.0, 2.0]):
        assert np.all(deq[:, h] == want)


def test_reshape_and_cache_int8_quantises_product():
    rng = np.random.default_rng(16)
    B, NB, H, d = 4, 3, 2, 8
    src = rng.standard_normal((3, H, d)).astype(np.float16)
    inv = np.array([31.0, 7.5], dtype=np.float32)
    zp = np.array([-3, 9], dtype=np.int32)
    kc = np.zeros((NB, H, B, d), dtype=np.int8)
    k2, _ = oracle.reshape_and_cache(src, src, kc, kc, [1, 5, 10], B, src_fmt="f16", kv_fmt="i8",
                                     k_inv_scale=inv, v_inv_scale=inv, k_zero_point=zp, v_zero_point=zp)
    for n, sl in enumerate([1, 5, 10]):
        for h in range(H):
            y = torch.from_numpy(src[n, h].astype(np.float32)) * float(inv[h])      # float32 product
            ref = torch.quantize_per_tensor(y, 1.0, int(zp[h]), torch.qint8).int_repr().numpy()
            assert np.array_equal(k2[sl // B, h, sl % B], ref)


def _int8_ties_away(y, zp):
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    r = np.sign(y) * np.floor(np.abs(y) + 0.5) + np.asarray(zp, dtype=np.float64)
    return np.clip(r, -128, 127).astype(np.int8)


def test_int8_pins_catch_planted_mistake():
    assert check_int8_vs_torch(_int8_ties_away) > 0


def test_int8_attention_equals_float_cache_of_same_values():
    """An i8 cache (scale s, zero point z) attends exactly like an f16 cache holding (code - z) * s."""
    rng = np.random.default_rng(32)
    q, kc16, vc16, tables, lens = _tiny_paged(rng, 3, 4, 2, 8, 4, 30)
    kcode = rng.integers(-128, 128, size=kc16.shape).astype(np.int8)
    vcode = rng.integers(-128, 128, size=vc16.shape).astype(np.int8)
    ks, vs = np.array([0.25, 0.5], np.float32), np.array([0.125, 1.0], np.float32)
    kz, vz = np.array([3, -5], np.int32), np.array([0, 7], np.int32)
    kf = ((kcode.astype(np.float64) - kz[None, :, None, None]) * ks[None, :, None, None]).astype(np.float16)
    vf = ((vcode.astype(np.float64) - vz[None, :, None, None]) * vs[None, :, None, None]).astype(np.float16)
    a = oracle.paged_decode_attention(q, kcode, vcode, tables, lens, 0.5, 4, kv_fmt="i8", k_scale=ks,
                                      v_scale=vs, k_zero_point=kz, v_zero_point=vz)
    b = oracle.paged_decode_attention(q, kf, vf, tables, lens, 0.5, 4)
    assert np.array_equal(a, b)


# ----------------------------------------------------------------------------- fused append + decode

def test_append_decode_single_token_returns_new_row():
    """T = 1: the only row attended is the appended one, so out = v_new exactly (whatever the cache held)."""
    rng = np.random.default_rng(33)
    q, kc, vc, tables, _ = _tiny_paged(rng, 3, 4, 2, 8, 4, 12)
    kc[:] = np.nan
    vc[:] = np.nan
    lens = np.ones(3, dtype=np.int32)
    kn = rng.standard_normal((3, 2, 8)).astype(np.float16)
    vn = rng.standard_normal((3, 2, 8)).astype(np.float16)
    out, k2, v2 = oracle.paged_append_decode(q, kn, vn, kc, vc, tables, lens, 0.5, 4)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(out[s, h], vn[s, h // 2].astype(np.float64))
        assert np.array_equal(k2[tables[s][0], :, 0], kn[s]) and np.array_equal(v2[tables[s][0], :, 0], vn[s])


def test_append_decode_writes_only_the_newest_slot():
    rng = np.random.default_rng(34)
    q, kc, vc, tables, lens = _tiny_paged(rng, 4, 4, 2, 8, 4, 30)
    kn = rng.standard_normal((4, 2, 8)).astype(np.float16)
    vn = rng.standard_normal((4, 2, 8)).astype(np.float16)
    _, k2, v2 = oracle.paged_append_decode(q, kn, vn, kc, vc, tables, lens, 0.5, 4)
    changed = np.argwhere(np.any(k2 != kc, axis=(1, 3)) | np.any(v2 != vc, axis=(1, 3)))
    want = {(int(tables[s][(int(lens[s]) - 1) // 4]), (int(lens[s]) - 1) % 4) for s in range(4)}
    assert {(int(b), int(r)) for b, r in changed} <= want


# ----------------------------------------------------------------------------- several queries per sequence

def _tiny_multi(rng, S, L, Hq, Hkv, d, B, max_len):
    q1, kc, vc, tables, lens = _tiny_paged(rng, S, Hq, Hkv, d, B, max_len)
    lens = np.maximum(lens, L).astype(np.int32)
    nbs = -(-lens // B)
    need = int(nbs.sum()) + 2
    kc = rng.standard_normal((need, Hkv, B, d)).astype(np.float16)
    vc = rng.standard_normal((need, Hkv, B, d)).astype(np.float16)
    perm = rng.permutation(need)
    tables = np.full((S, int(nbs.max())), -1, dtype=np.int32)
    c = 0
    for s in range(S):
        tables[s, :nbs[s]] = perm[c:c + nbs[s]]
        c += nbs[s]
    q = rng.standard_normal((S, L, Hq, d)).astype(np.float16)
    return q, kc, vc, tables, lens


def test_multi_query_one_query_is_decode():
    rng = np.random.default_rng(35)
    q, kc, vc, tables, lens = _tiny_multi(rng, 3, 1, 4, 2, 8, 4, 30)
    a = oracle.paged_multi_query_attention(q, kc, vc, tables, lens, 0.5, 4)
    b = oracle.paged_decode_attention(q[:, 0], kc, vc, tables, lens, 0.5, 4)
    assert np.array_equal(a[:, 0], b)


def check_multi_query_prefix(fn, seed=36, window=0):
    """Query i equals single-query decode of the same sequence cut to length T-L+i+1."""
    rng = np.random.default_rng(seed)
    worst = 0.0
    for L in (2, 3, 5):
        q, kc, vc, tables, lens = _tiny_multi(rng, 3, L, 4, 2, 8, 4, 30)
        out = fn(q, kc, vc, tables, lens, 0.5, 4, window=window)
        for i in range(L):
            cut = (lens - L + i + 1).astype(np.int32)
            ref = oracle.paged_decode_attention(q[:, i], kc, vc, tables, cut, 0.5, 4, window=window)
            worst = max(worst, float(np.max(np.abs(out[:, i] - ref))))
    return worst


def test_multi_query_equals_decode_of_each_prefix():
    assert check_multi_query_prefix(oracle.paged_multi_query_attention) == 0.0
    assert check_multi_query_prefix(oracle.paged_multi_query_attention, window=6) == 0.0


def test_multi_query_brute_force():
    rng = np.random.default_rng(37)
    q, kc, vc, tables, lens = _tiny_multi(rng, 2, 3, 2, 1, 4, 2, 12)
    out = oracle.paged_multi_query_attention(q, kc, vc, tables, lens, 0.7, 2)
    for s in range(2):
        T = int(lens[s])
        for i in range(3):
            for h in range(2):
                rk, rv = [], []
                for p in range(T - 3 + i + 1):
                    blk = int(tables[s][p // 2])
                    rk.append([float(x) for x in kc[blk, 0, p % 2]])
                    rv.append([float(x) for x in vc[blk, 0, p % 2]])
                ref = _brute_force_one([float(x) for x in q[s, i, h]], rk, rv, float(np.float32(0.7)))
                assert np.max(np.abs(np.array(ref) - out[s, i, h])) <= 1e-12


def _multi_not_causal(q, kc, vc, tables, lens, scale, B, window=0, **kw):
    # planted: every query sees the whole sequence
    S, L = q.shape[:2]
    return np.stack([oracle.paged_decode_attention(q[:, i], kc, vc, tables, lens, scale, B, window=window)
                     for i in range(L)], axis=1)


def test_multi_query_pins_catch_planted_mistake():
    assert check_multi_query_prefix(_multi_not_causal) > 1e-3

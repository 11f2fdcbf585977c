"""GPU-vs-oracle parity through the C ABI (small sizes: every output compared)."""

import numpy as np
import pytest

import oracle
import workloads
from paged_cases import PA_TOL, bits_equal, out_tolerance, run_gpu, run_oracle, to_torch

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_144_gb300 as pa  # noqa: E402


def _check(batch, vals, *, out_fmt="f32", partition_size=0, workspace="auto", tol=None):
    out, kc, vc, err = run_gpu(batch, vals, out_fmt=out_fmt, partition_size=partition_size, workspace=workspace)
    ref, okc, ovc = run_oracle(batch, vals)
    assert err == 0, f"device error bits {err}"
    assert bits_equal(kc, okc), "k_cache bytes differ from the oracle"
    assert bits_equal(vc, ovc), "v_cache bytes differ from the oracle"
    assert np.all(np.isfinite(out))
    bound = out_tolerance(ref, out_fmt) if tol is None else tol
    diff = np.abs(out - ref)
    assert np.all(diff <= bound), f"max abs err {diff.max():.3e}"
    return diff.max()


def test_tiny_workload():
    b = workloads.make_batch("tiny", seed=0)
    _check(b, workloads.host_values(b, seed=0))


@pytest.mark.parametrize("mode", [0, 512, 64, "single"])
def test_gqa_small_all_modes(mode):
    b = workloads.make_batch("gqa_32x4k", seed=1, num_seqs=8, lengths=("uniform", 1, 700))
    v = workloads.host_values(b, seed=1)
    if mode == "single":
        _check(b, v, partition_size=0, workspace=None)
    else:
        _check(b, v, partition_size=mode)


@pytest.mark.parametrize("q_mult", [1.0, 30.0])
def test_long_group8_extreme_logits(q_mult):
    b = workloads.make_batch("long_32k", seed=2, num_seqs=2, lengths=("const", 3000))
    _check(b, workloads.host_values(b, seed=2, q_mult=q_mult))


@pytest.mark.parametrize("wl,P", [("long_32k", 16), ("fp8_mix", 64), ("int8_mix", 64)])
def test_fixed_small_partitions_many_merges_per_warp(wl, P):
    """Fixed partitions of one unit or so: every warp processes and later merges many split segments
    (its list of won merges is sized from the partition count)."""
    kw = dict(num_seqs=4, lengths=("const", 3000)) if wl == "long_32k" else \
        dict(num_seqs=24, lengths=("lognormal", 6.5, 1.0, 16, 3000))
    b = workloads.make_batch(wl, seed=71, **kw)
    _check(b, workloads.host_values(b, seed=71), partition_size=P)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (6, 2), (16, 4), (10, 2), (16, 2)])
def test_shapes_grid(fmt, D, B, Hq, Hkv):
    b = workloads.make_batch("gqa_32x4k", seed=3, num_seqs=5, num_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                             block_size=B, q_fmt=fmt, kv_fmt=fmt, lengths=("uniform", 1, 300),
                             scale=1.0 / np.sqrt(D))
    _check(b, workloads.host_values(b, seed=3))


@pytest.mark.parametrize("out_fmt", ["f16", "bf16"])
def test_reduced_precision_outputs(out_fmt):
    b = workloads.make_batch("gqa_32x4k", seed=4, num_seqs=4, lengths=("uniform", 1, 500))
    _check(b, workloads.host_values(b, seed=4), out_fmt=out_fmt)


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("qfmt", ["bf16", "f16"])
def test_fp8_cache(B, qfmt):
    b = workloads.make_batch("fp8_mix", seed=5, num_seqs=8, block_size=B, q_fmt=qfmt,
                             lengths=("lognormal", 6.0, 1.0, 16, 1500))
    _check(b, workloads.host_values(b, seed=5))


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("qfmt", ["bf16", "f16"])
def test_int8_cache(B, qfmt):
    """INT8 cache (per-head scale + zero point): cache bytes bit-exact, attention within 2e-3."""
    b = workloads.make_batch("int8_mix", seed=6, num_seqs=8, block_size=B, q_fmt=qfmt,
                             lengths=("lognormal", 6.0, 1.0, 16, 1500))
    _check(b, workloads.host_values(b, seed=6))


def test_int8_split_modes_and_extreme_zero_points():
    b = workloads.make_batch("int8_mix", seed=7, num_seqs=6, lengths=("lognormal", 6.0, 1.0, 16, 2000))
    v = workloads.host_values(b, seed=7)
    v["k_zero_point"] = np.array([-128, 127, 0, 5, -5, 100, -100, 1][: b.num_kv_heads], dtype=np.int32)
    v["v_zero_point"] = np.array([127, -128, 3, -3, 64, -64, 0, 2][: b.num_kv_heads], dtype=np.int32)
    for mode in (0, 256):
        _check(b, v, partition_size=mode)


def test_many_short_sequences_cross_warp_ranges():
    b = workloads.make_batch("gqa_32x4k", seed=6, num_seqs=300, lengths=("uniform", 1, 60))
    _check(b, workloads.host_values(b, seed=6))


def test_lengths_on_block_boundaries_and_single_tokens():
    lens = np.array([1, 16, 17, 32, 15, 48, 2, 512, 513], dtype=np.int64)
    rng = np.random.default_rng(7)
    tables, nb, free = workloads.build_block_tables(lens, 16, rng, pool=("slack", 0.2), max_blocks_per_seq=40)
    b = workloads.make_batch("gqa_32x4k", seed=7, num_seqs=len(lens), lengths=("uniform", 1, 2))
    b.seq_lens = lens.astype(np.int32)
    b.block_tables, b.num_blocks, b.free_blocks = tables, nb, free
    b.new_slots = np.array([workloads.slot_of(tables[s], int(lens[s]) - 1, 16) for s in range(len(lens))],
                           dtype=np.int64)
    _check(b, workloads.host_values(b, seed=7))


def test_empty_sequences_give_zero():
    b = workloads.make_batch("gqa_32x4k", seed=8, num_seqs=6, lengths=("uniform", 1, 200))
    v = workloads.host_values(b, seed=8)
    out, kc, vc, err = run_gpu(b, v)
    # now zero two sequences' lengths: the decode must write zeros for them
    b2 = workloads.make_batch("gqa_32x4k", seed=8, num_seqs=6, lengths=("uniform", 1, 200))
    b2.seq_lens = b.seq_lens.copy()
    b2.seq_lens[[1, 4]] = 0
    b2.new_slots = b.new_slots.copy()
    b2.new_slots[[1, 4]] = -1   # padding tokens: not written
    out2, _, _, err2 = run_gpu(b2, v)
    ref, _, _ = run_oracle(b2, v)
    assert err2 == 0
    assert np.all(out2[[1, 4]] == 0.0)
    assert np.max(np.abs(out2 - ref)) <= PA_TOL


def test_deterministic_and_block_relabelling_invariant():
    b = workloads.make_batch("gqa_32x4k", seed=9, num_seqs=6, lengths=("uniform", 100, 900))
    v = workloads.host_values(b, seed=9)
    o1, *_ = run_gpu(b, v)
    o2, *_ = run_gpu(b, v)
    assert np.array_equal(o1, o2)
    # relabel physical blocks with a permutation
    rng = np.random.default_rng(10)
    pi = rng.permutation(b.num_blocks)
    b3 = workloads.make_batch("gqa_32x4k", seed=9, num_seqs=6, lengths=("uniform", 100, 900))
    b3.block_tables = np.where(b.block_tables >= 0, pi[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    b3.new_slots = np.array([pi[s // 16] * 16 + s % 16 for s in b.new_slots], dtype=np.int64)
    v3 = dict(v)
    for k in ("k_cache", "v_cache"):
        arr = np.empty_like(v[k])
        arr[pi] = v[k]
        v3[k] = arr
    o3, *_ = run_gpu(b3, v3)
    assert np.array_equal(o1, o3)


def test_beam_cow_workload():
    """Shared prompt, CoW of the partial block, private tails, 1 appended token, decode."""
    sc = workloads.beam_cow_scenario(0)
    dev = "cuda"
    B, P, H, D = sc["block_size"], sc["prompt_len"], sc["num_kv_heads"], sc["head_dim"]
    nbeams, NB = sc["num_beams"], sc["num_blocks"]
    bm = pa.BlockManager(NB, B, free_order=sc["free_order"])
    om = oracle.RefcountBlockManager(sc["free_order"])
    kc = torch.zeros((NB, H, B, D), dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    okc = np.zeros((NB, H, B, D), dtype=np.float16)
    ovc = np.zeros_like(okc)
    # (1) prompt
    slots = bm.add_sequence(0, P)
    ot = {0: [om.allocate() for _ in range(-(-P // B))]}
    oslots = [workloads.slot_of(ot[0], p, B) for p in range(P)]
    assert slots == oslots
    pa.reshape_and_cache(to_torch(sc["prompt_k"], "f16", dev), to_torch(sc["prompt_v"], "f16", dev), kc, vc,
                         torch.tensor(slots, dtype=torch.int64, device=dev), B)
    okc, ovc = oracle.reshape_and_cache(sc["prompt_k"], sc["prompt_v"], okc, ovc, oslots, B)
    for bb in range(1, nbeams):
        bm.fork(0, bb)
        ot[bb] = list(ot[0])
        for blk in ot[bb]:
            om.share(blk)
    # (2) CoW of the shared partial block, one batched copy
    last = P // B
    pairs = [p for p in (bm.copy_on_write(bb, last) for bb in range(nbeams)) if p]
    for bb in range(nbeams):
        oracle.copy_on_write(ot, bb, last, om)
    assert pairs == om.copies and len(pairs) == nbeams - 1
    pa.copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int32, device=dev))
    okc, ovc = oracle.copy_blocks(okc, ovc, pairs)
    assert bits_equal(kc.cpu().numpy(), okc) and bits_equal(vc.cpu().numpy(), ovc)
    # (3) private tails, (4) one appended token per beam
    for rows_k, rows_v, positions in (
        ([sc["tail_k"][bb] for bb in range(nbeams)], [sc["tail_v"][bb] for bb in range(nbeams)],
         [range(P, P + int(sc["tails"][bb])) for bb in range(nbeams)]),
        ([sc["new_k"][bb:bb + 1] for bb in range(nbeams)], [sc["new_v"][bb:bb + 1] for bb in range(nbeams)],
         [range(P + int(sc["tails"][bb]), P + int(sc["tails"][bb]) + 1) for bb in range(nbeams)]),
    ):
        gslots, oslots = [], []
        for bb in range(nbeams):
            for pos in positions[bb]:
                s, pair = bm.append_slot(bb)
                assert pair is None
                while len(ot[bb]) <= pos // B:
                    ot[bb].append(om.allocate())
                gslots.append(s)
                oslots.append(workloads.slot_of(ot[bb], pos, B))
        assert gslots == oslots
        k_rows = np.concatenate(rows_k)
        v_rows = np.concatenate(rows_v)
        pa.reshape_and_cache(to_torch(k_rows, "f16", dev), to_torch(v_rows, "f16", dev), kc, vc,
                             torch.tensor(gslots, dtype=torch.int64, device=dev), B)
        okc, ovc = oracle.reshape_and_cache(k_rows, v_rows, okc, ovc, oslots, B)
    assert bits_equal(kc.cpu().numpy(), okc) and bits_equal(vc.cpu().numpy(), ovc)
    # (5) decode
    lens = np.array([P + int(t) + 1 for t in sc["tails"]], dtype=np.int32)
    width = max(len(ot[bb]) for bb in range(nbeams))
    tables = np.array([bm.block_table(bb, width) for bb in range(nbeams)], dtype=np.int32)
    assert all(tables[bb, :len(ot[bb])].tolist() == ot[bb] for bb in range(nbeams))
    out = torch.empty((nbeams, sc["num_heads"], D), dtype=torch.float32, device=dev)
    n = pa.decode_workspace_bytes(nbeams, sc["num_heads"], H, D, B, width, 0, pa.PA_F16)
    ws = pa.new_workspace(n, dev)
    pa.decode(out, to_torch(sc["q"], "f16", dev), kc, vc, torch.from_numpy(tables).to(dev),
              torch.from_numpy(lens).to(dev), H, sc["scale"], B, workspace=ws)
    assert pa.get_device_error() == 0
    ref = oracle.paged_decode_attention(sc["q"], okc, ovc, tables, lens, sc["scale"], B)
    assert np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)) <= PA_TOL
    # isolation: every beam's own copy of the partial block still holds the prompt's rows
    keep = P % B
    want = sc["prompt_k"][P - keep:P].transpose(1, 0, 2)
    gk = kc.cpu().numpy()
    for bb in range(nbeams):
        assert np.array_equal(gk[tables[bb, last], :, :keep], want)


def test_bad_block_id_sets_error_bit_without_fault():
    b = workloads.make_batch("gqa_32x4k", seed=11, num_seqs=3, lengths=("uniform", 20, 80))
    v = workloads.host_values(b, seed=11)
    b.block_tables = b.block_tables.copy()
    b.block_tables[1, 0] = b.num_blocks + 5
    out, _, _, err = run_gpu(b, v)
    assert err & pa.PA_DEVERR_BLOCK_ID
    assert pa.get_device_error() == 0          # read-and-clear


def test_bad_slot_and_pair_set_error_bits():
    dev = "cuda"
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    k = torch.ones((2, 2, 64), dtype=torch.float16, device=dev)
    pa.reshape_and_cache(k, k, kc, vc, torch.tensor([3, 4 * 16 + 1], dtype=torch.int64, device=dev), 16)
    assert pa.get_device_error() & pa.PA_DEVERR_SLOT
    assert kc[0, :, 3].eq(1).all()
    pa.copy_blocks(kc, vc, torch.tensor([[0, 9]], dtype=torch.int32, device=dev))
    assert pa.get_device_error() & pa.PA_DEVERR_PAIR


def test_seq_len_beyond_table_capacity_flags_error():
    b = workloads.make_batch("gqa_32x4k", seed=12, num_seqs=2, lengths=("uniform", 10, 20))
    v = workloads.host_values(b, seed=12)
    b.seq_lens = b.seq_lens.copy()
    b.seq_lens[0] = b.max_blocks_per_seq * 16 + 100
    _, _, _, err = run_gpu(b, v)
    assert err & pa.PA_DEVERR_SEQ_LEN


@pytest.mark.parametrize("wl", ["fp8_mix", "int8_mix"])
@pytest.mark.parametrize("e", [17, -20])
def test_8bit_cache_bf16_query_outside_f16_range(wl, e):
    """bf16 queries beyond f16's range on 8-bit caches, whose products run in f16: q = N(0,1)·2^e with the
    softmax scale 2^-e/√d, so the scores are those of an ordinary batch while every |q| is above 65504
    somewhere (e = 17) or below f16's smallest normal 2^-14 everywhere (e = -20)."""
    b = workloads.make_batch(wl, seed=13, num_seqs=6, lengths=("lognormal", 6.0, 1.0, 16, 1200))
    b.scale = float(np.float32(2.0 ** -e / np.sqrt(128.0)))
    v = workloads.host_values(b, seed=13)
    q = oracle.bf16_bits_to_f64(v["q"]) * 2.0 ** e          # exact: a power of two times a bf16 value
    v["q"] = workloads.bf16_bits_from_f32(q.astype(np.float32))
    assert np.array_equal(oracle.bf16_bits_to_f64(v["q"]), q)
    aq = np.abs(q)
    if e > 0:
        assert aq.max() > 65504.0
    else:
        assert aq.max() < 2.0 ** -14
    _check(b, v)

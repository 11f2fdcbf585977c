"""Host-side tests (no GPU): library exports, argument validation, block manager."""

import ctypes

import numpy as np
import pytest

import oracle
import workloads
import paged_kv_cache_144_gb300 as pa
from paged_kv_cache_144_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    return pa.load()


def test_library_exports_every_header_function(lib):
    names = pa.header_functions()
    assert {"pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_decode_workspace_bytes",
            "pa_status_string", "pa_get_device_error", "pa_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(-7, 1):
        assert pa.status_string(code).startswith("PA_")
    assert pa.pa_version() >= 100


A = ctypes.c_void_p(0x10000)  # aligned fake device pointers: validation fails before any use
A2 = ctypes.c_void_p(0x20000)
MIS = ctypes.c_void_p(0x10008)


def _decode(**kw):
    args = dict(out=A, out_dtype=pa.PA_F32, q=A, q_dtype=pa.PA_BF16, q_stride=32 * 128, k=A, v=A2,
                kv_dtype=pa.PA_BF16, nb=100, ks=None, vs=None, bt=A, mb=16, sl=A, S=4, Hq=32, Hkv=8, D=128,
                scale=0.1, B=16, P=0, ws=None, wsb=0, stream=None)
    args.update(kw)
    a = args
    return pa.pa_decode(a["out"], a["out_dtype"], a["q"], a["q_dtype"], a["q_stride"], a["k"], a["v"],
                        a["kv_dtype"], a["nb"], a["ks"], a["vs"], a["bt"], a["mb"], a["sl"], a["S"], a["Hq"],
                        a["Hkv"], a["D"], a["scale"], a["B"], a["P"], a["ws"], a["wsb"], a["stream"])


def test_decode_validation(lib):
    assert _decode(S=0) == pa.PA_OK                      # nothing to do, nothing touched
    assert _decode(Hq=30) == pa.PA_ERR_SHAPE             # H_q not a multiple of H_kv
    assert _decode(Hq=128) == pa.PA_ERR_UNSUPPORTED      # G = 16
    assert _decode(D=96, q_stride=32 * 96) == pa.PA_ERR_UNSUPPORTED
    assert _decode(B=12) == pa.PA_ERR_UNSUPPORTED         # block size: a power of two from 8 to 1024
    assert _decode(B=96) == pa.PA_ERR_UNSUPPORTED
    assert _decode(B=4) == pa.PA_ERR_UNSUPPORTED
    assert _decode(B=2048) == pa.PA_ERR_UNSUPPORTED
    assert _decode(P=100) == pa.PA_ERR_SHAPE             # not a multiple of B
    assert _decode(mb=0) == pa.PA_ERR_SHAPE
    assert _decode(out=None) == pa.PA_ERR_NULL
    assert _decode(bt=None) == pa.PA_ERR_NULL
    assert _decode(out_dtype=pa.PA_FP8_E4M3) == pa.PA_ERR_DTYPE
    assert _decode(q_dtype=pa.PA_F16) == pa.PA_ERR_DTYPE  # 16-bit cache must match q
    assert _decode(kv_dtype=pa.PA_FP8_E4M3) == pa.PA_ERR_NULL   # scales required
    assert _decode(kv_dtype=pa.PA_FP8_E4M3, D=64, q_stride=32 * 64, ks=A, vs=A) == pa.PA_ERR_UNSUPPORTED
    assert _decode(q_stride=100) == pa.PA_ERR_SHAPE
    assert _decode(q=MIS) == pa.PA_ERR_ALIGN
    assert _decode(k=MIS) == pa.PA_ERR_ALIGN
    assert _decode(q_stride=32 * 128 + 1) == pa.PA_ERR_ALIGN
    assert _decode(nb=0) == pa.PA_ERR_SHAPE
    assert _decode(nb=2 ** 40) == pa.PA_ERR_SHAPE         # row coordinates must fit in int32
    assert _decode(S=20000) == pa.PA_ERR_UNSUPPORTED


def _decode_ex(opt, **kw):
    args = dict(out=A, out_dtype=pa.PA_F32, q=A, q_dtype=pa.PA_BF16, q_stride=32 * 128, k=A, v=A2,
                kv_dtype=pa.PA_BF16, nb=100, ks=None, vs=None, bt=A, mb=16, sl=A, S=4, Hq=32, Hkv=8, D=128,
                scale=0.1, B=16, P=0, ws=None, wsb=0, stream=None)
    args.update(kw)
    a = args
    return pa.pa_decode_ex(a["out"], a["out_dtype"], a["q"], a["q_dtype"], a["q_stride"], a["k"], a["v"],
                           a["kv_dtype"], a["nb"], a["ks"], a["vs"], a["bt"], a["mb"], a["sl"], a["S"], a["Hq"],
                           a["Hkv"], a["D"], a["scale"], a["B"], a["P"], a["ws"], a["wsb"],
                           None if opt is None else ctypes.byref(opt), a["stream"])


def test_decode_ex_options_validation(lib):
    assert _decode_ex(None, S=0) == pa.PA_OK
    assert _decode_ex(pa.DecodeOptions(window=5), S=0) == pa.PA_OK
    assert _decode_ex(pa.DecodeOptions(window=-1)) == pa.PA_ERR_SHAPE
    bad = pa.DecodeOptions(window=5)
    bad.struct_size = 0
    assert _decode_ex(bad) == pa.PA_ERR_SHAPE
    # option checks come before the shape checks that pa_decode shares
    assert _decode_ex(pa.DecodeOptions(window=3), Hq=30) == pa.PA_ERR_SHAPE
    assert _decode_ex(pa.DecodeOptions(window=3), B=12) == pa.PA_ERR_UNSUPPORTED
    assert ctypes.sizeof(pa.DecodeOptions) >= 12
    # INT8 caches need scales and zero points
    assert _decode_ex(None, kv_dtype=pa.PA_INT8, ks=A, vs=A) == pa.PA_ERR_NULL
    assert _decode_ex(pa.DecodeOptions(k_zero_point=0x10000, v_zero_point=0x20000), kv_dtype=pa.PA_INT8) == \
        pa.PA_ERR_NULL
    assert _decode_ex(pa.DecodeOptions(k_zero_point=0x10000, v_zero_point=0x20000), kv_dtype=pa.PA_INT8, ks=A,
                      vs=A, D=64, q_stride=32 * 64) == pa.PA_ERR_UNSUPPORTED


def test_decode_ex_multi_query_validation(lib):
    # 32 q heads / 8 KV heads: G = 4, so q_len 16 fills 64 (query, head) rows and q_len 17 is too many
    assert _decode_ex(pa.DecodeOptions(q_len=17), q_stride=17 * 32 * 128) == pa.PA_ERR_UNSUPPORTED
    assert _decode_ex(pa.DecodeOptions(q_len=4), q_stride=3 * 32 * 128) == pa.PA_ERR_SHAPE
    assert _decode_ex(pa.DecodeOptions(q_len=-1)) == pa.PA_ERR_SHAPE
    assert _decode_ex(pa.DecodeOptions(q_len=2, k_new=0x10000, v_new=0x20000, new_dtype=pa.PA_BF16,
                                       new_stride=8 * 128), q_stride=2 * 32 * 128) == pa.PA_ERR_UNSUPPORTED
    assert _decode_ex(pa.DecodeOptions(q_len=4), q_stride=4 * 32 * 128, S=0) == pa.PA_OK


def test_cache_write_int8_validation(lib):
    def rc(opt, **kw):
        a = dict(k=A, v=A2, src=pa.PA_BF16, ks=8 * 128, vs=8 * 128, kc=A, vc=A2, kv=pa.PA_INT8, nb=10, sm=A, N=3,
                 Hkv=8, D=128, B=16, ki=A, vi=A)
        a.update(kw)
        return pa.pa_reshape_and_cache_ex(a["k"], a["v"], a["src"], a["ks"], a["vs"], a["kc"], a["vc"], a["kv"],
                                          a["nb"], a["sm"], a["N"], a["Hkv"], a["D"], a["B"], a["ki"], a["vi"],
                                          None if opt is None else ctypes.byref(opt), None)
    assert rc(None) == pa.PA_ERR_NULL                      # zero points required
    assert rc(pa.CacheWriteOptions(k_zero_point=0x10000, v_zero_point=0x20000), ki=None) == pa.PA_ERR_NULL
    bad = pa.CacheWriteOptions(k_zero_point=0x10000, v_zero_point=0x20000)
    bad.struct_size = 0
    assert rc(bad) == pa.PA_ERR_SHAPE
    assert rc(pa.CacheWriteOptions(k_zero_point=0x10000, v_zero_point=0x20000), N=0) == pa.PA_OK


def _rc(**kw):
    a = dict(k=A, v=A2, src=pa.PA_F16, ks=8 * 128, vs=8 * 128, kc=A, vc=A2, kv=pa.PA_F16, nb=10, sm=A, N=3,
             Hkv=8, D=128, B=16, ki=None, vi=None, stream=None)
    a.update(kw)
    return pa.pa_reshape_and_cache(a["k"], a["v"], a["src"], a["ks"], a["vs"], a["kc"], a["vc"], a["kv"], a["nb"],
                                   a["sm"], a["N"], a["Hkv"], a["D"], a["B"], a["ki"], a["vi"], a["stream"])


def test_reshape_and_cache_validation(lib):
    assert _rc(N=0) == pa.PA_OK
    assert _rc(N=-1) == pa.PA_ERR_SHAPE
    assert _rc(D=80) == pa.PA_ERR_UNSUPPORTED
    assert _rc(sm=None) == pa.PA_ERR_NULL
    assert _rc(src=pa.PA_F32) == pa.PA_ERR_DTYPE
    assert _rc(kv=pa.PA_BF16) == pa.PA_ERR_DTYPE
    assert _rc(kv=pa.PA_FP8_E4M3) == pa.PA_ERR_NULL
    assert _rc(ks=100) == pa.PA_ERR_SHAPE
    assert _rc(k=MIS) == pa.PA_ERR_ALIGN
    assert _rc(ks=8 * 128 + 4) == pa.PA_ERR_ALIGN


def test_copy_blocks_validation(lib):
    assert pa.pa_copy_blocks(A, A2, 10, 4096, A, 0, None) == pa.PA_OK
    assert pa.pa_copy_blocks(A, A2, 10, 4097, A, 1, None) == pa.PA_ERR_ALIGN
    assert pa.pa_copy_blocks(A, A2, 10, 4096, None, 1, None) == pa.PA_ERR_NULL
    assert pa.pa_copy_blocks(A, A2, 10, 4096, A, 70000, None) == pa.PA_ERR_UNSUPPORTED
    assert pa.pa_copy_blocks(A, A2, 0, 4096, A, 1, None) == pa.PA_ERR_SHAPE
    assert pa.pa_copy_blocks(MIS, A2, 10, 4096, A, 1, None) == pa.PA_ERR_ALIGN


def test_workspace_query_without_device_is_rejected_or_sized(lib):
    n = pa.pa_decode_workspace_bytes(4, 32, 8, 128, 16, 16, 0, pa.PA_BF16)
    assert n == _lib.SIZE_MAX or n > 0
    assert pa.pa_decode_workspace_bytes(4, 30, 8, 128, 16, 16, 0, pa.PA_BF16) == _lib.SIZE_MAX


# ----------------------------------------------------------------------------- block manager

def test_block_manager_cow_matches_oracle():
    free = [5, 2, 9, 1, 7, 3, 8, 0, 4, 6]
    bm = pa.BlockManager(10, 4, free_order=free)
    om = oracle.RefcountBlockManager(free)
    # one sequence with 6 tokens (2 blocks), then 2 forks
    bm.add_sequence("a", 6)
    ot = {"a": [om.allocate(), om.allocate()]}
    bm.fork("a", "b")
    bm.fork("a", "c")
    for s in ("b", "c"):
        ot[s] = list(ot["a"])
        for blk in ot[s]:
            om.share(blk)
    assert bm.tables == {k: v for k, v in ot.items()}
    # each sequence writes into its last (shared, partial) block
    pairs = [bm.copy_on_write(s, 1) for s in ("a", "b", "c")]
    want = [oracle.copy_on_write(ot, s, 1, om) for s in ("a", "b", "c")]
    assert [p[1] if p else ot[s][1] for p, s in zip(pairs, "abc")] == want
    assert [p for p in pairs if p] == om.copies
    assert bm.tables == ot
    assert bm.refcount == om.refcount


def test_block_manager_append_slots():
    bm = pa.BlockManager(8, 4, free_order=[3, 1, 6, 0, 2, 4, 5, 7])
    slots = bm.add_sequence(0, 6)
    assert bm.block_table(0) == [3, 1]
    assert slots == [12, 13, 14, 15, 4, 5]
    bm.fork(0, 1)
    s, pair = bm.append_slot(1)          # writes into shared block 1 -> CoW
    assert pair == (1, 6) and s == 6 * 4 + 2
    s, pair = bm.append_slot(0)          # block 1 now held by 0 only
    assert pair is None and s == 1 * 4 + 2
    bm.free(1)
    assert 6 in bm._free


def test_beam_scenario_host_logic_matches_oracle():
    sc = workloads.beam_cow_scenario(0)
    B, P = sc["block_size"], sc["prompt_len"]
    bm = pa.BlockManager(sc["num_blocks"], B, free_order=sc["free_order"])
    om = oracle.RefcountBlockManager(sc["free_order"])
    bm.add_sequence(0, P)
    ot = {0: [om.allocate() for _ in range(-(-P // B))]}
    for b in range(1, sc["num_beams"]):
        bm.fork(0, b)
        ot[b] = list(ot[0])
        for blk in ot[b]:
            om.share(blk)
    last = P // B
    got = [bm.copy_on_write(b, last) for b in range(sc["num_beams"])]
    want = [oracle.copy_on_write(ot, b, last, om) for b in range(sc["num_beams"])]
    assert len([g for g in got if g]) == sc["num_beams"] - 1
    assert [g for g in got if g] == om.copies
    assert [bm.tables[b][last] for b in range(sc["num_beams"])] == want


# ----------------------------------------------------------------------------- generators

def test_generators_are_seeded_and_consistent():
    a = workloads.make_batch("gqa_32x4k", seed=3)
    b = workloads.make_batch("gqa_32x4k", seed=3)
    assert np.array_equal(a.seq_lens, b.seq_lens) and np.array_equal(a.block_tables, b.block_tables)
    used = np.concatenate([a.block_tables[s, : -(-int(a.seq_lens[s]) // 16)] for s in range(a.num_seqs)])
    assert len(np.unique(used)) == len(used) and used.min() >= 0 and used.max() < a.num_blocks
    assert a.seq_lens.min() >= 1 and a.seq_lens.max() <= 4096
    t = workloads.make_batch("tiny", seed=0)
    assert t.num_blocks == 64 and t.seq_lens.max() <= 129
    f = workloads.make_batch("fp8_mix", seed=0)
    assert f.seq_lens.min() >= 16 and f.seq_lens.max() <= 8192
    l3 = workloads.make_batch("long_32k", seed=0)
    assert np.all(l3.seq_lens == 32768)


def test_shard_sequences_covers_all():
    for n, w in [(32, 2), (7, 3), (1, 4)]:
        spans = [workloads.shard_sequences(n, r, w) for r in range(w)]
        assert spans[0][0] == 0 and spans[-1][1] == n
        assert all(spans[i][1] == spans[i + 1][0] for i in range(w - 1))


def _c_layout(struct_name, fields):
    """sizeof and offsetof of a pa.h struct, from a C program compiled with the system compiler."""
    import os
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    body = "".join(f'  printf("%zu\\n", offsetof({struct_name}, {f}));\n' for f in fields)
    src = ("#include <stddef.h>\n#include <stdio.h>\n#include \"pa.h\"\n"
           f"int main(void) {{\n  printf(\"%zu\\n\", sizeof({struct_name}));\n{body}  return 0;\n}}\n")
    with tempfile.TemporaryDirectory() as d:
        c, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(c, "w") as fh:
            fh.write(src)
        subprocess.run([cc, "-std=c99", "-I", inc, c, "-o", exe], check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    return int(out[0]), [int(x) for x in out[1:]]


@pytest.mark.parametrize("cls,cname", [(pa.DecodeOptions, "pa_decode_options"),
                                       (_lib.CacheWriteOptions, "pa_cache_write_options")])
def test_option_structs_match_the_header_layout(cls, cname):
    names = [n for n, _ in cls._fields_]
    size, offsets = _c_layout(cname, names)
    assert ctypes.sizeof(cls) == size
    assert [getattr(cls, n).offset for n in names] == offsets


def test_decode_ex_pdl_option_validation(lib):
    # the launch mode changes no argument rule: empty batches succeed, bad shapes still fail
    assert _decode_ex(pa.DecodeOptions(pdl=1), S=0) == pa.PA_OK
    assert _decode_ex(pa.DecodeOptions(pdl=1, window=-1)) == pa.PA_ERR_SHAPE
    assert _decode_ex(pa.DecodeOptions(pdl=1), B=12) == pa.PA_ERR_UNSUPPORTED
    # a caller compiled before the field existed (shorter struct_size) reads it as 0
    old = pa.DecodeOptions(pdl=1)
    old.struct_size = pa.DecodeOptions.pdl.offset
    assert _decode_ex(old, S=0) == pa.PA_OK


def test_cache_write_pdl_option_validation(lib):
    # the launch mode changes no argument rule
    opt = _lib.CacheWriteOptions(pdl=1)
    st = pa.pa_reshape_and_cache_ex(0x10000, 0x20000, pa.PA_BF16, 8 * 128, 8 * 128, 0x30000, 0x40000, pa.PA_BF16,
                                    16, 0x50000, 0, 8, 128, 16, None, None, ctypes.byref(opt), None)
    assert st == pa.PA_OK                    # no tokens: nothing to launch
    st = pa.pa_reshape_and_cache_ex(0x10000, 0x20000, pa.PA_BF16, 8 * 128, 8 * 128, 0x30000, 0x40000, pa.PA_BF16,
                                    16, 0x50000, 4, 8, 96, 16, None, None, ctypes.byref(opt), None)
    assert st == pa.PA_ERR_UNSUPPORTED       # head_dim 96


def test_decode_ex_fused_append_validation(lib):
    def app(**kw):
        o = dict(k_new=0x10000, v_new=0x20000, new_dtype=pa.PA_BF16, new_stride=8 * 128)
        o.update(kw)
        return pa.DecodeOptions(**o)
    assert _decode_ex(app(v_new=None)) == pa.PA_ERR_NULL                 # both rows or neither
    assert _decode_ex(app(new_dtype=pa.PA_F32)) == pa.PA_ERR_DTYPE       # 16-bit source rows only
    assert _decode_ex(app(new_dtype=pa.PA_F16)) == pa.PA_ERR_DTYPE       # a 16-bit cache takes its own type
    assert _decode_ex(app(), kv_dtype=pa.PA_FP8_E4M3, ks=A, vs=A) == pa.PA_ERR_NULL  # quantising needs 1/scale
    assert _decode_ex(app(new_stride=8 * 128 - 8)) == pa.PA_ERR_SHAPE    # a sequence's rows overlap
    assert _decode_ex(app(k_new=0x10008)) == pa.PA_ERR_ALIGN             # 16-byte bases
    assert _decode_ex(app(new_stride=8 * 128 + 4)) == pa.PA_ERR_ALIGN    # 16-byte row strides
    assert _decode_ex(app(), S=0) == pa.PA_OK                           # nothing to append or attend


def test_cache_write_and_copy_validation_edges(lib):
    st = pa.pa_reshape_and_cache(0x10000, 0x20000, pa.PA_BF16, 8 * 128 - 8, 8 * 128, 0x30000, 0x40000, pa.PA_BF16,
                                 16, 0x50000, 4, 8, 128, 16, None, None, None)
    assert st == pa.PA_ERR_SHAPE          # k rows of a token overlap the next token's
    st = pa.pa_reshape_and_cache(0x10000, 0x20000, pa.PA_BF16, 8 * 128, 8 * 128, 0x30000, 0x40000, pa.PA_INT8,
                                 16, 0x50000, 4, 8, 128, 16, 0x60000, 0x70000, None)
    assert st == pa.PA_ERR_NULL           # INT8 needs zero points (pa_reshape_and_cache_ex)
    assert pa.pa_copy_blocks(0x30000, 0x40000, 16, 32 * 1024, 0x50000, 65536, None) == pa.PA_ERR_UNSUPPORTED
    assert pa.pa_copy_blocks(0x30000, 0x40000, 16, 32 * 1024 + 8, 0x50000, 2, None) == pa.PA_ERR_ALIGN
    assert pa.pa_copy_blocks(0x30000, 0x40000, 16, 32 * 1024, 0x50000, 0, None) == pa.PA_OK

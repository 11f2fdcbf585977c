"""ctypes binding of libpagedattn (include/pa.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels.  If the library
cannot be loaded the calls raise; there is no CPU or PyTorch fallback.
"""

from __future__ import annotations

import ctypes
import os
import re

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libpagedattn.so")
HEADER = os.path.join(os.path.dirname(PKG_DIR), "include", "pa.h")

PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3, PA_INT8 = 0, 1, 2, 3, 4
PA_OK = 0
PA_ERR_NULL, PA_ERR_SHAPE, PA_ERR_DTYPE, PA_ERR_UNSUPPORTED = -1, -2, -3, -4
PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_ALIGN = -5, -6, -7
PA_DEVERR_BLOCK_ID, PA_DEVERR_SLOT, PA_DEVERR_SEQ_LEN, PA_DEVERR_TIMEOUT, PA_DEVERR_PAIR = 1, 2, 4, 8, 16
SIZE_MAX = ctypes.c_size_t(-1).value

_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

class DecodeOptions(ctypes.Structure):
    """pa_decode_options (include/pa.h); struct_size is filled in by the constructor."""
    _fields_ = [("struct_size", ctypes.c_size_t), ("window", ctypes.c_int32),
                ("k_zero_point", ctypes.c_void_p), ("v_zero_point", ctypes.c_void_p),
                ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("new_dtype", ctypes.c_int32),
                ("new_stride", ctypes.c_int64), ("k_inv_scale", ctypes.c_void_p), ("v_inv_scale", ctypes.c_void_p),
                ("q_len", ctypes.c_int32), ("pdl", ctypes.c_int32), ("early_kv", ctypes.c_int32)]

    def __init__(self, **kw):
        super().__init__(struct_size=ctypes.sizeof(DecodeOptions), **kw)


class CacheWriteOptions(ctypes.Structure):
    """pa_cache_write_options (include/pa.h)."""
    _fields_ = [("struct_size", ctypes.c_size_t), ("k_zero_point", ctypes.c_void_p),
                ("v_zero_point", ctypes.c_void_p), ("pdl", ctypes.c_int32)]

    def __init__(self, **kw):
        super().__init__(struct_size=ctypes.sizeof(CacheWriteOptions), **kw)


_SIGNATURES = {
    "pa_decode_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pa_decode_workspace_bytes_ex": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                           ctypes.POINTER(DecodeOptions)]),
    "pa_decode": (_i32, [_vp, _i32, _vp, _i32, _i64, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _i32, _vp,
                         _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp, _sz, _vp]),
    "pa_decode_ex": (_i32, [_vp, _i32, _vp, _i32, _i64, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _i32, _vp,
                            _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp, _sz, ctypes.POINTER(DecodeOptions), _vp]),
    "pa_reshape_and_cache": (_i32, [_vp, _vp, _i32, _i64, _i64, _vp, _vp, _i32, _i64, _vp, _i32, _i32, _i32,
                                    _i32, _vp, _vp, _vp]),
    "pa_reshape_and_cache_ex": (_i32, [_vp, _vp, _i32, _i64, _i64, _vp, _vp, _i32, _i64, _vp, _i32, _i32, _i32,
                                       _i32, _vp, _vp, ctypes.POINTER(CacheWriteOptions), _vp]),
    "pa_copy_blocks": (_i32, [_vp, _vp, _i64, _sz, _vp, _i32, _vp]),
    "pa_status_string": (ctypes.c_char_p, [_i32]),
    "pa_get_device_error": (_i32, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "pa_version": (_i32, []),
    "pa_last_error_detail": (ctypes.c_char_p, []),
    "pa_decode_noalloc": (_i32, [_vp, _i32, _vp, _i32, _i64, _vp, _vp, _i32, _i64, _vp, _vp, _vp, _i32, _vp,
                                 _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp]),
    "pa_decode_noalloc_capacity": (_sz, []),
    "pa_debug_set_decode_wait": (None, [ctypes.c_uint64, _i32]),
    "pa_decode_launch_config": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                       ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)]),
}

_LIB = None


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions that include/pa.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree libpagedattn.so."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        if not build_if_missing:
            raise OSError(f"{LIB_PATH} is missing; run paged_kv_cache_144_gb300.build")
        from .build import build
        build()
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != PA_OK:
        msg = status_string(status)
        if status == PA_ERR_CUDA:
            msg += ": " + load().pa_last_error_detail().decode()
        raise PagedAttnError(fn, status, msg)


# ----------------------------------------------------------------------------- raw C-ABI calls

def pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                              partition_size, kv_dtype) -> int:
    return int(load().pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                max_blocks_per_seq, partition_size, kv_dtype))


def pa_decode(*args) -> int:
    return int(load().pa_decode(*args))


def pa_decode_ex(*args) -> int:
    return int(load().pa_decode_ex(*args))


def pa_decode_noalloc(*args) -> int:
    return int(load().pa_decode_noalloc(*args))


def pa_decode_noalloc_capacity() -> int:
    return int(load().pa_decode_noalloc_capacity())


def pa_reshape_and_cache(*args) -> int:
    return int(load().pa_reshape_and_cache(*args))


def pa_reshape_and_cache_ex(*args) -> int:
    return int(load().pa_reshape_and_cache_ex(*args))


def pa_copy_blocks(*args) -> int:
    return int(load().pa_copy_blocks(*args))


def pa_get_device_error(stream) -> int:
    bits = ctypes.c_uint(0)
    _check("pa_get_device_error", int(load().pa_get_device_error(stream, ctypes.byref(bits))))
    return int(bits.value)


def pa_decode_launch_config(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                            partition_size, q_dtype, kv_dtype) -> dict:
    c, w, ns, sm = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    _check("pa_decode_launch_config", int(load().pa_decode_launch_config(
        num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, partition_size, q_dtype,
        kv_dtype, ctypes.byref(c), ctypes.byref(w), ctypes.byref(ns), ctypes.byref(sm))))
    return {"ctas": c.value, "warps_per_cta": w.value, "stages": ns.value, "smem_bytes": sm.value}


def pa_version() -> int:
    return int(load().pa_version())


def pa_debug_set_decode_wait(limit_ns: int, withhold_copies: bool) -> None:
    """Testing hook: wait limit of the next decode launches (0 = default) and whether their copies are withheld."""
    load().pa_debug_set_decode_wait(int(limit_ns), 1 if withhold_copies else 0)


# ----------------------------------------------------------------------------- torch marshalling

def _torch():
    import torch
    return torch


_DTYPE_CODES = None


def dtype_code(t) -> int:
    global _DTYPE_CODES
    m = _DTYPE_CODES
    if m is None:  # built once: this runs on every call of the step
        torch = _torch()
        m = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.uint8: PA_FP8_E4M3,
             torch.int8: PA_INT8}
        f8 = getattr(torch, "float8_e4m3fn", None)
        if f8 is not None:
            m[f8] = PA_FP8_E4M3
        _DTYPE_CODES = m
    code = m.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return code


def _ptr(t):
    # a plain integer: the signatures declare void*, so ctypes converts it
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = _torch().cuda.current_stream()
    return stream.cuda_stream


def _require_cuda(name, t, contiguous=True):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _require_cuda_all(named):
    """_require_cuda over (name, tensor) pairs in one call (the per-step path)."""
    for name, t in named:
        if t is not None and not (t.is_cuda and t.is_contiguous()):
            _require_cuda(name, t)


def decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                           partition_size=0, kv_dtype=PA_BF16, q_len=1) -> int:
    if q_len > 1:
        opt = DecodeOptions(q_len=int(q_len))
        n = int(load().pa_decode_workspace_bytes_ex(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                    max_blocks_per_seq, partition_size, kv_dtype, ctypes.byref(opt)))
    else:
        n = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                      partition_size, kv_dtype)
    if n == SIZE_MAX:
        raise PagedAttnError("pa_decode_workspace_bytes", PA_ERR_SHAPE, "sizes rejected or no usable device")
    return n


def new_workspace(nbytes: int, device):
    """Zero-filled workspace (allocated by torch, not by the library)."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads, scale, block_size, *,
           k_scale=None, v_scale=None, partition_size=0, workspace=None, stream=None, window=0,
           k_zero_point=None, v_zero_point=None, k_new=None, v_new=None, k_inv_scale=None, v_inv_scale=None,
           pdl=False, early_kv=False):
    """out[s,h] = softmax(scale * K_s q[s,h]) V_s through the block tables (pa_decode).

    window > 0: sliding-window decode over the last `window` positions (pa_decode_ex).
    INT8 caches (torch.int8) take k/v scales and int32 per-KV-head zero points (pa_decode_ex).
    k_new / v_new ([S, H_kv, d], F16/BF16): fused append -- the rows of position seq_lens[s]-1 are
    written into their cache slots (quantised with k_inv_scale / v_inv_scale for 8-bit caches) and
    attended in the same launch (pa_decode_ex).
    pdl=True: programmatic dependent launch (pa_decode_ex): the set-up overlaps the kernel launched just
    before on the stream, so seq_lens and block_tables must not be written by that kernel.
    early_kv=True (with pdl, one query, no fused append): that kernel also writes no cache row but each
    sequence's newest one (the step's cache write), so K/V copies of the other rows start before it ends.
    """
    _require_cuda_all((("out", out), ("k_cache", k_cache), ("v_cache", v_cache), ("block_tables", block_tables),
                       ("seq_lens", seq_lens), ("k_scale", k_scale), ("v_scale", v_scale),
                       ("k_zero_point", k_zero_point), ("v_zero_point", v_zero_point), ("k_inv_scale", k_inv_scale),
                       ("v_inv_scale", v_inv_scale)))
    _require_cuda("q", q, contiguous=False)
    q_len = 1
    if q.dim() == 4:                       # [S, L, H_q, d]: several queries per sequence
        q_len = q.shape[1]
        if q.stride(3) != 1 or q.stride(2) != q.shape[3] or q.stride(1) != q.shape[2] * q.shape[3]:
            raise ValueError("the queries of a sequence must be contiguous")
        q = q.view(q.shape[0], q_len * q.shape[2], q.shape[3]) if q.is_contiguous() else q
    new_stride, new_dtype = 0, PA_F16
    if k_new is not None or v_new is not None:
        _require_cuda("k_new", k_new, contiguous=False)
        _require_cuda("v_new", v_new, contiguous=False)
        for t in (k_new, v_new):
            if t.stride(2) != 1 or t.stride(1) != t.shape[2] or t.stride(0) != k_new.stride(0):
                raise ValueError("k_new/v_new rows must be contiguous per sequence with equal strides")
        new_stride, new_dtype = k_new.stride(0), dtype_code(k_new)
    if q.stride(2) != 1 or q.stride(1) != q.shape[2]:
        raise ValueError("q rows must be contiguous per sequence")
    S, Hq, D = q.shape
    Hq //= q_len
    NB = k_cache.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(out), dtype_code(out), _ptr(q), dtype_code(q), q.stride(0),
            _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache), NB,
            _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
            S, Hq, int(num_kv_heads), D, float(scale), int(block_size), int(partition_size),
            _ptr(workspace), ws_bytes)
    if window or k_zero_point is not None or v_zero_point is not None or k_new is not None or q_len > 1 or pdl:
        opt = DecodeOptions(window=int(window), k_zero_point=_ptr(k_zero_point), v_zero_point=_ptr(v_zero_point),
                            k_new=_ptr(k_new), v_new=_ptr(v_new), new_dtype=new_dtype, new_stride=new_stride,
                            k_inv_scale=_ptr(k_inv_scale), v_inv_scale=_ptr(v_inv_scale), q_len=q_len,
                            pdl=1 if pdl else 0, early_kv=1 if early_kv else 0)
        st = pa_decode_ex(*args, ctypes.byref(opt), _stream(stream))
        _check("pa_decode_ex", st)
    else:
        st = pa_decode(*args, _stream(stream))
        _check("pa_decode", st)
    return out


def decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads, scale, block_size, *,
                   k_scale=None, v_scale=None, partition_size=0, stream=None):
    """pa_decode on the library's fixed device array (for callers that cannot allocate)."""
    for n, t in (("out", out), ("k_cache", k_cache), ("v_cache", v_cache), ("block_tables", block_tables),
                 ("seq_lens", seq_lens), ("k_scale", k_scale), ("v_scale", v_scale)):
        _require_cuda(n, t)
    _require_cuda("q", q, contiguous=False)
    if q.stride(2) != 1 or q.stride(1) != q.shape[2]:
        raise ValueError("q rows must be contiguous per sequence")
    S, Hq, D = q.shape
    st = pa_decode_noalloc(_ptr(out), dtype_code(out), _ptr(q), dtype_code(q), q.stride(0),
                           _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache), k_cache.shape[0],
                           _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                           S, Hq, int(num_kv_heads), D, float(scale), int(block_size), int(partition_size),
                           _stream(stream))
    _check("pa_decode_noalloc", st)
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, block_size, *, k_inv_scale=None, v_inv_scale=None,
                      k_zero_point=None, v_zero_point=None, stream=None, pdl=False):
    """Write rows k[n], v[n] ([N, H_kv, d]) to cache slots slot_mapping[n] (pa_reshape_and_cache).

    INT8 caches (torch.int8) also take int32 per-KV-head zero points (pa_reshape_and_cache_ex).
    pdl=True: programmatic dependent launch (pa_reshape_and_cache_ex): the kernel waits for the kernel before
    it on the stream before touching memory, so only its launch overlaps that kernel's end.
    """
    _require_cuda_all((("k_cache", k_cache), ("v_cache", v_cache), ("slot_mapping", slot_mapping),
                       ("k_inv_scale", k_inv_scale), ("v_inv_scale", v_inv_scale), ("k_zero_point", k_zero_point),
                       ("v_zero_point", v_zero_point)))
    _require_cuda("k", k, contiguous=False)
    _require_cuda("v", v, contiguous=False)
    N, Hkv, D = k.shape
    for t in (k, v):
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError("k/v rows must be contiguous per token")
    args = (_ptr(k), _ptr(v), dtype_code(k), k.stride(0), v.stride(0),
            _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache), k_cache.shape[0],
            _ptr(slot_mapping), N, Hkv, D, int(block_size), _ptr(k_inv_scale), _ptr(v_inv_scale))
    if k_zero_point is not None or v_zero_point is not None or pdl:
        opt = CacheWriteOptions(k_zero_point=_ptr(k_zero_point), v_zero_point=_ptr(v_zero_point),
                                pdl=1 if pdl else 0)
        st = pa_reshape_and_cache_ex(*args, ctypes.byref(opt), _stream(stream))
        _check("pa_reshape_and_cache_ex", st)
    else:
        st = pa_reshape_and_cache(*args, _stream(stream))
        _check("pa_reshape_and_cache", st)


def copy_blocks(k_cache, v_cache, src_dst_pairs, *, stream=None):
    """Copy whole physical blocks src -> dst in both pools (pa_copy_blocks)."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("src_dst_pairs", src_dst_pairs)):
        _require_cuda(n, t)
    n_pairs = src_dst_pairs.shape[0] if src_dst_pairs.numel() else 0
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    st = pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), k_cache.shape[0], block_bytes, _ptr(src_dst_pairs),
                        n_pairs, _stream(stream))
    _check("pa_copy_blocks", st)


def get_device_error(stream=None) -> int:
    return pa_get_device_error(_stream(stream))

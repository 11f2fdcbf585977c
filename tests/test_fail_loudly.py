"""The product path has no CPU or PyTorch fallback: host tensors are refused
and a missing library is an error, never a silent substitute."""

import pytest
import torch

import paged_kv_cache_144_gb300 as pa
from paged_kv_cache_144_gb300 import _lib


def _host_batch():
    q = torch.zeros((2, 4, 64), dtype=torch.float16)
    kc = torch.zeros((8, 4, 16, 64), dtype=torch.float16)
    tables = torch.zeros((2, 4), dtype=torch.int32)
    lens = torch.ones((2,), dtype=torch.int32)
    return q, kc, tables, lens


def test_decode_refuses_host_tensors():
    q, kc, tables, lens = _host_batch()
    out = torch.empty_like(q, dtype=torch.float32)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        pa.decode(out, q, kc, kc, tables, lens, 4, 0.125, 16)


def test_cache_write_refuses_host_tensors():
    q, kc, tables, lens = _host_batch()
    rows = torch.zeros((2, 4, 64), dtype=torch.float16)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        pa.reshape_and_cache(rows, rows, kc, kc, torch.zeros((2,), dtype=torch.int64), 16)


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libpagedattn.so"))
    with pytest.raises(OSError, match="is missing"):
        _lib.load(build_if_missing=False)

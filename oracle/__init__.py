"""Float64 CPU oracle for paged decode attention and its cache operations.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code, constants or helpers with the CUDA path.

Sources (the pages this oracle restates; cited per function):
  [P1] "論文解説: Efficient Memory Management for Large Language Model Serving
       with PagedAttention" (0h-n0.github.io)
  [P2] "KVキャッシュとPagedAttention — 推論メモリのすべて" (youngju.dev)
  [P3] "PagedAttention" reading notes (dihengye.cn)
  [P4] "メモリ予算内での言語モデルのサービング：注意機構、ページング、スケジューリング"
       (auturnal.com), equations (1)-(4)

Every function is pinned by ``tests/test_oracle_pins.py`` against something
other than itself (closed forms, the pages' worked examples, library routines,
brute force).  Parity status per function is listed in each module header.
"""

from .codecs import (
    bf16_bits_to_f64,
    f16_to_f64,
    e4m3_decode,
    e4m3_encode_f32,
    int8_decode,
    int8_encode_f32,
    E4M3_MAX,
)
from .attention import (
    gather_sequence,
    dense_decode_attention,
    paged_decode_attention,
    paged_decode_attention_one,
    paged_append_decode,
    paged_multi_query_attention,
    dequantize_kv,
)
from .online_softmax import online_softmax_attention, merge_partials, partial_state
from .cache_ops import reshape_and_cache, copy_blocks
from .accounting import (
    kv_bytes,
    kv_bytes_per_token,
    tail_waste,
    tail_waste_one,
    mean_tail_waste_uniform,
    mean_reserve_waste_uniform,
)
from .cow import RefcountBlockManager, copy_on_write

__all__ = [
    "bf16_bits_to_f64", "f16_to_f64", "e4m3_decode", "e4m3_encode_f32", "E4M3_MAX",
    "gather_sequence", "dense_decode_attention", "paged_decode_attention",
    "paged_decode_attention_one", "dequantize_kv",
    "online_softmax_attention", "merge_partials", "partial_state",
    "reshape_and_cache", "copy_blocks",
    "kv_bytes", "kv_bytes_per_token", "tail_waste", "tail_waste_one",
    "mean_tail_waste_uniform", "mean_reserve_waste_uniform",
    "RefcountBlockManager", "copy_on_write",
]

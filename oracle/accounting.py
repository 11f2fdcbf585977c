"""KV-cache size and page-tail waste accounting.

Test infrastructure (see ``oracle/__init__``).

[P4] equation (1): M_KV = 2 L H_KV d_h b sum_i T_i (keys and values only, no
weights, activations, metadata or padding).  [P2] §"KVキャッシュはなぜメモリを消費
するのか" gives the same product per token and layer.

[P4] equation (2): W_tail = sum_i (B ceil(T_i/B) - T_i) <= N (B - 1) for N
non-empty requests of integer length; [P4] equation (3): for one request
with length uniform on 1..kB, E[W_tail] = (B - 1)/2 exactly; [P4] §5: the
scheme that reserves 512 slots per request wastes 255.5 slots on average
under lengths uniform on 1..512.

Pins: the pages' worked numbers (131072 B per token; 0.5 GiB for 4096 tokens;
2 GiB with 32 KV heads; about 16 GB for 32 such requests) and exhaustive
checks of the bound and the exact means (``tests/test_oracle_pins.py``).
"""

from __future__ import annotations

from fractions import Fraction


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, bytes_per_scalar: int) -> int:
    """2 * L * H_kv * d * b."""
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_scalar


def kv_bytes(num_layers: int, num_kv_heads: int, head_dim: int, bytes_per_scalar: int, lengths) -> int:
    """M_KV of equation (1)."""
    return kv_bytes_per_token(num_layers, num_kv_heads, head_dim, bytes_per_scalar) * sum(int(t) for t in lengths)


def tail_waste_one(length: int, block_size: int) -> int:
    """Unused slots in the last block of one request: B ceil(T/B) - T."""
    length = int(length)
    return block_size * (-(-length // block_size)) - length


def tail_waste(lengths, block_size: int) -> int:
    """W_tail of equation (2)."""
    return sum(tail_waste_one(t, block_size) for t in lengths)


def mean_tail_waste_uniform(block_size: int, max_len: int) -> Fraction:
    """Exact E[W_tail] for one request with length uniform on 1..max_len."""
    total = sum(tail_waste_one(t, block_size) for t in range(1, max_len + 1))
    return Fraction(total, max_len)


def mean_reserve_waste_uniform(reserved: int, max_len: int) -> Fraction:
    """Exact mean of (reserved - T) for T uniform on 1..max_len (reservation scheme)."""
    total = sum(reserved - t for t in range(1, max_len + 1))
    return Fraction(total, max_len)

"""Seeded synthetic inputs for paged decode attention (shared by tests, bench, smoke).

This module builds *inputs only*: sequence lengths, block-pool permutations,
block tables, slot numbers of appended tokens, random K/V/q values and FP8
calibration scales.  It holds none of the attention, softmax, quantisation or
copy arithmetic: the CUDA path and the oracle each implement those on their
own and both receive what this module produces.

Workloads (shapes and distributions of the pages' examples):
  tiny        4 seqs, cached len ~U{1..128} + 1 appended, 4 heads MHA, d=64,
              B=16, fp16, pool of 64 blocks in a seeded random permutation,
              scale 1/8.
  gqa_32x4k   32 seqs, len ~U{1..4096}, 32 q heads / 8 KV heads, d=128, B=16,
              bf16, pool = blocks needed + 10 % free, permuted tables,
              scale 1/sqrt(128).
  long_32k    8 seqs of exactly 32768 tokens, 64 q / 8 KV heads, d=128, B=16,
              bf16; q ~ N(0,1) or N(0,1)*30 (extreme logits).
  beam_cow    6 beams sharing a 1000-token prompt (63 blocks, the last holding
              8 tokens), private tails ~U{1..256}, 40 heads MHA, d=128, B=16,
              fp16; CoW of the shared partial block, one appended token each.
  fp8_mix     256 seqs, len = clip(round(lognormal(7, 1)), 16, 8192), 32 q /
              8 KV heads, d=128, K/V FP8-e4m3 with per-KV-head float32 scales
              calibrated as amax/448 over bf16-rounded N(0,1) values, bf16 q,
              B in {16, 32}.

Slot encoding (a reading; the pages give none): a token at position p of a
sequence goes to slot table[p // B] * B + p % B, as int64.
"""

from .configs import (  # noqa: F401
    WORKLOADS,
    DecodeBatch,
    make_batch,
    build_block_tables,
    slot_of,
    host_values,
    device_values,
    beam_cow_scenario,
    fp8_scales_from_amax,
    bf16_bits_from_f32,
    shard_sequences,
)

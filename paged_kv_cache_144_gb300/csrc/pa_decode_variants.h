// pa_decode_variants.h - the compiled (q dtype, kv dtype, head_dim, block_size,
// max group) variants of the decode kernel.  A group G is served by the
// smallest compiled maximum >= G (1, 4 or 8).
#pragma once

#define PA_DECODE_VARIANTS_F16(X)                                                    \
  X(f16_t, f16_t, 64, 16, 1) X(f16_t, f16_t, 64, 16, 4) X(f16_t, f16_t, 64, 16, 8)   \
  X(f16_t, f16_t, 64, 32, 1) X(f16_t, f16_t, 64, 32, 4) X(f16_t, f16_t, 64, 32, 8)   \
  X(f16_t, f16_t, 128, 16, 1) X(f16_t, f16_t, 128, 16, 4) X(f16_t, f16_t, 128, 16, 8) \
  X(f16_t, f16_t, 128, 32, 1) X(f16_t, f16_t, 128, 32, 4) X(f16_t, f16_t, 128, 32, 8)

#define PA_DECODE_VARIANTS_BF16(X)                                                        \
  X(bf16_t, bf16_t, 64, 16, 1) X(bf16_t, bf16_t, 64, 16, 4) X(bf16_t, bf16_t, 64, 16, 8)   \
  X(bf16_t, bf16_t, 64, 32, 1) X(bf16_t, bf16_t, 64, 32, 4) X(bf16_t, bf16_t, 64, 32, 8)   \
  X(bf16_t, bf16_t, 128, 16, 1) X(bf16_t, bf16_t, 128, 16, 4) X(bf16_t, bf16_t, 128, 16, 8) \
  X(bf16_t, bf16_t, 128, 32, 1) X(bf16_t, bf16_t, 128, 32, 4) X(bf16_t, bf16_t, 128, 32, 8)

#define PA_DECODE_VARIANTS_FP8(X)                                                         \
  X(bf16_t, e4m3_t, 128, 16, 1) X(bf16_t, e4m3_t, 128, 16, 4) X(bf16_t, e4m3_t, 128, 16, 8) \
  X(bf16_t, e4m3_t, 128, 32, 1) X(bf16_t, e4m3_t, 128, 32, 4) X(bf16_t, e4m3_t, 128, 32, 8) \
  X(f16_t, e4m3_t, 128, 16, 1) X(f16_t, e4m3_t, 128, 16, 4) X(f16_t, e4m3_t, 128, 16, 8)    \
  X(f16_t, e4m3_t, 128, 32, 1) X(f16_t, e4m3_t, 128, 32, 4) X(f16_t, e4m3_t, 128, 32, 8)

#define PA_DECODE_VARIANTS(X) PA_DECODE_VARIANTS_F16(X) PA_DECODE_VARIANTS_BF16(X) PA_DECODE_VARIANTS_FP8(X)

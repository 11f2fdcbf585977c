// pa_decode_variants.h - the compiled (q dtype, kv dtype, head_dim, max group,
// unit rows) variants of the decode kernel (the block size is a runtime
// parameter; 64-row units are compiled for 8-bit caches only).  A group G is served by the
// smallest compiled maximum >= G (1, 4 or 8).
#pragma once

#include "pa_common.cuh"
#include "pa_kernels.h"

#define PA_DECODE_VARIANTS_F16(X) \
  X(f16_t, f16_t, 64, 1, 16) X(f16_t, f16_t, 64, 1, 32) X(f16_t, f16_t, 64, 4, 16) X(f16_t, f16_t, 64, 4, 32) \
  X(f16_t, f16_t, 64, 8, 16) X(f16_t, f16_t, 64, 8, 32) X(f16_t, f16_t, 128, 1, 16) \
  X(f16_t, f16_t, 128, 1, 32) X(f16_t, f16_t, 128, 4, 16) X(f16_t, f16_t, 128, 4, 32) \
  X(f16_t, f16_t, 128, 8, 16) X(f16_t, f16_t, 128, 8, 32)

#define PA_DECODE_VARIANTS_BF16(X) \
  X(bf16_t, bf16_t, 64, 1, 16) X(bf16_t, bf16_t, 64, 1, 32) X(bf16_t, bf16_t, 64, 4, 16) \
  X(bf16_t, bf16_t, 64, 4, 32) X(bf16_t, bf16_t, 64, 8, 16) X(bf16_t, bf16_t, 64, 8, 32) \
  X(bf16_t, bf16_t, 128, 1, 16) X(bf16_t, bf16_t, 128, 1, 32) X(bf16_t, bf16_t, 128, 4, 16) \
  X(bf16_t, bf16_t, 128, 4, 32) X(bf16_t, bf16_t, 128, 8, 16) X(bf16_t, bf16_t, 128, 8, 32)

#define PA_DECODE_VARIANTS_FP8(X) \
  X(bf16_t, e4m3_t, 128, 1, 16) X(bf16_t, e4m3_t, 128, 1, 32) X(bf16_t, e4m3_t, 128, 4, 16) \
  X(bf16_t, e4m3_t, 128, 4, 32) X(bf16_t, e4m3_t, 128, 8, 16) X(bf16_t, e4m3_t, 128, 8, 32) \
  X(f16_t, e4m3_t, 128, 1, 16) X(f16_t, e4m3_t, 128, 1, 32) X(f16_t, e4m3_t, 128, 4, 16) \
  X(f16_t, e4m3_t, 128, 4, 32) X(f16_t, e4m3_t, 128, 8, 16) X(f16_t, e4m3_t, 128, 8, 32) \
  X(bf16_t, e4m3_t, 128, 1, 64) X(bf16_t, e4m3_t, 128, 4, 64) X(bf16_t, e4m3_t, 128, 8, 64) \
  X(f16_t, e4m3_t, 128, 1, 64) X(f16_t, e4m3_t, 128, 4, 64) X(f16_t, e4m3_t, 128, 8, 64)

#define PA_DECODE_VARIANTS_INT8(X) \
  X(bf16_t, i8_t, 128, 1, 16) X(bf16_t, i8_t, 128, 1, 32) X(bf16_t, i8_t, 128, 1, 64) \
  X(bf16_t, i8_t, 128, 4, 16) X(bf16_t, i8_t, 128, 4, 32) X(bf16_t, i8_t, 128, 4, 64) \
  X(bf16_t, i8_t, 128, 8, 16) X(bf16_t, i8_t, 128, 8, 32) X(bf16_t, i8_t, 128, 8, 64) \
  X(f16_t, i8_t, 128, 1, 16) X(f16_t, i8_t, 128, 1, 32) X(f16_t, i8_t, 128, 1, 64) \
  X(f16_t, i8_t, 128, 4, 16) X(f16_t, i8_t, 128, 4, 32) X(f16_t, i8_t, 128, 4, 64) \
  X(f16_t, i8_t, 128, 8, 16) X(f16_t, i8_t, 128, 8, 32) X(f16_t, i8_t, 128, 8, 64)

#define PA_DECODE_VARIANTS(X) \
  PA_DECODE_VARIANTS_F16(X) PA_DECODE_VARIANTS_BF16(X) PA_DECODE_VARIANTS_FP8(X) PA_DECODE_VARIANTS_INT8(X)

// Each variant translation unit defines these two plain functions; the
// dispatcher sees only the declarations, so every kernel is instantiated and
// registered in exactly one translation unit.
#define PA_DECLARE_VARIANT(QT, KVT, D, GM, UR)                                                   \
  bool decode_geometry_##QT##_##KVT##_##D##_##GM##_##UR(int num_seqs, int append, DecodeGeometry* geo); \
  cudaError_t decode_launch_##QT##_##KVT##_##D##_##GM##_##UR(const DecodeGeometry& geo,           \
                                                              const DecodeParams& p,              \
                                                              const CUtensorMap& tk,              \
                                                              const CUtensorMap& tv, cudaStream_t stream);
#define PA_DEFINE_VARIANT(QT, KVT, D, GM, UR)                                                      \
  bool decode_geometry_##QT##_##KVT##_##D##_##GM##_##UR(int num_seqs, int append, DecodeGeometry* geo) { \
    return DecodeVariant<QT, KVT, D, GM, UR>::geometry(num_seqs, append, geo);                     \
  }                                                                                                \
  cudaError_t decode_launch_##QT##_##KVT##_##D##_##GM##_##UR(const DecodeGeometry& geo,           \
                                                              const DecodeParams& p,              \
                                                              const CUtensorMap& tk,              \
                                                              const CUtensorMap& tv, cudaStream_t stream) { \
    return DecodeVariant<QT, KVT, D, GM, UR>::launch(geo, p, tk, tv, stream);                      \
  }

namespace pa {
PA_DECODE_VARIANTS(PA_DECLARE_VARIANT)
}  // namespace pa

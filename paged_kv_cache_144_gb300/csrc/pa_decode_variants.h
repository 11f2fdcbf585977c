// pa_decode_variants.h - the compiled (q dtype, kv dtype, head_dim, max A
// rows, unit rows, fused append) variants of the decode kernel (the block
// size is a runtime parameter; units of 32 rows, and of 64 rows for 8-bit
// caches; fused-append variants for the default unit rows only).  The A rows of
// a segment, q_len * G (query, head) pairs, are served by the smallest
// compiled maximum >= q_len * G (1, 4, 8 or 16).
#pragma once

#include "pa_common.cuh"
#include "pa_kernels.h"

#define PA_DECODE_VARIANTS_F16(X) \
  X(f16_t, f16_t, 64, 1, 32, 0) X(f16_t, f16_t, 64, 4, 32, 0) X(f16_t, f16_t, 64, 8, 32, 0) \
  X(f16_t, f16_t, 128, 1, 32, 0) X(f16_t, f16_t, 128, 4, 32, 0) X(f16_t, f16_t, 128, 8, 32, 0)

#define PA_DECODE_VARIANTS_BF16(X) \
  X(bf16_t, bf16_t, 64, 1, 32, 0) X(bf16_t, bf16_t, 64, 4, 32, 0) X(bf16_t, bf16_t, 64, 8, 32, 0) \
  X(bf16_t, bf16_t, 128, 1, 32, 0) X(bf16_t, bf16_t, 128, 4, 32, 0) X(bf16_t, bf16_t, 128, 8, 32, 0)

#define PA_DECODE_VARIANTS_FP8(X) \
  X(bf16_t, e4m3_t, 128, 1, 32, 0) X(bf16_t, e4m3_t, 128, 1, 64, 0) \
  X(bf16_t, e4m3_t, 128, 4, 32, 0) X(bf16_t, e4m3_t, 128, 4, 64, 0) \
  X(bf16_t, e4m3_t, 128, 8, 32, 0) X(bf16_t, e4m3_t, 128, 8, 64, 0) \
  X(f16_t, e4m3_t, 128, 1, 32, 0) X(f16_t, e4m3_t, 128, 1, 64, 0) \
  X(f16_t, e4m3_t, 128, 4, 32, 0) X(f16_t, e4m3_t, 128, 4, 64, 0) \
  X(f16_t, e4m3_t, 128, 8, 32, 0) X(f16_t, e4m3_t, 128, 8, 64, 0)

#define PA_DECODE_VARIANTS_INT8(X) \
  X(bf16_t, i8_t, 128, 1, 32, 0) X(bf16_t, i8_t, 128, 1, 64, 0) \
  X(bf16_t, i8_t, 128, 4, 32, 0) X(bf16_t, i8_t, 128, 4, 64, 0) \
  X(bf16_t, i8_t, 128, 8, 32, 0) X(bf16_t, i8_t, 128, 8, 64, 0) \
  X(f16_t, i8_t, 128, 1, 32, 0) X(f16_t, i8_t, 128, 1, 64, 0) \
  X(f16_t, i8_t, 128, 4, 32, 0) X(f16_t, i8_t, 128, 4, 64, 0) \
  X(f16_t, i8_t, 128, 8, 32, 0) X(f16_t, i8_t, 128, 8, 64, 0)

// 16 A rows per warp: several queries per sequence (q_len * G <= 64, 16 rows per warp of a ring)
#define PA_DECODE_VARIANTS_ROWS16(X) \
  X(f16_t, f16_t, 64, 16, 32, 0) X(f16_t, f16_t, 128, 16, 32, 0) X(bf16_t, bf16_t, 64, 16, 32, 0) \
  X(bf16_t, bf16_t, 128, 16, 32, 0) X(bf16_t, e4m3_t, 128, 16, 32, 0) X(bf16_t, i8_t, 128, 16, 32, 0) \
  X(f16_t, e4m3_t, 128, 16, 32, 0) X(f16_t, i8_t, 128, 16, 32, 0)

// fused append (cache write of the newest rows in the same launch), default unit rows
#define PA_DECODE_VARIANTS_APPEND16(X) \
  X(f16_t, f16_t, 64, 1, 32, 1) X(f16_t, f16_t, 64, 4, 32, 1) X(f16_t, f16_t, 64, 8, 32, 1) \
  X(f16_t, f16_t, 128, 1, 32, 1) X(f16_t, f16_t, 128, 4, 32, 1) X(f16_t, f16_t, 128, 8, 32, 1) \
  X(bf16_t, bf16_t, 64, 1, 32, 1) X(bf16_t, bf16_t, 64, 4, 32, 1) X(bf16_t, bf16_t, 64, 8, 32, 1) \
  X(bf16_t, bf16_t, 128, 1, 32, 1) X(bf16_t, bf16_t, 128, 4, 32, 1) X(bf16_t, bf16_t, 128, 8, 32, 1)

#define PA_DECODE_VARIANTS_APPEND8(X) \
  X(bf16_t, e4m3_t, 128, 1, 32, 1) X(bf16_t, e4m3_t, 128, 1, 64, 1) X(bf16_t, e4m3_t, 128, 4, 32, 1) \
  X(bf16_t, e4m3_t, 128, 4, 64, 1) X(bf16_t, e4m3_t, 128, 8, 32, 1) X(bf16_t, e4m3_t, 128, 8, 64, 1) \
  X(bf16_t, i8_t, 128, 1, 32, 1) X(bf16_t, i8_t, 128, 1, 64, 1) X(bf16_t, i8_t, 128, 4, 32, 1) \
  X(bf16_t, i8_t, 128, 4, 64, 1) X(bf16_t, i8_t, 128, 8, 32, 1) X(bf16_t, i8_t, 128, 8, 64, 1) \
  X(f16_t, e4m3_t, 128, 1, 32, 1) X(f16_t, e4m3_t, 128, 1, 64, 1) X(f16_t, e4m3_t, 128, 4, 32, 1) \
  X(f16_t, e4m3_t, 128, 4, 64, 1) X(f16_t, e4m3_t, 128, 8, 32, 1) X(f16_t, e4m3_t, 128, 8, 64, 1) \
  X(f16_t, i8_t, 128, 1, 32, 1) X(f16_t, i8_t, 128, 1, 64, 1) X(f16_t, i8_t, 128, 4, 32, 1) \
  X(f16_t, i8_t, 128, 4, 64, 1) X(f16_t, i8_t, 128, 8, 32, 1) X(f16_t, i8_t, 128, 8, 64, 1)

#define PA_DECODE_VARIANTS(X) \
  PA_DECODE_VARIANTS_F16(X) PA_DECODE_VARIANTS_BF16(X) PA_DECODE_VARIANTS_FP8(X) PA_DECODE_VARIANTS_INT8(X) \
  PA_DECODE_VARIANTS_ROWS16(X) PA_DECODE_VARIANTS_APPEND16(X) PA_DECODE_VARIANTS_APPEND8(X)

// Each variant translation unit defines these two plain functions; the
// dispatcher sees only the declarations, so every kernel is instantiated and
// registered in exactly one translation unit.
#define PA_DECLARE_VARIANT(QT, KVT, D, GM, UR, AP) \
  bool decode_geometry_##QT##_##KVT##_##D##_##GM##_##UR##_##AP(int num_seqs, int nc, DecodeGeometry* geo); \
  cudaError_t decode_launch_##QT##_##KVT##_##D##_##GM##_##UR##_##AP(const DecodeGeometry& geo, \
                                                              const DecodeParams& p, \
                                                              const CUtensorMap& tk, \
                                                              const CUtensorMap& tv, cudaStream_t stream, \
                                                              bool pdl);
#define PA_DEFINE_VARIANT(QT, KVT, D, GM, UR, AP) \
  bool decode_geometry_##QT##_##KVT##_##D##_##GM##_##UR##_##AP(int num_seqs, int nc, DecodeGeometry* geo) { \
    return DecodeVariant<QT, KVT, D, GM, UR, AP>::geometry(num_seqs, nc, geo); \
  } \
  cudaError_t decode_launch_##QT##_##KVT##_##D##_##GM##_##UR##_##AP(const DecodeGeometry& geo, \
                                                              const DecodeParams& p, \
                                                              const CUtensorMap& tk, \
                                                              const CUtensorMap& tv, cudaStream_t stream, \
                                                              bool pdl) { \
    return DecodeVariant<QT, KVT, D, GM, UR, AP>::launch(geo, p, tk, tv, stream, pdl); \
  }

namespace pa {
PA_DECODE_VARIANTS(PA_DECLARE_VARIANT)
}  // namespace pa

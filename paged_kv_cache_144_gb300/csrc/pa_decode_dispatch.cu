// pa_decode_dispatch.cu - maps a runtime DecodeKey to its compiled variant.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {

#define PA_EXTERN(QT, KVT, D, BS, GM) extern template struct DecodeVariant<QT, KVT, D, BS, GM>;
PA_DECODE_VARIANTS(PA_EXTERN)
#undef PA_EXTERN

template <typename T> constexpr int dtype_code();
template <> constexpr int dtype_code<f16_t>() { return PA_F16; }
template <> constexpr int dtype_code<bf16_t>() { return PA_BF16; }
template <> constexpr int dtype_code<e4m3_t>() { return PA_FP8_E4M3; }

#define PA_MATCH(QT, KVT, D, BS, GM)                                                        \
  (key.q_dtype == dtype_code<QT>() && key.kv_dtype == dtype_code<KVT>() && key.head_dim == D && \
   key.block_size == BS && key.gmax == GM)

bool decode_geometry(const DecodeKey& key, int num_seqs, DecodeGeometry* geo) {
#define PA_GEO(QT, KVT, D, BS, GM) \
  if (PA_MATCH(QT, KVT, D, BS, GM)) return DecodeVariant<QT, KVT, D, BS, GM>::geometry(num_seqs, geo);
  PA_DECODE_VARIANTS(PA_GEO)
#undef PA_GEO
  return false;
}

cudaError_t launch_decode(const DecodeKey& key, const DecodeGeometry& geo, const DecodeParams& p,
                          const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
#define PA_LAUNCH(QT, KVT, D, BS, GM) \
  if (PA_MATCH(QT, KVT, D, BS, GM)) return DecodeVariant<QT, KVT, D, BS, GM>::launch(geo, p, tk, tv, stream);
  PA_DECODE_VARIANTS(PA_LAUNCH)
#undef PA_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace pa

// pa_decode_bf16.cu - explicit instantiation of the BF16 decode variants (one
// translation unit per cache type so the build compiles them in parallel).
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
#define PA_INSTANTIATE(QT, KVT, D, BS, GM) template struct DecodeVariant<QT, KVT, D, BS, GM>;
PA_DECODE_VARIANTS_BF16(PA_INSTANTIATE)
#undef PA_INSTANTIATE
}  // namespace pa

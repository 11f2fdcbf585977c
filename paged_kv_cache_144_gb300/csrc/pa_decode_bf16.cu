// pa_decode_bf16.cu - the BF16 decode variants (one translation unit per cache
// type so the build compiles them in parallel).  This file is the only place
// these kernels are instantiated.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
PA_DECODE_VARIANTS_BF16(PA_DEFINE_VARIANT)
}  // namespace pa

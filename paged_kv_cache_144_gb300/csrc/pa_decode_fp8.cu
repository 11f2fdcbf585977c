// pa_decode_fp8.cu - the FP8 decode variants (one translation unit per cache
// type so the build compiles them in parallel).  This file is the only place
// these kernels are instantiated.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
PA_DECODE_VARIANTS_FP8(PA_DEFINE_VARIANT)
}  // namespace pa

// pa_decode_f16.cu - the F16 decode variants (one translation unit per cache
// type so the build compiles them in parallel).  This file is the only place
// these kernels are instantiated.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
PA_DECODE_VARIANTS_F16(PA_DEFINE_VARIANT)
}  // namespace pa

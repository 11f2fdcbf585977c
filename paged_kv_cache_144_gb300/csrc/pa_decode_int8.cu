// pa_decode_int8.cu - the INT8 decode variants (one translation unit per cache
// type so the build compiles them in parallel).  This file is the only place
// these kernels are instantiated.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
PA_DECODE_VARIANTS_INT8(PA_DEFINE_VARIANT)
}  // namespace pa

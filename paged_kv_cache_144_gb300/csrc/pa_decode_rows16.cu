// pa_decode_rows16.cu - the 16-row decode variants (several queries per
// sequence), in their own translation unit so the build compiles them in
// parallel.  This file is the only place these kernels are instantiated.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
PA_DECODE_VARIANTS_ROWS16(PA_DEFINE_VARIANT)
}  // namespace pa

// pa_decode_append16.cu - the fused-append decode variants for 16-bit caches, in
// their own translation unit so the build compiles them in parallel.  This
// file is the only place these kernels are instantiated.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
PA_DECODE_VARIANTS_APPEND16(PA_DEFINE_VARIANT)
}  // namespace pa

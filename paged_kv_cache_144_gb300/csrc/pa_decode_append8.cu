// pa_decode_append8.cu - the fused-append decode variants for 8-bit caches, in
// their own translation unit so the build compiles them in parallel.  This
// file is the only place these kernels are instantiated.
#include "pa_decode.cuh"
#include "pa_decode_variants.h"

namespace pa {
PA_DECODE_VARIANTS_APPEND8(PA_DEFINE_VARIANT)
}  // namespace pa

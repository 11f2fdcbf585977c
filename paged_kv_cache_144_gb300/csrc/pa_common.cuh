// pa_common.cuh - small device helpers shared by the libpagedattn kernels:
// mbarrier + TMA wrappers (inline PTX for sm_103a), packed f32x2 FMA, element
// conversions and the per-device error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Record PA_DEVERR_* bits in the per-device error word (its address is a
// kernel argument; the word itself lives in pa_api.cu).
__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bits) {
  atomicOr(err, bits);
}

// ----------------------------------------------------------------- mbarrier / TMA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Non-blocking probe: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of barrier `bar` to complete, giving up after
// `limit_ns` nanoseconds.  Returns false on timeout (the caller records it).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// 2-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 3-D tiled TMA load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ----------------------------------------------------------------- packed fp32 math

// d = a * b + c on two fp32 lanes at once (sm_100+ packed FMA).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra = *reinterpret_cast<uint64_t*>(&a);
  uint64_t rb = *reinterpret_cast<uint64_t*>(&b);
  uint64_t rc = *reinterpret_cast<uint64_t*>(&c);
  uint64_t rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2*>(&rd);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t ra = *reinterpret_cast<uint64_t*>(&a);
  uint64_t rb = *reinterpret_cast<uint64_t*>(&b);
  uint64_t rd;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2*>(&rd);
}

// 2^x with the hardware approximation (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ----------------------------------------------------------------- element types

struct f16_t {};
struct bf16_t {};
struct e4m3_t {};

template <typename T> struct elem;
template <> struct elem<f16_t> { static constexpr int bytes = 2; using storage = uint16_t; };
template <> struct elem<bf16_t> { static constexpr int bytes = 2; using storage = uint16_t; };
template <> struct elem<e4m3_t> { static constexpr int bytes = 1; using storage = uint8_t; };

// Widen two packed 16-bit values (one 32-bit word) to a float2 (x = low half).
template <typename T> __device__ __forceinline__ float2 widen2(uint32_t w);
template <> __device__ __forceinline__ float2 widen2<bf16_t>(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <> __device__ __forceinline__ float2 widen2<f16_t>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}
// Two e4m3 codes (low 16 bits of w) -> float2, exact (via f16x2).
__device__ __forceinline__ float2 widen2_e4m3(uint32_t w16) {
  __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w16 & 0xffffu), __NV_E4M3);
  __half2 h = *reinterpret_cast<__half2*>(&hr);
  return __half22float2(h);
}

// 16 bytes of cache elements -> 8 (16-bit) or 16 (fp8) floats as float2 pairs.
template <typename T> struct Chunk;
template <> struct Chunk<bf16_t> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void cvt(const uint4& r, float2* o) {
    o[0] = widen2<bf16_t>(r.x); o[1] = widen2<bf16_t>(r.y);
    o[2] = widen2<bf16_t>(r.z); o[3] = widen2<bf16_t>(r.w);
  }
};
template <> struct Chunk<f16_t> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void cvt(const uint4& r, float2* o) {
    o[0] = widen2<f16_t>(r.x); o[1] = widen2<f16_t>(r.y);
    o[2] = widen2<f16_t>(r.z); o[3] = widen2<f16_t>(r.w);
  }
};
template <> struct Chunk<e4m3_t> {
  static constexpr int N = 16;
  __device__ __forceinline__ static void cvt(const uint4& r, float2* o) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = widen2_e4m3(w[i] & 0xffffu);
      o[2 * i + 1] = widen2_e4m3(w[i] >> 16);
    }
  }
};

template <typename T> __device__ __forceinline__ float load_scalar(const void* p, int64_t i);
template <> __device__ __forceinline__ float load_scalar<f16_t>(const void* p, int64_t i) {
  return __half2float(reinterpret_cast<const __half*>(p)[i]);
}
template <> __device__ __forceinline__ float load_scalar<bf16_t>(const void* p, int64_t i) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}

// Store float -> out dtype (round to nearest even).
__device__ __forceinline__ void store_out(void* out, int dtype, int64_t i, float v) {
  if (dtype == PA_F32) {
    reinterpret_cast<float*>(out)[i] = v;
  } else if (dtype == PA_F16) {
    reinterpret_cast<__half*>(out)[i] = __float2half_rn(v);
  } else {
    reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

}  // namespace pa

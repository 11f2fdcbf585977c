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

// Raises the transaction bytes the current phase waits for, without an
// arrival (the arrival comes later, from the same thread).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

// 4-byte asynchronous copy global -> shared (no register destination).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// 16-byte asynchronous copy global -> shared, cached in L2 only (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch.  griddep_wait: returns once the grid this
// one was allowed to overlap (launched just before it on the stream with the
// programmatic-serialization attribute on this one) has finished and its
// writes are visible; returns at once when there is no such grid.
// griddep_launch_dependents: lets a grid launched after this one with that
// attribute start now instead of when this grid's blocks exit.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier among `threads` threads (whole warps) of the CTA on named barrier `id` (1..15).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Prefetch of the 128-byte line holding addr into L2.
__device__ __forceinline__ void prefetch_l2(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
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
struct i8_t {};  // INT8 code with a per-KV-head scale and zero point

template <typename T> struct elem;
template <> struct elem<f16_t> { static constexpr int bytes = 2; using storage = uint16_t; };
template <> struct elem<bf16_t> { static constexpr int bytes = 2; using storage = uint16_t; };
template <> struct elem<e4m3_t> { static constexpr int bytes = 1; using storage = uint8_t; };
template <> struct elem<i8_t> { static constexpr int bytes = 1; using storage = int8_t; };

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

// ----------------------------------------------------------------- tensor-core fragments
//
// mma.sync m16n8k16 with fp32 accumulators.  With g = lane/4 and t = lane%4,
// a thread holds A rows g and g+8 at columns 2t, 2t+1 (a0, a1) and 2t+8,
// 2t+9 (a2, a3); B column g at rows 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1); C
// rows g (c0, c1) and g+8 (c2, c3) at columns 2t, 2t+1.  The lower k index
// sits in the low half of each 32-bit operand register.

template <bool BF16>
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Four 8x8 16-bit matrices; lanes 8i..8i+7 give the row addresses of matrix i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Same, each matrix transposed on the way into registers.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Transpose of an 8x8 matrix of 16-bit elements held in the fragment layout
// (lane (g, t) holds row g, elements 2t and 2t + 1): the result holds the
// transposed matrix in the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr) : "memory");
  return r;
}

// atomic add with release semantics at GPU scope: this thread's earlier
// writes (and those ordered before it by a warp barrier) become visible to
// whoever observes the new value and then acquires (fence_acq_rel_gpu)
__device__ __forceinline__ int atom_add_release_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

// atomic add with acquire-release semantics at GPU scope: as above, and this
// thread's later reads see what the arrivals before it released
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

// Acquire-release fence at GPU scope: after observing values written by
// release operations, this thread's later reads see what they released.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Orders this thread's generic-proxy view of global memory before its later
// async-proxy operations (bulk copies that read global memory).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void st_shared_s32(uint32_t addr, int v) {
  asm volatile("st.shared.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Byte permute: result byte i = byte sel[i] of the 8-byte value {b, a}.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four 8-bit cache codes w (byte i = element i) -> two f16x2 words: elements
// (0, 1) in lo and (2, 3) in hi, low index in the low half, exact.
//  * e4m3: hardware conversion of each 16-bit half (exact: every e4m3 value is an f16).
//  * int8 (value = code - zero point): each code c is placed as the low byte
//    of the f16 pattern 0x64xx after flipping its sign bit, which reads as
//    1024 + (c + 128); subtracting zp2 = f16x2(1152 + zero point) leaves
//    c - zero point.  Every step is exact (integers below 2048).
template <typename T>
__device__ __forceinline__ void widen4(uint32_t w, uint32_t zp2, uint32_t& lo, uint32_t& hi);
template <>
__device__ __forceinline__ void widen4<e4m3_t>(uint32_t w, uint32_t /*zp2*/, uint32_t& lo, uint32_t& hi) {
  // the two byte pairs are the word's 16-bit halves: no masking or shifting
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
template <>
__device__ __forceinline__ void widen4<i8_t>(uint32_t w, uint32_t zp2, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = prmt(u, 0x64646464u, 0x5140u);
  const uint32_t b = prmt(u, 0x64646464u, 0x7362u);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(zp2));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(zp2));
}

// Four INT8 codes -> f16 (1152 + code), exact (an integer below 2048): the
// widening above without its subtraction.  Used for V, whose zero point and
// bias leave the output once, (1152 + zp) * v_scale after the divide by the
// row sum (the product sum and the row sum carry the same weights).
__device__ __forceinline__ void widen4_i8_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = prmt(u, 0x64646464u, 0x5140u);
  hi = prmt(u, 0x64646464u, 0x7362u);
}

// float32 y (= x * inv_scale, already rounded to float32) -> INT8 code:
// nearest integer (ties to even) plus the zero point, saturated to the int8
// range; NaN saturates upward.
__device__ __forceinline__ int int8_code(float y, int zp) {
  if (y != y) return 127;
  const float r = rintf(y) + static_cast<float>(zp);
  return static_cast<int>(fminf(fmaxf(r, -128.f), 127.f));
}

// Two float32 products -> two e4m3 codes (low byte = first), RNE, saturating.
__device__ __forceinline__ uint32_t e4m3x2_code(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// (lo, hi) fp32 -> packed 16-bit pair, round to nearest even; lo in the low half.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t d;
  if constexpr (BF16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  }
  return d;
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
}

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

// Four consecutive outputs from element i (a multiple of 4); one 16-byte (F32)
// or 8-byte (F16/BF16) store when `aligned` (the buffer is 16-byte aligned).
__device__ __forceinline__ void store_out4(void* out, int dtype, int64_t i, float4 v, bool aligned) {
  if (!aligned) {
    store_out(out, dtype, i, v.x);
    store_out(out, dtype, i + 1, v.y);
    store_out(out, dtype, i + 2, v.z);
    store_out(out, dtype, i + 3, v.w);
  } else if (dtype == PA_F32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + i) = v;
  } else if (dtype == PA_F16) {
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(out) + i) = w;
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + i) = w;
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

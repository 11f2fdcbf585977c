// pa_cache.cu - the cache write (reshape_and_cache) and the copy-on-write
// block copy (copy_blocks).
//
// reshape_and_cache follows "KVキャッシュとPagedAttention" (youngju.dev),
// §"PagedAttention: OS仮想メモリ式の管理": blocks are handed out as tokens
// accumulate and each token position maps to a slot of a physical block.
// One warp writes one (token, head, K|V) row: a single coalesced load of the
// source row and a single coalesced store into the cache row.  FP8 caches
// (§"KV量子化: FP8とINT8") quantise float32(x) * inv_scale[h] with
// round-to-nearest-even and saturation to +-448; INT8 caches store
// clamp(rne(float32(x) * inv_scale[h]) + zero_point[h], -128, 127).
//
// copy_blocks follows the PagedAttention explainer (0h-n0.github.io),
// §"Copy-on-Write（CoW）によるメモリ共有": the contents of a shared block are
// copied into a freshly allocated block before the first private write.  Each
// CTA moves a 16 KiB piece of one block of one pool with 16-byte vector
// loads/stores.
#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {

namespace {

enum CacheMode { kCopy = 0, kToFp8 = 1, kToInt8 = 2 };

template <typename SRC, int MODE, int D>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const void* __restrict__ k, const void* __restrict__ v, int64_t k_stride, int64_t v_stride,
    void* __restrict__ k_cache, void* __restrict__ v_cache, int64_t num_blocks,
    const int64_t* __restrict__ slot_mapping, int num_tokens, int num_kv_heads, int block_size,
    const float* __restrict__ k_inv_scale, const float* __restrict__ v_inv_scale,
    const int32_t* __restrict__ k_zero_point, const int32_t* __restrict__ v_zero_point, unsigned int* err) {
  constexpr int EPL = D / 32;  // elements per lane: 2 or 4
  // A decode launched after this write with programmatic serialization may
  // start its set-up now (it waits for this grid before it reads the cache).
  // Under a programmatic dependent launch of this write, nothing is read or
  // written before the kernel before it on the stream has finished (an
  // ordinary launch returns at once).
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads * 2;
  if (row >= rows) return;
  const int which = static_cast<int>(row & 1);  // 0 = K, 1 = V
  const int64_t th = row >> 1;
  const int h = static_cast<int>(th % num_kv_heads);
  const int64_t n = th / num_kv_heads;

  const void* src = which ? v : k;
  const int64_t src_elem = n * (which ? v_stride : k_stride) + static_cast<int64_t>(h) * D + lane * EPL;
  // The source row (and the quantisation constants) do not depend on the
  // slot: all of them are loaded before the slot is examined, so the row
  // costs one memory round trip, not two (the step's decode waits for it).
  const int64_t slot = slot_mapping[n];
  uint32_t raw[EPL / 2];  // kCopy: the row's 16-bit values as they are
  float x[EPL];           // quantising modes: float32(value) * inv_scale
  int zp = 0;
  if constexpr (MODE == kCopy) {
    if constexpr (EPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(src) + src_elem);
      raw[0] = w.x;
      raw[1] = w.y;
    } else {
      raw[0] = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(src) + src_elem);
    }
  } else {
    const float inv = (which ? v_inv_scale : k_inv_scale)[h];
    if constexpr (MODE == kToInt8) zp = (which ? v_zero_point : k_zero_point)[h];
#pragma unroll
    for (int i = 0; i < EPL; ++i) x[i] = __fmul_rn(load_scalar<SRC>(src, src_elem + i), inv);
  }
  if (slot < 0) return;  // padding token
  if (slot >= num_blocks * block_size) {
    if (lane == 0) raise_error(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / block_size;
  const int64_t off = slot - blk * block_size;
  const int64_t dst_elem = ((blk * num_kv_heads + h) * block_size + off) * D + lane * EPL;
  void* cache = which ? v_cache : k_cache;

  if constexpr (MODE == kCopy) {
    if constexpr (EPL == 4) {
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(cache) + dst_elem) = make_uint2(raw[0], raw[1]);
    } else {
      *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(cache) + dst_elem) = raw[0];
    }
  } else if constexpr (MODE == kToInt8) {
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int c = int8_code(x[i], zp);
      packed |= (static_cast<uint32_t>(c) & 0xffu) << (8 * i);
    }
    uint8_t* dst = static_cast<uint8_t*>(cache) + dst_elem;
    if constexpr (EPL == 4) {
      *reinterpret_cast<uint32_t*>(dst) = packed;
    } else {
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
    }
  } else {
    uint8_t* dst = static_cast<uint8_t*>(cache) + dst_elem;
    if constexpr (EPL == 4) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[0], x[1]), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x[2], x[3]), __NV_SATFINITE, __NV_E4M3);
      *reinterpret_cast<uint32_t*>(dst) = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    } else {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[0], x[1]), __NV_SATFINITE, __NV_E4M3);
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(lo);
    }
  }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyBytesPerCta = 16384;  // 256 threads x 16 B x 4

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, int64_t num_blocks,
    int64_t block_bytes, const int32_t* __restrict__ pairs, unsigned int* err) {
  griddep_launch_dependents();  // as in the cache write: dependents wait before reading the pools
  const int pair = blockIdx.y;
  const int32_t src = pairs[2 * pair];
  const int32_t dst = pairs[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) raise_error(err, PA_DEVERR_PAIR);
    return;
  }
  uint8_t* base = blockIdx.z ? v_cache : k_cache;
  const uint4* s = reinterpret_cast<const uint4*>(base + static_cast<int64_t>(src) * block_bytes);
  uint4* d = reinterpret_cast<uint4*>(base + static_cast<int64_t>(dst) * block_bytes);
  const int64_t n16 = block_bytes >> 4;
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * (kCopyBytesPerCta >> 4);
  const int64_t end = min(n16, begin + (kCopyBytesPerCta >> 4));
  uint4 buf[4];
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t idx = begin + threadIdx.x + static_cast<int64_t>(i) * kCopyThreads;
    if (idx < end) { buf[i] = s[idx]; cnt = i + 1; }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t idx = begin + threadIdx.x + static_cast<int64_t>(i) * kCopyThreads;
    if (i < cnt && idx < end) d[idx] = buf[i];
  }
}

}  // namespace

// One cache-write launch, optionally with programmatic stream serialisation.
template <typename... KArgs, typename... Args>
cudaError_t launch_rc(void (*kern)(KArgs...), unsigned grid, bool pdl, cudaStream_t stream, Args... args) {
  if (!pdl) {
    kern<<<grid, 256, 0, stream>>>(args...);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.num_tokens) * a.num_kv_heads * 2;
  if (rows == 0) return cudaSuccess;
  const int warps_per_cta = 8;
  const int64_t grid = (rows + warps_per_cta - 1) / warps_per_cta;
#define PA_RC_LAUNCH(SRC, MODE, D)                                                                    \
  le = launch_rc(reshape_and_cache_kernel<SRC, MODE, D>, static_cast<unsigned>(grid), a.pdl, stream, a.k, a.v, \
            a.k_stride, a.v_stride, a.k_cache, a.v_cache, a.num_blocks, a.slot_mapping, a.num_tokens,        \
            a.num_kv_heads, a.block_size, a.k_inv_scale, a.v_inv_scale, a.k_zero_point, a.v_zero_point, a.err)
#define PA_RC_D(SRC, MODE) \
  if (a.head_dim == 128) PA_RC_LAUNCH(SRC, MODE, 128); else PA_RC_LAUNCH(SRC, MODE, 64);
  const int mode = a.kv_dtype == PA_FP8_E4M3 ? kToFp8 : (a.kv_dtype == PA_INT8 ? kToInt8 : kCopy);
  (void)cudaGetLastError();
  cudaError_t le = cudaSuccess;
  if (a.src_dtype == PA_F16) {
    if (mode == kToFp8) { PA_RC_D(f16_t, kToFp8) } else if (mode == kToInt8) { PA_RC_D(f16_t, kToInt8) }
    else { PA_RC_D(f16_t, kCopy) }
  } else {
    if (mode == kToFp8) { PA_RC_D(bf16_t, kToFp8) } else if (mode == kToInt8) { PA_RC_D(bf16_t, kToInt8) }
    else { PA_RC_D(bf16_t, kCopy) }
  }
#undef PA_RC_D
#undef PA_RC_LAUNCH
  return le;
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks, int64_t block_bytes,
                               const int32_t* pairs, int num_pairs, unsigned int* err, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t chunks = (block_bytes + kCopyBytesPerCta - 1) / kCopyBytesPerCta;
  dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(num_pairs), 2);
  (void)cudaGetLastError();
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(static_cast<uint8_t*>(k_cache),
                                                         static_cast<uint8_t*>(v_cache), num_blocks,
                                                         block_bytes, pairs, err);
  return cudaGetLastError();
}

}  // namespace pa

// pa_decode_dispatch.cu - maps a runtime DecodeKey to its compiled variant.
#include "pa_decode_variants.h"

#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>
#include <unordered_map>

namespace pa {

int tuning_override(const char* name) {
  static std::mutex mu;
  static std::unordered_map<std::string, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(name);
  if (it != cache.end()) return it->second;
  const char* v = std::getenv(name);
  const int x = v ? std::atoi(v) : -1;
  cache.emplace(name, x);
  return x;
}

namespace {
thread_local char g_launch_note[256] = "";
}

void note_launch_failure(int ctas, int threads, size_t smem, int stages, int max_threads, int max_dyn_smem,
                         int regs, size_t local_bytes) {
  snprintf(g_launch_note, sizeof(g_launch_note),
           "grid %d x %d threads, dyn smem %zu, stages %d; kernel: max threads %d, max dyn smem %d, regs %d, "
           "local %zu",
           ctas, threads, smem, stages, max_threads, max_dyn_smem, regs, local_bytes);
}

const char* launch_failure_note() { return g_launch_note; }


template <typename T> constexpr int dtype_code();
template <> constexpr int dtype_code<f16_t>() { return PA_F16; }
template <> constexpr int dtype_code<bf16_t>() { return PA_BF16; }
template <> constexpr int dtype_code<e4m3_t>() { return PA_FP8_E4M3; }
template <> constexpr int dtype_code<i8_t>() { return PA_INT8; }

#define PA_MATCH(QT, KVT, D, GM, UR, AP)                                                                   \
  (key.q_dtype == dtype_code<QT>() && key.kv_dtype == dtype_code<KVT>() && key.head_dim == D && key.gmax == GM && \
   key.unit_rows == UR && key.append == AP)

namespace {
bool compute_geometry(const DecodeKey& key, int num_seqs, DecodeGeometry* geo) {
#define PA_GEO(QT, KVT, D, GM, UR, AP) \
  if (PA_MATCH(QT, KVT, D, GM, UR, AP))                                                                            \
    return decode_geometry_##QT##_##KVT##_##D##_##GM##_##UR##_##AP(num_seqs, key.row_groups, geo);
  PA_DECODE_VARIANTS(PA_GEO)
#undef PA_GEO
  return false;
}
}  // namespace

// The geometry depends only on the device, the variant and the batch size
// (the prologue's per-sequence arrays live in shared memory), so it is
// computed once per combination: the occupancy queries cost far more host
// time than a small decode launch.
bool decode_geometry(const DecodeKey& key, int num_seqs, DecodeGeometry* geo) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t k = (static_cast<uint64_t>(dev & 0xff) << 56) | (static_cast<uint64_t>(key.q_dtype & 0xf) << 52) |
                     (static_cast<uint64_t>(key.kv_dtype & 0xf) << 48) |
                     (static_cast<uint64_t>(key.head_dim & 0xfff) << 36) |
                     (static_cast<uint64_t>(key.gmax & 0xf) << 32) | (static_cast<uint64_t>(key.unit_rows & 0xff) << 24) |
                     (static_cast<uint64_t>(key.append & 1) << 23) | (static_cast<uint64_t>(key.row_groups & 7) << 20) |
                     static_cast<uint64_t>(num_seqs & 0xfffff);
  static std::mutex mu;
  static std::unordered_map<uint64_t, DecodeGeometry> cache;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(k);
    if (it != cache.end()) {
      *geo = it->second;
      return true;
    }
  }
  if (!compute_geometry(key, num_seqs, geo)) return false;
  std::lock_guard<std::mutex> lock(mu);
  cache.emplace(k, *geo);
  return true;
}

cudaError_t launch_decode(const DecodeKey& key, const DecodeGeometry& geo, const DecodeParams& p,
                          const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream, bool pdl) {
#define PA_LAUNCH(QT, KVT, D, GM, UR, AP) \
  if (PA_MATCH(QT, KVT, D, GM, UR, AP))    \
    return decode_launch_##QT##_##KVT##_##D##_##GM##_##UR##_##AP(geo, p, tk, tv, stream, pdl);
  PA_DECODE_VARIANTS(PA_LAUNCH)
#undef PA_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace pa

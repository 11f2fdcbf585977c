// pa_api.cu - the extern "C" entry points declared in include/pa.h: argument
// validation, TMA descriptor encoding, workspace accounting and dispatch to
// the kernels.  No call here allocates device memory.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pa_common.cuh"
#include "pa_kernels.h"

#define PA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// Per-device error word (PA_DEVERR_* bits).  Kernels receive its address.
__device__ unsigned int g_device_error = 0u;

constexpr int kMaxDevices = 64;

// Device address of g_device_error on the current device (nullptr on failure).
unsigned int* device_error_word() {
  static unsigned int* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned int*>(p);
  }
  return addr[dev];
}

// Text of the last CUDA error a call on this thread returned PA_ERR_CUDA for.
thread_local char g_last_error[512] = "";

int cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return PA_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
  return PA_ERR_CUDA;
}

constexpr int kMaxSeqs = 16384;  // prefix sums of the batch live in shared memory
constexpr int kMaxQueryRows = 64;  // q_len * G: up to four 16-row consumer warps share a ring

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int dtype_bytes(int dt) {
  switch (dt) {
    case PA_F32: return 4;
    case PA_F16: return 2;
    case PA_BF16: return 2;
    case PA_FP8_E4M3: return 1;
    case PA_INT8: return 1;
    default: return 0;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D view of a cache pool: {128 bytes of a row, rows, 128-byte halves of a
// row}, with num_blocks*Hkv*B rows of head_dim elements.  One TMA box =
// box_rows whole rows with the 128-byte swizzle, landing in shared memory as
// [half][row][128 bytes], so that each half-plane is swizzled by row.
bool encode_cache_map(CUtensorMap* map, const void* cache, int64_t num_blocks, int num_kv_heads,
                      int block_size, int head_dim, int elem_bytes, int box_rows) {
  if (box_rows % pa::kBoxRowQuantum != 0 || box_rows > 256) return false;
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int row_bytes = head_dim * elem_bytes;
  if (row_bytes % 128 != 0) return false;
  const cuuint32_t half_elems = static_cast<cuuint32_t>(128 / elem_bytes);
  const cuuint32_t halves = static_cast<cuuint32_t>(row_bytes / 128);
  cuuint64_t dims[3] = {half_elems, static_cast<cuuint64_t>(num_blocks) * num_kv_heads * block_size, halves};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), 128};
  cuuint32_t box[3] = {half_elems, static_cast<cuuint32_t>(box_rows), halves};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
                         const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Compiled maximum of A rows (q_len * G (query, head) pairs) serving `rows`.
int gmax_for_rows(int rows) { return rows <= 1 ? 1 : (rows <= 4 ? 4 : (rows <= 8 ? 8 : 16)); }

// Rows per work unit: 32 for 16-bit caches (16 KB of K + V per stage at
// d = 128), 64 for 8-bit caches with B >= 16 (the same 16 KB per stage, half
// the refills per byte of 32 rows).  A unit spans at most four blocks, so
// 64-row units need B >= 16.  Several queries per sequence (16 rows per
// consumer warp, nc warps sharing a ring, the query rows in one buffer per
// ring): 32-row units (measured on the GB300 at d = 128 against 16-row
// units: 32 rows per KV head on 8 x 32K tokens 227 -> 208 us, on the 32 x 4K
// GQA batch 84 -> 77 us).  PA_DECODE_UNIT_ROWS (32; 64 for 8-bit caches with
// B >= 16) overrides it (tuning).
int unit_rows_for(int kv_dtype, int block_size, int gmax, bool append) {
  const bool q8 = kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_INT8;  // 8-bit cache
  const int env = append ? -1 : pa::tuning_override("PA_DECODE_UNIT_ROWS");  // fused append: defaults only
  if (env == 32) return env;
  if (env == 64 && q8 && block_size >= 16 && gmax <= 8) return 64;
  if (gmax > 8) return 32;
  return q8 && block_size >= 16 ? 64 : 32;
}

// Shape checks shared by pa_decode and pa_decode_workspace_bytes.
int check_decode_shape(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                       int max_blocks_per_seq, int partition_size, int kv_dtype) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
  if (num_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  if (num_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if ((kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_INT8) && (head_dim != 128 || num_kv_heads > pa::kMaxHeadParams))
    return PA_ERR_UNSUPPORTED;
  // a power of two from 8 to 1024: a work unit (16, 32 or 64 rows) then covers
  // whole blocks or a whole fraction of one
  if (block_size < 8 || block_size > 1024 || (block_size & (block_size - 1)) != 0) return PA_ERR_UNSUPPORTED;
  if (partition_size < 0 || (partition_size > 0 && partition_size % block_size != 0)) return PA_ERR_SHAPE;
  if (num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_seqs) * num_kv_heads * max_blocks_per_seq * block_size / 8 >= (int64_t{1} << 31))
    return PA_ERR_SHAPE;
  return PA_OK;
}

struct DecodePlan {
  pa::DecodeKey key;
  pa::DecodeGeometry geo;
  int partition_units;      // as passed to the kernel (0 = balanced), in 8-row units
  size_t counters_bytes;
  size_t records;
  int pending_cap;          // segments one consumer warp may have to merge
  size_t pending_offset;    // bytes from the workspace start to the pending lists
  size_t bytes;             // total workspace bytes required
};

// Resolves the variant, launch geometry and workspace need.  `have_ws` tells
// whether the caller supplied a workspace (balanced mode needs one).
int make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
              int partition_size, int q_dtype, int kv_dtype, bool have_ws, DecodePlan* plan, bool append = false,
              int q_len = 1) {
  plan->key.append = append ? 1 : 0;
  plan->key.q_dtype = q_dtype;
  plan->key.kv_dtype = kv_dtype;
  plan->key.head_dim = head_dim;
  // several queries per sequence are served by the 16-row variants only, 16
  // rows per consumer warp: ceil(q_len * G / 16) warps share a ring
  plan->key.gmax = q_len > 1 ? 16 : gmax_for_rows(num_heads / num_kv_heads);
  const int rows = q_len * (num_heads / num_kv_heads);
  plan->key.row_groups = q_len > 1 ? (rows + 15) / 16 : 1;
  plan->key.unit_rows = unit_rows_for(kv_dtype, block_size, plan->key.gmax, append);
  if (!pa::decode_geometry(plan->key, num_seqs, &plan->geo)) return PA_ERR_UNSUPPORTED;
  const int ur = plan->geo.unit_rows;
  const int max_units = static_cast<int>((static_cast<int64_t>(max_blocks_per_seq) * block_size + ur - 1) / ur);
  int pu = (partition_size + ur - 1) / ur;  // fixed partitions rounded up to whole units
  if (partition_size == 0 && !have_ws) pu = max_units;  // single pass without workspace
  if (pu >= max_units) pu = max_units;
  plan->partition_units = pu;
  if (pu == max_units) {  // one fragment per segment: no partial records
    plan->counters_bytes = 0;
    plan->records = 0;
    plan->pending_cap = 0;
    plan->pending_offset = 0;
    plan->bytes = 0;
    return PA_OK;
  }
  // arrival counters and records are per (segment, row group of its ring)
  const int nc = plan->geo.row_groups;
  plan->counters_bytes = (static_cast<size_t>(num_seqs) * num_kv_heads * nc * sizeof(int) + 255) / 256 * 256;
  const size_t warps = static_cast<size_t>(plan->geo.ctas) * plan->geo.warps_per_cta;
  const size_t rings = warps / nc;
  if (pu == 0) {
    // balanced split: only the first and the last fragment of a ring's range
    // can be part of a split segment
    plan->records = 2 * warps;
    plan->pending_cap = 2;
  } else {
    // fixed partitions: dealt round-robin over the rings
    const size_t parts = static_cast<size_t>(num_seqs) * num_kv_heads * ((max_units + pu - 1) / pu);
    plan->records = parts * nc;
    plan->pending_cap = static_cast<int>((parts + rings - 1) / rings);
  }
  plan->pending_offset = plan->counters_bytes + (plan->records * plan->geo.record_floats * sizeof(float) + 255) / 256 * 256;
  plan->bytes = plan->pending_offset + warps * plan->pending_cap * sizeof(int);
  return PA_OK;
}

}  // namespace

PA_EXPORT int pa_version(void) { return 100; }

PA_EXPORT const char* pa_last_error_detail(void) { return g_last_error; }

PA_EXPORT const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: inconsistent or out-of-range sizes";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE: dtype combination not accepted";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: outside the compiled variants";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime or launch failure";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: pointer or stride not 16-byte aligned";
    default: return "unknown pa_status";
  }
}

PA_EXPORT size_t pa_decode_workspace_bytes_ex(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                              int block_size, int max_blocks_per_seq, int partition_size,
                                              pa_dtype kv_dtype, const pa_decode_options* opt) {
  pa_decode_options o;
  memset(&o, 0, sizeof(o));
  if (opt) {
    if (opt->struct_size < sizeof(size_t)) return static_cast<size_t>(-1);
    memcpy(&o, opt, opt->struct_size < sizeof(o) ? opt->struct_size : sizeof(o));
  }
  const int q_len = o.q_len <= 0 ? 1 : o.q_len;
  if (num_kv_heads > 0 && q_len * (num_heads / num_kv_heads) > kMaxQueryRows) return static_cast<size_t>(-1);
  if (check_decode_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                         partition_size, kv_dtype) != PA_OK)
    return static_cast<size_t>(-1);
  const int q_dtype = (kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_INT8) ? PA_BF16 : kv_dtype;
  if (q_dtype != PA_F16 && q_dtype != PA_BF16) return static_cast<size_t>(-1);
  DecodePlan plan;
  if (make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, partition_size, q_dtype,
                kv_dtype, true, &plan, false, q_len) != PA_OK)
    return static_cast<size_t>(-1);
  return plan.bytes;
}

PA_EXPORT size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                           int block_size, int max_blocks_per_seq, int partition_size,
                                           pa_dtype kv_dtype) {
  return pa_decode_workspace_bytes_ex(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                      partition_size, kv_dtype, nullptr);
}

PA_EXPORT int pa_decode_launch_config(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                      int max_blocks_per_seq, int partition_size, pa_dtype q_dtype,
                                      pa_dtype kv_dtype, int* ctas, int* warps_per_cta, int* stages,
                                      size_t* smem_bytes) {
  const int sh = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                    partition_size, kv_dtype);
  if (sh != PA_OK) return sh;
  if (!ctas || !warps_per_cta || !stages || !smem_bytes) return PA_ERR_NULL;
  if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_DTYPE;
  if (kv_dtype != q_dtype && kv_dtype != PA_FP8_E4M3 && kv_dtype != PA_INT8) return PA_ERR_DTYPE;
  DecodePlan plan;
  const int pr = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                           partition_size, q_dtype, kv_dtype, true, &plan);
  if (pr != PA_OK) return pr;
  *ctas = plan.geo.ctas;
  *warps_per_cta = plan.geo.warps_per_cta;
  *stages = plan.geo.stages;
  *smem_bytes = plan.geo.smem_bytes;
  return PA_OK;
}

namespace {

// Wait limit and copy withholding of the next decode launches (testing hook,
// pa_debug_set_decode_wait); 0 = the default limit.
std::atomic<uint64_t> g_wait_limit_ns{0};
std::atomic<int> g_withhold_copies{0};

// Everything one decode launch needs, validated: the plan, the kernel
// parameters and the two tensor maps.  Filling it enqueues nothing.
struct PreparedDecode {
  DecodePlan plan;
  pa::DecodeParams p;
  CUtensorMap tk, tv;
  bool pdl;
  bool empty;  // num_seqs == 0: nothing to launch
};

// All host-side checks of pa_decode_ex, then the launch plan, parameters and
// tensor maps.  Returns a pa_status; nothing is enqueued on any stream.
int prepare_decode(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype, int64_t q_stride,
                   const void* k_cache, const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                   const float* k_scale, const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* seq_lens, int num_seqs, int num_heads, int num_kv_heads, int head_dim, float scale,
                   int block_size, int partition_size, void* workspace, size_t workspace_bytes,
                   const pa_decode_options* opt, PreparedDecode* d) {
  d->empty = false;
  // options: fields beyond the caller's struct_size read as 0
  pa_decode_options o;
  memset(&o, 0, sizeof(o));
  if (opt) {
    if (opt->struct_size < sizeof(size_t)) return PA_ERR_SHAPE;
    memcpy(&o, opt, opt->struct_size < sizeof(o) ? opt->struct_size : sizeof(o));
  }
  if (o.window < 0 || o.q_len < 0) return PA_ERR_SHAPE;
  const int q_len = o.q_len == 0 ? 1 : o.q_len;
  if (num_kv_heads > 0 && q_len * (num_heads / num_kv_heads) > kMaxQueryRows) return PA_ERR_UNSUPPORTED;
  const bool append = o.k_new != nullptr || o.v_new != nullptr;
  if (append && q_len != 1) return PA_ERR_UNSUPPORTED;
  if (append) {
    if (!o.k_new || !o.v_new) return PA_ERR_NULL;
    if (o.new_dtype != PA_F16 && o.new_dtype != PA_BF16) return PA_ERR_DTYPE;
    const bool q8 = kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_INT8;
    if (!q8 && o.new_dtype != kv_dtype) return PA_ERR_DTYPE;
    if (q8 && (!o.k_inv_scale || !o.v_inv_scale)) return PA_ERR_NULL;
    if (o.new_stride < static_cast<int64_t>(num_kv_heads) * head_dim) return PA_ERR_SHAPE;
    if (!aligned16(o.k_new) || !aligned16(o.v_new) || (o.new_stride * 2) % 16 != 0) return PA_ERR_ALIGN;
  }
  const int sh = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                    partition_size, kv_dtype);
  if (sh != PA_OK) return sh;
  if (num_seqs == 0) {
    d->empty = true;
    return PA_OK;
  }
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_NULL;
  if (out_dtype != PA_F32 && out_dtype != PA_F16 && out_dtype != PA_BF16) return PA_ERR_DTYPE;
  if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_DTYPE;
  if (kv_dtype != q_dtype && kv_dtype != PA_FP8_E4M3 && kv_dtype != PA_INT8) return PA_ERR_DTYPE;
  if ((kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_INT8) && (!k_scale || !v_scale)) return PA_ERR_NULL;
  if (kv_dtype == PA_INT8 && (!o.k_zero_point || !o.v_zero_point)) return PA_ERR_NULL;
  if (num_blocks <= 0 || num_blocks * num_kv_heads * block_size >= (int64_t{1} << 31)) return PA_ERR_SHAPE;
  if (q_stride < static_cast<int64_t>(q_len) * num_heads * head_dim) return PA_ERR_SHAPE;
  if (!aligned16(q) || (q_stride * 2) % 16 != 0 || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;

  DecodePlan& plan = d->plan;
  const bool have_ws = workspace != nullptr && workspace_bytes > 0;
  const int pr = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                           partition_size, q_dtype, kv_dtype, have_ws, &plan, append, q_len);
  if (pr != PA_OK) return pr;
  if (plan.bytes > 0 && (!have_ws || workspace_bytes < plan.bytes || !aligned16(workspace))) return PA_ERR_WORKSPACE;

  const int eb = dtype_bytes(kv_dtype);
  const int box_rows = block_size < plan.geo.unit_rows ? block_size : plan.geo.unit_rows;
  if (!encode_cache_map(&d->tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim, eb, box_rows) ||
      !encode_cache_map(&d->tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim, eb, box_rows))
    return PA_ERR_CUDA;

  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  pa::DecodeParams& p = d->p;
  p.err = err;
  p.out = out;
  p.out_dtype = out_dtype;
  p.q = q;
  p.q_stride = q_stride;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.k_zero_point = o.k_zero_point;
  p.v_zero_point = o.v_zero_point;
  p.block_tables = block_tables;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.seq_lens = seq_lens;
  p.num_blocks = num_blocks;
  p.num_seqs = num_seqs;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  p.block_size = block_size;
  p.block_shift = __builtin_ctz(static_cast<unsigned>(block_size));
  p.partition_units = plan.partition_units;
  // Balanced split: every fragment (one ring's share of one segment) is
  // charged frag_cost units of work besides its own units (query set-up, the
  // masked last unit, the output or the record).  Measured per ring on the
  // GB300 with the plain split, a fragment cost 3.2 us against 1.6 us per unit
  // for FP8 (64-row units), 4.9 against 2.3 for INT8 and 1.1 against 0.9 for
  // bf16 (32-row units); charges of 0..4 units timed on the three mixes gave
  // their best at 2..3, so every cache type is charged 3.
  // PA_DECODE_FRAG_COST overrides it (tuning).
  {
    const int env = pa::tuning_override("PA_DECODE_FRAG_COST");
    p.frag_cost = plan.partition_units != 0 ? 0 : (env >= 0 && env <= 64 ? env : 3);
  }
  p.window = o.window;
  p.q_len = q_len;
  p.k_new = append ? o.k_new : nullptr;
  p.v_new = append ? o.v_new : nullptr;
  p.new_stride = o.new_stride;
  p.new_dtype = o.new_dtype;
  p.k_inv_scale = o.k_inv_scale;
  p.v_inv_scale = o.v_inv_scale;
  p.k_cache = const_cast<void*>(k_cache);
  p.v_cache = const_cast<void*>(v_cache);
  p.stages = plan.geo.stages;
  p.row_groups = plan.geo.row_groups;
  p.stage_bytes = plan.geo.stage_bytes;
  p.seg_counters = plan.bytes ? static_cast<int*>(workspace) : nullptr;
  p.pending = plan.bytes ? reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + plan.pending_offset) : nullptr;
  p.pending_cap = plan.pending_cap;
  p.part_records = plan.bytes ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.counters_bytes)
                              : nullptr;
  const uint64_t lim = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.wait_limit_ns = lim ? lim : pa::kDefaultWaitLimitNs;
  p.withhold_copies = g_withhold_copies.load(std::memory_order_relaxed);
  p.early_kv = (o.early_kv != 0 && o.pdl != 0 && q_len == 1 && !append) ? 1 : 0;
  d->pdl = o.pdl != 0;
  return PA_OK;
}

int launch_prepared(const PreparedDecode& d, void* stream) {
  const int st = cuda_status(pa::launch_decode(d.plan.key, d.plan.geo, d.p, d.tk, d.tv,
                                              static_cast<cudaStream_t>(stream), d.pdl),
                              "pa_decode launch");
  if (st != PA_OK) {
    const size_t n = strlen(g_last_error);
    snprintf(g_last_error + n, sizeof(g_last_error) - n, "; %s", pa::launch_failure_note());
  }
  return st;
}

}  // namespace

PA_EXPORT int pa_decode_ex(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype, int64_t q_stride,
                           const void* k_cache, const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                           const float* k_scale, const float* v_scale, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, float scale, int block_size, int partition_size,
                           void* workspace, size_t workspace_bytes, const pa_decode_options* opt, void* stream) {
  PreparedDecode d;
  const int st = prepare_decode(out, out_dtype, q, q_dtype, q_stride, k_cache, v_cache, kv_dtype, num_blocks, k_scale,
                                v_scale, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_heads,
                                num_kv_heads, head_dim, scale, block_size, partition_size, workspace, workspace_bytes,
                                opt, &d);
  if (st != PA_OK || d.empty) return st;
  return launch_prepared(d, stream);
}

PA_EXPORT void pa_debug_set_decode_wait(uint64_t limit_ns, int withhold_copies) {
  g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
  g_withhold_copies.store(withhold_copies ? 1 : 0, std::memory_order_relaxed);
}

PA_EXPORT int pa_decode(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype, int64_t q_stride,
                        const void* k_cache, const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_heads,
                        int num_kv_heads, int head_dim, float scale, int block_size, int partition_size,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return pa_decode_ex(out, out_dtype, q, q_dtype, q_stride, k_cache, v_cache, kv_dtype, num_blocks, k_scale, v_scale,
                      block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_heads, num_kv_heads, head_dim, scale,
                      block_size, partition_size, workspace, workspace_bytes, nullptr, stream);
}

PA_EXPORT int pa_reshape_and_cache_ex(const void* k, const void* v, pa_dtype src_dtype, int64_t k_stride,
                                      int64_t v_stride, void* k_cache, void* v_cache, pa_dtype kv_dtype,
                                      int64_t num_blocks, const int64_t* slot_mapping, int num_tokens,
                                      int num_kv_heads, int head_dim, int block_size, const float* k_inv_scale,
                                      const float* v_inv_scale, const pa_cache_write_options* opt, void* stream) {
  pa_cache_write_options o;
  memset(&o, 0, sizeof(o));
  if (opt) {
    if (opt->struct_size < sizeof(size_t)) return PA_ERR_SHAPE;
    memcpy(&o, opt, opt->struct_size < sizeof(o) ? opt->struct_size : sizeof(o));
  }
  if (num_tokens < 0 || num_kv_heads <= 0 || block_size <= 0 || num_blocks <= 0) return PA_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_NULL;
  if (src_dtype != PA_F16 && src_dtype != PA_BF16) return PA_ERR_DTYPE;
  const bool quant = kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_INT8;
  if (kv_dtype != src_dtype && !quant) return PA_ERR_DTYPE;
  if (quant && (!k_inv_scale || !v_inv_scale)) return PA_ERR_NULL;
  if (kv_dtype == PA_INT8 && (!o.k_zero_point || !o.v_zero_point)) return PA_ERR_NULL;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (k_stride < row || v_stride < row) return PA_ERR_SHAPE;
  if (!aligned16(k) || !aligned16(v) || (k_stride * 2) % 16 != 0 || (v_stride * 2) % 16 != 0 ||
      !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_ALIGN;
  if (static_cast<int64_t>(num_tokens) * num_kv_heads * 2 / 8 >= (int64_t{1} << 31)) return PA_ERR_SHAPE;
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  pa::ReshapeArgs a;
  a.err = err;
  a.k = k;
  a.v = v;
  a.src_dtype = src_dtype;
  a.k_stride = k_stride;
  a.v_stride = v_stride;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.kv_dtype = kv_dtype;
  a.num_blocks = num_blocks;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.k_inv_scale = k_inv_scale;
  a.v_inv_scale = v_inv_scale;
  a.k_zero_point = o.k_zero_point;
  a.v_zero_point = o.v_zero_point;
  a.pdl = o.pdl != 0;
  return cuda_status(pa::launch_reshape_and_cache(a, static_cast<cudaStream_t>(stream)),
                     "pa_reshape_and_cache launch");
}

PA_EXPORT int pa_reshape_and_cache(const void* k, const void* v, pa_dtype src_dtype, int64_t k_stride,
                                   int64_t v_stride, void* k_cache, void* v_cache, pa_dtype kv_dtype,
                                   int64_t num_blocks, const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                   int head_dim, int block_size, const float* k_inv_scale,
                                   const float* v_inv_scale, void* stream) {
  return pa_reshape_and_cache_ex(k, v, src_dtype, k_stride, v_stride, k_cache, v_cache, kv_dtype, num_blocks,
                                 slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, k_inv_scale,
                                 v_inv_scale, nullptr, stream);
}

PA_EXPORT int pa_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks, size_t block_bytes,
                             const int32_t* src_dst_pairs, int num_pairs, void* stream) {
  if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0) return PA_ERR_SHAPE;
  if (num_pairs > 65535) return PA_ERR_UNSUPPORTED;
  if (block_bytes % 16 != 0) return PA_ERR_ALIGN;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_dst_pairs) return PA_ERR_NULL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  return cuda_status(pa::launch_copy_blocks(k_cache, v_cache, num_blocks, static_cast<int64_t>(block_bytes),
                                            src_dst_pairs, num_pairs, err, static_cast<cudaStream_t>(stream)),
                     "pa_copy_blocks launch");
}

PA_EXPORT int pa_get_device_error(void* stream, unsigned int* error_bits) {
  if (!error_bits) return PA_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int h = 0u;
  if (cudaMemcpyFromSymbolAsync(&h, g_device_error, sizeof(h), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  const unsigned int zero = 0u;
  if (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  *error_bits = h;
  return PA_OK;
}

// ----------------------------------------------------------------- allocation-free decode
//
// Some callers cannot allocate device memory at decode time: code that runs
// where cudaMalloc is not allowed or would stall (inside a real-time serving
// loop that must not touch the allocator, in a process whose memory pool is
// owned and locked by another framework, or in a plugin that only receives
// its input and output buffers).  For them pa_decode_noalloc keeps the split
// workspace in a fixed array that the library itself defines in device
// memory, so the caller passes only inputs and outputs.

namespace {

// Device memory for the split records and arrival counters of
// pa_decode_noalloc.  Every device that loads the library holds this array
// until the process exits.  Host code must not use its name as an address:
// the device address is looked up per device (noalloc_scratch_address).
constexpr size_t kNoallocScratchBytes = size_t{16} << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.  nullptr if the lookup fails.
void* noalloc_scratch_address() {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      cuda_status(e, "pa_decode_noalloc scratch lookup");
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

PA_EXPORT size_t pa_decode_noalloc_capacity(void) { return kNoallocScratchBytes; }

PA_EXPORT int pa_decode_noalloc(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype, int64_t q_stride,
                                const void* k_cache, const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                                const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, float scale, int block_size, int partition_size,
                                void* stream) {
  const int sh = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                    partition_size, kv_dtype);
  if (sh != PA_OK) return sh;
  // INT8 caches need zero points, which this entry point has no arguments for
  if (kv_dtype == PA_INT8) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  void* scratch = noalloc_scratch_address();
  if (!scratch) return PA_ERR_CUDA;
  // every check of pa_decode first: a rejected call enqueues nothing
  PreparedDecode d;
  const int st = prepare_decode(out, out_dtype, q, q_dtype, q_stride, k_cache, v_cache, kv_dtype, num_blocks, k_scale,
                                v_scale, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_heads,
                                num_kv_heads, head_dim, scale, block_size, partition_size, scratch,
                                kNoallocScratchBytes, nullptr, &d);
  if (st == PA_ERR_WORKSPACE && d.plan.bytes > kNoallocScratchBytes) {
    snprintf(g_last_error, sizeof(g_last_error),
             "pa_decode_noalloc: this call needs %zu bytes of split workspace, more than the fixed %zu",
             d.plan.bytes, kNoallocScratchBytes);
  }
  if (st != PA_OK || d.empty) return st;
  // the arrival counters must start at zero; the records need no clearing
  if (d.plan.counters_bytes > 0) {
    const int ms = cuda_status(
        cudaMemsetAsync(scratch, 0, d.plan.counters_bytes, static_cast<cudaStream_t>(stream)), "pa_decode_noalloc memset");
    if (ms != PA_OK) return ms;
  }
  return launch_prepared(d, stream);
}

// pa_decode.cuh - paged single-query decode attention for sm_103a.
//
// What it computes ("Attention計算" of the PagedAttention explainer,
// 0h-n0.github.io; "分块 Attention 计算" of the dihengye.cn notes): for every
// sequence s and query head h,
//     out[s,h] = softmax(scale * K_s q[s,h]) V_s,
// where the rows of K_s / V_s are scattered over physical blocks of B tokens
// that the sequence's block table names.  Rows are consumed a tile at a time
// and folded into a running (m, l, acc) state with the online-softmax
// recurrence (equation (4) of the auturnal.com review: m' = max(m, max s_j),
// l' = e^{m-m'} l + sum e^{s_j-m'}, acc rescaled by the same factor); the
// recurrence runs in base 2 with log2(e) folded into the query.
//
// How it is laid out on GB300 (this is not the pages' A100 kernel design):
//  * Work unit = UR (16 or 32) consecutive rows of one (sequence, KV head).
//    A unit is filled by 3-D TMA boxes of min(UR, B) whole rows (each row is
//    one or two 128-byte halves, 128-byte swizzle): part of one block when
//    B >= UR, one box per block when a unit spans several blocks; one TMA
//    instruction per box for K and one for V.  The units of the whole
//    batch, ordered (s, kvh, unit), are split into equal contiguous ranges, one
//    per resident warp, so long and short sequences load every SM equally
//    ("balanced" mode).  A range crosses (s, kvh) segments freely.  Optionally
//    each warp instead takes fixed partitions of P tokens.
//  * Warp specialisation: each CTA has W consumer warps and one producer
//    warp.  Consumer warp c owns a ring of stages in shared memory (one unit
//    of K, of V and, at a segment start, the query group per stage).  Lane c
//    of the producer warp walks consumer c's units: it waits for the stage's
//    "empty" mbarrier, reads the block table, and issues the TMA copies
//    (cp.async.bulk.tensor) plus a 1-D bulk copy of the query group, all
//    completing on the stage's "full" mbarrier.  Consumers only wait, compute
//    and release.  No CTA-wide barrier is used after the prologue.
//  * QK: 32/UR lanes per token (one for UR=32), each a part of the row, form
//    the dot products with all G query heads of the group in packed fp32x2
//    FMAs (several independent accumulators per head); the pre-scaled fp32
//    query group is read from shared memory with broadcasts; the lane ->
//    (token, half) order is chosen so that, with the swizzle, every quarter
//    warp's K reads hit distinct banks.
//  * PV: each lane owns D/32 output columns of all G heads (fp32 registers)
//    and walks the tile's valid tokens, reading p from shared memory.
//  * FP8 tiles are widened in registers (e4m3 -> f16x2 -> f32); the per-head
//    K scale is folded into the query and the V scale into the final divide.
//  * Split segments: a warp whose range covers only part of a segment writes
//    its (m, l, acc) record to the workspace and bumps the segment's arrival
//    counter; the warp that arrives last merges all records with the same
//    recurrence, writes out[s, kvh*G .. kvh*G+G-1] and resets the counter.
//    Nothing waits on another warp, so the kernel cannot deadlock.
//  * Every wait on an mbarrier is bounded by %globaltimer; on expiry the warp
//    records PA_DEVERR_TIMEOUT, waits (bounded) for its own copies and
//    returns.
#pragma once

#include <type_traits>

#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {

constexpr int kMinUnitsPerWarp = 2;            // smallest balanced share (small batches spread wide)
constexpr int kStageBytesPerWarp = 24 * 1024;  // default K/V pipeline bytes per consumer warp
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Integer tuning override from the environment (read once per name), or -1.
int tuning_override(const char* name);

// Records the geometry and kernel attributes of a rejected launch (error detail).
void note_launch_failure(int ctas, int threads, size_t smem, int stages, int max_threads, int max_dyn_smem,
                         int regs, size_t local_bytes);

__host__ __device__ constexpr int align_up_c(int x, int a) { return (x + a - 1) / a * a; }

template <typename QT, typename KVT, int D, int GM, int UR_>
struct DecodeTraits {
  static constexpr int KVB = elem<KVT>::bytes;
  static constexpr int ROW = D * KVB;  // bytes of one cache row
  static_assert(ROW == 128 || ROW == 256, "cache rows must be 128 or 256 bytes");
  static constexpr int UR = UR_;                 // rows per work unit (16 or 32)
  static_assert(UR == 16 || UR == 32, "unit rows");
  static constexpr int NSUB = ROW / 128;         // 128-byte halves per row
  static constexpr int SUB_ELEMS = 128 / KVB;    // elements per half
  static constexpr int TILE = UR * ROW;          // bytes of one unit of K (or V)
  static constexpr int QRAW = GM * D * 2;        // bytes of one raw query group
  static constexpr int STAGE = align_up_c(2 * TILE + QRAW, 1024);  // K tile + V tile + raw q
  static constexpr int MAX_NS = 8;               // stages per consumer (chosen at launch, 2..MAX_NS)
  static constexpr int MAX_W = 8;                // consumer warps per CTA (chosen at launch)
  static constexpr int LPT = 32 / UR;            // lanes per token in QK (2 or 1)
  static constexpr int CHUNKS = ROW / 16;        // 16-byte chunks per row
  static constexpr int EPC = 16 / KVB;           // elements per chunk
  static constexpr int EPL = D / 32;             // PV columns per lane
  // The query group lives in shared memory as NPART padded parts per head:
  // the part a QK lane reads (LPT = 2) or the half it reads (LPT = 1).
  static constexpr int NPART = (LPT == 2 || NSUB == 2) ? 2 : 1;
  static constexpr int PART = D / NPART;         // elements per part
  static constexpr int CPP = CHUNKS / NPART;     // chunks per part
  static constexpr int QROW = NPART * (PART + 4);  // floats per head (4 floats of padding per part)
  static constexpr int NACC = (GM >= 8) ? 2 : 4;  // independent QK accumulators per head
  // per-consumer shared memory: [fp32 q | p | full[MAX_NS] | empty[MAX_NS] | NS stages]
  static constexpr int OFF_QF32 = 0;
  static constexpr int OFF_PBUF = OFF_QF32 + GM * QROW * 4;
  static constexpr int OFF_FULL = align_up_c(OFF_PBUF + UR * GM * 8, 8);
  static constexpr int OFF_EMPTY = OFF_FULL + MAX_NS * 8;
  static constexpr int OFF_STAGES = align_up_c(OFF_EMPTY + MAX_NS * 8, 1024);
  __host__ __device__ static constexpr int warp_smem(int ns) { return OFF_STAGES + ns * STAGE; }
  static constexpr int REC = align_up_c(GM * (D + 2), 4);  // floats per partial record
  static_assert(EPL == 2 || EPL == 4, "D/32 columns per lane");
  static_assert(EPC % 4 == 0 && PART % 4 == 0, "chunk split");
};

// Length of sequence s clamped to the table's capacity (error bit if outside).
__device__ __forceinline__ int clamped_len(const DecodeParams& p, int s, bool report) {
  int T = __ldg(p.seq_lens + s);
  const int cap = p.max_blocks_per_seq * p.block_size;
  if (T < 0 || T > cap) {
    if (report) raise_error(p.err, PA_DEVERR_SEQ_LEN);
    T = T < 0 ? 0 : cap;
  }
  return T;
}

// Fragment = a run of consecutive units [j, jend) of segment (s, kvh) that a
// warp processes.  Walks either the warp's balanced unit range or its fixed
// partitions.
struct WorkIter {
  int s, kvh, j, jend, j0, nu, T;
  int nblk;       // blocks that hold rows of sequence s
  int frag_idx;   // ordinal of the current fragment within this warp
  int slot;       // partial-record slot, -1 when the fragment is a whole segment
  bool valid;
  // balanced mode
  long long u, u1;  // unit index of unit j0 of the current fragment; end of the warp's range
  int gw;           // global warp id
  // fixed mode
  int r, rstride, R;
};

__device__ __forceinline__ int find_seq(const int* prefix, int S, long long u) {
  // last s in [0, S) with prefix[s] <= u (that sequence is non-empty)
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void frag_balanced(WorkIter& it, const int* prefix, const DecodeParams& p) {
  const int Hkv = p.num_kv_heads;
  const int s = find_seq(prefix, p.num_seqs, it.u);
  const int nu = (prefix[s + 1] - prefix[s]) / Hkv;
  const long long r = it.u - prefix[s];
  it.s = s;
  it.nu = nu;
  it.kvh = static_cast<int>(r / nu);
  it.j0 = static_cast<int>(r % nu);
  it.j = it.j0;
  const long long seg_start = prefix[s] + static_cast<long long>(it.kvh) * nu;
  const long long seg_end = seg_start + nu;
  const long long fend = min(it.u1, seg_end);
  it.jend = it.j0 + static_cast<int>(fend - it.u);
  const bool whole = (it.u == seg_start) && (fend == seg_end);
  it.slot = whole ? -1 : it.gw * 2 + (it.frag_idx == 0 ? 0 : 1);
  it.T = clamped_len(p, s, false);
  it.nblk = (it.T + p.block_size - 1) >> p.block_shift;
}

__device__ __forceinline__ void frag_fixed(WorkIter& it, const int* prefix, const DecodeParams& p, int UR) {
  const int Hkv = p.num_kv_heads;
  const int s = find_seq(prefix, p.num_seqs, it.r);
  const int parts = (prefix[s + 1] - prefix[s]) / Hkv;
  const int rr = it.r - prefix[s];
  it.s = s;
  it.kvh = rr / parts;
  const int part = rr % parts;
  it.T = clamped_len(p, s, false);
  it.nu = (it.T + UR - 1) / UR;
  it.nblk = (it.T + p.block_size - 1) >> p.block_shift;
  it.j0 = part * p.partition_units;
  it.j = it.j0;
  it.jend = min(it.nu, it.j0 + p.partition_units);
  it.slot = (parts == 1) ? -1 : it.r;
}

__device__ __forceinline__ void iter_next_fragment(WorkIter& it, const int* prefix, const DecodeParams& p,
                                                   bool fixed, int UR) {
  it.frag_idx++;
  if (fixed) {
    it.r += it.rstride;
    if (it.r >= it.R) { it.valid = false; return; }
    frag_fixed(it, prefix, p, UR);
  } else {
    it.u += it.jend - it.j0;
    if (it.u >= it.u1) { it.valid = false; return; }
    frag_balanced(it, prefix, p);
  }
}

template <typename QT, typename KVT, int D, int GM, int UR_>
__global__ void __launch_bounds__((DecodeTraits<QT, KVT, D, GM, UR_>::MAX_W + 1) * 32, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const DecodeParams p) {
  using Tr = DecodeTraits<QT, KVT, D, GM, UR_>;
  constexpr bool kFp8 = elem<KVT>::bytes == 1;
  constexpr int UR = Tr::UR;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NWARP = blockDim.x >> 5;
  const int W = NWARP - 1;         // consumer warps (warp 0 produces)
  const int S = p.num_seqs;
  const int Hkv = p.num_kv_heads;
  const int G = p.group;
  const int B = p.block_size;
  // A unit spans part of one block (B >= UR) or several whole blocks (B < UR);
  // one TMA box per block it touches, BOX rows high.  B is a power of two.
  const bool unit_in_block = B >= UR;
  const int BOX = unit_in_block ? UR : B;
  const int upb_shift = unit_in_block ? p.block_shift - (UR == 32 ? 5 : 4) : 0;  // log2(units per block)
  const int bpu_shift = unit_in_block ? 0 : (UR == 32 ? 5 : 4) - p.block_shift;  // log2(blocks per unit)
  const bool fixed = p.partition_units > 0;

  const int NS = p.stages;  // pipeline depth per consumer
  const int wsm = Tr::warp_smem(NS);
  int* prefix = reinterpret_cast<int*>(base + W * wsm);
  int* scan_tmp = prefix + (S + 1);

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }

  // ---- 1. units per sequence and their exclusive prefix sums (every CTA)
  {
    int carry = 0;
    for (int b0 = 0; b0 < S; b0 += blockDim.x) {
      const int s = b0 + threadIdx.x;
      int units = 0;
      if (s < S) {
        const int T = clamped_len(p, s, blockIdx.x == 0);
        const int nu = (T + UR - 1) / UR;
        units = (fixed ? (nu + p.partition_units - 1) / p.partition_units : nu) * Hkv;
      }
      int x = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) scan_tmp[warp] = x;
      __syncthreads();
      int wo = 0, tot = 0;
      for (int w = 0; w < NWARP; ++w) {
        const int v = scan_tmp[w];
        wo += (w < warp) ? v : 0;
        tot += v;
      }
      if (s < S) prefix[s] = carry + wo + x - units;
      carry += tot;
      __syncthreads();
    }
    if (threadIdx.x == 0) prefix[S] = carry;
  }

  // ---- 2. empty sequences attend to nothing: their outputs are zero
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < S; s += gridDim.x * blockDim.x) {
    if (clamped_len(p, s, false) == 0) {
      const int64_t n = static_cast<int64_t>(p.num_heads) * D;
      for (int64_t i = 0; i < n; ++i) store_out(p.out, p.out_dtype, static_cast<int64_t>(s) * n + i, 0.f);
    }
  }

  // ---- 3. barriers of every consumer ring
  if (threadIdx.x == 0) {
    for (int c = 0; c < W; ++c) {
      const uint32_t cb = base_u32 + c * wsm;
      for (int i = 0; i < NS; ++i) {
        mbar_init(cb + Tr::OFF_FULL + 8 * i, 1);
        mbar_init(cb + Tr::OFF_EMPTY + 8 * i, 1);
      }
    }
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  // ---- 4. the share of consumer c (global consumer id gc)
  const int nw_total = gridDim.x * W;
  const long long U = prefix[S];
  long long want = (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp;
  const int nw_eff = fixed ? nw_total : static_cast<int>(want < 1 ? 1 : (want < nw_total ? want : nw_total));
  auto start_iter = [&](WorkIter& w, int gc) {
    w.frag_idx = 0;
    w.gw = gc;
    w.valid = false;
    if (fixed) {
      w.R = static_cast<int>(U);
      w.rstride = nw_total;
      w.r = gc;
      if (w.r < w.R) { w.valid = true; frag_fixed(w, prefix, p, UR); }
    } else if (U > 0 && gc < nw_eff) {
      w.u = gc * U / nw_eff;
      w.u1 = (gc + 1) * U / nw_eff;
      if (w.u < w.u1) { w.valid = true; frag_balanced(w, prefix, p); }
    }
  };

  if (warp == 0) {
    // =================================================================== producer
    // Lane c feeds consumer c: one unit per free stage of its ring.
    WorkIter it;
    it.valid = false;
    if (lane < W) start_iter(it, blockIdx.x * W + lane);
    const uint32_t cbase = base_u32 + (lane < W ? lane : 0) * wsm;
    int pst = 0, pph = 1, issued = 0;
    uint64_t wait_since = 0;
    int nx_s = -1, nx_bj = -1;  // table entries of the next unit, loaded ahead
    int nx_phys[4] = {0, 0, 0, 0};
    while (__any_sync(0xffffffffu, it.valid)) {
      bool did = false;
      if (it.valid) {
        bool ready = issued < NS || mbar_test_wait(cbase + Tr::OFF_EMPTY + 8 * pst, pph);
        if (!ready) {
          const uint64_t now = global_timer_ns();
          if (wait_since == 0) {
            wait_since = now;
          } else if (now - wait_since > kWaitLimitNs) {
            raise_error(p.err, PA_DEVERR_TIMEOUT);
            it.valid = false;  // give up on this consumer; it times out on its own
          }
        } else {
          wait_since = 0;
          const bool new_frag = (it.j == it.j0);
          const uint32_t bar = cbase + Tr::OFF_FULL + 8 * pst;
          const uint32_t kdst = cbase + Tr::OFF_STAGES + pst * Tr::STAGE;
          const uint32_t vdst = kdst + Tr::TILE;
          const int bj0 = unit_in_block ? (it.j >> upb_shift) : (it.j << bpu_shift);
          const int nbox = unit_in_block ? 1 : min(1 << bpu_shift, it.nblk - bj0);
          const int row_in_block = unit_in_block ? (it.j - (bj0 << upb_shift)) * UR : 0;
          const uint32_t qbytes = new_frag ? static_cast<uint32_t>(G * D * 2) : 0u;
          int phys[4];
          if (nx_s == it.s && nx_bj == bj0) {  // entries loaded while issuing the previous unit
#pragma unroll
            for (int i = 0; i < 4; ++i) phys[i] = nx_phys[i];
          } else {
            const int32_t* trow = p.block_tables + static_cast<int64_t>(it.s) * p.max_blocks_per_seq + bj0;
#pragma unroll
            for (int i = 0; i < 4; ++i) phys[i] = (i < nbox) ? __ldg(trow + i) : 0;
          }
          mbar_arrive_expect_tx(bar, 2u * nbox * BOX * Tr::ROW + qbytes);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (i < nbox) {
              int pb = phys[i];
              if (pb < 0 || pb >= p.num_blocks) {
                raise_error(p.err, PA_DEVERR_BLOCK_ID);
                pb = 0;
              }
              const int z = (pb * Hkv + it.kvh) * B + row_in_block;
              tma_load_3d(kdst + i * BOX * Tr::ROW, &tmap_k, 0, 0, z, bar);
              tma_load_3d(vdst + i * BOX * Tr::ROW, &tmap_v, 0, 0, z, bar);
            }
          }
          if (new_frag) {
            const uint8_t* qsrc = static_cast<const uint8_t*>(p.q) +
                                  (static_cast<int64_t>(it.s) * p.q_stride + static_cast<int64_t>(it.kvh) * G * D) * 2;
            bulk_load(kdst + 2 * Tr::TILE, qsrc, qbytes, bar);
          }
          ++issued;
          if (++pst == NS) {
            pst = 0;
            pph ^= 1;
          }
          // load the next unit's table entries now; they are used one refill later
          nx_s = -1;
          if (it.j + 1 < it.jend) {
            const int nj = it.j + 1;
            const int nbj0 = unit_in_block ? (nj >> upb_shift) : (nj << bpu_shift);
            if (nbj0 != bj0) {
              const int nnbox = unit_in_block ? 1 : min(1 << bpu_shift, it.nblk - nbj0);
              const int32_t* trow = p.block_tables + static_cast<int64_t>(it.s) * p.max_blocks_per_seq + nbj0;
#pragma unroll
              for (int i = 0; i < 4; ++i) nx_phys[i] = (i < nnbox) ? __ldg(trow + i) : 0;
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) nx_phys[i] = phys[i];
            }
            nx_s = it.s;
            nx_bj = nbj0;
          }
          if (++it.j == it.jend) iter_next_fragment(it, prefix, p, fixed, UR);
          did = true;
        }
      }
      if (!__any_sync(0xffffffffu, did)) __nanosleep(64);
    }
    return;
  }

  // ===================================================================== consumer
  const int c = warp - 1;
  WorkIter it;
  start_iter(it, blockIdx.x * W + c);
  if (!it.valid) return;
  uint8_t* wbase = base + c * wsm;
  const uint32_t wbase_u32 = base_u32 + c * wsm;
  float* qf = reinterpret_cast<float*>(wbase + Tr::OFF_QF32);
  float2* pbuf = reinterpret_cast<float2*>(wbase + Tr::OFF_PBUF);
  int cst = 0, cpar = 0;
  // QK lane roles.  LPT = 2: lane pairs share a token (t = lane/2), each one
  // part of the row (qd = lane & 1).  LPT = 1: one token per lane, visiting
  // the halves of a 256-byte row in an order rotated by bit 2 of the token.
  const int t = (Tr::LPT == 2) ? (lane >> 1) : lane;
  const int qd = (Tr::LPT == 2) ? (lane & 1) : 0;
  const int rot = (Tr::LPT == 1 && Tr::NPART == 2) ? ((t >> 2) & 1) : 0;
  const int e0 = lane * Tr::EPL;  // first PV column of this lane
  // byte offset of K chunk ch of half h in row t of a stage (128-byte swizzle)
  auto kaddr = [&](int h, int ch) -> uint32_t {
    return t * Tr::ROW + h * 128 + (((ch ^ (t * Tr::NSUB + h)) & 7) << 4);
  };
  // V: this lane's columns of row r; the swizzle phase repeats every 8/NSUB rows
  constexpr int VPER = 8 / Tr::NSUB;
  const int vbyte = e0 * Tr::KVB;
  const int vh = vbyte >> 7;
  const int vch = (vbyte & 127) >> 4;
  uint32_t vofs[VPER];
#pragma unroll
  for (int k = 0; k < VPER; ++k) vofs[k] = Tr::TILE + vh * 128 + (((vch ^ (k * Tr::NSUB + vh)) & 7) << 4) + (vbyte & 15);
  // q parts this lane reads: LPT = 2 -> part qd; LPT = 1 -> parts (pi ^ rot)
  const float* qpart0 = qf + ((Tr::LPT == 2 ? qd : rot) * (Tr::PART + 4));
  const float* qpart1 = qf + ((Tr::LPT == 2 ? qd : (rot ^ 1)) * (Tr::PART + 4));

  float m[GM], l[GM];
  float2 acc[GM][Tr::EPL / 2];

  // V row -> EPL floats as float2 pairs
  auto load_v = [&](const uint8_t* row_ptr, float2* vf) {
    if constexpr (Tr::KVB == 2) {
      if constexpr (Tr::EPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(row_ptr);
        vf[0] = widen2<KVT>(w.x);
        vf[1] = widen2<KVT>(w.y);
      } else {
        vf[0] = widen2<KVT>(*reinterpret_cast<const uint32_t*>(row_ptr));
      }
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(row_ptr);
      vf[0] = widen2_e4m3(w & 0xffffu);
      vf[1] = widen2_e4m3(w >> 16);
    }
  };
  // acc[g] += p[tok][g] * v for all heads (p stored as (p, p) pairs)
  auto accumulate = [&](const float2* prow, const float2* vf) {
#pragma unroll
    for (int g = 0; g < GM; g += 2) {
      if (g + 1 < GM) {
        const float4 pp = *reinterpret_cast<const float4*>(prow + g);
#pragma unroll
        for (int i = 0; i < Tr::EPL / 2; ++i) {
          acc[g][i] = ffma2(make_float2(pp.x, pp.y), vf[i], acc[g][i]);
          acc[g + 1][i] = ffma2(make_float2(pp.z, pp.w), vf[i], acc[g + 1][i]);
        }
      } else {
        const float2 pp = prow[g];
#pragma unroll
        for (int i = 0; i < Tr::EPL / 2; ++i) acc[g][i] = ffma2(pp, vf[i], acc[g][i]);
      }
    }
  };

  // One unit (8 rows): scores, online-softmax update, p . V.  FULL: all 8 rows valid.
  auto unit_step = [&](auto full_tag, const uint8_t* stage, int n_valid) {
    constexpr bool FULL = decltype(full_tag)::value;
    // ---- scores: the lane dots its part(s) of token t's K row with all G query heads
    float2 sacc[Tr::NACC][GM];
#pragma unroll
    for (int a = 0; a < Tr::NACC; ++a)
#pragma unroll
      for (int g = 0; g < GM; ++g) sacc[a][g] = make_float2(0.f, 0.f);
    constexpr int NPI = (Tr::LPT == 2) ? 1 : Tr::NPART;  // parts this lane visits
#pragma unroll
    for (int pi = 0; pi < NPI; ++pi) {
      const int pp = (Tr::LPT == 2) ? qd : (pi ^ rot);   // part index
      const float* qp0 = pi == 0 ? qpart0 : qpart1;
#pragma unroll
      for (int c = 0; c < Tr::CPP; ++c) {
        // chunk c of part pp -> half h, chunk-in-half ch
        const int cb = pp * Tr::CPP + c;                  // chunk within the row
        const uint4 raw = *reinterpret_cast<const uint4*>(stage + kaddr(cb >> 3, cb & 7));
        float2 kf[Tr::EPC / 2];
        Chunk<KVT>::cvt(raw, kf);
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          const float4* qp = reinterpret_cast<const float4*>(qp0 + g * Tr::QROW + c * Tr::EPC);
#pragma unroll
          for (int i = 0; i < Tr::EPC / 4; ++i) {
            const float4 q4 = qp[i];
            float2& sa = sacc[(2 * i) % Tr::NACC][g];
            sa = ffma2(make_float2(q4.x, q4.y), kf[2 * i], sa);
            float2& sb = sacc[(2 * i + 1) % Tr::NACC][g];
            sb = ffma2(make_float2(q4.z, q4.w), kf[2 * i + 1], sb);
          }
        }
      }
    }
    float sv[GM];
    bool up = false;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      float2 s2 = sacc[0][g];
#pragma unroll
      for (int a = 1; a < Tr::NACC; ++a) s2 = make_float2(s2.x + sacc[a][g].x, s2.y + sacc[a][g].y);
      float x = s2.x + s2.y;
      if constexpr (Tr::LPT == 2) x += __shfl_xor_sync(0xffffffffu, x, 1);
      if constexpr (!FULL) x = (t < n_valid) ? x : -INFINITY;
      sv[g] = x;
      up |= x > m[g];
    }
    // ---- online softmax: the running maximum only moves when some score exceeds it
    if (__any_sync(0xffffffffu, up)) {
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        float bm = sv[g];
#pragma unroll
        for (int o = Tr::LPT; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
        const float mn = fmaxf(m[g], bm);
        const float alpha = fast_exp2(m[g] - mn);
        m[g] = mn;
        l[g] *= alpha;
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < Tr::EPL / 2; ++i) acc[g][i] = fmul2(acc[g][i], a2);
      }
    }
    float pg[GM];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      pg[g] = fast_exp2(sv[g] - m[g]);
      l[g] += (qd == 0) ? pg[g] : 0.f;
    }
    if (qd == 0) {
      float2* prow = pbuf + t * GM;
#pragma unroll
      for (int g = 0; g < GM; g += 2) {
        if (g + 1 < GM) {
          *reinterpret_cast<float4*>(prow + g) = make_float4(pg[g], pg[g], pg[g + 1], pg[g + 1]);
        } else {
          prow[g] = make_float2(pg[g], pg[g]);
        }
      }
    }
    __syncwarp();
    // ---- p . V: lane owns columns e0..e0+EPL-1 of all G heads
#pragma unroll
    for (int tt = 0; tt < UR; ++tt) {
      if (FULL || tt < n_valid) {
        float2 vf[Tr::EPL / 2];
        load_v(stage + vofs[tt % VPER] + tt * Tr::ROW, vf);
        accumulate(pbuf + tt * GM, vf);
      }
    }
  };

  while (it.valid) {
    if (!mbar_wait_bounded(wbase_u32 + Tr::OFF_FULL + 8 * cst, cpar, kWaitLimitNs)) {
      if (lane == 0) raise_error(p.err, PA_DEVERR_TIMEOUT);
      break;  // the producer stops feeding this ring when its empty barrier times out
    }
    const uint8_t* stage = wbase + Tr::OFF_STAGES + cst * Tr::STAGE;
    if (it.j == it.j0) {
      // new fragment: widen + pre-scale the query group, reset the state
      float qs = p.qk_scale_log2;
      if constexpr (kFp8) qs *= __ldg(p.k_scale + it.kvh);
      const uint8_t* qr = stage + 2 * Tr::TILE;  // the query group rode on this stage
      for (int idx = lane; idx < GM * D / 2; idx += 32) {
        const int e = 2 * idx;
        const int g = e / D;
        const int ed = e % D;
        float2 v2 = make_float2(0.f, 0.f);
        if (g < G) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(qr + 4 * idx);
          v2 = widen2<QT>(w);
          v2.x *= qs;
          v2.y *= qs;
        }
        *reinterpret_cast<float2*>(qf + g * Tr::QROW + (ed / Tr::PART) * (Tr::PART + 4) + ed % Tr::PART) = v2;
      }
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < Tr::EPL / 2; ++i) acc[g][i] = make_float2(0.f, 0.f);
      }
      __syncwarp();
    }

    const int n_valid = min(UR, it.T - it.j * UR);
    if (n_valid == UR) {
      unit_step(std::true_type{}, stage, UR);
    } else {
      unit_step(std::false_type{}, stage, n_valid);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(wbase_u32 + Tr::OFF_EMPTY + 8 * cst);  // the stage may be refilled
    if (++cst == NS) {
      cst = 0;
      cpar ^= 1;
    }

    // ---- end of fragment: write the output or a partial record
    if (it.j + 1 == it.jend) {
      float lt[GM];
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        float x = l[g];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        lt[g] = x;
      }
      float vs = 1.f;
      if constexpr (kFp8) vs = __ldg(p.v_scale + it.kvh);
      const int64_t orow = static_cast<int64_t>(it.s) * p.num_heads + static_cast<int64_t>(it.kvh) * G;
      if (it.slot < 0) {
#pragma unroll
        for (int g = 0; g < GM; ++g) {
          if (g < G) {
            const float inv = vs / lt[g];
#pragma unroll
            for (int i = 0; i < Tr::EPL / 2; ++i) {
              store_out(p.out, p.out_dtype, (orow + g) * D + e0 + 2 * i, acc[g][i].x * inv);
              store_out(p.out, p.out_dtype, (orow + g) * D + e0 + 2 * i + 1, acc[g][i].y * inv);
            }
          }
        }
      } else {
        float* rec = p.part_records + static_cast<int64_t>(it.slot) * Tr::REC;
#pragma unroll
        for (int g = 0; g < GM; ++g) {
#pragma unroll
          for (int i = 0; i < Tr::EPL / 2; ++i)
            *reinterpret_cast<float2*>(rec + g * D + e0 + 2 * i) = acc[g][i];
          if (lane == g) {
            rec[GM * D + g] = m[g];
            rec[GM * D + GM + g] = lt[g];
          }
        }
        __threadfence();
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atomicAdd(p.seg_counters + it.s * Hkv + it.kvh, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        // fragments of this segment and where their records live
        int nfr, first_slot_w = 0;
        long long seg_start = 0;
        int parts = 0;
        if (fixed) {
          parts = (prefix[it.s + 1] - prefix[it.s]) / Hkv;
          nfr = parts;
        } else {
          seg_start = prefix[it.s] + static_cast<long long>(it.kvh) * it.nu;
          const long long seg_last = seg_start + it.nu - 1;
          const int wf = static_cast<int>(((seg_start + 1) * nw_eff - 1) / U);
          const int wl = static_cast<int>(((seg_last + 1) * nw_eff - 1) / U);
          nfr = wl - wf + 1;
          first_slot_w = wf;
        }
        if (old == nfr - 1) {
          __threadfence();
          float M[GM], L[GM];
          float2 o2[GM][Tr::EPL / 2];
#pragma unroll
          for (int g = 0; g < GM; ++g) {
            M[g] = -INFINITY;
            L[g] = 0.f;
#pragma unroll
            for (int i = 0; i < Tr::EPL / 2; ++i) o2[g][i] = make_float2(0.f, 0.f);
          }
          auto slot_of = [&](int f) -> int {
            if (fixed) return prefix[it.s] + it.kvh * parts + f;
            const int w = first_slot_w + f;
            const long long rs = static_cast<long long>(w) * U / nw_eff;
            return 2 * w + (rs < seg_start ? 1 : 0);
          };
          for (int f = 0; f < nfr; ++f) {
            const float* rf = p.part_records + static_cast<int64_t>(slot_of(f)) * Tr::REC;
#pragma unroll
            for (int g = 0; g < GM; ++g) M[g] = fmaxf(M[g], __ldcg(rf + GM * D + g));
          }
          for (int f = 0; f < nfr; ++f) {
            const float* rf = p.part_records + static_cast<int64_t>(slot_of(f)) * Tr::REC;
#pragma unroll
            for (int g = 0; g < GM; ++g) {
              const float w = exp2f(__ldcg(rf + GM * D + g) - M[g]);
              L[g] += w * __ldcg(rf + GM * D + GM + g);
              const float2 w2 = make_float2(w, w);
#pragma unroll
              for (int i = 0; i < Tr::EPL / 2; ++i)
                o2[g][i] = ffma2(w2, __ldcg(reinterpret_cast<const float2*>(rf + g * D + e0 + 2 * i)), o2[g][i]);
            }
          }
#pragma unroll
          for (int g = 0; g < GM; ++g) {
            if (g < G) {
              const float inv = vs / L[g];
#pragma unroll
              for (int i = 0; i < Tr::EPL / 2; ++i) {
                store_out(p.out, p.out_dtype, (orow + g) * D + e0 + 2 * i, o2[g][i].x * inv);
                store_out(p.out, p.out_dtype, (orow + g) * D + e0 + 2 * i + 1, o2[g][i].y * inv);
              }
            }
          }
          if (lane == 0) p.seg_counters[it.s * Hkv + it.kvh] = 0;
        }
      }
    }
    if (++it.j == it.jend) iter_next_fragment(it, prefix, p, fixed, UR);
  }
}


// ----------------------------------------------------------------- host side of one variant

template <typename QT, typename KVT, int D, int GM, int UR>
struct DecodeVariant {
  using Tr = DecodeTraits<QT, KVT, D, GM, UR>;

  static size_t smem_bytes(int num_seqs, int warps, int stages) {
    return 1024 + static_cast<size_t>(warps) * Tr::warp_smem(stages) +
           static_cast<size_t>(align_up_c((num_seqs + 1 + warps + 1) * 4, 16));
  }

  // Launch geometry: pipeline depth (stages per consumer) and consumer warps
  // per CTA (plus one producer warp).  Default depth keeps about
  // kStageBytesPerWarp of K/V per consumer; the consumers per CTA maximise
  // resident consumer warps per SM (ties: more per CTA, i.e. fewer producer
  // warps).  PA_DECODE_STAGES / PA_DECODE_WARPS override both (tuning).
  static bool geometry(int num_seqs, DecodeGeometry* g) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    auto kern = paged_decode_kernel<QT, KVT, D, GM, UR>;
    int ns = kStageBytesPerWarp / Tr::STAGE;
    ns = ns < 2 ? 2 : (ns > Tr::MAX_NS ? Tr::MAX_NS : ns);
    const int env_ns = tuning_override("PA_DECODE_STAGES");
    if (env_ns >= 2 && env_ns <= Tr::MAX_NS) ns = env_ns;
    const int env_w = tuning_override("PA_DECODE_WARPS");
    int best_w = 0, best_occ = 0, best_warps = 0;
    for (int w = 1; w <= Tr::MAX_W; ++w) {
      if (env_w > 0 && w != env_w) continue;
      const size_t smem = smem_bytes(num_seqs, w, ns);
      if (smem > 227 * 1024) break;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
        return false;
      int occ = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, (w + 1) * 32, smem) != cudaSuccess) return false;
      if (occ * w >= best_warps && occ > 0) {
        best_warps = occ * w;
        best_w = w;
        best_occ = occ;
      }
    }
    if (best_w == 0) return false;
    const size_t smem = smem_bytes(num_seqs, best_w, ns);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
      return false;
    g->warps_per_cta = best_w;
    g->stages = ns;
    g->ctas = sms * best_occ;
    g->smem_bytes = smem;
    g->record_floats = Tr::REC;
    g->unit_rows = UR;
    return true;
  }

  static cudaError_t launch(const DecodeGeometry& g, const DecodeParams& p, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t stream) {
    (void)cudaGetLastError();  // an earlier unrelated error must not be reported as this launch's
    paged_decode_kernel<QT, KVT, D, GM, UR><<<g.ctas, (g.warps_per_cta + 1) * 32, g.smem_bytes, stream>>>(tk, tv, p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, paged_decode_kernel<QT, KVT, D, GM, UR>) == cudaSuccess)
        note_launch_failure(g.ctas, (g.warps_per_cta + 1) * 32, g.smem_bytes, g.stages, fa.maxThreadsPerBlock,
                            fa.maxDynamicSharedSizeBytes, fa.numRegs, fa.localSizeBytes);
    }
    return e;
  }
};

}  // namespace pa

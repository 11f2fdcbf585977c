// pa_decode.cuh - paged single-query decode attention for sm_103a.
//
// What it computes ("Attention計算" of the PagedAttention explainer,
// 0h-n0.github.io; "分块 Attention 计算" of the dihengye.cn notes): for every
// sequence s and query head h,
//     out[s,h] = softmax(scale * K_s q[s,h]) V_s,
// where the rows of K_s / V_s are scattered over physical blocks of B tokens
// that the sequence's block table names.  Blocks are consumed one at a time
// and folded into a running (m, l, acc) state with the online-softmax
// recurrence (equation (4) of the auturnal.com review: m' = max(m, max s_j),
// l' = e^{m-m'} l + sum e^{s_j-m'}, acc rescaled by the same factor); the
// recurrence runs in base 2 with log2(e) folded into the query.
//
// How it is laid out on GB300 (this is not the pages' A100 kernel design):
//  * Work unit = one (sequence, KV head, block) triple.  The units of the
//    whole batch, ordered (s, kvh, block), are split into equal contiguous
//    ranges, one per resident warp (152 SMs x occupancy x 4 warps), so long
//    and short sequences load every SM equally ("balanced" mode).  A range
//    crosses (s, kvh) segments freely.  Optionally each warp instead takes
//    fixed partitions of P tokens (the pages' "V2" style).
//  * Each warp owns a private ring of NS stages in shared memory and streams
//    the K and V tiles of its units into it with 2-D TMA copies
//    (cp.async.bulk.tensor, 128-byte swizzle) completing on one mbarrier per
//    stage; the query group of a new segment rides on the same barrier as a
//    1-D bulk copy.  No CTA-wide barrier is used after the prologue.
//  * QK: each lane owns one token of the 16/32-token tile (two lanes per
//    token for B=16, one d-half each) and forms the dot products of all G
//    query heads of the group with packed fp32x2 FMAs; the query group sits
//    pre-scaled in fp32 in shared memory (broadcast reads); the swizzle makes
//    the per-lane K row reads bank-conflict free.
//  * PV: each lane owns D/32 output columns for all G heads (fp32 registers)
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

#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {

constexpr int kMinUnitsPerWarp = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__host__ __device__ constexpr int align_up_c(int x, int a) { return (x + a - 1) / a * a; }

template <typename QT, typename KVT, int D, int BS, int GM>
struct DecodeTraits {
  static constexpr int KVB = elem<KVT>::bytes;
  static constexpr int ROW = D * KVB;  // bytes of one cache row
  static_assert(ROW == 128 || ROW == 256, "cache rows must be 128 or 256 bytes");
  static_assert(BS == 16 || BS == 32, "block size 16 or 32");
  static constexpr int NSUB = ROW / 128;         // 128-byte sub-tiles per row
  static constexpr int SUB_ELEMS = 128 / KVB;    // elements per sub-tile row
  static constexpr int TILE = BS * ROW;          // bytes of one (block, head) tile
  static constexpr int STAGE = 2 * TILE;         // K tile + V tile
  static constexpr int NS = (STAGE <= 4096) ? 4 : (STAGE <= 8192 ? 2 : 2);
  static constexpr int W = 4;                    // warps per CTA
  static constexpr int LPT = 32 / BS;            // lanes per token in QK
  static constexpr int CHUNKS = ROW / 16;        // 16-byte chunks per row
  static constexpr int CPL = CHUNKS / LPT;       // chunks per lane in QK
  static constexpr int EPC = 16 / KVB;           // elements per chunk
  static constexpr int EPL = D / 32;             // PV columns per lane
  static constexpr int HALF = D / LPT;           // row elements one QK lane covers
  static constexpr int QPAD = (LPT == 2) ? 4 : 0;  // keeps the two halves in other banks
  static constexpr int QROW = LPT * (HALF + QPAD);  // floats per head in q smem
  static constexpr int QRAW = GM * D * 2;        // bytes of one raw query group
  static constexpr int OFF_QRAW = NS * STAGE;
  static constexpr int OFF_QF32 = OFF_QRAW + 2 * align_up_c(QRAW, 128);
  static constexpr int OFF_PBUF = OFF_QF32 + GM * QROW * 4;
  static constexpr int OFF_BAR = OFF_PBUF + BS * GM * 8;
  static constexpr int WARP_SMEM = align_up_c(OFF_BAR + NS * 8, 1024);
  static constexpr int REC = align_up_c(GM * (D + 2), 4);  // floats per partial record
  static_assert(EPL == 2 || EPL == 4, "D/32 columns per lane");
};

// Length of sequence s clamped to the table's capacity (error bit if outside).
template <int BS>
__device__ __forceinline__ int clamped_len(const DecodeParams& p, int s, bool report) {
  int T = __ldg(p.seq_lens + s);
  const int cap = p.max_blocks_per_seq * BS;
  if (T < 0 || T > cap) {
    if (report) raise_error(p.err, PA_DEVERR_SEQ_LEN);
    T = T < 0 ? 0 : cap;
  }
  return T;
}

// Fragment = a run of consecutive blocks [j, jend) of segment (s, kvh) that a
// warp processes.  Walks either the warp's balanced unit range or its fixed
// partitions.
struct WorkIter {
  int s, kvh, j, jend, j0, nb, T;
  int frag_idx;   // ordinal of the current fragment within this warp
  int slot;       // partial-record slot, -1 when the fragment is a whole segment
  bool valid;
  // balanced mode
  long long u, u1;  // unit of block j0 of the current fragment; end of the warp's range
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

template <int BS>
__device__ __forceinline__ void frag_balanced(WorkIter& it, const int* prefix, const DecodeParams& p) {
  const int Hkv = p.num_kv_heads;
  const int s = find_seq(prefix, p.num_seqs, it.u);
  const int nb = (prefix[s + 1] - prefix[s]) / Hkv;
  const long long r = it.u - prefix[s];
  it.s = s;
  it.nb = nb;
  it.kvh = static_cast<int>(r / nb);
  it.j0 = static_cast<int>(r % nb);
  it.j = it.j0;
  const long long seg_start = prefix[s] + static_cast<long long>(it.kvh) * nb;
  const long long seg_end = seg_start + nb;
  const long long fend = min(it.u1, seg_end);
  it.jend = it.j0 + static_cast<int>(fend - it.u);
  const bool whole = (it.u == seg_start) && (fend == seg_end);
  it.slot = whole ? -1 : it.gw * 2 + (it.frag_idx == 0 ? 0 : 1);
  it.T = clamped_len<BS>(p, s, false);
}

template <int BS>
__device__ __forceinline__ void frag_fixed(WorkIter& it, const int* prefix, const DecodeParams& p) {
  const int Hkv = p.num_kv_heads;
  const int s = find_seq(prefix, p.num_seqs, it.r);
  const int parts = (prefix[s + 1] - prefix[s]) / Hkv;
  const int rr = it.r - prefix[s];
  it.s = s;
  it.kvh = rr / parts;
  const int part = rr % parts;
  it.T = clamped_len<BS>(p, s, false);
  it.nb = (it.T + BS - 1) / BS;
  it.j0 = part * p.partition_blocks;
  it.j = it.j0;
  it.jend = min(it.nb, it.j0 + p.partition_blocks);
  it.slot = (parts == 1) ? -1 : it.r;
}

template <int BS>
__device__ __forceinline__ void iter_next_fragment(WorkIter& it, const int* prefix, const DecodeParams& p,
                                                   bool fixed) {
  it.frag_idx++;
  if (fixed) {
    it.r += it.rstride;
    if (it.r >= it.R) { it.valid = false; return; }
    frag_fixed<BS>(it, prefix, p);
  } else {
    it.u += it.jend - it.j0;
    if (it.u >= it.u1) { it.valid = false; return; }
    frag_balanced<BS>(it, prefix, p);
  }
}

template <typename QT, typename KVT, int D, int BS, int GM>
__global__ void __launch_bounds__(DecodeTraits<QT, KVT, D, BS, GM>::W * 32)
paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const DecodeParams p) {
  using Tr = DecodeTraits<QT, KVT, D, BS, GM>;
  constexpr bool kFp8 = elem<KVT>::bytes == 1;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.num_seqs;
  const int Hkv = p.num_kv_heads;
  const int G = p.group;
  const bool fixed = p.partition_blocks > 0;

  int* prefix = reinterpret_cast<int*>(base + Tr::W * Tr::WARP_SMEM);
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
        const int T = clamped_len<BS>(p, s, blockIdx.x == 0);
        const int nb = (T + BS - 1) / BS;
        units = (fixed ? (nb + p.partition_blocks - 1) / p.partition_blocks : nb) * Hkv;
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
#pragma unroll
      for (int w = 0; w < Tr::W; ++w) {
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
    if (clamped_len<BS>(p, s, false) == 0) {
      const int64_t n = static_cast<int64_t>(p.num_heads) * D;
      for (int64_t i = 0; i < n; ++i) store_out(p.out, p.out_dtype, static_cast<int64_t>(s) * n + i, 0.f);
    }
  }
  __syncthreads();

  // ---- 3. this warp's share of the work
  const int nw_total = gridDim.x * Tr::W;
  const int gw = blockIdx.x * Tr::W + warp;
  const long long U = prefix[S];
  WorkIter it;
  it.frag_idx = 0;
  it.gw = gw;
  it.valid = false;
  int nw_eff = nw_total;
  if (fixed) {
    it.R = static_cast<int>(U);
    it.rstride = nw_total;
    it.r = gw;
    if (it.r < it.R) { it.valid = true; frag_fixed<BS>(it, prefix, p); }
  } else if (U > 0) {
    const long long want = (U + kMinUnitsPerWarp - 1) / kMinUnitsPerWarp;
    nw_eff = static_cast<int>(want < nw_total ? want : static_cast<long long>(nw_total));
    if (nw_eff < 1) nw_eff = 1;
    if (gw < nw_eff) {
      it.u = gw * U / nw_eff;
      it.u1 = (gw + 1) * U / nw_eff;
      if (it.u < it.u1) { it.valid = true; frag_balanced<BS>(it, prefix, p); }
    }
  }
  if (!it.valid) return;

  uint8_t* wbase = base + warp * Tr::WARP_SMEM;
  const uint32_t wbase_u32 = base_u32 + warp * Tr::WARP_SMEM;
  const uint32_t bar0 = wbase_u32 + Tr::OFF_BAR;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < Tr::NS; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();

  float* qf = reinterpret_cast<float*>(wbase + Tr::OFF_QF32);
  float2* pbuf = reinterpret_cast<float2*>(wbase + Tr::OFF_PBUF);
  const uint8_t* qraw_base = wbase + Tr::OFF_QRAW;
  const uint32_t qraw_u32 = wbase_u32 + Tr::OFF_QRAW;
  constexpr int kQrawStride = align_up_c(Tr::QRAW, 128);

  // producer state
  WorkIter prod = it;
  int tb_seq = -1, tb_base = 0, tb_val = -1;  // cached table slice: lane i holds entry tb_base+i
  int issued = 0, consumed = 0;
  bool timed_out = false;

  auto produce = [&](void) {
    // Fill free stages while the producer has units and the query slot is free.
    while (prod.valid && issued - consumed < Tr::NS) {
      const bool new_frag = (prod.j == prod.j0);
      if (new_frag && prod.frag_idx >= it.frag_idx + 2) break;  // raw-q double buffer busy
      // block-table entry (warp-collective cached slice)
      if (prod.s != tb_seq || prod.j < tb_base || prod.j >= tb_base + 32) {
        tb_seq = prod.s;
        tb_base = prod.j;
        const int jj = prod.j + lane;
        tb_val = (jj < prod.nb) ? __ldg(p.block_tables + static_cast<int64_t>(prod.s) * p.max_blocks_per_seq + jj) : -1;
      }
      int phys = __shfl_sync(0xffffffffu, tb_val, prod.j - tb_base);
      if (phys < 0 || phys >= p.num_blocks) {
        if (lane == 0) raise_error(p.err, PA_DEVERR_BLOCK_ID);
        phys = 0;
      }
      if (lane == 0) {
        const int st = issued % Tr::NS;
        const uint32_t bar = bar0 + 8 * st;
        const uint32_t kdst = wbase_u32 + st * Tr::STAGE;
        const uint32_t vdst = kdst + Tr::TILE;
        const uint32_t qbytes = new_frag ? static_cast<uint32_t>(G * D * 2) : 0u;
        mbar_arrive_expect_tx(bar, 2u * Tr::TILE + qbytes);
        const int row = (phys * Hkv + prod.kvh) * BS;
#pragma unroll
        for (int sub = 0; sub < Tr::NSUB; ++sub) {
          tma_load_2d(kdst + sub * (BS * 128), &tmap_k, sub * Tr::SUB_ELEMS, row, bar);
          tma_load_2d(vdst + sub * (BS * 128), &tmap_v, sub * Tr::SUB_ELEMS, row, bar);
        }
        if (new_frag) {
          const uint8_t* qsrc = static_cast<const uint8_t*>(p.q) +
                                (static_cast<int64_t>(prod.s) * p.q_stride + static_cast<int64_t>(prod.kvh) * G * D) * 2;
          bulk_load(qraw_u32 + (prod.frag_idx & 1) * kQrawStride, qsrc, qbytes, bar);
        }
      }
      ++issued;
      if (++prod.j == prod.jend) iter_next_fragment<BS>(prod, prefix, p, fixed);
    }
  };

  produce();

  const int t = lane % BS;     // token of this lane in QK
  const int half = lane / BS;  // d-half of this lane in QK (B=16)
  const int e0 = lane * Tr::EPL;  // first PV column of this lane
  const int vsub = e0 / Tr::SUB_ELEMS;
  const int vbyte = (e0 % Tr::SUB_ELEMS) * Tr::KVB;

  float m[GM], l[GM];
  float2 acc[GM][Tr::EPL / 2];

  while (it.valid) {
    const int st = consumed % Tr::NS;
    const uint32_t parity = (consumed / Tr::NS) & 1;
    if (!mbar_wait_bounded(bar0 + 8 * st, parity, kWaitLimitNs)) {
      timed_out = true;
      break;
    }
    if (it.j == it.j0) {
      // new fragment: widen + pre-scale the query group, reset the state
      float qs = p.qk_scale_log2;
      if constexpr (kFp8) qs *= __ldg(p.k_scale + it.kvh);
      const uint8_t* qr = qraw_base + (it.frag_idx & 1) * kQrawStride;
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
        *reinterpret_cast<float2*>(qf + g * Tr::QROW + (ed / Tr::HALF) * (Tr::HALF + Tr::QPAD) + ed % Tr::HALF) = v2;
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

    const int n_valid = min(BS, it.T - it.j * BS);
    const uint32_t kst = wbase_u32 + st * Tr::STAGE;
    const uint32_t vst = kst + Tr::TILE;

    // ---- scores: lane (t, half) dots its half-row of K with all G query heads
    float2 sacc[GM];
#pragma unroll
    for (int g = 0; g < GM; ++g) sacc[g] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < Tr::CPL; ++c) {
      const int cg = half * Tr::CPL + c;
      const uint32_t kaddr = kst + (cg >> 3) * (BS * 128) + t * 128 + (((cg & 7) ^ (t & 7)) << 4);
      const uint4 raw = lds128(kaddr);
      float2 kf[Tr::EPC / 2];
      Chunk<KVT>::cvt(raw, kf);
      const int qoff = half * (Tr::HALF + Tr::QPAD) + c * Tr::EPC;
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        const float4* qp = reinterpret_cast<const float4*>(qf + g * Tr::QROW + qoff);
#pragma unroll
        for (int i = 0; i < Tr::EPC / 4; ++i) {
          const float4 q4 = qp[i];
          sacc[g] = ffma2(make_float2(q4.x, q4.y), kf[2 * i], sacc[g]);
          sacc[g] = ffma2(make_float2(q4.z, q4.w), kf[2 * i + 1], sacc[g]);
        }
      }
    }
    const bool tok_ok = t < n_valid;
    float alpha[GM];
    bool rescale = false;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      float sv = sacc[g].x + sacc[g].y;
      if constexpr (Tr::LPT == 2) sv += __shfl_xor_sync(0xffffffffu, sv, 16);
      sv = tok_ok ? sv : -INFINITY;
      float bm = sv;
#pragma unroll
      for (int o = 1; o < BS; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
      const float mn = fmaxf(m[g], bm);
      alpha[g] = exp2f(m[g] - mn);
      rescale |= (alpha[g] != 1.f);
      m[g] = mn;
      const float pg = tok_ok ? exp2f(sv - mn) : 0.f;
      l[g] = l[g] * alpha[g] + (half == 0 ? pg : 0.f);
      sacc[g].x = pg;  // keep p for the store below
    }
    if (half == 0) {
#pragma unroll
      for (int g = 0; g < GM; g += 2) {
        const float pa = sacc[g].x;
        const float pb = (g + 1 < GM) ? sacc[g + 1].x : 0.f;
        if (g + 1 < GM) {
          *reinterpret_cast<float4*>(pbuf + t * GM + g) = make_float4(pa, pa, pb, pb);
        } else {
          pbuf[t * GM + g] = make_float2(pa, pa);
        }
      }
    }
    __syncwarp();
    if (rescale) {
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
        for (int i = 0; i < Tr::EPL / 2; ++i) acc[g][i] = fmul2(acc[g][i], a2);
      }
    }

    // ---- p . V: lane owns columns e0..e0+EPL-1 of all G heads
    for (int tt = 0; tt < n_valid; ++tt) {
      const uint32_t vaddr = vst + vsub * (BS * 128) + tt * 128 + ((((vbyte >> 4) ^ (tt & 7))) << 4) + (vbyte & 15);
      float2 vf[Tr::EPL / 2];
      if constexpr (Tr::KVB == 2) {
        if constexpr (Tr::EPL == 4) {
          uint32_t w0, w1;
          asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(vaddr));
          vf[0] = widen2<KVT>(w0);
          vf[1] = widen2<KVT>(w1);
        } else {
          uint32_t w0;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(vaddr));
          vf[0] = widen2<KVT>(w0);
        }
      } else {
        static_assert(Tr::EPL == 4 || Tr::KVB == 2, "fp8 path needs 4 columns per lane");
        uint32_t w0;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(vaddr));
        vf[0] = widen2_e4m3(w0 & 0xffffu);
        vf[1] = widen2_e4m3(w0 >> 16);
      }
#pragma unroll
      for (int g = 0; g < GM; g += 2) {
        if (g + 1 < GM) {
          const float4 pp = *reinterpret_cast<const float4*>(pbuf + tt * GM + g);
#pragma unroll
          for (int i = 0; i < Tr::EPL / 2; ++i) {
            acc[g][i] = ffma2(make_float2(pp.x, pp.y), vf[i], acc[g][i]);
            acc[g + 1][i] = ffma2(make_float2(pp.z, pp.w), vf[i], acc[g + 1][i]);
          }
        } else {
          const float2 pp = pbuf[tt * GM + g];
#pragma unroll
          for (int i = 0; i < Tr::EPL / 2; ++i) acc[g][i] = ffma2(pp, vf[i], acc[g][i]);
        }
      }
    }
    __syncwarp();
    ++consumed;

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
          seg_start = prefix[it.s] + static_cast<long long>(it.kvh) * it.nb;
          const long long seg_last = seg_start + it.nb - 1;
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
    if (++it.j == it.jend) iter_next_fragment<BS>(it, prefix, p, fixed);
    produce();
  }

  if (timed_out) {
    if (lane == 0) raise_error(p.err, PA_DEVERR_TIMEOUT);
    // let this warp's copies in flight land before the CTA can exit
    for (int k = consumed; k < issued; ++k)
      (void)mbar_wait_bounded(bar0 + 8 * (k % Tr::NS), (k / Tr::NS) & 1, kWaitLimitNs);
  }
}

// ----------------------------------------------------------------- host side of one variant

template <typename QT, typename KVT, int D, int BS, int GM>
struct DecodeVariant {
  using Tr = DecodeTraits<QT, KVT, D, BS, GM>;

  static size_t smem_bytes(int num_seqs) {
    return 1024 + static_cast<size_t>(Tr::W) * Tr::WARP_SMEM +
           static_cast<size_t>(align_up_c((num_seqs + 1 + Tr::W) * 4, 16));
  }

  static bool geometry(int num_seqs, DecodeGeometry* g) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    const size_t smem = smem_bytes(num_seqs);
    auto kern = paged_decode_kernel<QT, KVT, D, BS, GM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
      return false;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Tr::W * 32, smem) != cudaSuccess || occ < 1)
      return false;
    g->warps_per_cta = Tr::W;
    g->ctas = sms * occ;
    g->smem_bytes = smem;
    g->record_floats = Tr::REC;
    return true;
  }

  static cudaError_t launch(const DecodeGeometry& g, const DecodeParams& p, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t stream) {
    paged_decode_kernel<QT, KVT, D, BS, GM><<<g.ctas, Tr::W * 32, g.smem_bytes, stream>>>(tk, tv, p);
    return cudaGetLastError();
  }
};

}  // namespace pa

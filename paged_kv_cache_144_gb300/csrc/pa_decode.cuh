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
// recurrence runs in base 2 with log2(e) folded into the scale.
//
// How it is laid out on GB300 (this is not the pages' A100 kernel design):
//  * Work unit = UR (32; 64 for 8-bit caches) consecutive rows of one (sequence, KV head).
//    A unit is filled by 3-D TMA boxes of min(UR, B) whole rows: part of one
//    block when B >= UR, one box per block when a unit spans several blocks;
//    one TMA instruction per box for K and one for V.  A box lands as
//    [128-byte half of the row][row][128 bytes] with the 128-byte swizzle, so
//    each half-plane is swizzled by row.  The units of the whole batch,
//    ordered (s, kvh, unit), are split into equal contiguous ranges, one per
//    resident warp, so long and short sequences load every SM equally
//    ("balanced" mode).  A range crosses (s, kvh) segments freely.
//    Optionally each warp instead takes fixed partitions of P tokens.
//  * Warp specialisation: each CTA has W consumer warps and one producer
//    warp.  Consumer warp c owns a ring of stages in shared memory (one unit
//    of K, of V and, at a segment start, the query group per stage; several
//    queries per sequence keep their query rows in one buffer per ring).
//    Lane c of the producer warp walks consumer c's units: it waits for the
//    stage's "empty" mbarrier, reads the block table, and issues the TMA
//    copies (cp.async.bulk.tensor) plus a 1-D bulk copy of the query group,
//    all completing on the stage's "full" mbarrier.  Consumers only wait,
//    compute and release.  No CTA-wide barrier is used after the prologue.
//    Under a programmatic dependent launch the producer may issue the K/V of
//    its first units before the kernel before has finished when the caller
//    guarantees that kernel writes no row of them (early_kv).
//  * The two contractions of a unit run on the tensor cores (mma.sync
//    m16n8k16, fp32 accumulate) in the register layout of that instruction.
//    One query per sequence: S = K Q^T with 16 tokens per m-tile and the
//    G <= 8 query rows as N; each 8 x 8 half of the probabilities is
//    transposed in registers (movmatrix) into the B operand of
//    O^T += V^T P^T (16 head_dim columns per m-tile).  Several queries:
//    S^T = Q K^T with 16 (query, head) rows per warp as M, whose C fragment
//    is the B operand of O^T += V^T P^T as it is.  At the GB300's ratio of
//    issue slots to HBM bytes the fp32-FMA formulation of these products is
//    instruction-bound; the tensor-core one is not.  The probabilities enter
//    the second product as a hi + lo pair of 16-bit values (two MMAs), which
//    keeps their rounding error near 2^-16 relative.
//  * 16-bit caches feed the MMAs with ldmatrix (K) and ldmatrix.trans (V)
//    straight from the swizzled tiles.  8-bit caches are widened in registers
//    (e4m3 -> f16x2; INT8 K as code - zero point, INT8 V as 1152 + code with
//    (1152 + zero point) * v_scale subtracted from the output, all exact) with
//    the head_dim order of QK permuted so that a lane reads 16 contiguous
//    bytes of a K row, and V transposed in registers with byte permutes; the
//    per-head K scale multiplies the scores, the V scale the final divide,
//    and a bf16 query enters the f16 product scaled by a power of two that
//    puts the group's largest element at 2^14 .. 2^15 (no overflow, no lost
//    bits within 2^28 of that element).
//  * Split segments: a warp whose range covers only part of a segment writes
//    its (m, l, acc) record to the workspace and arrives on the segment's
//    counter (a release atomic whose result it reads one fragment later, so
//    arriving never stalls it; the ring's final fragment arrives with an
//    acquire as well); the warp that arrived last merges all records with the
//    same recurrence after its own unit loop, one row per lane, writes
//    out[s, kvh*G .. kvh*G+G-1] and resets the counter.  Nothing waits on
//    another warp, so the kernel cannot deadlock.
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
constexpr int kTablePrefetch = 3;              // units whose table entries the producer fetches ahead
constexpr int64_t kTableL2Bytes = 2 << 20;     // block tables up to this size are prefetched into L2 at entry

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
  static constexpr int UR = UR_;                 // rows per work unit (32; 64 for 8-bit caches)
  static_assert(UR == 32 || (UR == 64 && KVB == 1), "unit rows");
  static constexpr int UR_SHIFT = UR == 64 ? 6 : 5;
  static constexpr int NSUB = ROW / 128;         // 128-byte halves per row
  static constexpr int TILE = UR * ROW;          // bytes of one unit of K (or V)
  static constexpr int QRAW = GM * D * 2;        // bytes of one raw query group
  static constexpr int STAGE = align_up_c(2 * TILE + QRAW, 1024);  // K tile + V tile + raw q
  // fused append: each stage can also stage the new K and V rows (16-bit
  // source format) and the physical block that receives them
  static constexpr int OFF_NEW = 2 * TILE + QRAW;
  static constexpr int NEWB = 2 * D * 2 + 16;
  static constexpr int STAGE_APPEND = align_up_c(2 * TILE + QRAW + NEWB, 1024);
  static constexpr int MAX_NS = 8;               // stages per consumer (chosen at launch, 2..MAX_NS)
  static constexpr int MAX_W = 7;                // consumer warps per CTA (with the producer: 8 warps, up to 255 registers)
  static constexpr int KS = D / 16;              // k-steps of S^T = Q K^T, m-tiles of O^T
  static constexpr int NT = UR / 8;              // 8-token n-tiles of a unit
  static constexpr int NSB = UR / 16;            // 16-token sub-tiles (one PV k-step each)
  static constexpr bool B8 = KVB == 1;          // FP8-e4m3 or INT8 cache
  static constexpr bool MMA_BF16 = !B8 && std::is_same<KVT, bf16_t>::value;  // else f16
  static_assert(!B8 || D == 128, "8-bit caches: head_dim 128");
  // per-consumer shared memory: [full[MAX_NS] | empty[MAX_NS] | NS stages]
  static constexpr int OFF_FULL = 0;
  static constexpr int OFF_EMPTY = OFF_FULL + MAX_NS * 8;
  static constexpr int OFF_MERGE = OFF_EMPTY + MAX_NS * 8;  // one barrier per warp of the ring: its merge copies
  static constexpr int OFF_QEMPTY = OFF_MERGE + 4 * 8;      // several queries: the ring's query buffer is free
  static constexpr int OFF_STAGES = 1024;
  static_assert(OFF_QEMPTY + 8 <= OFF_STAGES, "barriers");
  // Several queries per sequence (16-row variants): the query rows of a
  // fragment (16 per consumer warp of the ring) live in one buffer per ring,
  // after its stages, instead of an area in every stage.
  __host__ __device__ static constexpr int qbuf_bytes(int nc) { return GM > 8 ? align_up_c(16 * nc * D * 2, 1024) : 0; }
  __host__ __device__ static constexpr int warp_smem(int ns, int stage) { return OFF_STAGES + ns * stage; }
  // partial record: acc as [D][GM] (head fastest), then m[GM], l[GM]
  static constexpr int REC = align_up_c(GM * (D + 2), 4);
  // the split merge stages records in a consumer's (at least two) idle stages
  static_assert(2 * STAGE >= REC * 4, "a record fits the stages of one consumer");
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
  int s, kvh, j, jend, j0, T;
  int nu;         // units of the segment that are attended (from unit ulo on)
  int ulo;        // first attended unit of the sequence
  int lo;         // first attended position (sliding window), 0 without one
  int nblk;       // blocks that hold rows of sequence s
  int frag_idx;   // ordinal of the current fragment within this warp
  int slot;       // partial-record slot, -1 when the fragment is a whole segment
  bool valid;
  // balanced mode: positions in the cost order (see frag_balanced)
  long long u, u1;  // start of the current fragment; end of the ring's range
  long long fend;   // end of the current fragment
  int gw;           // global ring id
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

// First attended position of a sequence of length T: that of its first
// query (position T - q_len) under a sliding window, else 0.
__device__ __forceinline__ int window_lo(const DecodeParams& p, int T) {
  const int first = T - p.q_len + 1;
  return (p.window > 0 && first > p.window) ? first - p.window : 0;
}

// Balanced split in cost order.  The units of the batch are laid out
// segment by segment, (s, kvh) in order, each segment charged its nu
// attended units plus p.frag_cost for the work a fragment costs besides its
// units (query set-up, the last partial unit, the output or record): segment
// x occupies positions [c_x, c_x + frag_cost + nu), its unit j at
// c_x + frag_cost + j.  The positions are split into equal contiguous
// ranges, one per ring, and a ring owns the units whose positions fall in its
// range, so a ring whose range crosses many short segments gets fewer units.
// A range boundary inside a segment's leading overhead assigns the whole
// segment to the later ring.  prefix[s] = position of sequence s's first
// segment (its H_kv segments are consecutive, each of the same cost).
//
// Fills the fragment starting at it.u (the first of its units at or after
// it.u); returns false when the ring's range holds no further unit.  it.s is
// a sequence with prefix[it.s] <= it.u (the ring's positions only grow): the
// sequence of it.u is found by scanning forward from it, one or two
// shared-memory reads per fragment, not a search over the whole batch.
__device__ __forceinline__ bool frag_balanced(WorkIter& it, const int* prefix, const DecodeParams& p, int ur_shift) {
  const int Hkv = p.num_kv_heads;
  const int beta = p.frag_cost;
  int s = it.s;
  while (it.u < it.u1) {
    while (s + 1 < p.num_seqs && prefix[s + 1] <= it.u) ++s;  // last s with prefix[s] <= u
    const int seg = (prefix[s + 1] - prefix[s]) / Hkv;  // frag_cost + nu of each segment of sequence s
    const int r = static_cast<int>(it.u - prefix[s]);  // < 2^31: positions are int32
    const int kvh = r / seg;
    const int off = r - kvh * seg;
    const long long seg_start = prefix[s] + static_cast<long long>(kvh) * seg;
    const long long fend = min(it.u1, seg_start + seg);
    const int ja = max(0, off - beta);                        // first unit of the segment in the range
    const int jb = static_cast<int>(fend - seg_start) - beta;  // units of the segment before fend
    if (jb <= ja) {  // the range ends inside the segment's overhead: none of its units
      it.u = fend;
      continue;
    }
    const int nu = seg - beta;
    it.s = s;
    it.nu = nu;
    it.T = prefix[p.num_seqs + 1 + s];  // clamped length, cached by the prologue
    it.lo = window_lo(p, it.T);
    it.ulo = it.lo >> ur_shift;
    it.kvh = kvh;
    it.j0 = it.ulo + ja;
    it.j = it.j0;
    it.jend = it.ulo + jb;
    it.fend = fend;
    const bool whole = ja == 0 && jb == nu;
    it.slot = whole ? -1 : it.gw * 2 + (it.frag_idx == 0 ? 0 : 1);
    it.nblk = (it.T + p.block_size - 1) >> p.block_shift;
    return true;
  }
  return false;
}

// INT8 caches: (1152 + zp) * v_scale, from the staged f16x2(1152 + zp) word
// (1152 + zp is exact in f16).  V enters the products as 1152 + code, so the
// output is acc * v_scale / l minus this.
__device__ __forceinline__ float v_bias_offset(uint32_t zp2, float vs) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(zp2 & 0xffffu))) * vs;
}

// Ring containing cost position x of a balanced split of C positions over nw rings.
__device__ __forceinline__ int ring_of(long long x, long long C, int nw) {
  return static_cast<int>(((x + 1) * nw - 1) / C);
}

__device__ __forceinline__ void frag_fixed(WorkIter& it, const int* prefix, const DecodeParams& p, int ur_shift) {
  const int Hkv = p.num_kv_heads;
  const int s = find_seq(prefix, p.num_seqs, it.r);
  const int parts = (prefix[s + 1] - prefix[s]) / Hkv;
  const int rr = it.r - prefix[s];
  it.s = s;
  it.kvh = rr / parts;
  const int part = rr % parts;
  it.T = prefix[p.num_seqs + 1 + s];  // clamped length, cached by the prologue
  it.lo = window_lo(p, it.T);
  it.ulo = it.lo >> ur_shift;
  const int nu_all = (it.T + (1 << ur_shift) - 1) >> ur_shift;
  it.nu = nu_all - it.ulo;
  it.nblk = (it.T + p.block_size - 1) >> p.block_shift;
  it.j0 = it.ulo + part * p.partition_units;
  it.j = it.j0;
  it.jend = min(nu_all, it.j0 + p.partition_units);
  it.slot = (parts == 1) ? -1 : it.r;
}

__device__ __forceinline__ void iter_next_fragment(WorkIter& it, const int* prefix, const DecodeParams& p,
                                                   bool fixed, int ur_shift) {
  it.frag_idx++;
  if (fixed) {
    it.r += it.rstride;
    if (it.r >= it.R) { it.valid = false; return; }
    frag_fixed(it, prefix, p, ur_shift);
  } else {
    it.u = it.fend;
    if (!frag_balanced(it, prefix, p, ur_shift)) it.valid = false;
  }
}

// Where the partial record of fragment f of a split segment lives.
struct MergeSlots {
  bool fixed;
  int fixed_base;       // fixed partitions: slot of partition 0 of the segment
  int first_w;          // balanced split: global warp id of the first fragment
  long long U;          // balanced split: total cost positions
  int nw_eff;           // balanced split: rings sharing them
  long long seg_start;  // balanced split: first unit of the segment
  int nc, rg;           // warps per ring and this warp's row group: records are per warp
  __device__ __forceinline__ int slot(int f) const {
    if (fixed) return (fixed_base + f) * nc + rg;
    const int w = first_w + f;
    const long long rs = static_cast<long long>(w) * U / nw_eff;
    return (2 * w + (rs < seg_start ? 1 : 0)) * nc + rg;
  }
};

// Merges the nfr partial (m, l, acc) records of one segment with the
// online-softmax recurrence and writes the output rows of its R (query, head)
// rows row0 .. row0 + R - 1 (of the segment's q_len * G rows).  Run by the
// warp that arrived last, after its unit loop, when its own pipeline stages
// are idle: the records are copied into those stages (buf / bufp, room for
// cap records) a batch at a time, lane k issuing one bulk copy of record k,
// all completing on the warp's merge barrier `mbar` (phase parity tracked in
// `mpar`), and folded from shared memory.
//
// A record's accumulator is [D][GM] floats (row fastest), so element
// lane + 32 j of it belongs to row lane % GM: each lane folds one row (its
// running maximum M, sum L and D * GM / 32 elements of it) and reads the
// batch with consecutive lanes on consecutive words (no bank conflicts, no
// shuffles: a lane computes its row's weights e^(m_k - M) itself).  A batch
// that raises M rescales what was folded before (the same recurrence across
// batches).  Records are folded in fragment order, so the result does not
// depend on which warp merges.  The rows leave through shared memory
// (swizzled by 16-byte chunk) as whole rows, 16 bytes per lane.
template <int GM, int D, int REC>
__device__ __forceinline__ void merge_segment(const float* records, const MergeSlots& ms, int nfr, int lane, int R,
                                              int G, int num_heads, float vs, float voff, void* out, int out_dtype,
                                              int64_t seq_row0, int row0, uint32_t buf, float* bufp,
                                              int cap, uint32_t mbar, uint32_t& mpar, unsigned int* err) {
  constexpr int PER = GM * D / 32;  // accumulator elements per lane
  static_assert(REC % 4 == 0, "records are whole 16-byte chunks");
  static_assert(32 % GM == 0 && D % 32 == 0 && GM * D <= REC, "one row per lane; output staging fits a record");
  cap = cap < 32 ? cap : 32;  // one bulk copy per lane
  const int g = lane % GM;    // the row this lane folds
  float M = -INFINITY, L = 0.f, o[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) o[j] = 0.f;
#pragma unroll 1
  for (int f0 = 0; f0 < nfr; f0 += cap) {
    const int nb = min(cap, nfr - f0);
    const int my_slot = lane < nb ? ms.slot(f0 + lane) : 0;
    if (lane == 0) mbar_arrive_expect_tx(mbar, static_cast<uint32_t>(nb * REC * 4));
    __syncwarp();
    if (lane < nb) bulk_load(buf + static_cast<uint32_t>(lane * REC) * 4, records + static_cast<int64_t>(my_slot) * REC,
                             REC * 4, mbar);
    if (!mbar_wait_bounded(mbar, mpar, kDefaultWaitLimitNs) && lane == 0) raise_error(err, PA_DEVERR_TIMEOUT);
    mpar ^= 1;
    __syncwarp();  // every lane sees the batch
    float mb = -INFINITY;
    for (int k = 0; k < nb; ++k) mb = fmaxf(mb, bufp[k * REC + GM * D + g]);
    const float mn = fmaxf(M, mb);
    const float resc = M == -INFINITY ? 0.f : exp2f(M - mn);  // nothing folded yet: 0
    L *= resc;
#pragma unroll
    for (int j = 0; j < PER; ++j) o[j] *= resc;
    M = mn;
    constexpr int kUnrollRecords = GM > 8 ? 2 : 4;  // records folded together (registers: PER per record)
#pragma unroll kUnrollRecords
    for (int k = 0; k < nb; ++k) {
      const float* rk = bufp + k * REC;
      const float mk = rk[GM * D + g];
      const float w = mk == -INFINITY ? 0.f : exp2f(mk - mn);  // an empty record (its rows saw nothing) weighs 0
      L = fmaf(w, rk[GM * D + GM + g], L);
#pragma unroll
      for (int j = 0; j < PER; ++j) o[j] = fmaf(w, rk[lane + 32 * j], o[j]);
    }
    __syncwarp();  // every lane has read the batch before the next one overwrites it
  }
  // rows through shared memory: element (row g, column d) at row g, 16-byte
  // chunk (d / 4) ^ (g % 8), so that both the writes and the row reads below
  // spread over the banks
  const float inv = L > 0.f ? vs / L : 0.f, off = L > 0.f ? voff : 0.f;  // a row that saw nothing: 0
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int d = (lane + 32 * j) / GM;
    bufp[g * D + ((((d >> 2) ^ (g & 7)) << 2) | (d & 3))] = fmaf(o[j], inv, -off);
  }
  __syncwarp();
  const bool vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  for (int r = 0; r < R; ++r) {
    // row row0 + r = (query (row0 + r) / G, head (row0 + r) % G) of the group
    const int64_t orow = GM > 8 ? seq_row0 + static_cast<int64_t>((row0 + r) / G) * num_heads + (row0 + r) % G
                                : seq_row0 + r;
    for (int c = lane; c < D / 4; c += 32) {
      const float4 v = *reinterpret_cast<const float4*>(bufp + r * D + ((c ^ (r & 7)) << 2));
      store_out4(out, out_dtype, orow * D + 4 * c, v, vec);
    }
  }
  // the next merge's bulk copies overwrite this staging area
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

template <typename QT, typename KVT, int D, int GM, int UR_, int AP>
__global__ void __launch_bounds__((DecodeTraits<QT, KVT, D, GM, UR_>::MAX_W + 1) * 32, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const DecodeParams p) {
  using Tr = DecodeTraits<QT, KVT, D, GM, UR_>;
  constexpr bool k8bit = elem<KVT>::bytes == 1;
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
  const int upb_shift = unit_in_block ? p.block_shift - Tr::UR_SHIFT : 0;  // log2(units per block)
  const int bpu_shift = unit_in_block ? 0 : Tr::UR_SHIFT - p.block_shift;  // log2(blocks per unit)
  const bool fixed = p.partition_units > 0;

  const int NS = p.stages;  // pipeline depth per ring
  // fused append (AP): stages also carry the new K/V rows
  constexpr bool append = AP != 0;
  // Several queries per sequence (16-row variants): the R = q_len * G rows of
  // a segment are served by NC = ceil(R / 16) consumer warps that share one
  // ring, warp k of the ring taking rows 16k .. 16k + 15 of every unit; the
  // ring's query buffer holds all 16 * NC rows.  Otherwise one warp per ring.
  constexpr bool kMQ = GM > 8;
  const int NC = kMQ ? p.row_groups : 1;
  const int RW = W / NC;  // rings per CTA, each fed by producer lane 0 .. RW-1
  const int STG = kMQ ? p.stage_bytes : (append ? Tr::STAGE_APPEND : Tr::STAGE);
  const int OFF_QBUF = Tr::warp_smem(NS, STG);       // several queries: the ring's query buffer
  const int wsm = OFF_QBUF + Tr::qbuf_bytes(NC);      // bytes per ring (a multiple of 1024)
  // shared: prefix[S+1] (units before sequence s), lens[S] (clamped seq_lens),
  // scan scratch, then the producer's block-table ring (16 ints per ring)
  int* prefix = reinterpret_cast<int*>(base + RW * wsm);
  int* lens = prefix + (S + 1);
  int* scan_tmp = lens + S;
  // 8-bit caches: the per-KV-head K scale, V scale and (INT8) zero-point
  // constants, staged once per CTA so that no fragment waits on them
  float* hp_ks = reinterpret_cast<float*>(scan_tmp + NWARP);
  float* hp_vs = hp_ks + kMaxHeadParams;
  uint32_t* hp_zk = reinterpret_cast<uint32_t*>(hp_vs + kMaxHeadParams);
  uint32_t* hp_zv = hp_zk + kMaxHeadParams;
  constexpr int kHeadWords = Tr::B8 ? 4 * kMaxHeadParams : 0;
  const uint32_t table_ring_u32 = base_u32 + RW * wsm + align_up_c((2 * S + 1 + NWARP + kHeadWords) * 4, 16);

  // A kernel launched after this one with programmatic serialization (the
  // next step's cache write) may be scheduled now; it waits for this grid
  // before it touches memory.
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }

  // ---- 0. the block tables are brought into L2 while the lengths are read,
  // so that the producers' first table reads (which need the lengths) hit L2
  // (tables up to kTableL2Bytes; the block tables are never written here)
  {
    const int64_t tbytes = static_cast<int64_t>(S) * p.max_blocks_per_seq * 4;
    if (tbytes <= kTableL2Bytes) {
      const char* tb = reinterpret_cast<const char*>(p.block_tables);
      for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i * 128 < tbytes;
           i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        prefetch_l2(tb + i * 128);
    }
  }

  // ---- 1. units per sequence and their exclusive prefix sums (every CTA)
  {
    int carry = 0;
    for (int b0 = 0; b0 < S; b0 += blockDim.x) {
      const int s = b0 + threadIdx.x;
      int units = 0;
      if (s < S) {
        const int T = clamped_len(p, s, blockIdx.x == 0);
        lens[s] = T;
        const int nu = ((T + UR - 1) >> Tr::UR_SHIFT) - (window_lo(p, T) >> Tr::UR_SHIFT);
        // fixed: partitions; balanced: cost positions (units + fragment overhead)
        units = (fixed ? (nu + p.partition_units - 1) / p.partition_units : (nu > 0 ? nu + p.frag_cost : 0)) * Hkv;
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

  // ---- 2. barriers of every ring: a stage is full once its copies land and
  // empty once each of the ring's NC consumer warps has released it
  if (threadIdx.x == 0) {
    for (int c = 0; c < RW; ++c) {
      const uint32_t cb = base_u32 + c * wsm;
      for (int i = 0; i < NS; ++i) {
        mbar_init(cb + Tr::OFF_FULL + 8 * i, 1);
        mbar_init(cb + Tr::OFF_EMPTY + 8 * i, NC);
      }
      for (int k = 0; k < NC; ++k) mbar_init(cb + Tr::OFF_MERGE + 8 * k, 1);
      if (kMQ) mbar_init(cb + Tr::OFF_QEMPTY, NC);
    }
    fence_mbar_init();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  // ---- 3. the share of ring c (global ring id gc)
  const int nw_total = gridDim.x * RW;
  const long long U = prefix[S];  // partitions (fixed) or cost positions (balanced) of the batch
  const int min_share = kMinUnitsPerWarp + (fixed ? 0 : p.frag_cost);
  long long want = (U + min_share - 1) / min_share;
  const int nw_eff = fixed ? nw_total : static_cast<int>(want < 1 ? 1 : (want < nw_total ? want : nw_total));
  auto start_iter = [&](WorkIter& w, int gc) {
    w.frag_idx = 0;
    w.gw = gc;
    w.valid = false;
    if (fixed) {
      w.R = static_cast<int>(U);
      w.rstride = nw_total;
      w.r = gc;
      if (w.r < w.R) { w.valid = true; frag_fixed(w, prefix, p, Tr::UR_SHIFT); }
    } else if (U > 0 && gc < nw_eff) {
      w.u = gc * U / nw_eff;
      w.u1 = (gc + 1) * U / nw_eff;
      w.s = find_seq(prefix, S, w.u);
      w.valid = frag_balanced(w, prefix, p, Tr::UR_SHIFT);
    }
  };

  if (warp == 0) {
    // =================================================================== producer
    // Lane c feeds consumer c: one unit per free stage of its ring.  The
    // block-table entries of a unit are copied into shared memory
    // (cp.async, no register dependency) kTablePrefetch units before the
    // unit is issued, so that a table read never stalls the warp.
    WorkIter it, ah;  // next unit to issue; next unit whose table entries to fetch
    it.valid = false;
    if (lane < RW) start_iter(it, blockIdx.x * RW + lane);
    ah = it;
    const uint32_t cbase = base_u32 + (lane < RW ? lane : 0) * wsm;
    const uint32_t ring = table_ring_u32 + (lane < RW ? lane : 0) * 64;  // 4 units x 4 entries
    int pst = 0, pph = 1, issued = 0;
    int pf = 0, rs_use = 0, rs_pf = 0;  // units fetched ahead; ring slots to read / fill
    uint64_t wait_since = 0;
    // boxes [first_box, nbox) of a unit hold attended rows: blocks wholly
    // before a sliding window are neither looked up nor loaded
    auto first_box = [&](const WorkIter& w, int bj) {
      return unit_in_block ? 0 : max(0, (w.lo >> p.block_shift) - bj);
    };
    auto fetch_tables = [&]() {
      const int bj = unit_in_block ? (ah.j >> upb_shift) : (ah.j << bpu_shift);
      const int nb = unit_in_block ? 1 : min(1 << bpu_shift, ah.nblk - bj);
      const int i0 = first_box(ah, bj);
      const int32_t* src = p.block_tables + static_cast<int64_t>(ah.s) * p.max_blocks_per_seq + bj;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i >= i0 && i < nb) cp_async4(ring + (rs_pf * 4 + i) * 4, src + i);
      cp_async_commit();
      rs_pf = (rs_pf + 1) & 3;
      ++pf;
      if (++ah.j == ah.jend) iter_next_fragment(ah, prefix, p, fixed, Tr::UR_SHIFT);
    };
    while (ah.valid && pf < kTablePrefetch) fetch_tables();
    int nq = 0;  // several queries: query loads issued into this lane's ring buffer
    // Issues unit `it` into stage pst (its K/V boxes, the query group at a
    // fragment start, the appended rows) and advances.  early: the grid
    // before this one may still be running (early_kv), so the stage is only
    // armed with its byte count; the query copy (early_q) and the producer's
    // arrival, which releases the head constants written after the wait,
    // come after the wait.
    int n_early = 0;
    int early_q[Tr::MAX_NS];  // per early stage: segment s * H_kv + kvh whose query group it carries, or -1
    auto issue_unit = [&](bool early) {
      const bool new_frag = (it.j == it.j0);
      const uint32_t bar = cbase + Tr::OFF_FULL + 8 * pst;
      const uint32_t kdst = cbase + Tr::OFF_STAGES + pst * STG;
      const uint32_t vdst = kdst + Tr::TILE;
      const int bj0 = unit_in_block ? (it.j >> upb_shift) : (it.j << bpu_shift);
      const int nbox = unit_in_block ? 1 : min(1 << bpu_shift, it.nblk - bj0);
      const int box0 = first_box(it, bj0);
      const int row_in_block = unit_in_block ? (it.j - (bj0 << upb_shift)) * UR : 0;
      const int qlen = GM > 8 ? p.q_len : 1;  // only 16-row variants serve several queries
      const uint32_t qbytes = new_frag ? static_cast<uint32_t>(qlen * G * D * 2) : 0u;
      // this unit's entries were fetched pf - 1 units before the newest fetch
      if (pf >= 3) {
        cp_async_wait<2>();
      } else if (pf == 2) {
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      int phys[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        phys[i] = (i >= box0 && i < nbox) ? static_cast<int>(lds32(ring + (rs_use * 4 + i) * 4)) : 0;
      rs_use = (rs_use + 1) & 3;
      --pf;
      // fused append: this unit holds position T-1; its new rows ride along
      const bool has_new = append && it.j == ((it.T - 1) >> Tr::UR_SHIFT);
      if (has_new) {
        const int pb = phys[((it.T - 1) >> p.block_shift) - bj0];
        st_shared_s32(kdst + Tr::OFF_NEW + 4 * D, (pb >= 0 && pb < p.num_blocks) ? pb : -1);
      }
      const uint32_t nbytes = has_new ? static_cast<uint32_t>(4 * D) : 0u;
      const uint32_t bytes = 2u * (nbox - box0) * BOX * Tr::ROW + qbytes + nbytes;
      if (early) {
        mbar_expect_tx(bar, bytes);  // armed only: the query copy and the arrival follow the wait
      } else {
        mbar_arrive_expect_tx(bar, bytes);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i >= box0 && i < nbox) {
          int pb = phys[i];
          if (pb < 0 || pb >= p.num_blocks) {
            raise_error(p.err, PA_DEVERR_BLOCK_ID);
            pb = 0;
          }
          const int z = (pb * Hkv + it.kvh) * B + row_in_block;
          tma_load_3d(kdst + i * BOX * Tr::ROW, &tmap_k, 0, z, 0, bar);
          tma_load_3d(vdst + i * BOX * Tr::ROW, &tmap_v, 0, z, 0, bar);
        }
      }
      if (early) {
        early_q[n_early++] = new_frag ? it.s * Hkv + it.kvh : -1;
      } else if (new_frag) {
        // rows (query i, head g) of the group, query-major: [q_len][G][D],
        // into the stage (one query) or the ring's query buffer (several)
        const uint32_t qdst = kMQ ? cbase + OFF_QBUF : kdst + 2 * Tr::TILE;
        for (int i = 0; i < qlen; ++i) {
          const uint8_t* qsrc =
              static_cast<const uint8_t*>(p.q) +
              (static_cast<int64_t>(it.s) * p.q_stride + (static_cast<int64_t>(i) * p.num_heads + it.kvh * G) * D) * 2;
          bulk_load(qdst + i * G * D * 2, qsrc, G * D * 2, bar);
        }
        ++nq;
      }
      if (has_new) {
        const int64_t off = (static_cast<int64_t>(it.s) * p.new_stride + static_cast<int64_t>(it.kvh) * D) * 2;
        bulk_load(kdst + Tr::OFF_NEW, static_cast<const uint8_t*>(p.k_new) + off, 2 * D, bar);
        bulk_load(kdst + Tr::OFF_NEW + 2 * D, static_cast<const uint8_t*>(p.v_new) + off, 2 * D, bar);
      }
      ++issued;
      if (++pst == NS) {
        pst = 0;
        pph ^= 1;
      }
      if (ah.valid) fetch_tables();
      if (++it.j == it.jend) iter_next_fragment(it, prefix, p, fixed, Tr::UR_SHIFT);
    };
    // Everything above reads only seq_lens and block_tables.  Under a
    // programmatic dependent launch the grid before this one on the stream
    // may still be running (it may be writing the cache, q or out); every
    // copy of q, of the scales and of the newest rows, and every write, comes
    // after it has finished.  With early_kv the caller guarantees that it
    // writes no cache row but each sequence's newest: the K/V of the ring's
    // first units that hold none of those rows are copied now.  The consumers
    // start only on stages this warp completes, so they are ordered after the
    // wait as well.
    if (p.early_kv && !append && !kMQ && !p.withhold_copies) {
      while (it.valid && issued < NS && ((it.T - 1) >> Tr::UR_SHIFT) != it.j) issue_unit(true);
    }
    griddep_wait();
    // empty sequences attend to nothing: their outputs are zero
    for (int s = blockIdx.x * 32 + lane; s < S; s += gridDim.x * 32) {
      if (lens[s] == 0) {
        const int64_t n = static_cast<int64_t>(p.q_len) * p.num_heads * D;
        for (int64_t i = 0; i < n; ++i) store_out(p.out, p.out_dtype, static_cast<int64_t>(s) * n + i, 0.f);
      }
    }
    // 8-bit caches: the per-head constants every consumer needs (read after
    // the wait: they are inputs like q).  The warp barrier orders every lane's
    // stores before each lane's first stage arrival, which the consumers
    // acquire.
    if constexpr (k8bit) {
      for (int h = lane; h < Hkv; h += 32) {
        hp_ks[h] = __ldg(p.k_scale + h);
        hp_vs[h] = __ldg(p.v_scale + h);
        if constexpr (std::is_same<KVT, i8_t>::value) {
          const uint32_t zk = __half_as_ushort(__float2half_rn(1152.f + static_cast<float>(__ldg(p.k_zero_point + h))));
          const uint32_t zv = __half_as_ushort(__float2half_rn(1152.f + static_cast<float>(__ldg(p.v_zero_point + h))));
          hp_zk[h] = zk | (zk << 16);
          hp_zv[h] = zv | (zv << 16);
        }
      }
      __syncwarp();
    }
    // the early stages: their query groups, then the arrival that completes them
    for (int i = 0; i < n_early; ++i) {
      const uint32_t bar = cbase + Tr::OFF_FULL + 8 * i;
      const int x = early_q[i];
      if (x >= 0) {
        const int s = x / Hkv, kvh = x - (x / Hkv) * Hkv;
        bulk_load(cbase + Tr::OFF_STAGES + i * STG + 2 * Tr::TILE,
                  static_cast<const uint8_t*>(p.q) +
                      (static_cast<int64_t>(s) * p.q_stride + static_cast<int64_t>(kvh) * G * D) * 2,
                  G * D * 2, bar);
      }
      mbar_arrive(bar);
    }
    if (p.withhold_copies) it.valid = false;  // testing hook: nothing is issued, every consumer wait runs out
    while (__any_sync(0xffffffffu, it.valid)) {
      bool did = false;
      if (it.valid) {
        bool ready = issued < NS || mbar_test_wait(cbase + Tr::OFF_EMPTY + 8 * pst, pph);
        // several queries: a fragment's first unit also needs the ring's query
        // buffer, free once every consumer of the ring has read the last load
        if (kMQ && ready && it.j == it.j0 && nq > 0) ready = mbar_test_wait(cbase + Tr::OFF_QEMPTY, (nq - 1) & 1);
        if (!ready) {
          const uint64_t now = global_timer_ns();
          if (wait_since == 0) {
            wait_since = now;
          } else if (now - wait_since > p.wait_limit_ns) {
            raise_error(p.err, PA_DEVERR_TIMEOUT);
            it.valid = false;  // give up on this consumer; it times out on its own
          }
        } else {
          wait_since = 0;
          issue_unit(false);
          did = true;
        }
      }
      if (!__any_sync(0xffffffffu, did)) __nanosleep(64);
    }
    // Nothing of ours may still land in shared memory after the CTA exits.
    // The table entries: cp.async groups.  The K/V/q copies: a consumer that
    // gave up (or a ring this lane gave up on) may leave stages in flight, so
    // the lane waits for the last phase it started on each stage of its
    // ring to complete, with the full limit (a copy lands within
    // microseconds; only a broken copy engine would exhaust it).
    cp_async_wait<0>();
    if (lane < RW) {
      for (int i = 0; i < NS; ++i) {
        const int n_i = issued / NS + (i < issued % NS ? 1 : 0);  // phases started on stage i
        if (n_i > 0 && !mbar_wait_bounded(cbase + Tr::OFF_FULL + 8 * i, (n_i - 1) & 1, kDefaultWaitLimitNs))
          raise_error(p.err, PA_DEVERR_TIMEOUT);
      }
    }
    return;
  }

  // ===================================================================== consumer
  constexpr bool MB = Tr::MMA_BF16;
  const int c = warp - 1;
  const int ring_id = c / NC;  // the ring this warp consumes
  const int rg = c - ring_id * NC;  // its 16-row group of the segment's rows (several queries)
  if (ring_id >= RW) return;
  WorkIter it;
  start_iter(it, blockIdx.x * RW + ring_id);
  if (!it.valid) return;
  // Under a programmatic dependent launch this CTA may be resident long
  // before the kernel before it has finished; the bounded waits below start
  // counting only after it has (at once otherwise).
  griddep_wait();
  const uint8_t* wbase = base + ring_id * wsm;
  const uint32_t wbase_u32 = base_u32 + ring_id * wsm;
  int cst = 0, cpar = 0;
  const int gid = lane >> 2;  // fragment row group: query head of S^T, column of O^T
  const int tig = lane & 3;

  // Byte offset of 16-byte chunk ch of row t in a K or V tile: a box of BOX
  // rows per block is stored as NSUB half-planes [BOX rows][128 B], each
  // swizzled by row (chunk ^ row % 8).
  const int bshift = unit_in_block ? Tr::UR_SHIFT : p.block_shift;  // log2(BOX)
  const int plane = BOX * 128;
  auto chunk_off = [&](int t, int ch) -> uint32_t {
    return static_cast<uint32_t>(((t >> bshift) * Tr::NSUB + (ch >> 3)) * plane + (t & (BOX - 1)) * 128 +
                                 (((ch & 7) ^ (t & 7)) << 4));
  };
  // offset between the two 16-row sub-tiles of a 32-row unit (same for every lane)
  const uint32_t sub_delta = BOX >= 32 ? 2048u : static_cast<uint32_t>(Tr::NSUB * 2048);

  // 16-bit tiles: the row address this lane gives to ldmatrix at k-step s
  // (K) or m-tile s (V).  Matrices 0..3 = (rows 0-7, cols lo), (rows 0-7,
  // cols hi), (rows 8-15, cols lo), (rows 8-15, cols hi) of a 16x16 block.
  uint32_t moff[Tr::KS];
  // single-query variants: K is the A operand of S = K Q^T (tokens as M);
  // matrices 0..3 = (rows 0-7, cols lo), (rows 8-15, cols lo), (rows 0-7,
  // cols hi), (rows 8-15, cols hi)
  uint32_t moffA[Tr::KS];
  // 8-bit tiles: n-position j of an 8-token n-tile holds token j ^ 4(j & 1),
  // which keeps both the K and the V loads below free of bank conflicts.
  auto sigma = [](int j) { return j ^ ((j & 1) << 2); };
  uint32_t kb8[2], vb8[2][Tr::KS / 2];
  if constexpr (!k8bit) {
    const int lt = (lane & 7) + ((lane >> 4) << 3);
    const int lhi = (lane >> 3) & 1;
#pragma unroll
    for (int s = 0; s < Tr::KS; ++s) moff[s] = chunk_off(lt, 2 * s + lhi);
    const int ltA = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int lhiA = lane >> 4;
#pragma unroll
    for (int s = 0; s < Tr::KS; ++s) moffA[s] = chunk_off(ltA, 2 * s + lhiA);
  } else {
    if constexpr (GM > 8) {
      // K as the B operand: token sigma(gid) of each n-tile, chunks tig and
      // 4 + tig (16 head_dim values each, consumed as 4 k-steps of 4 values).
      const int sg = sigma(gid);
#pragma unroll
      for (int g = 0; g < 2; ++g) kb8[g] = chunk_off(sg, 4 * g + tig);
    } else {
      // K as the A operand: m-row g of each 16-token m-tile holds token
      // sigma(g) (row g + 8: 8 + sigma(g)); the lane reads chunks 2t and
      // 2t + 1 of it, head_dim columns 32t .. 32t + 31, k-step s taking
      // columns 32t + 4s .. 32t + 4s + 3 (the same order on the query side).
      const int sg = sigma(gid);
#pragma unroll
      for (int c = 0; c < 2; ++c) kb8[c] = chunk_off(sg, 2 * tig + c);
    }
    // V: tokens sigma(2t), sigma(2t+1); 4 bytes at head_dim column 32 jj + 4 gid.
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int st = sigma(2 * tig + e);
#pragma unroll
      for (int jj = 0; jj < Tr::KS / 2; ++jj) vb8[e][jj] = chunk_off(st, 2 * jj + (gid >> 2)) + 4 * (gid & 3);
    }
  }
  // head_dim column of accumulator row (m-tile i, half hf) of O^T
  auto dim_of = [&](int i, int hf) -> int {
    if constexpr (!k8bit) return 16 * i + gid + 8 * hf;
    return 32 * (i >> 1) + 4 * gid + 2 * (i & 1) + hf;
  };

  // Rows of the A operand: r = query * G + head (r < R = q_len * G).  Lane
  // (g, t) holds rows g and, with 16-row variants, g + 8 (NH halves).  Only
  // the 16-row variants serve several queries per sequence (MQ); the others
  // compile the single-query case, whose rows share one set of bounds.
  constexpr int NH = GM > 8 ? 2 : 1;
  constexpr bool MQ = GM > 8;
  const int QL = MQ ? p.q_len : 1;
  const int R = QL * G;                          // rows of the segment
  const int row0 = MQ ? 16 * rg : 0;             // this warp's first row of them
  const int Rw = MQ ? min(16, R - row0) : R;     // and how many it owns
  uint32_t qa0[Tr::KS], qa1[Tr::KS];  // A operand, row g (zero when g >= R)
  uint32_t qb0[Tr::KS], qb1[Tr::KS];  // A operand, row g + 8 (NH == 2)
  // softmax state rows of this lane: g and g + 8 (several queries), else
  // 2t and 2t + 1 (the N columns of S = K Q^T)
  constexpr int NR = MQ ? NH : 2;
  float m[NR], l[NR];                 // running max / sum of those rows (log2 domain)
  float acc[Tr::KS][NH][4];           // O^T: rows = head_dim columns, cols = A rows 8h + 2t, 8h + 2t + 1
  int hi_abs[NH], lo_abs[NH];         // last / first position row g + 8h may see (MQ)
  float score_scale = p.qk_scale_log2;
  uint32_t zpk2 = 0u, zpv2 = 0u;  // INT8: f16x2(1152 + zero point) of this KV head

  // One unit: S^T = Q K^T, online-softmax update, O^T += V^T P^T.
  // FULL: all UR rows valid.
  auto unit_step = [&](auto full_tag, uint32_t kt, int n_valid, int lo_rel, int j) {
    constexpr bool FULL = decltype(full_tag)::value;
    const uint32_t vt = kt + Tr::TILE;
    // P^T as the B operand of each 16-token k-step of O^T += V^T P^T, split hi + lo
    uint32_t ph[Tr::NSB][NH][2], pl[Tr::NSB][NH][2];
    if constexpr (!MQ) {
      // ---- scores S = K Q^T: tokens as M (16 per m-tile), the G <= 8 query
      // rows as N.  Lane (g, t) holds the scores of m-rows g and g + 8 (tokens
      // g, g + 8; 8-bit: sigma(g), 8 + sigma(g)) for rows 2t and 2t + 1.
      constexpr int NMT = Tr::NSB;
      float sc[NMT][4];
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
      if constexpr (!k8bit) {
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
          for (int s = 0; s < Tr::KS; ++s) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kt + mt * sub_delta + moffA[s], a0, a1, a2, a3);
            mma16816<MB>(sc[mt], a0, a1, a2, a3, qa0[s], qa1[s]);
          }
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint4 w0 = lds128(kt + mt * 2048 + kb8[c]);         // token sigma(g)
            const uint4 w1 = lds128(kt + mt * 2048 + 1024 + kb8[c]);  // token 8 + sigma(g)
            const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w};
            const uint32_t x1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int s = 4 * c + r;
              uint32_t a0, a1, a2, a3;
              widen4<KVT>(x0[r], zpk2, a0, a2);
              widen4<KVT>(x1[r], zpk2, a1, a3);
              mma16816<false>(sc[mt], a0, a1, a2, a3, qa0[s], qa1[s]);
            }
          }
        }
      }
      // ---- online softmax: rows 2t (elements 0, 2) and 2t + 1 (1, 3), each
      // reduced over the 8 lanes of equal t
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = sc[mt][e] * score_scale;
          if constexpr (!FULL) {
            const int tok = 16 * mt + 8 * (e >> 1) + (k8bit ? sigma(gid) : gid);
            x = (tok < n_valid && tok >= lo_rel) ? x : -INFINITY;
          }
          sc[mt][e] = x;
          if (e & 1) {
            mx1 = fmaxf(mx1, x);
          } else {
            mx0 = fmaxf(mx0, x);
          }
        }
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      // every row sees a token in every unit it processes: the new maxima are finite
      if (__any_sync(0xffffffffu, mx0 > m[0] || mx1 > m[1])) {
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float a0 = fast_exp2(m[0] - mn0), a1 = fast_exp2(m[1] - mn1);
        m[0] = mn0;
        m[1] = mn1;
        l[0] *= a0;
        l[1] *= a1;
#pragma unroll
        for (int i = 0; i < Tr::KS; ++i) {
          acc[i][0][0] *= a0;
          acc[i][0][1] *= a1;
          acc[i][0][2] *= a0;
          acc[i][0][3] *= a1;
        }
      }
      // P, then its transposes: m-rows g (g + 8) of S become k-rows 2t, 2t + 1
      // (2t + 8, 2t + 9) of P^T, the token order the V loads use
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        const float p0 = fast_exp2(sc[mt][0] - m[0]);
        const float p1 = fast_exp2(sc[mt][1] - m[1]);
        const float p2 = fast_exp2(sc[mt][2] - m[0]);
        const float p3 = fast_exp2(sc[mt][3] - m[1]);
        l[0] += p0 + p2;
        l[1] += p1 + p3;
        const uint32_t h01 = pack2<MB>(p0, p1), h23 = pack2<MB>(p2, p3);
        const float2 f01 = unpack2<MB>(h01), f23 = unpack2<MB>(h23);
        ph[mt][0][0] = movmatrix_trans(h01);
        ph[mt][0][1] = movmatrix_trans(h23);
        pl[mt][0][0] = movmatrix_trans(pack2<MB>(p0 - f01.x, p1 - f01.y));
        pl[mt][0][1] = movmatrix_trans(pack2<MB>(p2 - f23.x, p3 - f23.y));
      }
    } else {
      float sc[Tr::NT][4];
#pragma unroll
      for (int nt = 0; nt < Tr::NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      // ---- scores
      if constexpr (!k8bit) {
#pragma unroll
        for (int sb = 0; sb < Tr::NSB; ++sb) {
#pragma unroll
          for (int s = 0; s < Tr::KS; ++s) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kt + sb * sub_delta + moff[s], b0, b1, b2, b3);
            const uint32_t a1 = NH == 2 ? qb0[s] : 0u, a3 = NH == 2 ? qb1[s] : 0u;
            mma16816<MB>(sc[2 * sb], qa0[s], a1, qa1[s], a3, b0, b1);
            mma16816<MB>(sc[2 * sb + 1], qa0[s], a1, qa1[s], a3, b2, b3);
          }
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < Tr::NT; ++nt) {
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const uint4 w = lds128(kt + nt * 1024 + kb8[g]);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int s = 4 * g + r;
              uint32_t b0, b1;
              widen4<KVT>(ws[r], zpk2, b0, b1);
              mma16816<false>(sc[nt], qa0[s], NH == 2 ? qb0[s] : 0u, qa1[s], NH == 2 ? qb1[s] : 0u, b0, b1);
            }
          }
        }
      }
      // ---- online softmax per row (the quad of lanes g*4 .. g*4+3 shares rows g, g+8)
      float mx[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        mx[h] = -INFINITY;
        int hr = 0, lr = 0;  // this row's bounds in the unit (several queries per sequence)
        if constexpr (MQ) {
          hr = hi_abs[h] - j * UR;
          lr = lo_abs[h] - j * UR;
        }
#pragma unroll
        for (int nt = 0; nt < Tr::NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x = sc[nt][2 * h + e] * score_scale;
            if constexpr (!FULL) {
              const int tok = nt * 8 + (k8bit ? sigma(2 * tig + e) : 2 * tig + e);
              bool ok = tok < n_valid && tok >= lo_rel;
              if constexpr (MQ) ok = ok && tok <= hr && tok >= lr;
              x = ok ? x : -INFINITY;
            }
            sc[nt][2 * h + e] = x;
            mx[h] = fmaxf(mx[h], x);
          }
        }
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      }
      bool up = mx[0] > m[0];
      if constexpr (NH == 2) up |= mx[1] > m[1];
      if (__any_sync(0xffffffffu, up)) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const float mn = fmaxf(m[h], mx[h]);
          // a row that has seen nothing yet keeps alpha = 1 (its state is still empty);
          // single-query rows see a token in every unit they process
          const float alpha = (MQ && mn == -INFINITY) ? 1.f : fast_exp2(m[h] - mn);
          m[h] = mn;
          l[h] *= alpha;
          const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * tig);      // row 8h + 2t
          const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * tig + 4);  // row 8h + 2t + 1
#pragma unroll
          for (int i = 0; i < Tr::KS; ++i) {
            acc[i][h][0] *= a0;
            acc[i][h][1] *= a1;
            acc[i][h][2] *= a0;
            acc[i][h][3] *= a1;
          }
        }
      }
      // P^T as the B operand of each 16-token k-step, per row half, split hi + lo
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const float ms = (MQ && m[h] == -INFINITY) ? 0.f : m[h];  // exp2(-inf - ms) = 0 for an empty row
#pragma unroll
        for (int nt = 0; nt < Tr::NT; ++nt) {
          const float p0 = fast_exp2(sc[nt][2 * h] - ms);
          const float p1 = fast_exp2(sc[nt][2 * h + 1] - ms);
          l[h] += p0 + p1;
          const uint32_t hp = pack2<MB>(p0, p1);
          const float2 hf = unpack2<MB>(hp);
          ph[nt >> 1][h][nt & 1] = hp;
          pl[nt >> 1][h][nt & 1] = pack2<MB>(p0 - hf.x, p1 - hf.y);
        }
      }
    }
    // rows past the end of the sequence, and rows before a sliding window,
    // may hold anything (or were not loaded): zero them in V
    if constexpr (!FULL) {
      const int nlo = max(lo_rel, 0);
      const int nz = (UR - n_valid + nlo) * Tr::NSUB * 8;
      for (int k = lane; k < nz; k += 32) {
        const int rr = k / (Tr::NSUB * 8);
        const int r = rr < nlo ? rr : n_valid + (rr - nlo);
        const int ch = k % (Tr::NSUB * 8);
        sts128_zero(vt + chunk_off(r, ch));
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    // ---- O^T += V^T P^T
    if constexpr (!k8bit) {
#pragma unroll
      for (int sb = 0; sb < Tr::NSB; ++sb) {
#pragma unroll
        for (int i = 0; i < Tr::KS; ++i) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vt + sb * sub_delta + moff[i], a0, a1, a2, a3);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            mma16816<MB>(acc[i][h], a0, a1, a2, a3, ph[sb][h][0], ph[sb][h][1]);
            mma16816<MB>(acc[i][h], a0, a1, a2, a3, pl[sb][h][0], pl[sb][h][1]);
          }
        }
      }
    } else {
#pragma unroll
      for (int sb = 0; sb < Tr::NSB; ++sb) {
#pragma unroll
        for (int jj = 0; jj < Tr::KS / 2; ++jj) {
          // tokens of k 2t, 2t+1 (n-tile 2 sb) and k 2t+8, 2t+9 (n-tile 2 sb + 1)
          const uint32_t x0 = lds32(vt + (2 * sb) * 1024 + vb8[0][jj]);
          const uint32_t x1 = lds32(vt + (2 * sb) * 1024 + vb8[1][jj]);
          const uint32_t y0 = lds32(vt + (2 * sb + 1) * 1024 + vb8[0][jj]);
          const uint32_t y1 = lds32(vt + (2 * sb + 1) * 1024 + vb8[1][jj]);
          const uint32_t lo01 = prmt(x0, x1, 0x5140u), lo23 = prmt(x0, x1, 0x7362u);
          const uint32_t hi01 = prmt(y0, y1, 0x5140u), hi23 = prmt(y0, y1, 0x7362u);
          uint32_t d0l, d1l, d2l, d3l, d0h, d1h, d2h, d3h;
          if constexpr (std::is_same<KVT, i8_t>::value) {
            // 1152 + code: the output subtracts (1152 + zp) * v_scale once
            widen4_i8_biased(lo01, d0l, d1l);
            widen4_i8_biased(lo23, d2l, d3l);
            widen4_i8_biased(hi01, d0h, d1h);
            widen4_i8_biased(hi23, d2h, d3h);
          } else {
            widen4<KVT>(lo01, zpv2, d0l, d1l);
            widen4<KVT>(lo23, zpv2, d2l, d3l);
            widen4<KVT>(hi01, zpv2, d0h, d1h);
            widen4<KVT>(hi23, zpv2, d2h, d3h);
          }
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            mma16816<false>(acc[2 * jj][h], d0l, d1l, d0h, d1h, ph[sb][h][0], ph[sb][h][1]);
            mma16816<false>(acc[2 * jj][h], d0l, d1l, d0h, d1h, pl[sb][h][0], pl[sb][h][1]);
            mma16816<false>(acc[2 * jj + 1][h], d2l, d3l, d2h, d3h, ph[sb][h][0], ph[sb][h][1]);
            mma16816<false>(acc[2 * jj + 1][h], d2l, d3l, d2h, d3h, pl[sb][h][0], pl[sb][h][1]);
          }
        }
      }
    }
  };

  // Fused append: the unit holding position T-1 carries the new K/V rows in
  // 16-bit source format.  Lanes convert them to the cache format (a copy, or
  // the cache write's quantisation for 8-bit caches), overwrite the stale
  // row of the tile and store the row into its cache slot.  Each unit is
  // processed by exactly one warp, so nothing else reads that slot here.
  auto append_row = [&](int st) {
    uint8_t* stage = const_cast<uint8_t*>(wbase) + Tr::OFF_STAGES + st * STG;
    const uint8_t* staged = stage + Tr::OFF_NEW;
    const int pos = it.T - 1;
    const int r = pos - it.j * UR;
    const int pb = *reinterpret_cast<const int*>(staged + 4 * D);
    constexpr int CH = Tr::ROW / 16;  // 16-byte chunks of a cache row
    if (lane < 2 * CH) {
      const int which = lane / CH, ch = lane % CH;  // 0: K, 1: V
      uint4 w;
      if constexpr (!k8bit) {
        w = *reinterpret_cast<const uint4*>(staged + which * 2 * D + ch * 16);
      } else {
        // 16 source values -> 16 cache bytes
        const uint4* src = reinterpret_cast<const uint4*>(staged + which * 2 * D + ch * 32);
        const uint4 a = src[0], b = src[1];
        const uint32_t pairs[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const float inv = __ldg((which ? p.v_inv_scale : p.k_inv_scale) + it.kvh);
        int zp = 0;
        if constexpr (std::is_same<KVT, i8_t>::value) zp = __ldg((which ? p.v_zero_point : p.k_zero_point) + it.kvh);
        uint32_t out4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 x0, x1;
          if (p.new_dtype == PA_BF16) {
            x0 = widen2<bf16_t>(pairs[2 * i]);
            x1 = widen2<bf16_t>(pairs[2 * i + 1]);
          } else {
            x0 = widen2<f16_t>(pairs[2 * i]);
            x1 = widen2<f16_t>(pairs[2 * i + 1]);
          }
          const float y0 = __fmul_rn(x0.x, inv), y1 = __fmul_rn(x0.y, inv);
          const float y2 = __fmul_rn(x1.x, inv), y3 = __fmul_rn(x1.y, inv);
          if constexpr (std::is_same<KVT, i8_t>::value) {
            out4[i] = (static_cast<uint32_t>(int8_code(y0, zp)) & 0xffu) |
                      ((static_cast<uint32_t>(int8_code(y1, zp)) & 0xffu) << 8) |
                      ((static_cast<uint32_t>(int8_code(y2, zp)) & 0xffu) << 16) |
                      ((static_cast<uint32_t>(int8_code(y3, zp)) & 0xffu) << 24);
          } else {
            out4[i] = e4m3x2_code(y0, y1) | (e4m3x2_code(y2, y3) << 16);
          }
        }
        w = make_uint4(out4[0], out4[1], out4[2], out4[3]);
      }
      *reinterpret_cast<uint4*>(stage + which * Tr::TILE + chunk_off(r, ch)) = w;
      if (pb >= 0) {
        const int64_t crow = (static_cast<int64_t>(pb) * Hkv + it.kvh) * B + (pos & (B - 1));
        uint8_t* cache = static_cast<uint8_t*>(which ? p.v_cache : p.k_cache);
        *reinterpret_cast<uint4*>(cache + crow * Tr::ROW + ch * 16) = w;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before TMA refills this stage
    __syncwarp();
  };

  // Merge of split segment x = s * H_kv + kvh by the warp that arrived last,
  // after the unit loop (list in the workspace): an inlined merge inside the
  // loop costs the loop registers, and the arrival itself does not wait: its
  // atomic's result is looked at only at the next fragment end ("settle").
  int npend = 0;
  uint32_t merge_par = 0;  // phase parity of this warp's merge barrier
  int* const pend = p.pending + static_cast<int64_t>(blockIdx.x * W + c) * p.pending_cap;
  int arr_old = 0, arr_x = -1, arr_nfr = 0;  // the arrival not settled yet (x < 0: none)
  bool arr_acq = false;    // that arrival was an acquire (the ring's final fragment)
  bool pend_fence = false;  // a pending merge was won by a release-only arrival
  auto settle = [&]() {
    if (arr_x >= 0) {
      const int old = __shfl_sync(0xffffffffu, arr_old, 0);
      if (old == arr_nfr - 1) {  // last to arrive: this warp merges the segment
        if (npend < p.pending_cap) {
          if (lane == 0) pend[npend] = arr_x;
          ++npend;
          pend_fence = pend_fence || !arr_acq;
        } else if (lane == 0) {
          raise_error(p.err, PA_DEVERR_INTERNAL);
        }
      }
      arr_x = -1;
    }
  };
  auto merge_seg = [&](int x) {
    const int s = x / Hkv, kvh = x - (x / Hkv) * Hkv;
    const int per = (prefix[s + 1] - prefix[s]) / Hkv;  // units (balanced) or partitions (fixed) per KV head
    MergeSlots ms;
    ms.fixed = fixed;
    ms.fixed_base = prefix[s] + kvh * per;
    ms.U = U;
    ms.nw_eff = nw_eff;
    ms.seg_start = prefix[s] + static_cast<long long>(kvh) * per;
    ms.first_w = 0;
    ms.nc = NC;
    ms.rg = rg;
    int nfr = per;
    if (!fixed) {
      // rings holding the segment's first and last units (positions seg_start + frag_cost, seg_start + per - 1)
      ms.first_w = ring_of(ms.seg_start + p.frag_cost, U, nw_eff);
      nfr = ring_of(ms.seg_start + per - 1, U, nw_eff) - ms.first_w + 1;
    }
    float vs = 1.f, voff = 0.f;
    if constexpr (k8bit) vs = hp_vs[kvh];
    if constexpr (std::is_same<KVT, i8_t>::value) voff = v_bias_offset(hp_zv[kvh], vs);
    const int64_t seq_row0 = static_cast<int64_t>(s) * QL * p.num_heads + static_cast<int64_t>(kvh) * G;
    // the ring's stages are idle after the unit loop (every warp of the ring
    // has passed the ring barrier): warp rg stages its records in its share
    const int share = (NS * STG) / NC / (Tr::REC * 4) * (Tr::REC * 4);
    merge_segment<GM, D, Tr::REC>(p.part_records, ms, nfr, lane, Rw, G, p.num_heads, vs, voff, p.out, p.out_dtype, seq_row0,
                                  row0, wbase_u32 + Tr::OFF_STAGES + rg * share,
                                  reinterpret_cast<float*>(const_cast<uint8_t*>(wbase) + Tr::OFF_STAGES + rg * share),
                                  share / (Tr::REC * 4), wbase_u32 + Tr::OFF_MERGE + 8 * rg, merge_par, p.err);
    if (lane == 0) p.seg_counters[x * NC + rg] = 0;
  };

  while (it.valid) {
    // ---- one fragment: units j0 .. jend-1 of segment (s, kvh)
    if (!mbar_wait_bounded(wbase_u32 + Tr::OFF_FULL + 8 * cst, cpar, p.wait_limit_ns)) {
      if (lane == 0) raise_error(p.err, PA_DEVERR_TIMEOUT);
      break;  // the producer stops feeding this ring when its empty barrier times out
    }
    // 8-bit caches with a bf16 query: the products run in f16 (the widened
    // cache values are exact f16), so the query group is brought into f16's
    // range first.  Every element is multiplied by 2^qexp, the power of two
    // that puts the group's largest |q| in [2^14, 2^15); the scores are
    // multiplied back by 2^-qexp.  Both steps are exact, and so is the f16
    // rounding of every element within 2^28 of the group's largest (bf16 has 8
    // significant bits, f16 11); smaller elements can lose bits as f16
    // subnormals, an absolute error below 2^-38 of the largest element.
    constexpr bool q_rescale = k8bit && std::is_same<QT, bf16_t>::value;
    int qexp = 0;
    {
      // the query group rode on the fragment's first stage (into the ring's
      // query buffer with several queries)
      const uint8_t* qr = kMQ ? wbase + OFF_QBUF : wbase + Tr::OFF_STAGES + cst * STG + 2 * Tr::TILE;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int row = gid + 8 * h;  // local row of the A operand
        const bool row_ok = row < Rw;
#pragma unroll
        for (int s = 0; s < Tr::KS; ++s) {
          // columns of k-step s held by this lane: (d, d+1) for a0/a1, (d2, d2+1) for a2/a3
          const int d = k8bit ? (MQ ? 16 * (4 * (s >> 2) + tig) + 4 * (s & 3) : 32 * tig + 4 * s) : 16 * s + 2 * tig;
          const int d2 = k8bit ? d + 2 : d + 8;
          uint32_t w0 = 0u, w1 = 0u;
          if (row_ok) {
            w0 = *reinterpret_cast<const uint32_t*>(qr + ((row0 + row) * D + d) * 2);
            w1 = *reinterpret_cast<const uint32_t*>(qr + ((row0 + row) * D + d2) * 2);
          }
          if (h == 0) {
            qa0[s] = w0;
            qa1[s] = w1;
          } else {
            qb0[s] = w0;
            qb1[s] = w1;
          }
        }
        // query i = row / G sits at position T - q_len + i and sees positions up to
        // it (and, under a window, the last `window` of them); padding rows see all
        if constexpr (MQ) {
          const int qi = row < Rw ? (row0 + row) / G : QL - 1;
          hi_abs[h] = it.T - QL + qi;
          lo_abs[h] = p.window > 0 ? hi_abs[h] - p.window + 1 : 0;
        }
      }
    }
    if constexpr (MQ) {
      // every lane's query rows are in registers: the ring's query buffer may
      // be refilled (each of the ring's NC warps arrives once per fragment)
      __syncwarp();
      if (lane == 0) mbar_arrive(wbase_u32 + Tr::OFF_QEMPTY);
    }
    if constexpr (q_rescale) {
      // largest |q| of the group (bf16 halves read as floats), over the warp
      auto amax2 = [](float a, uint32_t w) {
        return fmaxf(a, fmaxf(__uint_as_float((w << 16) & 0x7fffffffu), __uint_as_float(w & 0x7fff0000u)));
      };
      float qmax = 0.f;
#pragma unroll
      for (int s = 0; s < Tr::KS; ++s) {
        qmax = amax2(amax2(qmax, qa0[s]), qa1[s]);
        if constexpr (NH == 2) qmax = amax2(amax2(qmax, qb0[s]), qb1[s]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
      // qmax in [2^E, 2^(E+1)) -> qexp = 14 - E; all-zero groups keep qexp = 0;
      // the clamp keeps both 2^qexp and the scale below normal float32 numbers
      const int ebits = (__float_as_int(qmax) >> 23) & 0xff;
      qexp = qmax > 0.f ? min(100, max(-100, 141 - ebits)) : 0;
      const float mul = __int_as_float((127 + qexp) << 23);
      auto narrow = [&](uint32_t w) {
        const float2 f = widen2<bf16_t>(w);
        return pack2<false>(f.x * mul, f.y * mul);
      };
#pragma unroll
      for (int s = 0; s < Tr::KS; ++s) {
        qa0[s] = narrow(qa0[s]);
        qa1[s] = narrow(qa1[s]);
        if constexpr (NH == 2) {
          qb0[s] = narrow(qb0[s]);
          qb1[s] = narrow(qb1[s]);
        }
      }
    }
    score_scale = p.qk_scale_log2;
    if constexpr (k8bit) score_scale *= hp_ks[it.kvh];
    if constexpr (q_rescale) score_scale *= __int_as_float((127 - qexp) << 23);
    if constexpr (std::is_same<KVT, i8_t>::value) {
      zpk2 = hp_zk[it.kvh];
      zpv2 = hp_zv[it.kvh];
    }
#pragma unroll
    for (int h = 0; h < NR; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
#pragma unroll
      for (int i = 0; i < Tr::KS; ++i) acc[i][h][0] = acc[i][h][1] = acc[i][h][2] = acc[i][h][3] = 0.f;
    }
    // a unit is FULL when every row sees all of its tokens
    const int full_lo = p.window > 0 ? it.T - 1 - p.window + 1 : 0;  // first position the last query sees
    const int full_hi = it.T - QL;                                   // last position the first query sees
    bool timed_out = false;
    for (;;) {
      const uint32_t stage_u32 = wbase_u32 + Tr::OFF_STAGES + cst * STG;
      if (append && it.j == ((it.T - 1) >> Tr::UR_SHIFT)) append_row(cst);
      const int n_valid = min(UR, it.T - it.j * UR);
      const int lo_rel = it.lo - it.j * UR;  // positions before the window (> 0 only in its first unit)
      if constexpr (MQ) {
        // one (masked) copy of the unit step: two inlined copies do not fit the
        // registers of the 16-row variants
        (void)full_lo;
        (void)full_hi;
        unit_step(std::false_type{}, stage_u32, n_valid, lo_rel, it.j);
      } else if (n_valid == UR && lo_rel <= 0) {
        unit_step(std::true_type{}, stage_u32, UR, 0, it.j);
      } else {
        unit_step(std::false_type{}, stage_u32, n_valid, lo_rel, it.j);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(wbase_u32 + Tr::OFF_EMPTY + 8 * cst);  // the stage may be refilled
      if (++cst == NS) {
        cst = 0;
        cpar ^= 1;
      }
      if (it.j + 1 == it.jend) break;
      ++it.j;
      if (!mbar_wait_bounded(wbase_u32 + Tr::OFF_FULL + 8 * cst, cpar, p.wait_limit_ns)) {
        if (lane == 0) raise_error(p.err, PA_DEVERR_TIMEOUT);
        timed_out = true;
        break;
      }
    }
    if (timed_out) break;

    // ---- end of fragment: write the output or a partial record
    {
      // sums of this lane's softmax rows: several queries: rows g, g + 8
      // (over the quad); else rows 2t, 2t + 1 (over the 8 lanes of equal t)
      float lt[NR];
#pragma unroll
      for (int h = 0; h < NR; ++h) {
        if constexpr (MQ) {
          lt[h] = l[h] + __shfl_xor_sync(0xffffffffu, l[h], 1);
          lt[h] += __shfl_xor_sync(0xffffffffu, lt[h], 2);
        } else {
          lt[h] = l[h];
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) lt[h] += __shfl_xor_sync(0xffffffffu, lt[h], off);
        }
      }
      float vs = 1.f, voff = 0.f;  // out = acc * vs / l - voff (INT8: V entered as 1152 + code)
      if constexpr (k8bit) vs = hp_vs[it.kvh];
      if constexpr (std::is_same<KVT, i8_t>::value) voff = v_bias_offset(hp_zv[it.kvh], vs);
      // output row of A row r: out[s][r / G][kvh * G + r % G]
      const int64_t seq_row0 = static_cast<int64_t>(it.s) * QL * p.num_heads + static_cast<int64_t>(it.kvh) * G;
      auto out_row = [&](int r) -> int64_t {
        if constexpr (!MQ) return seq_row0 + r;  // one query: row = head
        return seq_row0 + static_cast<int64_t>((row0 + r) / G) * p.num_heads + (row0 + r) % G;
      };
      if (it.slot < 0) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int r0 = 8 * h + 2 * tig, r1 = r0 + 1;
          float l0, l1;  // sums of rows r0, r1
          if constexpr (MQ) {
            l0 = __shfl_sync(0xffffffffu, lt[h], 8 * tig);
            l1 = __shfl_sync(0xffffffffu, lt[h], 8 * tig + 4);
          } else {
            l0 = lt[0];
            l1 = lt[1];
          }
          const float i0 = l0 > 0.f ? vs / l0 : 0.f, i1 = l1 > 0.f ? vs / l1 : 0.f;  // a row that saw nothing: 0
          const float b0 = l0 > 0.f ? voff : 0.f, b1 = l1 > 0.f ? voff : 0.f;
          const int64_t o0 = out_row(r0) * D, o1 = out_row(r1) * D;
          const bool w0 = r0 < Rw, w1 = r1 < Rw;
#pragma unroll
          for (int i = 0; i < Tr::KS; ++i) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int d = dim_of(i, hf);
              if (w0) store_out(p.out, p.out_dtype, o0 + d, fmaf(acc[i][h][2 * hf], i0, -b0));
              if (w1) store_out(p.out, p.out_dtype, o1 + d, fmaf(acc[i][h][2 * hf + 1], i1, -b1));
            }
          }
        }
      } else {
        float* rec = p.part_records + (static_cast<int64_t>(it.slot) * NC + rg) * Tr::REC;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          const int r0 = 8 * h + 2 * tig;
#pragma unroll
          for (int i = 0; i < Tr::KS; ++i) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int d = dim_of(i, hf);
              if constexpr (GM == 1) {
                if (tig == 0) rec[d] = acc[i][h][2 * hf];
              } else {
                if (r0 < GM)
                  *reinterpret_cast<float2*>(rec + d * GM + r0) = make_float2(acc[i][h][2 * hf], acc[i][h][2 * hf + 1]);
              }
            }
          }
          if constexpr (MQ) {
            const int row = gid + 8 * h;
            if (tig == 0 && row < GM) {
              rec[GM * D + row] = m[h];
              rec[GM * D + GM + row] = lt[h];
            }
          }
        }
        if constexpr (!MQ) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int row = 2 * tig + e;
            if (gid == 0 && row < GM) {
              rec[GM * D + row] = m[e];
              rec[GM * D + GM + row] = lt[e];
            }
          }
        }
        // fragments of this segment
        int nfr;
        if (fixed) {
          nfr = (prefix[it.s + 1] - prefix[it.s]) / Hkv;
        } else {
          const long long seg_start = prefix[it.s] + static_cast<long long>(it.kvh) * (it.nu + p.frag_cost);
          nfr = ring_of(seg_start + p.frag_cost + it.nu - 1, U, nw_eff) - ring_of(seg_start + p.frag_cost, U, nw_eff) + 1;
        }
        settle();
        __syncwarp();  // every lane's record stores come before lane 0's release
        // The ring's final fragment (no unit after it to stall) arrives with
        // an acquire too, so a merge it wins needs no fence after the loop.
        // (Conservative: a range that ends in a later segment's overhead
        // arrives with a release and its merge takes the fence.)
        const bool final_frag = fixed ? it.r + it.rstride >= it.R : it.fend >= it.u1;
        int* const ctr = p.seg_counters + (it.s * Hkv + it.kvh) * NC + rg;
        if (lane == 0) arr_old = final_frag ? atom_add_acq_rel_gpu(ctr, 1) : atom_add_release_gpu(ctr, 1);
        arr_x = it.s * Hkv + it.kvh;
        arr_nfr = nfr;
        arr_acq = final_frag;
      }
    }
    ++it.j;
    iter_next_fragment(it, prefix, p, fixed, Tr::UR_SHIFT);
  }

  // ---- the split merges this warp won
  settle();
  // The ring's stages become merge staging space: every warp of a shared ring
  // first waits until all of them have left the unit loop (named barrier
  // 1 + ring, NC warps).  Each of them reaches it: a warp that stops early on
  // a timeout stops releasing stages, so the others time out too.
  if (MQ && NC > 1) named_barrier_sync(1 + ring_id, NC * 32);
  if (npend > 0) {
    // acquire: the other fragments' records, released by their arrivals.
    // Lane 0 observed those arrivals (its atomics' results); its fence (or
    // the final fragment's acquiring arrival), then the warp barrier, order
    // every lane's reads after them.  (An acquire on every arrival would
    // order the next unit's loads after the atomic and stall the unit loop.)
    if (pend_fence) fence_acq_rel_gpu();
    __syncwarp();
    // the records are read by bulk copies (the async proxy): each lane orders
    // them after its (acquired) view of global memory
    fence_proxy_async_global();
    for (int i = 0; i < npend; ++i) merge_seg(pend[i]);
  }
}


// ----------------------------------------------------------------- host side of one variant

template <typename QT, typename KVT, int D, int GM, int UR, int AP>
struct DecodeVariant {
  using Tr = DecodeTraits<QT, KVT, D, GM, UR>;

  static size_t smem_bytes(int num_seqs, int warps, int rings, int stages, int stage) {
    constexpr int head_words = Tr::B8 ? 4 * kMaxHeadParams : 0;
    return 1024 + static_cast<size_t>(rings) * (Tr::warp_smem(stages, stage) + Tr::qbuf_bytes(warps / rings)) +
           static_cast<size_t>(align_up_c((2 * num_seqs + 1 + warps + 1 + head_words) * 4, 16)) +
           static_cast<size_t>(rings) * 64;
  }

  // Launch geometry: pipeline depth (stages per ring) and consumer warps per
  // CTA (plus one producer warp).  One warp per ring: the default depth keeps
  // about kStageBytesPerWarp of K/V per consumer and the consumers per CTA
  // maximise resident consumer warps per SM (ties: more per CTA, i.e. fewer
  // producer warps).  Rings shared by nc warps (several queries per sequence,
  // nc = ceil(q_len * G / 16)): the consumers per CTA are a multiple of nc and
  // each choice takes the deepest ring that fits; the choice maximises the
  // K/V stages in flight per SM (ties: more warps).  PA_DECODE_STAGES /
  // PA_DECODE_WARPS override depth and warps (tuning).
  static bool geometry(int num_seqs, int nc, DecodeGeometry* g) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    int sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
    auto kern = paged_decode_kernel<QT, KVT, D, GM, UR, AP>;
    // allow every size the device allows, once: geometries of other batch
    // sizes are cached and launched later without touching the attribute
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess) return false;
    constexpr bool mq = GM > 8;
    if (nc < 1 || (!mq && nc != 1) || nc > 4) return false;
    // several queries: K and V only (the query rows have a buffer per ring)
    const int stage = mq ? align_up_c(2 * Tr::TILE, 1024) : (AP ? Tr::STAGE_APPEND : Tr::STAGE);
    const int env_ns = tuning_override("PA_DECODE_STAGES");
    const int env_w = tuning_override("PA_DECODE_WARPS");
    int best_w = 0, best_occ = 0, best_ns = 0;
    long long best_score = 0;
    for (int w = nc; w <= Tr::MAX_W; w += nc) {
      if (env_w > 0 && w != env_w) continue;
      const int rings = w / nc;
      int ns;
      if (env_ns >= 2 && env_ns <= Tr::MAX_NS) {
        ns = env_ns;
      } else if (!mq || nc == 1) {
        ns = kStageBytesPerWarp / stage;
        ns = ns < 2 ? 2 : (ns > Tr::MAX_NS ? Tr::MAX_NS : ns);
      } else {
        ns = Tr::MAX_NS;  // deepest ring that fits
        while (ns > 2 && smem_bytes(num_seqs, w, rings, ns, stage) > static_cast<size_t>(optin)) --ns;
      }
      // the merges stage at least one record per warp in the ring's stages
      if (static_cast<long long>(ns) * stage / nc < Tr::REC * 4) continue;
      const size_t smem = smem_bytes(num_seqs, w, rings, ns, stage);
      if (smem > static_cast<size_t>(optin)) continue;
      int occ = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, (w + 1) * 32, smem) != cudaSuccess) return false;
      if (occ <= 0) continue;
      // one warp per ring: resident consumer warps; shared rings: K/V stages in flight
      const long long score = (!mq || nc == 1) ? static_cast<long long>(occ) * w
                                                : static_cast<long long>(occ) * rings * (ns - 1) * 16 + w;
      if (score >= best_score) {
        best_score = score;
        best_w = w;
        best_occ = occ;
        best_ns = ns;
      }
    }
    if (best_w == 0) return false;
    const int ns = best_ns;
    const size_t smem = smem_bytes(num_seqs, best_w, best_w / nc, ns, stage);
    g->warps_per_cta = best_w;
    g->row_groups = nc;
    g->stage_bytes = stage;
    g->stages = ns;
    g->ctas = sms * best_occ;
    g->smem_bytes = smem;
    g->record_floats = Tr::REC;
    g->unit_rows = UR;
    return true;
  }

  static cudaError_t launch(const DecodeGeometry& g, const DecodeParams& p, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t stream, bool pdl) {
    (void)cudaGetLastError();  // an earlier unrelated error must not be reported as this launch's
    cudaError_t e;
    if (pdl) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(g.ctas);
      cfg.blockDim = dim3((g.warps_per_cta + 1) * 32);
      cfg.dynamicSmemBytes = g.smem_bytes;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, paged_decode_kernel<QT, KVT, D, GM, UR, AP>, tk, tv, p);
      if (e == cudaSuccess) e = cudaGetLastError();
    } else {
      paged_decode_kernel<QT, KVT, D, GM, UR, AP><<<g.ctas, (g.warps_per_cta + 1) * 32, g.smem_bytes, stream>>>(tk, tv, p);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, paged_decode_kernel<QT, KVT, D, GM, UR, AP>) == cudaSuccess)
        note_launch_failure(g.ctas, (g.warps_per_cta + 1) * 32, g.smem_bytes, g.stages, fa.maxThreadsPerBlock,
                            fa.maxDynamicSharedSizeBytes, fa.numRegs, fa.localSizeBytes);
    }
    return e;
  }
};

}  // namespace pa

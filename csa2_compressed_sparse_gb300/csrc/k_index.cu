// k_index.cu -- lightning-indexer scores on tcgen05 tensor cores.
// [A] "特殊模块 · indexer" Fig. 3b: logits[r, c] = sum_h w[r,h] * <q[r,h], k[c]> scaled by
// head_dim^-1/2 * n_heads^-1/2, each row scored only up to its own visible prefix;
// [C] A.15.2: ReLU on each head's dot product, candidates gathered before scoring;
// [A] Fig. 2c: REINDEX scores only the 2048 candidate blocks x 8 rows.
//
// Formulation (per work tile of 128 index rows and one query group):
//     S^T[128 rows x N] = K_tile[128 x 128] . Qg^T[128 x N],   N = nq * H <= 256
// with the index rows on the M side, so TMEM lane r holds every head score of row
// r and the ReLU, the head weights and the head sum are thread-local in the
// epilogue.  A query group is up to 256/H consecutive queries of one sequence
// (prefill); they share the K tile, which is then read once for all of them.
//
// Persistent CTA, one per SM, warp-specialised:
//   warp 0      TMA producer: K tiles (4-stage ring) and the group's Q block
//   warp 1      TMEM allocation; lane 0 issues the MMAs (8 x K=16 per tile)
//   warps 2..9  epilogue in two groups of four warps: group e reads TMEM accumulator e
//               (tiles of parity e) -> relu * w -> sum -> order-preserving key
//   warps 10..17 (MXFP4 planes only) convert packed E2M1 blocks to bf16 tiles
// TMEM holds two 256-column fp32 accumulators, so two tiles are in the epilogue while
// the MMAs of the next one run.  The scores are written as uint32 keys for the top-k.
#include <cuda_fp4.h>

#include "common.cuh"

CSA2_DEFINE_FAULT_FLAG(index)

namespace csa2 {
namespace {

constexpr int kTileRows = 128;
// Operand formats of the index plane.
constexpr int kModeBf16 = 0;  // bf16 rows
constexpr int kModeFp8 = 1;   // blocks of 8 E4M3 rows with fp32 row scales
constexpr int kModeFp4 = 2;   // blocks of 8 E2M1 rows with E8M0 scales per 32 dims
constexpr int kModeGather = 3;  // bf16 rows of candidate blocks, gathered by eight warps
constexpr int kModeFp8Gat = 4;  // FP8 candidate blocks, gathered by eight warps
constexpr int kFp4ConvWarps = 8;  // FP4: warps 10 .. 17 convert packed blocks to bf16
constexpr int kGatherWarps = 8;   // gather mode: warps 10 .. 17 copy the candidate blocks
__host__ __device__ constexpr int num_threads(int mode) {
  return mode == kModeFp4 ? 320 + 32 * kFp4ConvWarps
                          : (mode == kModeGather || mode == kModeFp8Gat ? 320 + 32 * kGatherWarps
                                                                     : 320);
}
// MMA operand ring: bf16 tiles are 32 KiB (two 64-dim blocks of 128-byte rows), FP8 tiles
// 16 KiB (one block).  bf16 and FP8 rings hold 128 KiB, filled by TMA.  FP4 tiles are
// converted to bf16 in shared memory: an 8-stage ring of packed blocks (filled by bulk
// copies) feeds a 2-stage ring of bf16 tiles.
constexpr int kBf16Tile = kTileRows * kDIdx * 2;
constexpr int kFp4BlockBytes = 8 * 64 + 8 * 4;      // 544: 8 rows of codes, 8 x 4 scales
constexpr int kFp4StgBytes = 16 * kFp4BlockBytes;    // 8704: the 16 blocks of a tile
constexpr int kFp4StgStages = 8;
constexpr int kFp4CvStages = 2;
__host__ __device__ constexpr int stage_bytes(int mode) {
  return mode == kModeFp8 || mode == kModeFp8Gat ? kTileRows * kDIdx : kBf16Tile;
}
__host__ __device__ constexpr int num_stages(int mode) {
  return mode == kModeFp4 ? kFp4CvStages : 4 * kBf16Tile / stage_bytes(mode);
}
__host__ __device__ constexpr int ring_bytes(int mode) {
  return mode == kModeFp4 ? kFp4CvStages * kBf16Tile + kFp4StgStages * kFp4StgBytes
                          : 4 * kBf16Tile;
}
constexpr int kMaxStages = 8;
static_assert(num_stages(kModeFp8) <= kMaxStages && num_stages(kModeFp8Gat) <= kMaxStages &&
                  kFp4StgStages <= kMaxStages, "ring");
static_assert(ring_bytes(kModeFp4) % 1024 == 0, "the Q block must stay 1024-byte aligned");
constexpr int kBBytes = 2 * 256 * 128;              // 64 KiB: two 64-dim blocks x 256 rows
constexpr int kMaxGroup = 8;
constexpr int kFp8BlockBytes = 8 * kDIdx + 8 * 4;   // 1056: 8 rows of codes, 8 scales

struct __align__(8) Bars {
  uint64_t full[kMaxStages];   // the ring the producer fills
  uint64_t empty[kMaxStages];
  uint64_t cv_full[kFp4CvStages];   // FP4: converted bf16 tiles
  uint64_t cv_empty[kFp4CvStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t b_full;
  uint64_t b_empty;
};

struct GroupInfo {
  int q0, nq, seq;
  int64_t tile0, tile1;
  int64_t rb;  // row_base of the group's sequence
};

__device__ __forceinline__ int64_t n_visible(int64_t pos, int ratio) { return (pos + 1) / ratio; }

// ---- prep: scored counts, query groups, tile prefix ---------------------------------
// One pass over blocks of 1024 queries.  A query group is a run of at most group_max
// consecutive queries of one sequence: query q starts a group when (q - run start) is
// a multiple of group_max, and the group ends at group_max members or at the end of
// the run.  The block's sequence ids and visible counts (plus a halo of kMaxGroup) sit
// in shared memory, so a leader finds its members without global round trips; group
// ids and tile offsets come from one block-wide exclusive scan of (leader, tiles).
// 256 threads: the prep CTA (8 K registers) fits beside a score CTA on its SM, so that
// score CTA starts at once instead of after the prep.
constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;

// Exclusive block sums of (x, y) over threads in index order, with the block totals.
__device__ __forceinline__ void block_excl_sum2(int x, long long y, int* redx, long long* redy,
                                                int& ex, long long& ey, int& tx, long long& ty) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ix = x;
  long long iy = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int tx1 = __shfl_up_sync(0xFFFFFFFFu, ix, o);
    const long long ty1 = __shfl_up_sync(0xFFFFFFFFu, iy, o);
    if (lane >= o) { ix += tx1; iy += ty1; }
  }
  if (lane == 31) { redx[warp] = ix; redy[warp] = iy; }
  __syncthreads();
  // every warp scans the warp totals itself
  const int wx = lane < kPrepWarps ? redx[lane] : 0;
  const long long wy = lane < kPrepWarps ? redy[lane] : 0;
  int sx = wx;
  long long sy = wy;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int tx1 = __shfl_up_sync(0xFFFFFFFFu, sx, o);
    const long long ty1 = __shfl_up_sync(0xFFFFFFFFu, sy, o);
    if (lane >= o) { sx += tx1; sy += ty1; }
  }
  ex = __shfl_sync(0xFFFFFFFFu, sx - wx, warp) + ix - x;
  ey = __shfl_sync(0xFFFFFFFFu, sy - wy, warp) + iy - y;
  tx = __shfl_sync(0xFFFFFFFFu, sx, 31);
  ty = __shfl_sync(0xFFFFFFFFu, sy, 31);
  __syncthreads();  // redx / redy may be rewritten by the next call
}

// Groups whose tile ranges the prep keeps in shared memory for the CTA-record pass (more
// groups are read back from the group records).
constexpr int kPrepGroupCache = 256;

__global__ void __launch_bounds__(kPrepThreads) index_prep_kernel(IndexArgs a) {
  __shared__ int s_seq[kPrepThreads + kMaxGroup];
  __shared__ int s_ns[kPrepThreads + kMaxGroup];
  __shared__ long long s_rb[kPrepThreads];       // row base of each query's sequence
  __shared__ long long s_t0[kPrepGroupCache], s_t1[kPrepGroupCache];
  __shared__ int s_gfirst[kMaxIndexCtas];
  __shared__ int redx[kPrepWarps];
  __shared__ long long redy[kPrepWarps];
  __shared__ int red_run[kPrepWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The first block reads only the call's inputs (positions, sequence ids, row bases),
  // so its loads and scans run while the preceding kernel drains; nothing is written to
  // the workspace before the wait (the preceding kernels may still read it).
  griddep_launch_dependents();
  int carry_run = 0, carry_groups = 0, prev_seq = -1;
  long long carry_tiles = 0;
  for (int base = 0; base < a.Q; base += kPrepThreads) {
    for (int i = tid; i < kPrepThreads + kMaxGroup; i += kPrepThreads) {
      const int q = base + i;
      if (q < a.Q) {
        int64_t ns;
        if (a.cand) {
          ns = (int64_t)a.ncb * 8;
        } else {
          ns = n_visible(a.q_pos[q], a.ratio);
          if (ns > a.ld) { if (i < kPrepThreads) raise_fault(kFaultBounds); ns = a.ld; }
        }
        s_seq[i] = a.q_seq[q];
        s_ns[i] = (int)ns;
        if (i < kPrepThreads) {
          s_rb[i] = a.row_base[s_seq[i]];
          if ((a.plane8 || a.plane4) && (s_rb[i] & 7) != 0)
            raise_fault(kFaultBounds);  // block planes start every sequence on a block
        }
      }
    }
    const int q = base + tid;
    const bool in = q < a.Q;
    __syncthreads();
    // run start of q: inclusive max-scan of the positions where the sequence changes
    int v = -1;
    if (in) {
      const int before = tid > 0 ? s_seq[tid - 1] : prev_seq;
      v = (q == 0 || s_seq[tid] != before) ? q : -1;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v = max(v, t);
    }
    if (lane == 31) red_run[warp] = v;
    __syncthreads();
    int rs = max(carry_run, v);
    {
      const int wv = lane < kPrepWarps ? red_run[lane] : -1;
      int sv = lane < warp ? wv : -1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sv = max(sv, __shfl_xor_sync(0xFFFFFFFFu, sv, o));
      rs = max(rs, sv);
    }
    // leaders: members and the group's largest visible count
    const bool lead = in && ((q - rs) % a.group_max) == 0;
    int nq = 0;
    long long tiles = 0;
    if (lead) {
      nq = 1;
      int mx = s_ns[tid];
      while (nq < a.group_max && q + nq < a.Q && s_seq[tid + nq] == s_seq[tid]) {
        mx = max(mx, s_ns[tid + nq]);
        ++nq;
      }
      tiles = (mx + kTileRows - 1) / kTileRows;
    }
    int ex, tx;
    long long ey, ty;
    block_excl_sum2(lead ? 1 : 0, tiles, redx, redy, ex, ey, tx, ty);
    if (base == 0) griddep_wait();  // the workspace writes of this call start here
    if (in) {
      a.n_scored[q] = (int32_t)s_ns[tid];
      a.topk_count[q] = 0;
      if (a.pool_count) a.pool_count[q] = 0;
    }
    if (lead) {
      GroupRec r;
      r.q0 = q;
      r.nq = nq;
      r.seq = s_seq[tid];
      r.pad0 = 0;
      r.tile0 = carry_tiles + ey;
      r.tile1 = r.tile0 + tiles;
      r.rb = s_rb[tid];
      r.pad1 = 0;
      a.grp[carry_groups + ex] = r;
      if (carry_groups + ex < kPrepGroupCache) {
        s_t0[carry_groups + ex] = r.tile0;
        s_t1[carry_groups + ex] = r.tile1;
      }
    }
    // carries into the next block (every thread keeps its own copy); block_excl_sum2
    // ended with a barrier, so red_run is free
    if (tid == kPrepThreads - 1) red_run[0] = rs;
    __syncthreads();
    carry_run = red_run[0];
    prev_seq = s_seq[kPrepThreads - 1];
    carry_groups += tx;
    carry_tiles += ty;
    __syncthreads();  // s_seq / s_ns / red_run are rewritten by the next block
  }
  if (tid == 0) a.n_groups[0] = carry_groups;
  // the score CTAs' ranges (ceil(total / nctas) tiles each) and the group each starts in,
  // so that a score CTA starts after two loads instead of a search
  const int64_t total = carry_tiles;
  const int64_t per = (total + a.nctas - 1) / a.nctas;
  for (int c = tid; c < a.nctas; c += kPrepThreads) s_gfirst[c] = 0;
  __syncthreads();  // the group records (global and cached) are visible to all threads
  if (per > 0) {
    const bool cached = carry_groups <= kPrepGroupCache;
    for (int g = tid; g < carry_groups; g += kPrepThreads) {
      const int64_t t0 = cached ? s_t0[g] : a.grp[g].tile0;
      const int64_t t1 = cached ? s_t1[g] : a.grp[g].tile1;
      // CTAs whose first tile c * per lies in [t0, t1)
      for (int64_t c = (t0 + per - 1) / per; c * per < t1 && c < a.nctas; ++c)
        s_gfirst[c] = g;
    }
  }
  __syncthreads();
  for (int c = tid; c < a.nctas; c += kPrepThreads) {
    CtaRec r;
    r.g_first = s_gfirst[c];
    r.pad0 = 0;
    r.it_lo = min(total, (int64_t)c * per);
    r.it_hi = min(total, r.it_lo + per);
    r.pad1 = 0;
    a.cta[c] = r;
  }
}

// ---- main kernel -----------------------------------------------------------------------

__device__ __forceinline__ void load_group(const IndexArgs& a, int g, GroupInfo& gi) {
  const GroupRec r = a.grp[g];
  gi.q0 = r.q0;
  gi.nq = r.nq;
  gi.seq = r.seq;
  gi.tile0 = r.tile0;
  gi.tile1 = r.tile1;
  gi.rb = r.rb;
}

// ---- FP8 quantisation: [A] indexer figure (FP8 rows of 128 E4M3 codes with one fp32
//      scale; the query quantised per (token, head)); [E] indexer compressor ("row amax
//      -> ue8m0 -> e4m3") ----------------------------------------------------------------

// Exponent of the power-of-two scale of a group whose largest magnitude is amax: the
// smallest e with amax <= 448 * 2^e (448 = 1.75 * 2^8, the largest E4M3 value), read off
// the bits of amax; 0 for amax == 0.
__device__ __forceinline__ int ue8m0_exp(float amax) {
  const uint32_t u = __float_as_uint(amax);
  if (u == 0u) return 0;
  int E;
  uint32_t m;
  if ((u >> 23) != 0u) {
    E = (int)(u >> 23) - 127;
    m = u & 0x7FFFFFu;
  } else {  // subnormal: normalise the fraction
    const int p = 31 - __clz((int)u);
    E = p - 149;
    m = (u << (23 - p)) & 0x7FFFFFu;
  }
  return E - 8 + (m > 0x600000u ? 1 : 0);
}

// One warp quantises one row of 128 bf16 values (live == false: a row of zeros); lane l
// returns the codes of values 4l .. 4l+3 as one word.  Returns the row's scale 2^e.
// Dividing by 2^e is exact (two power-of-two factors keep each one a normal float).
__device__ __forceinline__ float quant_row_e4m3(const uint16_t* src, bool live, uint32_t& codes) {
  const int lane = threadIdx.x & 31;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (live) {
    const uint2 r = __ldg(reinterpret_cast<const uint2*>(src) + lane);
    v[0] = __uint_as_float(r.x << 16); v[1] = __uint_as_float(r.x & 0xFFFF0000u);
    v[2] = __uint_as_float(r.y << 16); v[3] = __uint_as_float(r.y & 0xFFFF0000u);
  }
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int e = ue8m0_exp(amax);
  int ne = -e;
  float f1 = 1.f;
  if (ne > 100) { f1 = __uint_as_float((100u + 127u) << 23); ne -= 100; }
  const float f2 = __uint_as_float((uint32_t)(ne + 127) << 23);
  const uint32_t c01 = cvt_e4m3x2(v[0] * f1 * f2, v[1] * f1 * f2);
  const uint32_t c23 = cvt_e4m3x2(v[2] * f1 * f2, v[3] * f1 * f2);
  codes = c01 | (c23 << 16);
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23)
                   : __uint_as_float(1u << (e + 149));
}

// One CTA per block of the FP8 plane: warp w quantises row 8 * blockIdx.x + w.
__global__ void __launch_bounds__(256) plane_fp8_kernel(const uint16_t* k, int64_t n,
                                                        uint8_t* plane) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  uint32_t codes;
  const float sc = quant_row_e4m3(k + (r < n ? r : 0) * kDIdx, r < n, codes);
  uint8_t* blk = plane + (int64_t)blockIdx.x * kFp8BlockBytes;
  reinterpret_cast<uint32_t*>(blk + (r & 7) * kDIdx)[lane] = codes;
  if (lane == 0) reinterpret_cast<float*>(blk + 8 * kDIdx)[r & 7] = sc;
}

// The queries of an FP8 index call: row q * H + h -> codes [128] and a scale.
__global__ void __launch_bounds__(256) quant_q_kernel(IndexArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= (int64_t)a.Q * a.H) return;
  uint32_t codes;
  const float sc = quant_row_e4m3(a.iq + r * kDIdx, true, codes);
  reinterpret_cast<uint32_t*>(a.q8 + r * kDIdx)[lane] = codes;
  if (lane == 0) a.qscale[r] = sc;
}

// ---- MXFP4 quantisation: [A] indexer figure (FP4 index rows of 64 code bytes and 4 scale
//      bytes, paged in blocks of 8 rows); [A] indexer K (E2M1 values, one E8M0 scale per
//      32 dims) ----------------------------------------------------------------------------

// E8M0 code of a group whose largest magnitude is amax: the smallest e in [0, 254] with
// amax <= 6 * 2^(e - 127), and 127 for amax == 0.  With amax = M * 2^E (1 <= M < 2),
// 6 * 2^(E - 2) = 1.5 * 2^E covers M <= 1.5 and 3 * 2^E covers the rest.
__device__ __forceinline__ int e8m0_fp4(float amax) {
  const uint32_t u = __float_as_uint(amax);
  if (u == 0u) return 127;
  int E;
  uint32_t m;
  if ((u >> 23) != 0u) {
    E = (int)(u >> 23) - 127;
    m = u & 0x7FFFFFu;
  } else {
    const int p = 31 - __clz((int)u);
    E = p - 149;
    m = (u << (23 - p)) & 0x7FFFFFu;
  }
  const int e = 127 + E - 2 + (m > 0x400000u ? 1 : 0);
  return e < 0 ? 0 : (e > 254 ? 254 : e);
}

// One CTA per block of the plane: warp w quantises row 8 * blockIdx.x + w; lane l holds
// dims 4l .. 4l+3 of group l / 8.  Rows past n get zero codes and scale code 127.
__global__ void __launch_bounds__(256) plane_fp4_index_kernel(const uint16_t* k, int64_t n,
                                                              uint8_t* plane) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31, slot = threadIdx.x >> 5;
  const int64_t r = (int64_t)blockIdx.x * 8 + slot;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (r < n) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(k + r * kDIdx) + lane);
    v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
  }
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int e = e8m0_fp4(amax);
  // x / 2^(e - 127) as two exact power-of-two factors, each a normal float
  const int ne = 127 - e;  // in [-127, 127]
  const float f1 = __uint_as_float((uint32_t)((ne >> 1) + 127) << 23);
  const float f2 = __uint_as_float((uint32_t)((ne - (ne >> 1)) + 127) << 23);
  const __nv_fp4x2_storage_t c01 =
      __nv_cvt_float2_to_fp4x2(make_float2(v[0] * f1 * f2, v[1] * f1 * f2), __NV_E2M1,
                               cudaRoundNearest);
  const __nv_fp4x2_storage_t c23 =
      __nv_cvt_float2_to_fp4x2(make_float2(v[2] * f1 * f2, v[3] * f1 * f2), __NV_E2M1,
                               cudaRoundNearest);
  uint8_t* blk = plane + (int64_t)blockIdx.x * kFp4BlockBytes;
  reinterpret_cast<uint16_t*>(blk + slot * 64)[lane] =
      (uint16_t)((uint32_t)c01 | ((uint32_t)c23 << 8));
  if ((lane & 7) == 0) blk[512 + slot * 4 + (lane >> 3)] = (uint8_t)e;
}

// ---- FP4 tile conversion ------------------------------------------------------------------
// A code byte holds dims 2i (low nibble) and 2i+1.  The hardware conversion gives the
// E2M1 values as f16 (exact); shifting each f16 magnitude right by 3 gives the bf16 bits
// of the same value times 2^-112 (bias 15 against 127, 10 mantissa bits against 7, and an
// E2M1 value uses only the top mantissa bit), and a bf16 multiply by 2^(e - 15) then gives
// value * 2^(e - 127) exactly while the result is normal (2 <= e <= 142).  Groups with
// other scale codes take the float path.

// The eight E2M1 codes of a word as four f16 pairs.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b32 {c0, c1, c2, c3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Eight values of a group with scale code e in [2, 142], as one 16-byte bf16 chunk.
__device__ __forceinline__ uint4 fp4_word_fast(uint32_t w, uint32_t s2) {
  uint32_t h[4], o[4];
  e2m1x8_to_f16x2(w, h);
#pragma unroll
  for (int b = 0; b < 4; ++b)
    o[b] = mul_bf16x2(((h[b] & 0x7FFF7FFFu) >> 3) | (h[b] & 0x80008000u), s2);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The float path for any scale code (2^(e - 127), subnormal below -126), one chunk.
__device__ __noinline__ uint4 fp4_word_slow(uint32_t w, int e) {
  const int ex = e - 127;
  const float sf = ex >= -126 ? __uint_as_float((uint32_t)(ex + 127) << 23)
                              : __uint_as_float(1u << (ex + 149));
  uint32_t h[4], o[4];
  e2m1x8_to_f16x2(w, h);
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[b]));
    o[b] = pack_bf16x2(f.x * sf, f.y * sf);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// kModeFp8 / kModeFp8Gat: K tiles and queries are E4M3 codes (tcgen05 kind::f8f6f4, K = 32
// per MMA); the row scale of K and the query scales multiply the head sum in the epilogue.
// FULL tiles (kModeFp8, 320 threads) come by one TMA box over the block layout ([16 blocks]
// [8 rows][128 B], the scales skipped by the block stride); REINDEX tiles (kModeFp8Gat) are
// gathered by warps 10..17 as in the gather mode (one box per 1 KiB candidate block is as
// slow as the bf16 plane's).  Two instances, because the gather warps' threads leave the
// epilogue fewer registers, which costs the FULL instance's wide query groups (prefill).
// kModeFp4: the producer bulk-copies the tile's 16 packed blocks, warps 10..17 convert
// them to a bf16 tile (exact) and the MMAs and epilogue are those of the bf16 mode.
// kModeGather (REINDEX on the bf16 plane): the tile's 16 candidate blocks are 2 KiB each at
// random places, which a TMA copy per block fetches at about 20 GB/s per SM; instead warps
// 10..17 gather them by 16-byte asynchronous copies into the swizzled tile (each warp two
// blocks, up to four tiles in flight), and the producer only loads the Q blocks.
template <int kMode>
__global__ void __launch_bounds__(num_threads(kMode), 1)
    index_score_kernel(IndexArgs a, const __grid_constant__ CUtensorMap kmap_tile,
                       const __grid_constant__ CUtensorMap kmap_blk,
                       const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // rounded up to 1024 bytes by pointer arithmetic, so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr bool kFp8 = kMode == kModeFp8 || kMode == kModeFp8Gat;
  constexpr bool kFp4 = kMode == kModeFp4;
  constexpr bool kGat = kMode == kModeGather;
  // warps 10..17 fill the operand ring (candidate blocks on the bf16 or FP8 plane)
  constexpr bool fill = kGat || kMode == kModeFp8Gat;
  // the ring the producer fills: operand tiles, or the FP4 mode's packed blocks
  constexpr int kStages = kFp4 ? kFp4StgStages : num_stages(kMode);
  constexpr int kStageBytes = kFp4 ? kFp4StgBytes : stage_bytes(kMode);
  uint8_t* a_smem = smem;                              // MMA operand tiles
  uint8_t* fill_smem = kFp4 ? smem + kFp4CvStages * kBf16Tile : smem;
  uint8_t* b_smem = smem + ring_bytes(kMode);          // 64 KiB
  float* w_all = reinterpret_cast<float*>(b_smem + kBBytes);  // [8][256], per epilogue warp
  Bars* bars = reinterpret_cast<Bars*>(w_all + 8 * 256);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int64_t* gq_all = reinterpret_cast<int64_t*>(tmem_slot + 4);  // [8][kMaxGroup] row limit

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    if (!kFp4) {
      prefetch_tensormap(&kmap_tile);
      prefetch_tensormap(&kmap_blk);
    }
    prefetch_tensormap(&qmap);
  }
  // the barriers and the accumulators (shared memory and TMEM only) are set up while the
  // preceding kernel drains: the allocation never waits on another kernel, as no other
  // kernel that holds TMEM fits beside this one in shared memory
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->full[s]), fill ? 32 * kGatherWarps : 1);  // gathers: their threads
      mbar_init(smem_u32(&bars->empty[s]), kFp4 ? kFp4ConvWarps : 1);  // FP4: the converters
    }
    for (int s = 0; s < kFp4CvStages; ++s) {
      mbar_init(smem_u32(&bars->cv_full[s]), kFp4ConvWarps);
      mbar_init(smem_u32(&bars->cv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->acc_full[s]), 1);
      mbar_init(smem_u32(&bars->acc_empty[s]), 4);
    }
    mbar_init(smem_u32(&bars->b_full), 1);
    mbar_init(smem_u32(&bars->b_empty), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();
  // this CTA's tile range and first group, from the prep kernel
  const CtaRec cr = a.cta[blockIdx.x];
  const int64_t it_lo = cr.it_lo, it_hi = cr.it_hi;
  const int g_first = cr.g_first;
  if (it_lo >= it_hi) {
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }

  const float alpha = rsqrtf((float)kDIdx) * rsqrtf((float)a.H);

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      const uint64_t pol_k = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      GroupInfo gi;
      int g = g_first - 1;
      gi.tile1 = -1;
      int u = 0;  // groups loaded
      int64_t issued[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = -1;
      for (int64_t it = it_lo; it < it_hi; ++it) {
        if (*abort_flag) break;
        while (it >= gi.tile1) {
          ++g;
          load_group(a, g, gi);
        }
        if (it == it_lo || it == gi.tile0) {  // new group: load its Q block
          if (u > 0 && !mbar_wait(smem_u32(&bars->b_empty), (u - 1) & 1)) { *abort_flag = 1; break; }
          const uint32_t bb = smem_u32(&bars->b_full);
          mbar_arrive_expect_tx(bb, (uint32_t)(gi.nq * a.H * kDIdx * (kFp8 ? 1 : 2)));
          for (int i = 0; i < gi.nq; ++i) {
            if (kFp8) {
              tma_load_2d(smem_u32(b_smem + i * a.H * 128), &qmap, 0, (gi.q0 + i) * a.H, bb,
                          pol_q);
            } else {
              for (int db = 0; db < 2; ++db)
                tma_load_2d(smem_u32(b_smem + db * 32768 + i * a.H * 128), &qmap, db * 64,
                            (gi.q0 + i) * a.H, bb, pol_q);
            }
          }
          ++u;
        }
        if (fill) continue;  // the gather warps fill the ring
        const int64_t k = it - it_lo;
        const int s = (int)(k % kStages);
        const uint32_t round = (uint32_t)(k / kStages);
        if (!mbar_wait(smem_u32(&bars->empty[s]), (round & 1) ^ 1)) { *abort_flag = 1; break; }
        const uint32_t fb = smem_u32(&bars->full[s]);
        if (!kFp4) mbar_arrive_expect_tx(fb, kStageBytes);  // FP4: per copy below
        issued[s] = round;
        const int64_t tile = it - gi.tile0;
        uint8_t* dst = fill_smem + s * kStageBytes;
        if (kFp4) {
          // the tile's 16 packed blocks; copies never leave the plane (a block id outside
          // it is a caller error: flagged, and block 0 is read instead)
          const int64_t nbt = (a.index_rows + 7) >> 3;
          const int64_t b0 = gi.rb >> 3;
          if (!a.cand) {
            const int64_t first = b0 + tile * 16;
            const int64_t nblk = first < 0 ? 0 : (nbt - first < 16 ? nbt - first : 16);
            if (nblk > 0) {
              mbar_arrive_expect_tx(fb, (uint32_t)(nblk * kFp4BlockBytes));
              bulk_copy_g2s(smem_u32(dst), a.plane4 + first * kFp4BlockBytes,
                            (uint32_t)(nblk * kFp4BlockBytes), fb);
            } else {
              mbar_arrive(fb);
            }
          } else {
            const int32_t* cb = a.cand + (int64_t)gi.q0 * a.ncb + tile * 16;
            int32_t blk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) blk[i] = tile * 16 + i < a.ncb ? __ldg(cb + i) : -1;
            mbar_arrive_expect_tx(fb, (uint32_t)kFp4StgBytes);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              int64_t src = blk[i] >= 0 ? b0 + blk[i] : 0;
              if (src >= nbt) { raise_fault(kFaultBounds); src = 0; }
              bulk_copy_g2s(smem_u32(dst + i * kFp4BlockBytes), a.plane4 + src * kFp4BlockBytes,
                            (uint32_t)kFp4BlockBytes, fb);
            }
          }
        } else if (kFp8) {
          // FULL: blocks (row_base + 128 tile) / 8 .. + 15 as [16][8 rows][128 B]
          tma_load_3d(smem_u32(dst), &kmap_tile, 0, 0, (int32_t)((gi.rb >> 3) + tile * 16), fb,
                      pol_k);
        } else {  // bf16 FULL (candidate blocks are gathered, kModeGather)
          const int32_t y = (int32_t)(gi.rb + tile * kTileRows);
          for (int db = 0; db < 2; ++db)
            tma_load_2d(smem_u32(dst + db * 16384), &kmap_tile, db * 64, y, fb, pol_k);
        }
      }
      // do not leave the CTA with copies still landing in shared memory
      for (int s = 0; s < kStages; ++s)
        if (issued[s] >= 0) mbar_wait(smem_u32(&bars->full[s]), (uint32_t)(issued[s] & 1),
                                      100000000ull);
      if (u > 0) mbar_wait(smem_u32(&bars->b_full), (u - 1) & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    if (lane == 0) {
      GroupInfo gi;
      int g = g_first - 1;
      gi.tile1 = -1;
      int u = 0;
      uint32_t idesc = 0;
      for (int64_t it = it_lo; it < it_hi; ++it) {
        if (*abort_flag) break;
        while (it >= gi.tile1) {
          ++g;
          load_group(a, g, gi);
        }
        if (it == it_lo || it == gi.tile0) {
          if (!mbar_wait(smem_u32(&bars->b_full), u & 1)) { *abort_flag = 1; break; }
          ++u;
          idesc = kFp8 ? idesc_e4m3(128, gi.nq * a.H) : idesc_bf16(128, gi.nq * a.H, 0, 0);
        }
        const int64_t k = it - it_lo;
        const int s = (int)(k % kStages);
        const uint32_t round = (uint32_t)(k / kStages);
        const int ab = (int)(k & 1);
        const uint32_t use = (uint32_t)(k >> 1);
        // FP4: the converted tile k & 1 (its use k >> 1, the accumulator's)
        const uint32_t in_bar = kFp4 ? smem_u32(&bars->cv_full[ab]) : smem_u32(&bars->full[s]);
        if (!mbar_wait(in_bar, kFp4 ? (use & 1) : (round & 1))) { *abort_flag = 1; break; }
        if (!mbar_wait(smem_u32(&bars->acc_empty[ab]), (use & 1) ^ 1)) { *abort_flag = 1; break; }
        if (fill) fence_proxy_async_smem();  // the gathered tile was written by cp.async
        tc_fence_after();
        const uint32_t a_base = kFp4 ? smem_u32(a_smem + ab * kBf16Tile)
                                     : smem_u32(a_smem + s * kStageBytes);
        const uint32_t b_base = smem_u32(b_smem);
        const uint32_t d = tmem + (uint32_t)(ab * 256);
        if (kFp8) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 4 x K = 32 codes, 32 bytes apart
            const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
            umma_f8(d, ad, bd, idesc, kk != 0);
          }
        } else {
          // tile rows in 8-row atoms, 1 KiB apart in each 16 KiB dim half
          const uint32_t half = 16384u, sbo = 1024u;
#pragma unroll
          for (int db = 0; db < 2; ++db)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc_sw128(a_base + db * half + kk * 32, 16, sbo);
              const uint64_t bd = sdesc_sw128(b_base + db * 32768 + kk * 32, 16, 1024);
              umma_bf16(d, ad, bd, idesc, (db | kk) != 0);
            }
        }
        umma_commit(kFp4 ? smem_u32(&bars->cv_empty[ab]) : smem_u32(&bars->empty[s]));
        umma_commit(smem_u32(&bars->acc_full[ab]));
        if (it + 1 == it_hi || it + 1 == gi.tile1) umma_commit(smem_u32(&bars->b_empty));
      }
    }
  } else if (fill && warp >= 10) {
    // ============ tile gathers: warps 10..17 ============
    // Warp w copies blocks 2w and 2w + 1 of each tile: lane l, step j takes 16-byte piece
    // 32 j + l of the pair (a block is 8 rows x 16 pieces; a step covers two rows of one
    // block, 512 contiguous bytes) into row 8 (2w + j / 4) + r8 of the tile, dim half c / 8,
    // swizzled as a TMA tile.  A missing block (-1), or rows past the plane's end (those of
    // a partial newest block), are not copied: such rows are invalid in the epilogue and
    // an MMA row depends only on its own tile row.  Every thread's part of a tile arrives
    // on the tile's barrier when it lands (the MMA warp fences before reading it), so the
    // whole ring is in flight; the next tile's block ids are fetched meanwhile.
    // FP8 (FULL: the 16 consecutive blocks of the tile; REINDEX: 16 candidate blocks): a
    // block is 8 rows x 8 pieces of codes (its 32 scale bytes are read by the epilogue), a
    // step of the warp is four rows of one block; the tile is [128 rows][128 B].
    const int gw = warp - 10;
    GroupInfo gi;
    int g = g_first - 1;
    gi.tile1 = -1;
    const int64_t ntile = it_hi - it_lo;
    int32_t nb0 = -1, nb1 = -1;
    int64_t nrb = 0;
    auto fetch_ids = [&](int64_t it) {  // block ids of this warp's pair in tile it
      while (it >= gi.tile1) {
        ++g;
        load_group(a, g, gi);
      }
      const int64_t c0 = (it - gi.tile0) * 16 + 2 * gw;
      if (a.cand) {
        const int32_t* cb = a.cand + (int64_t)gi.q0 * a.ncb;
        nb0 = c0 < a.ncb ? __ldg(cb + c0) : -1;
        nb1 = c0 + 1 < a.ncb ? __ldg(cb + c0 + 1) : -1;
      } else {  // FULL (FP8): the tile's own blocks, from the sequence's first row
        nb0 = (int32_t)c0;
        nb1 = (int32_t)c0 + 1;
      }
      nrb = gi.rb;
    };
    if (ntile > 0) fetch_ids(it_lo);
    int64_t k = 0;
    for (; k < ntile; ++k) {
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
      const int s = (int)(k % kStages);
      const uint32_t round = (uint32_t)(k / kStages);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->empty[s]), (round & 1) ^ 1))) {
        *abort_flag = 1;
        break;
      }
      const int32_t b0 = nb0, b1 = nb1;
      const int64_t rb = nrb;
      const uint32_t stg = smem_u32(a_smem + s * kStageBytes);
      if (kFp8) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int pc = j * 32 + lane;
          const int32_t blk = j < 2 ? b0 : b1;
          const int r8 = (pc & 63) >> 3, c = pc & 7;
          const uint32_t row = (uint32_t)((2 * gw + (j >> 1)) * 8 + r8);
          const int64_t grow = rb + (int64_t)blk * 8 + r8;  // rb is a multiple of 8
          if (blk >= 0 && grow < a.index_rows)
            cp_async16(stg + sw128_off(row, (uint32_t)c),
                       a.plane8 + (grow >> 3) * kFp8BlockBytes + r8 * kDIdx + c * 16);
        }
      }
#pragma unroll
      for (int j = 0; j < 8 && !kFp8; ++j) {
        const int pc = j * 32 + lane;
        const int32_t blk = j < 4 ? b0 : b1;
        const int r8 = (pc & 127) >> 4, c = pc & 15;
        const uint32_t row = (uint32_t)((2 * gw + (j >> 2)) * 8 + r8);
        const int64_t grow = rb + (int64_t)blk * 8 + r8;
        if (blk >= 0 && grow < a.index_rows)
          cp_async16(stg + (uint32_t)(c >> 3) * 16384u + sw128_off(row, (uint32_t)(c & 7)),
                     a.index_k + grow * kDIdx + c * 8);
      }
      cp_async_arrive_noinc(smem_u32(&bars->full[s]));
      if (k + 1 < ntile) fetch_ids(it_lo + k + 1);
    }
    cp_async_wait_all();  // nothing may still be landing when the CTA exits
  } else if (kFp4 && warp >= 10) {
    // ============ FP4 converters: warps 10..17 ============
    // Warp c converts blocks c and c+8 of a tile; lane l takes row l / 4 of the
    // block and its dims 32 j .. 32 j + 31 (j = l % 4, one scale).  Each quarter-warp
    // reads 128 contiguous bytes; lanes with j >= 2 write their four 16-byte chunks in the
    // order 2, 3, 0, 1, so that each quarter-warp's stores fall in eight distinct chunk
    // positions of the swizzled rows (no bank conflicts).
    const int cw = warp - 10, j = lane & 3;
    for (int64_t it = it_lo; it < it_hi; ++it) {
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
      const int64_t k = it - it_lo;
      const int s = (int)(k % kStages);
      const uint32_t round = (uint32_t)(k / kStages);
      const int c = (int)(k & 1);
      const uint32_t use = (uint32_t)(k >> 1);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->full[s]), round & 1)) ||
          !__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->cv_empty[c]), (use & 1) ^ 1))) {
        *abort_flag = 1;
        break;
      }
      const uint8_t* src = fill_smem + s * kStageBytes;
      const uint32_t dst = smem_u32(a_smem + c * kBf16Tile) + (uint32_t)(j >> 1) * (kBf16Tile / 2);
      // all of the warp's blocks are loaded, then decoded, then stored, so that their
      // independent conversions overlap
      constexpr int kB = 16 / kFp4ConvWarps;
      uint4 cd[kB];
      int e[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const int blk = cw + kFp4ConvWarps * i;
        cd[i] = *reinterpret_cast<const uint4*>(src + blk * kFp4BlockBytes + lane * 16);
        e[i] = src[blk * kFp4BlockBytes + 512 + lane];
      }
      uint4 o[kB][4];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (j & 2) {
          const uint32_t x = cd[i].x, y = cd[i].y;
          cd[i].x = cd[i].z; cd[i].y = cd[i].w; cd[i].z = x; cd[i].w = y;
        }
        const uint32_t w4[4] = {cd[i].x, cd[i].y, cd[i].z, cd[i].w};
        const uint32_t sb = (uint32_t)(e[i] + 112) << 7, s2 = sb | (sb << 16);  // 2^(e - 15)
#pragma unroll
        for (int q = 0; q < 4; ++q) o[i][q] = fp4_word_fast(w4[q], s2);
        if (!(e[i] >= 2 && e[i] <= 142)) {  // rare: scale codes outside the fast path
#pragma unroll
          for (int q = 0; q < 4; ++q) o[i][q] = fp4_word_slow(w4[q], e[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const uint32_t row = (uint32_t)((cw + kFp4ConvWarps * i) * 8 + (lane >> 2));
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared16(dst + sw128_off(row, (uint32_t)((j & 1) * 4 + (q ^ (j & 2)))), o[i][q]);
      }
      fence_proxy_async_smem();  // the bf16 tile is read by the tensor cores
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->cv_full[c]));
        mbar_arrive(smem_u32(&bars->empty[s]));
      }
    }
  } else if (warp >= 2 && warp < 10) {
    // ============ epilogue: warps 2..5 (tiles k even), warps 6..9 (k odd) ============
    const int eg = (warp - 2) >> 2;       // epilogue group = TMEM accumulator it reads
    const int sub = warp & 3;             // TMEM sub-partition of this warp
    const int r = sub * 32 + lane;        // tile row = TMEM lane
    // every warp keeps its own copy of the group's weights and row limits, so a new
    // group needs no barrier across warps (an abort cannot strand one at a barrier)
    float* w_s = w_all + 256 * (warp - 2);
    int64_t* gq = gq_all + kMaxGroup * (warp - 2);
    GroupInfo gi;
    int g = g_first - 1;
    gi.tile1 = -1;
    int loaded = -1;  // query group whose weights sit in w_s
    for (int64_t it = it_lo + eg; it < it_hi; it += 2) {
      // warp-uniform exits: the loop body holds warp-collective TMEM loads and shuffles
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
      while (it >= gi.tile1) {
        ++g;
        load_group(a, g, gi);
      }
      if (g != loaded) {
        // all loads in flight at once (nq * H <= 256: eight per lane), then the stores
        const int nw = gi.nq * a.H;
        const float* wg = a.w + (int64_t)gi.q0 * a.H;
        float wv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) wv[u] = lane + 32 * u < nw ? __ldg(wg + lane + 32 * u) : 0.f;
        if (kFp8) {  // the queries' power-of-two scales fold into the weights exactly
          const float* qs = a.qscale + (int64_t)gi.q0 * a.H;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (lane + 32 * u < nw) wv[u] *= __ldg(qs + lane + 32 * u);
        }
        int64_t lim = 0;
        if (lane < gi.nq)
          lim = a.cand ? n_visible(a.q_pos[gi.q0 + lane], a.ratio)
                       : (int64_t)a.n_scored[gi.q0 + lane];
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (lane + 32 * u < nw) w_s[lane + 32 * u] = wv[u] * alpha;
        if (lane < gi.nq) gq[lane] = lim;
        __syncwarp();
        loaded = g;
      }
      const int64_t k = it - it_lo;
      const uint32_t use = (uint32_t)(k >> 1);
      const int64_t tile = it - gi.tile0;
      const int64_t pos = tile * kTileRows + r;
      // REINDEX groups hold one query: fetch its candidate block id before the wait
      const int32_t cblk = a.cand && (pos >> 3) < a.ncb
                               ? __ldg(a.cand + (int64_t)gi.q0 * a.ncb + (pos >> 3)) : -1;
      // FP8: this row's scale, from its block's tail (rows of a group share it)
      float sk = 1.f;
      if (kFp8) {
        const int64_t row = !a.cand ? gi.rb + pos
                                    : (cblk >= 0 ? gi.rb + (int64_t)cblk * 8 + (pos & 7) : -1);
        if (row >= 0 && row < a.index_rows)
          sk = __ldg(reinterpret_cast<const float*>(a.plane8 + (row >> 3) * kFp8BlockBytes +
                                                    8 * kDIdx) + (row & 7));
      }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bars->acc_full[eg]), use & 1))) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(sub * 32) << 16) + (uint32_t)(eg * 256);
      for (int i = 0; i < gi.nq; ++i) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const float4* w4 = reinterpret_cast<const float4*>(w_s + i * a.H);
        if (a.H == 64) {
          uint32_t v0[32], v1[32];
          tmem_ld32(tbase + (uint32_t)(i * 64), v0);
          tmem_ld32(tbase + (uint32_t)(i * 64 + 32), v1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 wa = w4[j >> 2], wb = w4[8 + (j >> 2)];
            float x0 = __uint_as_float(v0[j]), x1 = __uint_as_float(v0[j + 1]);
            float x2 = __uint_as_float(v0[j + 2]), x3 = __uint_as_float(v0[j + 3]);
            float y0 = __uint_as_float(v1[j]), y1 = __uint_as_float(v1[j + 1]);
            float y2 = __uint_as_float(v1[j + 2]), y3 = __uint_as_float(v1[j + 3]);
            if (a.relu) {
              x0 = fmaxf(x0, 0.f); x1 = fmaxf(x1, 0.f); x2 = fmaxf(x2, 0.f); x3 = fmaxf(x3, 0.f);
              y0 = fmaxf(y0, 0.f); y1 = fmaxf(y1, 0.f); y2 = fmaxf(y2, 0.f); y3 = fmaxf(y3, 0.f);
            }
            acc[0] = fmaf(wa.x, x0, acc[0]); acc[1] = fmaf(wa.y, x1, acc[1]);
            acc[2] = fmaf(wa.z, x2, acc[2]); acc[3] = fmaf(wa.w, x3, acc[3]);
            acc[0] = fmaf(wb.x, y0, acc[0]); acc[1] = fmaf(wb.y, y1, acc[1]);
            acc[2] = fmaf(wb.z, y2, acc[2]); acc[3] = fmaf(wb.w, y3, acc[3]);
          }
        } else {
          uint32_t v0[32];
          tmem_ld32(tbase + (uint32_t)(i * 32), v0);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 wa = w4[j >> 2];
            float x0 = __uint_as_float(v0[j]), x1 = __uint_as_float(v0[j + 1]);
            float x2 = __uint_as_float(v0[j + 2]), x3 = __uint_as_float(v0[j + 3]);
            if (a.relu) {
              x0 = fmaxf(x0, 0.f); x1 = fmaxf(x1, 0.f); x2 = fmaxf(x2, 0.f); x3 = fmaxf(x3, 0.f);
            }
            acc[0] = fmaf(wa.x, x0, acc[0]); acc[1] = fmaf(wa.y, x1, acc[1]);
            acc[2] = fmaf(wa.z, x2, acc[2]); acc[3] = fmaf(wa.w, x3, acc[3]);
          }
        }
        const float score = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * sk;
        const int q = gi.q0 + i;
        bool valid;
        if (!a.cand) {
          valid = pos < gq[i];
        } else {
          valid = cblk >= 0 && (int64_t)cblk * 8 + (pos & 7) < gq[i];
        }
        if (pos < a.ld) {
          a.keys[(int64_t)q * a.ldk + pos] = valid ? score_key(score) : 0u;
          if (valid && a.scores_out) a.scores_out[(int64_t)q * a.ld + pos] = score;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[eg]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t index_smem_bytes(int mode) {
  return 1024 + ring_bytes(mode) + kBBytes + 8 * 256 * 4 + sizeof(Bars) + 16 + 8 * 8 * kMaxGroup;
}

cudaError_t launch_index(const IndexArgs& args, int num_sms, cudaStream_t s) {
  if (args.Q == 0) return cudaSuccess;
  IndexArgs a = args;
  a.nctas = num_sms < kMaxIndexCtas ? num_sms : kMaxIndexCtas;  // one score CTA per SM
  cudaError_t e = launch_pdl(index_prep_kernel, dim3(1), dim3(kPrepThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  CUtensorMap kt, kb, qm;
  const int mode = a.plane8 ? (a.cand ? kModeFp8Gat : kModeFp8)
                            : (a.plane4 ? kModeFp4 : (a.cand ? kModeGather : kModeBf16));
  if (mode == kModeFp8 || mode == kModeFp8Gat) {
    const int64_t qrows = (int64_t)a.Q * a.H;
    e = launch_pdl(quant_q_kernel, dim3((unsigned)((qrows + 7) / 8)), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    // FULL tiles: the plane as [blocks][8 rows][128 B] (scales skipped by the block stride);
    // candidate blocks are gathered
    const uint64_t dims[3] = {(uint64_t)kDIdx, 8, (uint64_t)((a.index_rows + 7) / 8)};
    const uint64_t strides[2] = {(uint64_t)kDIdx, (uint64_t)kFp8BlockBytes};
    const uint32_t box_t[3] = {(uint32_t)kDIdx, 8, kTileRows / 8};
    const uint64_t qd[2] = {(uint64_t)kDIdx, (uint64_t)qrows};
    const uint64_t qs[1] = {(uint64_t)kDIdx};
    const uint32_t qbox[2] = {(uint32_t)kDIdx, (uint32_t)a.H};
    if (!encode_bytes(&kt, a.plane8, 3, dims, strides, box_t) ||
        !encode_bytes(&qm, a.q8, 2, qd, qs, qbox))
      return cudaErrorInvalidValue;
    kb = kt;
  } else if (mode == kModeFp4 || mode == kModeGather) {
    // K blocks arrive by bulk copies or gathers: only the query map is used (passed three
    // times)
    if (!encode_rows_bf16(&qm, a.iq, (uint64_t)a.Q * a.H, kDIdx, 64, (uint32_t)a.H))
      return cudaErrorInvalidValue;
    kt = qm;
    kb = qm;
  } else {
    if (!encode_rows_bf16(&kt, a.index_k, (uint64_t)a.index_rows, kDIdx, 64, kTileRows) ||
        !encode_rows_bf16(&qm, a.iq, (uint64_t)a.Q * a.H, kDIdx, 64, (uint32_t)a.H))
      return cudaErrorInvalidValue;
    kb = kt;  // FULL tiles only (candidate blocks are gathered)
  }
  const size_t smem = index_smem_bytes(mode);
  auto kern = mode == kModeFp8    ? index_score_kernel<kModeFp8>
              : mode == kModeFp8Gat ? index_score_kernel<kModeFp8Gat>
              : mode == kModeFp4  ? index_score_kernel<kModeFp4>
              : mode == kModeGather ? index_score_kernel<kModeGather>
                                    : index_score_kernel<kModeBf16>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.nctas), dim3(num_threads(mode)), smem, s, a, kt, kb, qm);
}

cudaError_t launch_plane_fp8(const uint16_t* k, int64_t n, uint8_t* plane, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t nb = (n + 7) / 8;
  return launch_pdl(plane_fp8_kernel, dim3((unsigned)nb), dim3(256), 0, s, k, n, plane);
}

cudaError_t launch_plane_fp4_index(const uint16_t* k, int64_t n, uint8_t* plane,
                                   cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t nb = (n + 7) / 8;
  return launch_pdl(plane_fp4_index_kernel, dim3((unsigned)nb), dim3(256), 0, s, k, n, plane);
}

}  // namespace csa2

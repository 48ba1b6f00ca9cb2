// k_attn.cu -- CSA2 sparse MQA attention (64 heads x 512 dims, K = V) over the
// layer's sliding window plus the selected compressed rows, one softmax with a
// per-head sink logit in the denominator.
// [A] "四种层合并出来的是什么形状" (one CSR, one softmax, K = V, <= 640 rows, sink only in
// the denominator); [B] §4.1 (two sources, no de-duplication), §4.4 step 4 (window
// slots); [C] §5.5-5.6 (logical concatenation, no physical copy), A.19.3 (gather by
// int32 index, online softmax with running max and sum, fused sink);
// [E] Fig. 2d (out_h = sum e^{s_j} v_j / (e^{sink_h} + sum e^{s_j})).
//
// A query's entries form up to ten chunks of 64 rows: chunks 0 and 1 are the window
// (positions p-127..p-64 and p-63..p), chunks 2..9 hold sel[64 (c-2) ..].  The chunks
// of one query are dealt round-robin to nsplit CTAs (grid = nsplit x Q); each CTA
// runs an online softmax over its chunks through a two-buffer pipeline:
//   gather   two teams of 256 threads, team b filling KV buffer b with every other
//            chunk in the 128-byte-swizzled layout [8 dim blocks][64 rows][128 B]
//            (bf16 rows by 16-byte cp.async, FP8 rows dequantised to bf16).  Row
//            gathers reach the HBM rate only with many requests in flight per SM, so
//            most of the CTA's threads are gatherers
//   S        = Q[64 x 512] . KV^T[512 x 64] -> TMEM buffer b as two M = 64 accumulators
//            (dims 0..255 and 256..511, issued by two threads): head h in lane
//            32 (h / 16) + h % 16, column = row
//   softmax  warps 0..3, four threads per pair of heads (16x256b TMEM loads): running
//            max and partial sums in registers, reductions over the thread's own
//            columns plus two shuffles where a head's four threads must agree.  P uses the
//            running max, which moves only when a score exceeds it by more than 64
//            (log2 units: P <= 2^64 keeps bf16 P and the fp32 sums finite).  P is
//            written in one pass with the current max; when a head's max moved the
//            chunk's pass is redone and warps 0..3 rescale O^T in TMEM (a barrier vote)
//   O^T     += V^T[512 x 64] . P^T[64 x 64] -> TMEM, four M = 128 tiles issued by two
//            threads; the KV buffer is the A operand again, read MN-major, and P
//            [head][row] is the B operand
// S of the next chunk runs while the softmax of this one does, and the gather of
// chunk c + 2 starts as soon as the PV of chunk c has released its buffer.
// Every CTA starts its running max at the sink logit.  With nsplit = 1 its running sum
// starts at the sink's mass (1) and the CTA writes the output.  With nsplit = 2 the two
// CTAs of a query run as a cluster and merge through distributed shared memory, each
// finishing half of the dims; the merge adds the sink's e^{sink_h} once.  With more
// queries than SMs (a prefill chunk) a second kernel runs nsplit = 1 on one CTA per SM
// that carries on from query to query (see sparse_attn_persist_kernel).
//
// Warps 0..3 softmax + O^T rescale + output, warps 4..19 gather (teams of eight
// warps), warps 20..23 issue the MMAs (lane 0 each; warp 20 also owns the TMEM).
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

CSA2_DEFINE_FAULT_FLAG(attn)

namespace csa2 {
namespace {

constexpr int kThreads = 768;             // 24 warps
constexpr int kGroupThreads = 128;        // warps 0..3
constexpr int kTeam = 256;                // threads per gather team
constexpr int kGatherWarp0 = 4;
constexpr int kMmaWarp = 20;              // warps 20..23 issue the MMAs
constexpr int kChunk = 64;                // rows per chunk
constexpr int kMaxChunks = 10;            // 2 window + 8 selected chunks
constexpr int kDimBlock = 64 * 128;       // one 64-dim block of 64 rows (8 KiB)
constexpr int kQBytes = 8 * kDimBlock;    // Q [8 dim blocks][64 heads][128 B]
constexpr int kBufBytes = 8 * kDimBlock;  // KV [8 dim blocks][64 rows][128 B]
constexpr int kPBytes = 64 * 128;         // P [64 heads][64 rows] bf16
constexpr uint32_t kColSa = 0;            // TMEM columns of S buffer b, dims 0..255: 64 b
constexpr uint32_t kColSb = 128;          // the same for dims 256..511: 128 + 64 b
constexpr uint32_t kColO = 256;           // O^T tiles at 256 + 64 * mt
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 64.0f;
constexpr int kRopeDim0 = 448;            // dims 448..511 carry the RoPE phase

struct __align__(16) Aux {
  float m_run[64];
  float l_run[64];
  float fac[2][64];  // rescale factor per head, by chunk parity (merge weights at the end)
  float rope_c[32];  // inverse RoPE of the output at the query position: cos, sin of
  float rope_s[32];  // p theta_i for pair i (dims 448 + 2i, 449 + 2i)
  float peer_m[64];  // cluster merge: the other CTA's running max and sum (filled by a
  float peer_l[64];  // store of its m_run, l_run: the pairs must stay adjacent)
  float sink2[64];   // sink logit per head in log2 units (-inf without a sink)
  int32_t rowidx[kMaxChunks][kChunk];  // source row per slot (chunk = rank + slot * nsplit)
  uint32_t rowmask[kMaxChunks][2];     // valid rows of each slot
  uint64_t q_full;      // Q landed (TMA transaction count)
  uint64_t kv_full[2];  // KV buffer filled (one arrival of the team)
  uint64_t s_full[2];   // both S halves of the buffer written (two commits)
  uint64_t p_full[2];   // P buffer written and O^T rescaled (128 arrivals)
  uint64_t pv_done[2];  // PV of the buffer's chunk complete (two commits)
  uint64_t fin[4];      // every MMA of an issuer complete (commit)
  uint64_t merge_full[2];  // cluster merge: the peer's rows of each tile landed
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// OR of `pred` over warps 0..3 (a barrier of the group with a reduction)
__device__ __forceinline__ bool group_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 128, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// Source row of entry r of chunk c of query q (sequence b, position p, compressed rows
// from rb): chunks 0 and 1 are window slots, chunk c >= 2 holds sel[64 (c - 2) + r]; -1
// for none.  A row outside its buffer raises the bounds fault and gives -1.
__device__ __forceinline__ int32_t chunk_row(const AttnArgs& a, int q, int b, int64_t p,
                                             int64_t rb, int c, int r) {
  int32_t idx32 = -1;
  if (c < 2) {
    const int64_t pos = p - (kRing - 1) + kChunk * c + r;
    if (pos >= 0) {
      int64_t idx;
      bool ok = true;
      if (a.swa_mode == 0) {
        idx = (int64_t)b * kRing + (pos & (kRing - 1));
      } else {
        // a position before the sequence's first stored row would index the previous
        // sequence's rows: a caller error, skipped and flagged
        const int64_t p0 = a.lin_pos0[b];
        ok = pos >= p0;
        idx = a.lin_base[b] + (pos - p0);
      }
      if (ok && idx >= 0 && idx < a.swa_rows) idx32 = (int32_t)idx;
      else raise_fault(kFaultBounds);
    }
  } else {
    const int i = (c - 2) * kChunk + r;
    if (i < a.nsel) {
      const int32_t rr = a.sel[(int64_t)q * a.nsel + i];
      if (rr >= 0) {
        const int64_t idx = rb + rr;
        if (idx >= 0 && idx < a.plane_rows) idx32 = (int32_t)idx;
        else raise_fault(kFaultBounds);
      }
    }
  }
  return idx32;
}

// Valid-row bits of columns 8 g + 2 r4 and 8 g + 2 r4 + 1 of a chunk (bit 0, bit 1).
__device__ __forceinline__ uint32_t col_mask(bool full, uint32_t mlo, uint32_t mhi, int g,
                                             int r4) {
  return full ? 3u : ((g < 4 ? mlo : mhi) >> (8 * (g & 3) + 2 * r4)) & 3u;
}

// One pass of a softmax thread over its 16 columns of heads hA and hB of a chunk's S
// (the sum of the accumulators at sa and sb): P = 2^(s scale2 - m), zero for invalid
// rows, stored as bf16 pairs into the P rows at pA / pB (swizzle sw); returns the sum
// of the stored (rounded) values and the largest s scale2 - m over the valid columns.
__device__ __forceinline__ void p_pass(uint32_t sa, uint32_t sb, bool full, uint32_t mlo,
                                       uint32_t mhi, int r4, float scale2, float mA, float mB,
                                       uint32_t pA, uint32_t pB, int sw, float& mxA, float& mxB,
                                       float& lsA, float& lsB) {
  mxA = -INFINITY; mxB = -INFINITY; lsA = 0.f; lsB = 0.f;
#pragma unroll 1
  for (int gb = 0; gb < 8; gb += 4) {
    uint32_t x[4][4], y[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      tmem_ld_16x256b(sa + 8 * (gb + i), x[i]);
      tmem_ld_16x256b(sb + 8 * (gb + i), y[i]);
    }
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int g = gb + i;
      const uint32_t mk = col_mask(full, mlo, mhi, g, r4);
      const float t0 = fmaf(__uint_as_float(x[i][0]) + __uint_as_float(y[i][0]), scale2, -mA);
      const float t1 = fmaf(__uint_as_float(x[i][1]) + __uint_as_float(y[i][1]), scale2, -mA);
      const float t2 = fmaf(__uint_as_float(x[i][2]) + __uint_as_float(y[i][2]), scale2, -mB);
      const float t3 = fmaf(__uint_as_float(x[i][3]) + __uint_as_float(y[i][3]), scale2, -mB);
      if (mk & 1u) { mxA = fmaxf(mxA, t0); mxB = fmaxf(mxB, t2); }
      if (mk & 2u) { mxA = fmaxf(mxA, t1); mxB = fmaxf(mxB, t3); }
      const uint32_t qa = pack_bf16x2((mk & 1u) ? ex2(t0) : 0.f, (mk & 2u) ? ex2(t1) : 0.f);
      const uint32_t qb = pack_bf16x2((mk & 1u) ? ex2(t2) : 0.f, (mk & 2u) ? ex2(t3) : 0.f);
      lsA += __uint_as_float(qa << 16) + __uint_as_float(qa & 0xFFFF0000u);
      lsB += __uint_as_float(qb << 16) + __uint_as_float(qb & 0xFFFF0000u);
      st_shared32(pA + ((g ^ sw) << 4), qa);
      st_shared32(pB + ((g ^ sw) << 4), qb);
    }
  }
}

// cos, sin of p theta_i for the 32 RoPE pairs (one warp: lane i), for the output's inverse
// rotation at the query position p.
__device__ __forceinline__ void rope_table(const float* inv_freq, int64_t p, int lane, float* rc,
                                           float* rs) {
  float s, c;
  sincosf(rope_angle(rope_turn(inv_freq[lane]), (uint64_t)p), &s, &c);
  rc[lane] = c;
  rs[lane] = s;
}

// Staged O^T rows: fp32, 64 heads per dim (256 B), 16-byte pieces of 4 heads; piece c
// of row d sits at position c ^ ot_swz(d), which keeps both the writer (32 consecutive
// dims, one piece each) and the reader (eight consecutive dims per thread, threads eight
// dims apart) free of bank conflicts.
__device__ __forceinline__ int ot_swz(int d) { return (d ^ (d >> 3)) & 7; }

// O^T tiles mt0 .. mt0 + ntile - 1 from TMEM into shared memory as staged rows; row =
// dim - 128 mt0.  `warp` is the caller's lane quarter (warp index % 4: TMEM lanes
// 32 warp ..); with n == 0 the tiles are zero.
__device__ __forceinline__ void stage_ot(uint32_t tmem_o, int warp, int lane, int mt0, int ntile,
                                         uint32_t stage, bool have) {
  const uint32_t lrow = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
  for (int mi = 0; mi < ntile; ++mi) {
    const int d = mi * 128 + warp * 32 + lane;
    const uint32_t row = stage + d * 256;
    const int sw = ot_swz(d);
#pragma unroll 1
    for (int hb = 0; hb < 64; hb += 32) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(tmem_o + lrow + 64 * (mt0 + mi) + hb, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const int c = (hb >> 2) + j4;  // heads 4c .. 4c + 3
        st_shared16(row + ((c ^ sw) << 4),
                    make_uint4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]));
      }
    }
  }
}

// out[q][h][dbase + d] = bf16(own[d][h] w0[h] + peer[d][h] w1[h]) for nd dims, from rows
// staged by stage_ot (peer may be null), by threads tid of nthreads.  A thread takes four
// heads x eight dims (eight 16-byte loads from each source) and stores four 16-byte runs;
// a warp covers consecutive dim groups of the same four heads, so each store is one
// contiguous 512-byte run per head.  With rc / rs (cos, sin of p theta_i), pair i of
// dims 448.. is rotated back: times e^{-i p theta_i}.
__device__ __forceinline__ void out_pass(const float* own, const float* peer, const float* w0,
                                         const float* w1, const float* rc, const float* rs,
                                         uint16_t* out_q, int nd, int dbase, int tid,
                                         int nthreads) {
  const int ng = nd >> 3;  // groups of eight dims
  for (int it = tid; it < 16 * ng; it += nthreads) {
    const int c = it / ng, g = it - c * ng;
    float wa[4], wb[4];
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      wa[hh] = w0[4 * c + hh];
      wb[hh] = peer ? w1[4 * c + hh] : 0.f;
    }
    float o[4][8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int d = 8 * g + j;
      const int off = d * 64 + ((c ^ ot_swz(d)) << 2);
      const float4 x = *reinterpret_cast<const float4*>(own + off);
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
      if (peer) y = *reinterpret_cast<const float4*>(peer + off);
      o[0][j] = x.x * wa[0] + y.x * wb[0];
      o[1][j] = x.y * wa[1] + y.y * wb[1];
      o[2][j] = x.z * wa[2] + y.z * wb[2];
      o[3][j] = x.w * wa[3] + y.w * wb[3];
    }
    const int gd = dbase + 8 * g;  // first output dim of the group
    if (rc && gd >= kRopeDim0) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const int i = (gd + j - kRopeDim0) >> 1;
        const float cs = rc[i], sn = rs[i];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const float o0 = o[hh][j] * cs + o[hh][j + 1] * sn;
          const float o1 = o[hh][j + 1] * cs - o[hh][j] * sn;
          o[hh][j] = o0;
          o[hh][j + 1] = o1;
        }
      }
    }
    // streaming stores: the output is not read again here and should not push the
    // plane's rows out of L2
#pragma unroll
    for (int hh = 0; hh < 4; ++hh)
      __stcs(reinterpret_cast<uint4*>(out_q + (4 * c + hh) * kDLat + gd),
             make_uint4(pack_bf16x2(o[hh][0], o[hh][1]), pack_bf16x2(o[hh][2], o[hh][3]),
                        pack_bf16x2(o[hh][4], o[hh][5]), pack_bf16x2(o[hh][6], o[hh][7])));
  }
}

// Rows of one chunk into the KV buffer at `kvb` by the threads of a team (t = 0..255);
// a row index below zero gives a row of zeros.  stream: bf16 rows are evicted from L2 first
// (a call that reads each row about once).
__device__ __forceinline__ void gather_chunk(const int32_t* rows, int fp8, bool fp4,
                                             const uint8_t* base, uint32_t kvb, int t,
                                             bool stream) {
  if (fp4) {
    // FP4 plane rows: 64 rows x 32 groups of 16 dims (8 code bytes + 1 scale byte); each
    // group becomes two 16-byte bf16 chunks.  E2M1 x E4M3 has at most six significant
    // bits, so the bf16 values are exact.  All of a thread's loads are issued before the
    // first conversion.
    constexpr int kItems = 64 * 32 / kTeam;
    uint2 codes[kItems];
    uint32_t scb[kItems];
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
      const int flat = i * kTeam + t;
      const int r = flat >> 5, g = flat & 31;
      codes[i] = make_uint2(0u, 0u);
      scb[i] = 0u;
      if (rows[r] >= 0) {
        const uint8_t* src = base + (int64_t)rows[r] * 288;
        codes[i] = __ldg(reinterpret_cast<const uint2*>(src + 8 * g));
        scb[i] = __ldg(src + 256 + g);
      }
    }
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
      const int flat = i * kTeam + t;
      const int r = flat >> 5, g = flat & 31;
      const uint32_t d0 = kvb + (g >> 2) * kDimBlock + sw128_off(r, (2 * g) & 7);
      const uint32_t d1 = kvb + (g >> 2) * kDimBlock + sw128_off(r, (2 * g + 1) & 7);
      // a missing row has zero codes and scale code 0: its values are zero
      const __half2_raw sr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)scb[i], __NV_E4M3);
      const float sc = __low2float(*reinterpret_cast<const __half2*>(&sr));
      const uint32_t w2[2] = {codes[i].x, codes[i].y};
      uint32_t packed[8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {  // byte b of word j: dims 8 j + 2 b, + 1
          const __half2_raw hr = __nv_cvt_fp4x2_to_halfraw2(
              (__nv_fp4x2_storage_t)((w2[j] >> (8 * b)) & 0xFFu), __NV_E2M1);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
          packed[4 * j + b] = pack_bf16x2(f.x * sc, f.y * sc);
        }
      }
      st_shared16(d0, make_uint4(packed[0], packed[1], packed[2], packed[3]));
      st_shared16(d1, make_uint4(packed[4], packed[5], packed[6], packed[7]));
    }
  } else if (fp8) {
    // 64 rows x 32 pieces of 16 codes; each piece becomes two 16-byte bf16 chunks
#pragma unroll 2
    for (int i = 0; i < 64 * 32 / kTeam; ++i) {
      const int flat = i * kTeam + t;
      const int r = flat >> 5, c16 = flat & 31;
      const int64_t off = rows[r] < 0 ? -1 : (int64_t)rows[r] * 528;
      const uint32_t d0 = kvb + (c16 >> 2) * kDimBlock + sw128_off(r, (2 * c16) & 7);
      const uint32_t d1 = kvb + (c16 >> 2) * kDimBlock + sw128_off(r, (2 * c16 + 1) & 7);
      if (off < 0) { st_shared_zero16(d0); st_shared_zero16(d1); continue; }
      const uint8_t* src = base + off;
      const uint4 codes = *reinterpret_cast<const uint4*>(src + c16 * 16);
      // fp8 == 1: one fp32 scale per 128 dims; 2: one E8M0 byte per 32 dims (2^(e - 127))
      const float sc = fp8 == 1
                           ? *reinterpret_cast<const float*>(src + 512 + 4 * (c16 >> 3))
                           : (src[512 + (c16 >> 1)] == 0
                                  ? __uint_as_float(0x00400000u)  // 2^-127 (subnormal)
                                  : __uint_as_float((uint32_t)src[512 + (c16 >> 1)] << 23));
      const uint32_t w4[4] = {codes.x, codes.y, codes.z, codes.w};
      uint32_t packed[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const __nv_fp8x2_storage_t two = (__nv_fp8x2_storage_t)((w4[j] >> (16 * hh)) & 0xFFFFu);
          const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
          packed[2 * j + hh] = pack_bf16x2(f.x * sc, f.y * sc);
        }
      }
      st_shared16(d0, make_uint4(packed[0], packed[1], packed[2], packed[3]));
      st_shared16(d1, make_uint4(packed[4], packed[5], packed[6], packed[7]));
    }
  } else {
    // four 1 KiB rows per iteration of the team
    const uint64_t pol = stream ? policy_evict_first() : policy_evict_normal();
#pragma unroll
    for (int i = 0; i < 64 * 64 / kTeam; ++i) {
      const int flat = i * kTeam + t;
      const int r = flat >> 6, c = flat & 63;
      const int64_t off = rows[r] < 0 ? -1 : (int64_t)rows[r] * 1024;
      const uint32_t dst = kvb + (c >> 3) * kDimBlock + sw128_off(r, c & 7);
      if (off < 0) st_shared_zero16(dst);
      else cp_async16_hint(dst, base + off + c * 16, pol);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap wmap,
                       const __grid_constant__ CUtensorMap omap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // rounded up to 1024 bytes by pointer arithmetic, so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + kQBytes;            // two buffers
  uint8_t* p_s = kv_s + 2 * kBufBytes;       // two buffers
  Aux& X = *reinterpret_cast<Aux*>(p_s + 2 * kPBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = blockIdx.y;
  const int rank = blockIdx.x;
  const int nsplit = gridDim.x;
  griddep_launch_dependents();
  if (tid == 0) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&wmap);
    mbar_init(smem_u32(&X.q_full), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&X.kv_full[b]), 1);
      mbar_init(smem_u32(&X.s_full[b]), 2);
      mbar_init(smem_u32(&X.p_full[b]), kGroupThreads);
      mbar_init(smem_u32(&X.pv_done[b]), 2);
    }
    for (int r = 0; r < 4; ++r) mbar_init(smem_u32(&X.fin[r]), 1);
    for (int t = 0; t < 2; ++t) mbar_init(smem_u32(&X.merge_full[t]), 1);
    X.abort = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&X.tmem_slot), 512);
    tmem_relinquish();
  }
  // ---- before the dependency wait: only this call's inputs (q, positions, the window),
  // never the selection a preceding kernel may still be writing ----
  const uint32_t qb = smem_u32(q_s), kv0 = smem_u32(kv_s), p0 = smem_u32(p_s);
  if (tid == 0) {
    // Q [64 heads][512] of this query: eight 64 x 64 boxes, one per dim block
    const uint32_t qf = smem_u32(&X.q_full);
    mbar_arrive_expect_tx(qf, kQBytes);
    const uint64_t pol = policy_evict_first();
#pragma unroll
    for (int db = 0; db < 8; ++db) tma_load_2d(qb + db * kDimBlock, &qmap, 64 * db, q * kHeads, qf, pol);
  }
  const int b = a.q_seq[q];
  const int64_t p = a.q_pos[q];
  const float scale2 = a.scale * kLog2e;
  const int nchunks_total = 2 + (a.nsel + kChunk - 1) / kChunk;
  // row sources of this CTA's chunks (chunk = rank + slot * nsplit): the window slots
  // (chunks 0, 1) now, the selected ones after the wait
  const int nslot = (nchunks_total - rank + nsplit - 1) / nsplit;
  int nwin = 0;  // window slots come first
  while (nwin < nslot && rank + nwin * nsplit < 2) ++nwin;
  const int64_t rb = a.row_base ? a.row_base[b] : 0;  // no row_base: no selected rows
  auto row_source = [&](int e) {
    const int slot = e >> 6, r = e & 63;
    const int32_t idx32 = chunk_row(a, q, b, p, rb, rank + slot * nsplit, r);
    X.rowidx[slot][r] = idx32;
    // the 32 lanes of a warp cover one half of a slot (768 threads = 24 warps)
    const uint32_t vm = __ballot_sync(0xFFFFFFFFu, idx32 >= 0);
    if (lane == 0) X.rowmask[slot][r >> 5] = vm;
  };
  for (int e = tid; e < nwin * kChunk; e += kThreads) row_source(e);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Every slot of the CTA is a chunk (an empty one runs as a fully masked chunk), the
  // window slots first; gather team t owns slots t, t + 2, ..  The window slots run before
  // the wait: team t (t < nwin) lands window slot t now.
  const bool is_gather = warp >= kGatherWarp0 && warp < kMmaWarp;
  const int team = is_gather ? (warp - kGatherWarp0) / (kTeam / 32) : 0;
  const int t_in_team = tid - kGatherWarp0 * 32 - kTeam * team;
  const int n = nslot;
  const uint32_t tmem = X.tmem_slot;
  auto issue_gather = [&](int slot) -> bool {  // true: a TMA box load (arrives by itself)
    const int c = rank + slot * nsplit;
    const uint32_t kvb = kv0 + team * kBufBytes;
    const uint32_t full_bar = smem_u32(&X.kv_full[team]);
    // a full window chunk of a LINEAR bf16 window is 64 consecutive rows: one TMA box
    // of 64 x 64 per dim block
    if (c < 2 && a.swa_mode == 1 && a.swa_dtype == 0 &&
        (X.rowmask[slot][0] & X.rowmask[slot][1]) == 0xFFFFFFFFu) {
      if (t_in_team == 0) {
        mbar_arrive_expect_tx(full_bar, kBufBytes);
        const int32_t y0 = X.rowidx[slot][0];
        const uint64_t pol = policy_evict_first();
#pragma unroll
        for (int db = 0; db < 8; ++db)
          tma_load_2d(kvb + db * kDimBlock, &wmap, 64 * db, y0, full_bar, pol);
      }
      return true;
    }
    const int fp8 = c < 2 ? a.swa_dtype : 0;  // 1, 2: the FP8 window layouts
    const uint8_t* base = c < 2 ? a.swa : reinterpret_cast<const uint8_t*>(a.plane);
    gather_chunk(X.rowidx[slot], fp8, c >= 2 && a.plane_dtype == 1, base, kvb, t_in_team,
                 a.stream_rows != 0);
    cp_async_commit();
    return false;
  };
  if (is_gather && team < nwin && !issue_gather(team)) {
    cp_async_wait_group<0>();
    fence_proxy_async_smem();
    if (team == 0) asm volatile("bar.sync 2, 256;" ::: "memory");
    else asm volatile("bar.sync 3, 256;" ::: "memory");
    if (t_in_team == 0) mbar_arrive(smem_u32(&X.kv_full[team]));
  }

  if (is_gather) {
    // =================== gather: team 0 = warps 4..11; team 1 = warps 12..19 ===================
    // Only the gathers read what the preceding kernels write (the selection, the
    // compressed plane), so only they wait for them.  Each team then reads the row
    // sources of its own selected slots (at most four, one entry per thread, the loads in
    // flight together) and starts gathering.
    const int t = t_in_team;
    const uint32_t full_bar = smem_u32(&X.kv_full[team]);
    griddep_wait();
    {
      int s0 = team;  // the team's first selected slot
      while (s0 < nwin) s0 += 2;
      const int slot = s0 + 2 * (t >> 6);
      if (slot < nslot) row_source(slot * kChunk + (t & 63));  // uniform within a warp
      if (team == 0) asm volatile("bar.sync 2, 256;" ::: "memory");
      else asm volatile("bar.sync 3, 256;" ::: "memory");
    }
    int last = -1;  // last chunk of this team (its kv_full phase ends every copy of the team)
    for (int it = team; it < n; it += 2) {
      last = it;
      if (it < nwin) continue;  // a window slot: landed before the wait
      if (it >= 2 && !X.abort &&
          !mbar_wait(smem_u32(&X.pv_done[team]), (uint32_t)((it - 2) >> 1) & 1))
        X.abort = 1;
      if (issue_gather(it)) continue;
      cp_async_wait_group<0>();
      fence_proxy_async_smem();
      // every thread of the team has landed its rows
      if (team == 0) asm volatile("bar.sync 2, 256;" ::: "memory");
      else asm volatile("bar.sync 3, 256;" ::: "memory");
      if (t == 0) mbar_arrive(full_bar);
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (t == 0 && last >= 0) mbar_wait(full_bar, (uint32_t)(last >> 1) & 1, 100000000ull);
  } else if (warp >= kMmaWarp) {
    // ====== MMA issuers (lane 0): warp 20 S over dims 0..255, warp 21 S over dims
    // 256..511 (two accumulators, summed by the softmax), warps 22 and 23 PV into O^T
    // tiles 0, 1 and 2, 3 ======
    // One thread issues a tcgen05.mma about every 28 ns however small it is, so the
    // chunk's 48 small MMAs are spread over four threads.
    const int role = warp - kMmaWarp;
    if (lane == 0) {
      int issued = 0;
      if (role < 2) {
        const uint32_t id_s = idesc_bf16(64, 64, 0, 0);
        if (!mbar_wait(smem_u32(&X.q_full), 0)) X.abort = 1;
        for (int c = 0; !X.abort && c < n; ++c) {
          // kv_full of chunk c also means that the softmax of chunk c - 2 is done with
          // S buffer c & 1 (the gather of chunk c waited for the PV of chunk c - 2)
          if (!mbar_wait(smem_u32(&X.kv_full[c & 1]), (uint32_t)(c >> 1) & 1)) {
            X.abort = 1;
            break;
          }
          tc_fence_after();
          const uint32_t kvb = kv0 + (c & 1) * kBufBytes;
          const uint32_t d = tmem + (role ? kColSb : kColSa) + 64 * (c & 1);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int db = 4 * role + i;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(d, sdesc_sw128(qb + db * kDimBlock + kk * 32, 16, 1024),
                        sdesc_sw128(kvb + db * kDimBlock + kk * 32, 16, 1024), id_s,
                        (i | kk) != 0);
          }
          umma_commit(smem_u32(&X.s_full[c & 1]));
          ++issued;
        }
      } else {
        const uint32_t id_o = idesc_bf16(128, 64, 1, 0);
        for (int c = 0; !X.abort && c < n; ++c) {
          if (!mbar_wait(smem_u32(&X.p_full[c & 1]), (uint32_t)(c >> 1) & 1)) {
            X.abort = 1;
            break;
          }
          tc_fence_after();
          const uint32_t kvb = kv0 + (c & 1) * kBufBytes;
          const uint32_t pb = p0 + (c & 1) * kPBytes;
#pragma unroll
          for (int mt = 2 * (role - 2); mt < 2 * (role - 2) + 2; ++mt)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + kColO + 64 * mt,
                        sdesc_sw128(kvb + 2 * mt * kDimBlock + kk * 2048, kDimBlock, 1024),
                        sdesc_sw128(pb + kk * 32, 16, 1024), id_o, (c > 0 || kk > 0) ? 1 : 0);
          umma_commit(smem_u32(&X.pv_done[c & 1]));
          ++issued;
        }
      }
      // no MMA may still be running when the TMEM is released, whatever happened above
      if (issued > 0) {
        umma_commit(smem_u32(&X.fin[role]));
        mbar_wait(smem_u32(&X.fin[role]), 0, 100000000ull);
      }
    }
  } else {
    // ============ softmax + O^T rescale (warps 0..3) ============
    // S of a chunk is the sum of two M = 64 accumulators; head 16 w + i sits in TMEM lane
    // 32 w + i.  A 16x256b load of column group g gives thread t of warp w the columns
    // 8 g + 2 (t % 4) + {0, 1} of heads hA = 16 w + t / 4 and hB = hA + 8, so the four
    // threads with the same t / 4 share two heads: each keeps the running max of both
    // (kept equal across the four) and a partial running sum over its own columns.
    const int r4 = lane & 3;
    const int hA = 16 * warp + (lane >> 2), hB = hA + 8;
    const uint32_t lrow = (uint32_t)(warp * 32) << 16;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    if (a.sink) {
      // the running max starts at the sink logit, so no chunk needs a separate max pass;
      // the sink's own mass enters the sum here with one CTA per query, else once in the
      // merge
      mA = a.sink[hA] * kLog2e;
      mB = a.sink[hB] * kLog2e;
      if (nsplit == 1 && r4 == 0) { lA = 1.f; lB = 1.f; }
    }
    if (r4 == 0) {
      X.sink2[hA] = mA;
      X.sink2[hB] = mB;
    }
    for (int it = 0; it < n; ++it) {
      const int bsel = it & 1;
      const uint32_t ph = (uint32_t)(it >> 1) & 1;
      const uint32_t sa = tmem + lrow + kColSa + 64 * bsel;
      const uint32_t sb = tmem + lrow + kColSb + 64 * bsel;
      if (!X.abort && !mbar_wait(smem_u32(&X.s_full[bsel]), ph)) X.abort = 1;
      tc_fence_after();
      // the chunk's valid rows: written by its gather team before its rows landed (a
      // selected slot's only after the dependency wait), so read after S
      const uint32_t mlo = X.rowmask[it][0], mhi = X.rowmask[it][1];
      const bool full = (mlo & mhi) == 0xFFFFFFFFu;
      // the P buffer was last read by the PV of chunk it - 2
      if (it >= 2 && !X.abort &&
          !mbar_wait(smem_u32(&X.pv_done[bsel]), (uint32_t)((it - 2) >> 1) & 1))
        X.abort = 1;
      // P [head][row] bf16, 128-byte swizzled rows: thread t writes 4 bytes (two rows) of
      // heads hA and hB in each 16-byte chunk g
      const uint32_t pA = p0 + bsel * kPBytes + hA * 128 + 4 * r4;
      const uint32_t pB = p0 + bsel * kPBytes + hB * 128 + 4 * r4;
      const int sw = hA & 7;  // hB & 7 is the same
      float mxA, mxB, lsA, lsB, facA = 1.f, facB = 1.f;
      bool need;
      if (mA == -INFINITY) {
        // no running max yet (first chunk, no sink; the same for every head): the chunk's
        // largest score of each head first
        float smA = -INFINITY, smB = -INFINITY;
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
          uint32_t x[4], y[4];
          tmem_ld_16x256b(sa + 8 * g, x);
          tmem_ld_16x256b(sb + 8 * g, y);
          tmem_ld_wait();
          const uint32_t mk = col_mask(full, mlo, mhi, g, r4);
          if (mk & 1u) {
            smA = fmaxf(smA, (__uint_as_float(x[0]) + __uint_as_float(y[0])) * scale2);
            smB = fmaxf(smB, (__uint_as_float(x[2]) + __uint_as_float(y[2])) * scale2);
          }
          if (mk & 2u) {
            smA = fmaxf(smA, (__uint_as_float(x[1]) + __uint_as_float(y[1])) * scale2);
            smB = fmaxf(smB, (__uint_as_float(x[3]) + __uint_as_float(y[3])) * scale2);
          }
        }
        smA = fmaxf(smA, __shfl_xor_sync(0xFFFFFFFFu, smA, 1));
        smA = fmaxf(smA, __shfl_xor_sync(0xFFFFFFFFu, smA, 2));
        smB = fmaxf(smB, __shfl_xor_sync(0xFFFFFFFFu, smB, 1));
        smB = fmaxf(smB, __shfl_xor_sync(0xFFFFFFFFu, smB, 2));
        mA = smA;
        mB = smB;
        facA = 0.f;
        facB = 0.f;
        need = true;
        p_pass(sa, sb, full, mlo, mhi, r4, scale2, mA, mB, pA, pB, sw, mxA, mxB, lsA, lsB);
      } else {
        // P with the current running max; redone only if a head's four threads saw a
        // score above it by more than the lazy threshold
        p_pass(sa, sb, full, mlo, mhi, r4, scale2, mA, mB, pA, pB, sw, mxA, mxB, lsA, lsB);
        mxA = fmaxf(mxA, __shfl_xor_sync(0xFFFFFFFFu, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xFFFFFFFFu, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xFFFFFFFFu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xFFFFFFFFu, mxB, 2));
        const bool nA = !(mxA <= kLazy), nB = !(mxB <= kLazy);
        need = nA || nB;
        if (__any_sync(0xFFFFFFFFu, need)) {
          if (nA) { facA = ex2(-mxA); mA += mxA; }
          if (nB) { facB = ex2(-mxB); mB += mxB; }
          p_pass(sa, sb, full, mlo, mhi, r4, scale2, mA, mB, pA, pB, sw, mxA, mxB, lsA, lsB);
        }
      }
      lA = lA * facA + lsA;
      lB = lB * facB + lsB;
      if (r4 == 0) {
        X.fac[bsel][hA] = facA;
        X.fac[bsel][hB] = facB;
      }
      if (group_any(need) && it > 0) {
        // O^T columns are heads: scale column h of every O tile by fac[h] once the PV of
        // the previous chunk is complete.  Warp w covers TMEM lanes 32w.. of all tiles.
        if (!X.abort &&
            !mbar_wait(smem_u32(&X.pv_done[(it - 1) & 1]), (uint32_t)((it - 1) >> 1) & 1))
          X.abort = 1;
        tc_fence_after();
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
          for (int hb = 0; hb < 64; hb += 32) {
            uint32_t v[32];
            const uint32_t ta = tmem + lrow + kColO + 64 * mt + hb;
            tmem_ld32(ta, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = __float_as_uint(__uint_as_float(v[j]) * X.fac[bsel][hb + j]);
            tmem_st32(ta, v);
          }
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&X.p_full[bsel]));
    }
    // running sums of the four threads of each head
    lA += __shfl_xor_sync(0xFFFFFFFFu, lA, 1);
    lA += __shfl_xor_sync(0xFFFFFFFFu, lA, 2);
    lB += __shfl_xor_sync(0xFFFFFFFFu, lB, 1);
    lB += __shfl_xor_sync(0xFFFFFFFFu, lB, 2);
    if (r4 == 0) {
      X.m_run[hA] = mA;
      X.l_run[hA] = lA;
      X.m_run[hB] = mB;
      X.l_run[hB] = lB;
    }
    if (n > 0 && !X.abort)
      mbar_wait(smem_u32(&X.pv_done[(n - 1) & 1]), (uint32_t)((n - 1) >> 1) & 1);
    tc_fence_after();
  }

  // ---- epilogue (warp w reads TMEM lanes 32 (w % 4) .. = dims mt*128 + 32 (w % 4) ..) ----
  if (tid == 0 && n == 0) mbar_wait(smem_u32(&X.q_full), 0, 100000000ull);  // Q copy landed
  __syncthreads();
  tc_fence_after();  // every MMA is complete (the softmax warps waited for the last PV)
  if (nsplit == 1) {
    // O^T / l -> bf16 out[q][64 heads][512]: O^T staged in the KV buffers (all 512 dims;
    // warp w < 16 stages tile w / 4 from its lane quarter w % 4), then every thread writes
    if (tid < 64) X.fac[0][tid] = 1.f / X.l_run[tid];
    if (a.inv_freq && warp == 4) rope_table(a.inv_freq, p, lane, X.rope_c, X.rope_s);
    if (warp < 16)
      stage_ot(tmem + kColO, warp & 3, lane, warp >> 2, 1,
               smem_u32(kv_s) + (uint32_t)(warp >> 2) * 128u * 256u, n > 0);
    __syncthreads();
    out_pass(reinterpret_cast<const float*>(kv_s), nullptr, X.fac[0], nullptr,
             a.inv_freq ? X.rope_c : nullptr, X.rope_s, a.out + (int64_t)q * kHeads * kDLat,
             kDLat, 0, tid, kThreads);
    if (a.lse && tid < 64)
      a.lse[(int64_t)q * kHeads + tid] =
          (X.m_run[tid] + __log2f(X.l_run[tid])) * 0.6931471805599453f;
  } else {
    // Two CTAs per query as a cluster: CTA r finishes dims 256 r .. 256 r + 255 (the O^T
    // tiles 2 r and 2 r + 1).  Warps 0..7 stage the two tiles the peer finishes from TMEM
    // (warp w: TMEM lanes 32 (w % 4) .., tile w / 4) in the second KV buffer, and the
    // lanes of warp 16 store (m_run, l_run) into the peer's peer_m, peer_l.  After a
    // cluster barrier (both CTAs past their main loops, so the peer's Q buffer is free)
    // one bulk copy per tile ships the staged rows into the peer's Q buffer, each counted
    // by its own merge barrier, and warps 8 and 9 form the merge weights of the 64 heads,
    //   M = max(m_own, m_peer, sink),  Z = 2^(sink - M) + sum 2^(m - M) l,
    //   o = (2^(m_own - M) O_own + 2^(m_peer - M) O_peer) / Z.
    // Warps 8..11 and 16..19 merge their own first tile as soon as its peer rows land
    // (while the second tile's copy is in flight), warps 12..15 and 20..23 the second:
    // every thread takes one dim and 32 heads, one shuffle per pair of heads giving each
    // lane a bf16 pair of neighbouring dims, which go to a 128-byte-swizzled staging box
    // in shared memory; each tile leaves by two tensor stores.  A staged fp32 row holds
    // one dim's 64 heads as 16 pieces of four, piece c at c ^ (d % 8), which keeps the
    // 16-byte stores and loads free of bank conflicts.
    const uint32_t peer = (uint32_t)rank ^ 1u;
    constexpr uint32_t kTileBytes = 128 * 256;  // one staged tile: 128 dims x 64 heads fp32
    if (tid == 0) {
      mbar_arrive_expect_tx(smem_u32(&X.merge_full[0]), kTileBytes);
      mbar_arrive_expect_tx(smem_u32(&X.merge_full[1]), kTileBytes);
    }
    const int sp = warp & 3, tl = (warp >> 2) & 1;
    const int d = sp * 32 + lane;  // dim within the tile = TMEM lane
    const uint32_t rowb = (uint32_t)(tl * 128 + d) * 256;  // this dim's staged row
    if (warp < 8) {
      const uint32_t trow =
          tmem + ((uint32_t)(sp * 32) << 16) + kColO + 64 * (2 * (int)peer + tl);
      const uint32_t stage = smem_u32(kv_s + kBufBytes) + rowb;
#pragma unroll 1
      for (int hb = 0; hb < 64; hb += 32) {
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(trow + hb, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const int c = (hb >> 2) + c4;
          st_shared16(stage + ((c ^ (d & 7)) << 4),
                      make_uint4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]));
        }
      }
      fence_proxy_async_smem();  // the staged rows are read by the bulk copies
    } else if (warp == 16) {  // m_run[64], l_run[64]: 512 adjacent bytes -> peer_m, peer_l
      const uint4 ml = reinterpret_cast<const uint4*>(&X.m_run[0])[lane];
      st_cluster16(dsmem_addr(smem_u32(&X.peer_m[0]) + 16 * lane, peer), ml);
    } else if (a.inv_freq && warp == 17) {
      rope_table(a.inv_freq, p, lane, X.rope_c, X.rope_s);
    }
    cluster_sync();  // both main loops are done; the staged rows and (m, l) are visible
    tc_fence_after();
    if (tid == 0) {
#pragma unroll 1
      for (int t = 0; t < 2; ++t)
        bulk_copy_to_cluster(dsmem_addr(smem_u32(q_s) + t * kTileBytes, peer),
                             smem_u32(kv_s + kBufBytes) + t * kTileBytes, kTileBytes,
                             dsmem_addr(smem_u32(&X.merge_full[t]), peer));
    }
    if (warp >= 8) {
      // merge warps: warp 8 + 4 t + i (t = tile) and 16 + 4 t + i take TMEM lanes 32 i..
      // of their own tile t, for heads 0..31 and 32..63 respectively
      if (warp < 10) {  // merge weights of head tid - 256
        const int h = tid - 256;
        const float mo = X.m_run[h], mp = X.peer_m[h], sk = X.sink2[h];
        const float M = fmaxf(fmaxf(mo, mp), sk);
        const float wo = mo == -INFINITY ? 0.f : ex2(mo - M);
        const float wp = mp == -INFINITY ? 0.f : ex2(mp - M);
        const float Z =
            wo * X.l_run[h] + wp * X.peer_l[h] + (sk == -INFINITY ? 0.f : ex2(sk - M));
        const float inv = Z > 0.f ? 1.f / Z : 0.f;
        X.fac[0][h] = wo * inv;
        X.fac[1][h] = wp * inv;
        if (a.lse && rank == 0)
          a.lse[(int64_t)q * kHeads + h] = (M + __log2f(Z)) * 0.6931471805599453f;
      }
      asm volatile("bar.sync 5, 512;" ::: "memory");  // warps 8..23: the weights are written
      const uint32_t trow =
          tmem + ((uint32_t)(sp * 32) << 16) + kColO + 64 * (2 * rank + tl);
      const int gd = 256 * rank + 128 * tl + d;  // output dim; a warp's 32 dims share `rot`
      const bool rot = a.inv_freq && gd >= kRopeDim0;
      const float cs = rot ? X.rope_c[(gd - kRopeDim0) >> 1] : 1.f;
      const float sn = rot ? X.rope_s[(gd - kRopeDim0) >> 1] : 0.f;
      const float* pin = reinterpret_cast<const float*>(q_s + rowb);
      // bf16 output of this tile staged in the first KV buffer as two 128-byte-swizzled
      // boxes of 64 heads x 64 dims (box sp / 2 holds this warp's dims), written out by
      // two tensor stores
      const int dd = (sp * 32 + lane) & 63;  // dim within the box
      const uint32_t obox = smem_u32(kv_s) + (uint32_t)tl * 16384u + (uint32_t)(sp >> 1) * 8192u;
      if (!mbar_wait(smem_u32(&X.merge_full[tl]), 0)) X.abort = 1;
      {
        const int hb = warp >= 16 ? 32 : 0;
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(trow + hb, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
        // merged values replace the own ones in v (as float bits)
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const int c = (hb >> 2) + c4;
          const float4 y = *reinterpret_cast<const float4*>(pin + ((c ^ (d & 7)) << 2));
          const float4 f0 = *reinterpret_cast<const float4*>(&X.fac[0][4 * c]);
          const float4 f1 = *reinterpret_cast<const float4*>(&X.fac[1][4 * c]);
          v[4 * c4 + 0] = __float_as_uint(__uint_as_float(v[4 * c4 + 0]) * f0.x + y.x * f1.x);
          v[4 * c4 + 1] = __float_as_uint(__uint_as_float(v[4 * c4 + 1]) * f0.y + y.y * f1.y);
          v[4 * c4 + 2] = __float_as_uint(__uint_as_float(v[4 * c4 + 2]) * f0.z + y.z * f1.z);
          v[4 * c4 + 3] = __float_as_uint(__uint_as_float(v[4 * c4 + 3]) * f0.w + y.w * f1.w);
        }
        if (rot) {  // pair (2i, 2i + 1) times e^{-i p theta_i}: the partner is lane ^ 1
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = __uint_as_float(v[j]);
            const float pt = __shfl_xor_sync(0xFFFFFFFFu, x, 1);
            v[j] = __float_as_uint((lane & 1) ? x * cs - pt * sn : x * cs + pt * sn);
          }
        }
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int h = hb + j;
          const float a0 = __uint_as_float(v[j]), a1 = __uint_as_float(v[j + 1]);
          const float rcv = __shfl_xor_sync(0xFFFFFFFFu, (lane & 1) ? a0 : a1, 1);
          // the even lane writes head h at dims (d, d + 1), the odd one head h + 1 at
          // (d - 1, d): row hr, 4 bytes at the pair's even dim de
          const int hr = (lane & 1) ? h + 1 : h;
          const int de = dd & ~1;
          const uint32_t w = (lane & 1) ? pack_bf16x2(rcv, a1) : pack_bf16x2(a0, rcv);
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(obox + (uint32_t)hr * 128u +
                                                          ((uint32_t)((de >> 3) ^ (hr & 7)) << 4) +
                                                          (uint32_t)(de & 7) * 2u),
                       "r"(w)
                       : "memory");
        }
      }
      fence_proxy_async_smem();  // the staged boxes are read by the tensor stores
      if (tl == 0) asm volatile("bar.sync 6, 256;" ::: "memory");  // warps 8..11, 16..19
      else asm volatile("bar.sync 7, 256;" ::: "memory");          // warps 12..15, 20..23
      if (warp < 16 && sp == 0 && lane == 0) {
        const uint32_t tb = smem_u32(kv_s) + (uint32_t)tl * 16384u;
        const int x0 = 256 * rank + 128 * tl;
        tma_store_2d(&omap, x0, q * kHeads, tb);
        tma_store_2d(&omap, x0 + 64, q * kHeads, tb + 8192u);
        bulk_commit_group();
        bulk_wait_group_read0();  // the CTA may exit once the boxes have been read
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// ---- one CTA per SM carrying on from query to query (nsplit = 1, more queries than SMs) --
// CTA i takes queries i, i + G, i + 2G, .. (G = gridDim.x) with the same roles and
// per-chunk pipeline as above, but the barriers' phases run on a chunk count that goes on
// across queries, so the two KV buffers keep cycling: a gather team resolves its next
// query's row sources (into the other half of the row tables, by query parity) and starts
// that query's gathers as soon as its buffer's last PV is done, while the softmax warps
// finish the query.  Once the query's last S has completed the next query's Q is loaded
// into the Q buffer, so the next query's S products run while the softmax warps write this
// query's output themselves: O^T / l from TMEM, bf16 pairs of neighbouring dims after one
// shuffle per pair of heads, stored straight to global memory (64 contiguous bytes of two
// heads per warp store).

struct __align__(16) PAux {
  float inv_l[64];   // 1 / running sum per head of the query being written
  float fac[2][64];  // rescale factor per head, by chunk parity
  float rope_c[32];  // inverse RoPE of the output at the query position
  float rope_s[32];
  int32_t rowidx[2][kMaxChunks][kChunk];  // source rows, by query parity
  uint32_t rowmask[2][kMaxChunks][2];     // valid rows of each chunk, by query parity
  uint64_t q_full;      // Q of the CTA's current query landed (one load per query)
  uint64_t kv_full[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t fin[4];
  uint32_t tmem_slot;
  int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_persist_kernel(AttnArgs a, const __grid_constant__ CUtensorMap qmap,
                               const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + kQBytes;
  uint8_t* p_s = kv_s + 2 * kBufBytes;
  PAux& X = *reinterpret_cast<PAux*>(p_s + 2 * kPBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, q0 = blockIdx.x;
  const int nq = q0 < a.Q ? (a.Q - q0 + G - 1) / G : 0;  // queries of this CTA
  const int n = 2 + (a.nsel + kChunk - 1) / kChunk;      // chunks per query
  const uint32_t qb = smem_u32(q_s), kv0 = smem_u32(kv_s), p0 = smem_u32(p_s);
  griddep_launch_dependents();
  if (tid == 0) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&wmap);
    mbar_init(smem_u32(&X.q_full), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&X.kv_full[b]), 1);
      mbar_init(smem_u32(&X.s_full[b]), 2);
      mbar_init(smem_u32(&X.p_full[b]), kGroupThreads);
      mbar_init(smem_u32(&X.pv_done[b]), 2);
    }
    for (int r = 0; r < 4; ++r) mbar_init(smem_u32(&X.fin[r]), 1);
    X.abort = 0;
    mbar_fence_init();
    if (nq > 0) {  // the first query's Q (a call input: before the dependency wait)
      const uint32_t qf = smem_u32(&X.q_full);
      mbar_arrive_expect_tx(qf, kQBytes);
      const uint64_t pol = policy_evict_first();
#pragma unroll
      for (int db = 0; db < 8; ++db)
        tma_load_2d(qb + db * kDimBlock, &qmap, 64 * db, q0 * kHeads, qf, pol);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&X.tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = X.tmem_slot;
  const float scale2 = a.scale * kLog2e;
  const bool is_gather = warp >= kGatherWarp0 && warp < kMmaWarp;

  if (is_gather) {
    // ======== gather: team b owns KV buffer b and the chunks cg with cg % 2 == b ========
    const int team = (warp - kGatherWarp0) / (kTeam / 32);
    const int t = tid - kGatherWarp0 * 32 - kTeam * team;
    const uint32_t full_bar = smem_u32(&X.kv_full[team]);
    const uint32_t kvb = kv0 + team * kBufBytes;
    auto team_sync = [&]() {
      if (team == 0) asm volatile("bar.sync 2, 256;" ::: "memory");
      else asm volatile("bar.sync 3, 256;" ::: "memory");
    };
    griddep_wait();  // the selection and the plane come from the preceding kernels
    int last = -1;   // the team's last chunk (its kv_full phase ends every copy)
    for (int j = 0; j < nq; ++j) {
      const int q = q0 + j * G, par = j & 1, cg0 = j * n;
      const int c_first = (team - cg0) & 1;  // the team's chunks of this query: c_first + 2 k
      const int mine = c_first < n ? (n - c_first + 1) / 2 : 0;
      const int b = a.q_seq[q];
      const int64_t p = a.q_pos[q];
      const int64_t rb = a.row_base ? a.row_base[b] : 0;
      // row sources of the team's chunks, one entry per thread and step (whole warps)
      for (int e = t; e < mine * kChunk; e += kTeam) {
        const int c = c_first + 2 * (e >> 6), r = e & 63;
        const int32_t idx32 = chunk_row(a, q, b, p, rb, c, r);
        X.rowidx[par][c][r] = idx32;
        const uint32_t vm = __ballot_sync(0xFFFFFFFFu, idx32 >= 0);
        if (lane == 0) X.rowmask[par][c][r >> 5] = vm;
      }
      team_sync();
      for (int k = 0; k < mine; ++k) {
        const int c = c_first + 2 * k, cg = cg0 + c;
        last = cg;
        // the buffer's previous chunk (cg - 2) has been multiplied into O^T
        if (cg >= 2 && !X.abort &&
            !mbar_wait(smem_u32(&X.pv_done[team]), (uint32_t)((cg - 2) >> 1) & 1))
          X.abort = 1;
        const int32_t* rows = X.rowidx[par][c];
        // a full window chunk of a LINEAR bf16 window: 64 consecutive rows, one TMA box of
        // 64 x 64 per dim block (arriving on the barrier by itself)
        if (c < 2 && a.swa_mode == 1 && a.swa_dtype == 0 &&
            (X.rowmask[par][c][0] & X.rowmask[par][c][1]) == 0xFFFFFFFFu) {
          if (t == 0) {
            mbar_arrive_expect_tx(full_bar, kBufBytes);
            const uint64_t pol = policy_evict_first();
#pragma unroll
            for (int db = 0; db < 8; ++db)
              tma_load_2d(kvb + db * kDimBlock, &wmap, 64 * db, rows[0], full_bar, pol);
          }
          continue;
        }
        const int fp8 = c < 2 ? a.swa_dtype : 0;
        const uint8_t* base = c < 2 ? a.swa : reinterpret_cast<const uint8_t*>(a.plane);
        gather_chunk(rows, fp8, c >= 2 && a.plane_dtype == 1, base, kvb, t, a.stream_rows != 0);
        cp_async_commit();
        cp_async_wait_group<0>();
        fence_proxy_async_smem();
        team_sync();  // every thread of the team has landed its rows
        if (t == 0) mbar_arrive(full_bar);
      }
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (t == 0 && last >= 0) mbar_wait(full_bar, (uint32_t)(last >> 1) & 1, 100000000ull);
  } else if (warp >= kMmaWarp) {
    // ====== MMA issuers (lane 0), as above: warps 20 and 21 S, warps 22 and 23 PV ======
    const int role = warp - kMmaWarp;
    if (lane == 0) {
      int issued = 0;
      if (role < 2) {
        const uint32_t id_s = idesc_bf16(64, 64, 0, 0);
        for (int j = 0; j < nq && !X.abort; ++j) {
          if (!mbar_wait(smem_u32(&X.q_full), (uint32_t)j & 1)) {
            X.abort = 1;
            break;
          }
          for (int c = 0; c < n; ++c) {
            const int cg = j * n + c;
            // kv_full of chunk cg also means that the softmax of chunk cg - 2 is done with
            // S buffer cg & 1
            if (!mbar_wait(smem_u32(&X.kv_full[cg & 1]), (uint32_t)(cg >> 1) & 1)) {
              X.abort = 1;
              break;
            }
            tc_fence_after();
            const uint32_t kvb = kv0 + (cg & 1) * kBufBytes;
            const uint32_t d = tmem + (role ? kColSb : kColSa) + 64 * (cg & 1);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int db = 4 * role + i;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16(d, sdesc_sw128(qb + db * kDimBlock + kk * 32, 16, 1024),
                          sdesc_sw128(kvb + db * kDimBlock + kk * 32, 16, 1024), id_s,
                          (i | kk) != 0);
            }
            umma_commit(smem_u32(&X.s_full[cg & 1]));
            ++issued;
          }
        }
      } else {
        const uint32_t id_o = idesc_bf16(128, 64, 1, 0);
        for (int cg = 0; cg < nq * n && !X.abort; ++cg) {
          const int c = cg % n;  // a query's first chunk starts O^T afresh
          if (!mbar_wait(smem_u32(&X.p_full[cg & 1]), (uint32_t)(cg >> 1) & 1)) {
            X.abort = 1;
            break;
          }
          tc_fence_after();
          const uint32_t kvb = kv0 + (cg & 1) * kBufBytes;
          const uint32_t pb = p0 + (cg & 1) * kPBytes;
#pragma unroll
          for (int mt = 2 * (role - 2); mt < 2 * (role - 2) + 2; ++mt)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + kColO + 64 * mt,
                        sdesc_sw128(kvb + 2 * mt * kDimBlock + kk * 2048, kDimBlock, 1024),
                        sdesc_sw128(pb + kk * 32, 16, 1024), id_o, (c > 0 || kk > 0) ? 1 : 0);
          umma_commit(smem_u32(&X.pv_done[cg & 1]));
          ++issued;
        }
      }
      // no MMA may still be running when the TMEM is released, whatever happened above
      if (issued > 0) {
        umma_commit(smem_u32(&X.fin[role]));
        mbar_wait(smem_u32(&X.fin[role]), 0, 100000000ull);
      }
    }
  } else {
    // ============ softmax + O^T rescale + output (warps 0..3) ============
    const int r4 = lane & 3;
    const int hA = 16 * warp + (lane >> 2), hB = hA + 8;
    const uint32_t lrow = (uint32_t)(warp * 32) << 16;
    const float skA = a.sink ? a.sink[hA] * kLog2e : -INFINITY;
    const float skB = a.sink ? a.sink[hB] * kLog2e : -INFINITY;
    auto group_sync = [] { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    for (int j = 0; j < nq; ++j) {
      const int q = q0 + j * G, par = j & 1;
      // the running max starts at the sink logit and the sum at the sink's mass
      float mA = skA, mB = skB, lA = 0.f, lB = 0.f;
      if (a.sink && r4 == 0) { lA = 1.f; lB = 1.f; }
      for (int c = 0; c < n; ++c) {
        const int cg = j * n + c;
        const int bsel = cg & 1;
        const uint32_t ph = (uint32_t)(cg >> 1) & 1;
        const uint32_t sa = tmem + lrow + kColSa + 64 * bsel;
        const uint32_t sb = tmem + lrow + kColSb + 64 * bsel;
        if (!X.abort && !mbar_wait(smem_u32(&X.s_full[bsel]), ph)) X.abort = 1;
        tc_fence_after();
        if (c == n - 1 && tid == 0 && j + 1 < nq && !X.abort) {
          // every S of this query has completed: the Q buffer takes the next query's Q
          const uint32_t qf = smem_u32(&X.q_full);
          mbar_arrive_expect_tx(qf, kQBytes);
          const uint64_t pol = policy_evict_first();
#pragma unroll
          for (int db = 0; db < 8; ++db)
            tma_load_2d(qb + db * kDimBlock, &qmap, 64 * db, (q + G) * kHeads, qf, pol);
        }
        __syncwarp();  // warp-wide TMEM loads follow
        const uint32_t mlo = X.rowmask[par][c][0], mhi = X.rowmask[par][c][1];
        const bool full = (mlo & mhi) == 0xFFFFFFFFu;
        // the P buffer was last read by the PV of chunk cg - 2
        if (cg >= 2 && !X.abort &&
            !mbar_wait(smem_u32(&X.pv_done[bsel]), (uint32_t)((cg - 2) >> 1) & 1))
          X.abort = 1;
        const uint32_t pA = p0 + bsel * kPBytes + hA * 128 + 4 * r4;
        const uint32_t pB = p0 + bsel * kPBytes + hB * 128 + 4 * r4;
        const int sw = hA & 7;
        float mxA, mxB, lsA, lsB, facA = 1.f, facB = 1.f;
        bool need;
        if (mA == -INFINITY) {
          // no running max yet (first chunk, no sink): the chunk's largest score first
          float smA = -INFINITY, smB = -INFINITY;
#pragma unroll 1
          for (int g = 0; g < 8; ++g) {
            uint32_t x[4], y[4];
            tmem_ld_16x256b(sa + 8 * g, x);
            tmem_ld_16x256b(sb + 8 * g, y);
            tmem_ld_wait();
            const uint32_t mk = col_mask(full, mlo, mhi, g, r4);
            if (mk & 1u) {
              smA = fmaxf(smA, (__uint_as_float(x[0]) + __uint_as_float(y[0])) * scale2);
              smB = fmaxf(smB, (__uint_as_float(x[2]) + __uint_as_float(y[2])) * scale2);
            }
            if (mk & 2u) {
              smA = fmaxf(smA, (__uint_as_float(x[1]) + __uint_as_float(y[1])) * scale2);
              smB = fmaxf(smB, (__uint_as_float(x[3]) + __uint_as_float(y[3])) * scale2);
            }
          }
          smA = fmaxf(smA, __shfl_xor_sync(0xFFFFFFFFu, smA, 1));
          smA = fmaxf(smA, __shfl_xor_sync(0xFFFFFFFFu, smA, 2));
          smB = fmaxf(smB, __shfl_xor_sync(0xFFFFFFFFu, smB, 1));
          smB = fmaxf(smB, __shfl_xor_sync(0xFFFFFFFFu, smB, 2));
          mA = smA;
          mB = smB;
          facA = 0.f;
          facB = 0.f;
          need = true;
          p_pass(sa, sb, full, mlo, mhi, r4, scale2, mA, mB, pA, pB, sw, mxA, mxB, lsA, lsB);
        } else {
          p_pass(sa, sb, full, mlo, mhi, r4, scale2, mA, mB, pA, pB, sw, mxA, mxB, lsA, lsB);
          mxA = fmaxf(mxA, __shfl_xor_sync(0xFFFFFFFFu, mxA, 1));
          mxA = fmaxf(mxA, __shfl_xor_sync(0xFFFFFFFFu, mxA, 2));
          mxB = fmaxf(mxB, __shfl_xor_sync(0xFFFFFFFFu, mxB, 1));
          mxB = fmaxf(mxB, __shfl_xor_sync(0xFFFFFFFFu, mxB, 2));
          const bool nA = !(mxA <= kLazy), nB = !(mxB <= kLazy);
          need = nA || nB;
          if (__any_sync(0xFFFFFFFFu, need)) {
            if (nA) { facA = ex2(-mxA); mA += mxA; }
            if (nB) { facB = ex2(-mxB); mB += mxB; }
            p_pass(sa, sb, full, mlo, mhi, r4, scale2, mA, mB, pA, pB, sw, mxA, mxB, lsA, lsB);
          }
        }
        lA = lA * facA + lsA;
        lB = lB * facB + lsB;
        if (r4 == 0) {
          X.fac[bsel][hA] = facA;
          X.fac[bsel][hB] = facB;
        }
        if (group_any(need) && c > 0) {
          // scale column h of every O tile by fac[h] once the previous chunk's PV is done
          if (!X.abort && !mbar_wait(smem_u32(&X.pv_done[(cg - 1) & 1]),
                                     (uint32_t)((cg - 1) >> 1) & 1))
            X.abort = 1;
          tc_fence_after();
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
            for (int hb = 0; hb < 64; hb += 32) {
              uint32_t v[32];
              const uint32_t ta = tmem + lrow + kColO + 64 * mt + hb;
              tmem_ld32(ta, v);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                v[jj] = __float_as_uint(__uint_as_float(v[jj]) * X.fac[bsel][hb + jj]);
              tmem_st32(ta, v);
            }
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&X.p_full[bsel]));
      }
      // ---- the query's output: O^T / l, after its last PV ----
      lA += __shfl_xor_sync(0xFFFFFFFFu, lA, 1);
      lA += __shfl_xor_sync(0xFFFFFFFFu, lA, 2);
      lB += __shfl_xor_sync(0xFFFFFFFFu, lB, 1);
      lB += __shfl_xor_sync(0xFFFFFFFFu, lB, 2);
      const int cl = j * n + n - 1;
      if (!X.abort && !mbar_wait(smem_u32(&X.pv_done[cl & 1]), (uint32_t)(cl >> 1) & 1))
        X.abort = 1;
      tc_fence_after();
      if (r4 == 0) {
        X.inv_l[hA] = 1.f / lA;
        X.inv_l[hB] = 1.f / lB;
        if (a.lse) {
          a.lse[(int64_t)q * kHeads + hA] = (mA + __log2f(lA)) * 0.6931471805599453f;
          a.lse[(int64_t)q * kHeads + hB] = (mB + __log2f(lB)) * 0.6931471805599453f;
        }
      }
      if (a.inv_freq && warp == 0) rope_table(a.inv_freq, a.q_pos[q], lane, X.rope_c, X.rope_s);
      group_sync();  // inv_l and the RoPE table are written
      // warp w holds dims mt * 128 + 32 w + lane of tile mt (TMEM lanes 32 w ..); bf16
      // pairs of neighbouring dims after one shuffle per pair of heads, streamed out
      uint16_t* out_q = a.out + (int64_t)q * kHeads * kDLat;
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        const int d = mt * 128 + warp * 32 + lane;
        const bool rot = a.inv_freq && d >= kRopeDim0;  // uniform in a warp
        const float cs = rot ? X.rope_c[(d - kRopeDim0) >> 1] : 1.f;
        const float sn = rot ? X.rope_s[(d - kRopeDim0) >> 1] : 0.f;
        const int de = d & ~1;  // the pair's even dim
#pragma unroll 1
        for (int hb = 0; hb < 64; hb += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lrow + kColO + 64 * mt + hb, v);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            v[jj] = __float_as_uint(__uint_as_float(v[jj]) * X.inv_l[hb + jj]);
          if (rot) {  // pair (2i, 2i + 1) times e^{-i p theta_i}: the partner is lane ^ 1
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const float x = __uint_as_float(v[jj]);
              const float pt = __shfl_xor_sync(0xFFFFFFFFu, x, 1);
              v[jj] = __float_as_uint((lane & 1) ? x * cs - pt * sn : x * cs + pt * sn);
            }
          }
#pragma unroll
          for (int jj = 0; jj < 32; jj += 2) {
            const int h = hb + jj;
            const float a0 = __uint_as_float(v[jj]), a1 = __uint_as_float(v[jj + 1]);
            const float rcv = __shfl_xor_sync(0xFFFFFFFFu, (lane & 1) ? a0 : a1, 1);
            // the even lane writes head h at dims (d, d + 1), the odd one head h + 1 at
            // (d - 1, d)
            const int hr = (lane & 1) ? h + 1 : h;
            const uint32_t w = (lane & 1) ? pack_bf16x2(rcv, a1) : pack_bf16x2(a0, rcv);
            __stcs(reinterpret_cast<unsigned int*>(out_q + hr * kDLat + de), w);
          }
        }
      }
      tc_fence_before();  // the TMEM reads precede the next query's first PV
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t attn_smem_bytes() {
  return 1024 + kQBytes + 2 * kBufBytes + 2 * kPBytes + sizeof(Aux);
}
size_t attn_persist_smem_bytes() {
  return 1024 + kQBytes + 2 * kBufBytes + 2 * kPBytes + sizeof(PAux);
}

// CTAs per query: two (a cluster that merges in distributed shared memory) when both fit
// in one wave of one CTA per SM, else one.  More CTAs per query, each writing a partial
// that a second kernel merged, measured slower at every batch tried (4, 8 and 32 queries:
// 4, 8 and 6 us per step), the extra launch and the partials' round trip through
// memory costing more than the shorter chains of chunks save.
int attn_num_splits(int Q, int nsel, int num_sms) {
  (void)nsel;
  return Q > 0 && 2 * Q <= num_sms ? 2 : 1;
}

cudaError_t launch_attn(const AttnArgs& a, int nsplit, cudaStream_t s) {
  if (a.Q == 0) return cudaSuccess;
  // Q of each query as eight boxes of 64 heads x 64 dims; a LINEAR bf16 window as boxes of
  // 64 rows x 64 dims (the Q map stands in when there is none); the output likewise (the
  // cluster merge writes it by tensor stores)
  CUtensorMap qm, wm, om;
  if (!encode_rows_bf16(&qm, a.q, (uint64_t)a.Q * kHeads, kDLat, 64, 64) ||
      !encode_rows_bf16(&om, a.out, (uint64_t)a.Q * kHeads, kDLat, 64, 64))
    return cudaErrorInvalidValue;
  wm = qm;
  if (a.swa_mode == 1 && a.swa_dtype == 0 && a.swa_rows > 0 &&
      !encode_rows_bf16(&wm, a.swa, (uint64_t)a.swa_rows, kDLat, 64, 64))
    return cudaErrorInvalidValue;
  if (a.persist > 0) {  // one CTA per SM, each carrying on from query to query
    const size_t psmem = attn_persist_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_persist_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(sparse_attn_persist_kernel, dim3((unsigned)a.persist), dim3(kThreads), psmem,
                      s, a, qm, wm);
  }
  const size_t smem = attn_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (nsplit == 2) {  // the two CTAs of a query merge through distributed shared memory
    AttnArgs b = a;
    b.cluster = 1;
    return launch_pdl_cluster(sparse_attn_kernel, dim3(2u, (unsigned)a.Q), dim3(kThreads), smem, s,
                              2u, b, qm, wm, om);
  }
  return launch_pdl(sparse_attn_kernel, dim3(1u, (unsigned)a.Q), dim3(kThreads), smem, s, a, qm,
                    wm, om);
}

}  // namespace csa2

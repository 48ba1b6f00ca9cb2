// k_attn.cu -- CSA2 sparse MQA attention (64 heads x 512 dims, K = V) over the
// layer's sliding window plus the selected compressed rows, one softmax with a
// per-head sink logit in the denominator.
// [A] "四种层合并出来的是什么形状" (one CSR, one softmax, K = V, <= 640 rows, sink only in
// the denominator); [B] §4.1 (two sources, no de-duplication), §4.4 step 4 (window
// slots); [C] §5.5-5.6 (logical concatenation, no physical copy), A.19.3 (gather by
// int32 index, online softmax with running max and sum, fused sink);
// [E] Fig. 2d (out_h = sum e^{s_j} v_j / (e^{sink_h} + sum e^{s_j})).
//
// A query's entries form up to five tiles of 128 rows: tile 0 is the window
// (positions p-127..p), tiles 1..4 hold sel[0..511].  The tiles of one query are
// spread over nsplit CTAs (grid = nsplit x Q); each CTA keeps an online softmax over
// its tiles:
//   gather   rows (bf16, or FP8 dequantised to bf16) into a 128-byte-swizzled shared
//            tile [8 dim blocks][128 rows][128 B], in four groups of two dim blocks,
//            each signalled on its own mbarrier so the MMAs start on early groups
//   S^T      = KV[128 x 512] . Q^T[512 x 64]  -> TMEM (row = lane, head = column)
//   softmax  per head over the rows (warp butterfly + 4-warp combine); the running
//            max moves only when it grows by more than 8 (log2 units)
//   O^T     += V^T[512 x 128] . P^T[128 x 64] -> TMEM, four M = 128 tiles; the same
//            shared tile is the A operand again, read MN-major
// With nsplit = 1 the CTA starts from the sink (running max = sink, running sum = 1)
// and writes the output.  Otherwise every CTA writes its partial (max, sum, O) to the
// workspace and attn_combine_kernel merges them, adding the sink's e^{sink_h} once.
//
// Warps 0..7 gather and write the output, warps 0..3 also run the softmax, warp 8
// owns the TMEM allocation and its lane 0 issues every tcgen05.mma.
#include <cuda_fp8.h>

#include "common.cuh"

CSA2_DEFINE_FAULT_FLAG(attn)

namespace csa2 {
namespace {

constexpr int kThreads = 288;
constexpr int kWorkers = 256;             // warps 0..7
constexpr int kMaxTiles = 5;
constexpr int kQBytes = 8 * 64 * 128;     // 64 KiB
constexpr int kKVBytes = 8 * 128 * 128;   // 128 KiB (also the fp32 [64][512] partial O)
constexpr int kPBytes = 128 * 128;        // 16 KiB
constexpr uint32_t kColS = 0;             // TMEM columns of S^T (64)
constexpr uint32_t kColO = 64;            // O^T tiles at 64 + 64 * mt
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;

struct __align__(16) Aux {
  float red[4][64];
  float m_run[64];
  float l_run[64];
  float fac[64];
  int64_t rowsrc[kMaxTiles][128];  // per slot of this CTA (tile t = rank + slot * nsplit)
  int cnt[kMaxTiles];               // valid rows per slot
  int tiles[kMaxTiles];             // non-empty slots, in order
  uint64_t bar_g[4];   // gather group done (256 arrivals)
  uint64_t bar_s;      // S^T complete (commit)
  uint64_t bar_p;      // P^T written (128 arrivals)
  uint64_t bar_pv[4];  // PV M-tile complete (commit)
  uint32_t tmem_slot;
  int rescale;
  int ntile;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Butterfly reduce-scatter of 64 per-lane values across the warp: afterwards lane l
// holds the reduction over the 32 lanes of heads 2l and 2l+1 in v[0], v[1].
template <bool kMax>
__device__ __forceinline__ void warp_reduce_heads(float (&v)[64], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = 32 >> step;
    const int bit = 16 >> step;
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, bit);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

__device__ __forceinline__ void st_shared16(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Gather group g (dim blocks 2g, 2g+1) of the current tile.
__device__ __forceinline__ void gather_group(const AttnArgs& a, const Aux& X, int slot, int g,
                                             bool fp8, const uint8_t* base, uint32_t kvb,
                                             int tid) {
  const int64_t* src_of = X.rowsrc[slot];
  if (fp8) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int flat = i * kWorkers + tid;
      const int r = flat >> 3, c16 = 8 * g + (flat & 7);
      const int64_t off = src_of[r];
      const uint32_t d0 = kvb + (c16 >> 2) * 16384 + sw128_off(r, (2 * c16) & 7);
      const uint32_t d1 = kvb + (c16 >> 2) * 16384 + sw128_off(r, (2 * c16 + 1) & 7);
      if (off < 0) { st_shared_zero16(d0); st_shared_zero16(d1); continue; }
      const uint8_t* src = base + off;
      const uint4 codes = *reinterpret_cast<const uint4*>(src + c16 * 16);
      const float sc = *reinterpret_cast<const float*>(src + 512 + 4 * (c16 >> 3));
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
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int flat = i * kWorkers + tid;
      const int r = flat >> 4, c = 16 * g + (flat & 15);
      const int64_t off = src_of[r];
      const uint32_t dst = kvb + (c >> 3) * 16384 + sw128_off(r, c & 7);
      if (off < 0) st_shared_zero16(dst);
      else cp_async16(dst, base + off + c * 16);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + kQBytes;
  uint8_t* p_s = kv_s + kKVBytes;
  Aux& X = *reinterpret_cast<Aux*>(p_s + kPBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = blockIdx.y;
  const int rank = blockIdx.x;
  const int nsplit = gridDim.x;
  griddep_launch_dependents();
  if (tid == 0) {
    for (int g = 0; g < 4; ++g) {
      mbar_init(smem_u32(&X.bar_g[g]), kWorkers);
      mbar_init(smem_u32(&X.bar_pv[g]), 1);
    }
    mbar_init(smem_u32(&X.bar_s), 1);
    mbar_init(smem_u32(&X.bar_p), 128);
    X.rescale = 0;
    X.ntile = 0;
    for (int i = 0; i < kMaxTiles; ++i) X.cnt[i] = 0;
    mbar_fence_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(&X.tmem_slot), 512);
    tmem_relinquish();
  }
  griddep_wait();
  const int b = a.q_seq[q];
  const int64_t p = a.q_pos[q];
  const float scale2 = a.scale * kLog2e;
  const int ntiles_total = 1 + (a.nsel + 127) / 128;

  if (tid < 64) {
    if (nsplit == 1 && a.sink) { X.m_run[tid] = a.sink[tid] * kLog2e; X.l_run[tid] = 1.f; }
    else { X.m_run[tid] = -INFINITY; X.l_run[tid] = 0.f; }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = X.tmem_slot;

  // Q[64 heads][512] -> 8 dim blocks of [64 rows][128 B], swizzled.  These copies join
  // the first commit group of the first tile, so its group-0 barrier also covers Q.
  if (warp < 8) {
    const uint8_t* qg = reinterpret_cast<const uint8_t*>(a.q + (int64_t)q * kHeads * kDLat);
    const uint32_t qb = smem_u32(q_s);
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int flat = i * kWorkers + tid;
      const int h = flat >> 6, c = flat & 63;
      cp_async16(qb + (c >> 3) * 8192 + sw128_off(h, c & 7), qg + h * 1024 + c * 16);
    }
  }
  // ---- row sources of this CTA's tiles (t = rank + slot * nsplit), one pass ----
  {
    const int nslot = (ntiles_total - rank + nsplit - 1) / nsplit;
    const int64_t win_lo = p - (kRing - 1) < 0 ? 0 : p - (kRing - 1);
    const int row_bytes_swa = a.swa_dtype == 1 ? 528 : 1024;
    const int64_t rb = a.row_base[b];
    for (int e = tid; e < nslot * 128; e += kThreads) {
      const int slot = e >> 7, r = e & 127;
      const int t = rank + slot * nsplit;
      int64_t off = -1;
      if (t == 0) {
        const int64_t pos = win_lo + r;
        if (pos <= p) {
          int64_t idx;
          if (a.swa_mode == 0) idx = (int64_t)b * kRing + (pos & (kRing - 1));
          else idx = a.lin_base[b] + (pos - a.lin_pos0[b]);
          if (idx >= 0 && idx < a.swa_rows) off = idx * row_bytes_swa;
          else raise_fault(kFaultBounds);
        }
      } else {
        const int i = (t - 1) * 128 + r;
        if (i < a.nsel) {
          const int32_t rr = a.sel[(int64_t)q * a.nsel + i];
          if (rr >= 0) {
            const int64_t idx = rb + rr;
            if (idx < a.plane_rows) off = idx * 1024;
            else raise_fault(kFaultBounds);
          }
        }
      }
      X.rowsrc[slot][r] = off;
      // all 32 lanes of a warp share one slot (128 rows per slot)
      const uint32_t vm = __ballot_sync(0xFFFFFFFFu, off >= 0);
      if (lane == 0 && vm) atomicAdd(&X.cnt[slot], __popc(vm));
    }
    __syncthreads();
    if (tid == 0) {
      int n = 0;
      for (int slot = 0; slot < nslot; ++slot)
        if (X.cnt[slot] > 0) X.tiles[n++] = slot;
      X.ntile = n;
    }
    __syncthreads();
  }
  const int ntile = X.ntile;

  if (warp < 8) {
    // =================== gather (warps 0..7), softmax (warps 0..3) ===================
    const uint32_t kvb = smem_u32(kv_s);
    for (int it = 0; it < ntile; ++it) {
      const int slot = X.tiles[it];
      const int t = rank + slot * nsplit;
      const bool fp8 = (t == 0 && a.swa_dtype == 1);
      const uint8_t* base = t == 0 ? a.swa : reinterpret_cast<const uint8_t*>(a.plane);
      for (int g = 0; g < 4; ++g) {
        if (it > 0) mbar_wait(smem_u32(&X.bar_pv[g]), (it - 1) & 1);
        gather_group(a, X, slot, g, fp8, base, kvb, tid);
        cp_async_commit();
      }
      cp_async_wait_group<3>();
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&X.bar_g[0]));
      cp_async_wait_group<2>();
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&X.bar_g[1]));
      cp_async_wait_group<1>();
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&X.bar_g[2]));
      cp_async_wait_group<0>();
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&X.bar_g[3]));

      if (warp < 4) {
        mbar_wait(smem_u32(&X.bar_s), it & 1);
        tc_fence_after();
        const int r = warp * 32 + lane;
        const uint32_t lrow = (uint32_t)(warp * 32) << 16;
        float s[64];
        {
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lrow + kColS, v0);
          tmem_ld32(tmem + lrow + kColS + 32, v1);
          tmem_ld_wait();
          const bool ok = X.rowsrc[slot][r] >= 0;
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            s[h] = ok ? __uint_as_float(v0[h]) * scale2 : -INFINITY;
            s[h + 32] = ok ? __uint_as_float(v1[h]) * scale2 : -INFINITY;
          }
        }
        float red[64];
#pragma unroll
        for (int h = 0; h < 64; ++h) red[h] = s[h];
        warp_reduce_heads<true>(red, lane);
        X.red[warp][2 * lane] = red[0];
        X.red[warp][2 * lane + 1] = red[1];
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (tid < 64) {
          const float tm =
              fmaxf(fmaxf(X.red[0][tid], X.red[1][tid]), fmaxf(X.red[2][tid], X.red[3][tid]));
          const float mo = X.m_run[tid];
          const float mn = fmaxf(mo, tm);
          if (mn > mo + kLazy) {
            X.fac[tid] = ex2(mo - mn);
            X.m_run[tid] = mn;
            X.rescale = 1;
          } else {
            X.fac[tid] = 1.f;
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        uint32_t pk[32];
#pragma unroll
        for (int h = 0; h < 64; h += 2) {
          const float p0 = ex2(s[h] - X.m_run[h]);
          const float p1 = ex2(s[h + 1] - X.m_run[h + 1]);
          pk[h >> 1] = pack_bf16x2(p0, p1);
          red[h] = __uint_as_float(pk[h >> 1] << 16);
          red[h + 1] = __uint_as_float(pk[h >> 1] & 0xFFFF0000u);
        }
        const uint32_t pb = smem_u32(p_s);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared16(pb + sw128_off(r, c),
                      make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
        warp_reduce_heads<false>(red, lane);
        X.red[warp][2 * lane] = red[0];
        X.red[warp][2 * lane + 1] = red[1];
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const bool rescale = X.rescale != 0;
        if (tid < 64)
          X.l_run[tid] = X.l_run[tid] * X.fac[tid] + (X.red[0][tid] + X.red[1][tid]) +
                         (X.red[2][tid] + X.red[3][tid]);
        if (rescale && it > 0) {
          // O^T columns are heads: scale column h of every O tile by fac[h].  The PV of
          // the previous tile is complete (its last commit was waited for above).
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int hb = 0; hb < 64; hb += 32) {
              uint32_t v[32];
              const uint32_t ta = tmem + lrow + kColO + 64 * mt + hb;
              tmem_ld32(ta, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[j] = __float_as_uint(__uint_as_float(v[j]) * X.fac[hb + j]);
              tmem_st32(ta, v);
            }
          }
          tmem_st_wait();
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // all read X.rescale and X.red
        if (tid == 0) X.rescale = 0;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&X.bar_p));
      }
    }
    if (ntile > 0) mbar_wait(smem_u32(&X.bar_pv[3]), (ntile - 1) & 1);
    tc_fence_after();
  } else if (lane == 0) {
    // =================== MMA issuer (warp 8, lane 0) ===================
    const uint32_t kvb = smem_u32(kv_s);
    const uint32_t qb = smem_u32(q_s);
    const uint32_t pb = smem_u32(p_s);
    const uint32_t id_s = idesc_bf16(128, 64, 0, 0);
    const uint32_t id_o = idesc_bf16(128, 64, 1, 1);
    for (int it = 0; it < ntile; ++it) {
      for (int g = 0; g < 4; ++g) {
        mbar_wait(smem_u32(&X.bar_g[g]), it & 1);
        tc_fence_after();
#pragma unroll
        for (int d2 = 0; d2 < 2; ++d2) {
          const int db = 2 * g + d2;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + kColS, sdesc_sw128(kvb + db * 16384 + kk * 32, 16, 1024),
                      sdesc_sw128(qb + db * 8192 + kk * 32, 16, 1024), id_s, (db | kk) != 0);
        }
      }
      umma_commit(smem_u32(&X.bar_s));
      mbar_wait(smem_u32(&X.bar_p), it & 1);
      tc_fence_after();
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + kColO + 64 * mt,
                    sdesc_sw128(kvb + 2 * mt * 16384 + kk * 2048, 16384, 1024),
                    sdesc_sw128(pb + kk * 2048, 8192, 1024), id_o, (it > 0 || kk > 0) ? 1 : 0);
        umma_commit(smem_u32(&X.bar_pv[mt]));
      }
    }
  }

  // ---- epilogue ----
  __syncthreads();
  if (nsplit == 1) {
    // O^T / l -> bf16 [64 heads][512], staged in the KV tile, then coalesced stores
    if (tid < 64) X.fac[tid] = 1.f / X.l_run[tid];
    __syncthreads();
    uint16_t* stage = reinterpret_cast<uint16_t*>(kv_s);
    if (warp < 8) {
      const int sub = warp & 3;
      const uint32_t lrow = (uint32_t)(sub * 32) << 16;
#pragma unroll 1
      for (int mi = 0; mi < 2; ++mi) {
        const int mt = 2 * (warp >> 2) + mi;
        const int dim = mt * 128 + sub * 32 + lane;
#pragma unroll
        for (int hb = 0; hb < 64; hb += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lrow + kColO + 64 * mt + hb, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float o = ntile > 0 ? __uint_as_float(v[j]) * X.fac[hb + j] : 0.f;
            __nv_bfloat16 bv = __float2bfloat16_rn(o);
            stage[(hb + j) * kDLat + dim] = *reinterpret_cast<uint16_t*>(&bv);
          }
        }
      }
    }
    __syncthreads();
    const uint4* src = reinterpret_cast<const uint4*>(kv_s);
    uint4* dst = reinterpret_cast<uint4*>(a.out + (int64_t)q * kHeads * kDLat);
    for (int i = tid; i < kHeads * kDLat * 2 / 16; i += kThreads) dst[i] = src[i];
    if (a.lse && tid < 64)
      a.lse[(int64_t)q * kHeads + tid] =
          (X.m_run[tid] + __log2f(X.l_run[tid])) * 0.6931471805599453f;
  } else {
    // partial O^T (unnormalised fp32) -> workspace [Q][nsplit][64 heads][512], plus the
    // running max (log2 units) and sum per head
    float* po = a.part_o + ((int64_t)q * nsplit + rank) * kHeads * kDLat;
    if (warp < 8) {
      const int sub = warp & 3;
      const uint32_t lrow = (uint32_t)(sub * 32) << 16;
#pragma unroll 1
      for (int mi = 0; mi < 2; ++mi) {
        const int mt = 2 * (warp >> 2) + mi;
        const int dim = mt * 128 + sub * 32 + lane;
#pragma unroll
        for (int hb = 0; hb < 64; hb += 32) {
          uint32_t v[32];
          if (ntile > 0) {
            tmem_ld32(tmem + lrow + kColO + 64 * mt + hb, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) po[(hb + j) * kDLat + dim] = __uint_as_float(v[j]);
        }
      }
    }
    if (tid < 64) {
      a.part_ml[((int64_t)q * nsplit + rank) * 128 + tid] = X.m_run[tid];
      a.part_ml[((int64_t)q * nsplit + rank) * 128 + 64 + tid] = X.l_run[tid];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, 512);
}

// Merge of the nsplit partials of each query: grid = Q x 8, each CTA 8 heads.
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a, int nsplit) {
  __shared__ float coef[8][8];  // [split][head within the CTA]
  __shared__ float lse2[8];
  const int q = blockIdx.x, h0 = blockIdx.y * 8, tid = threadIdx.x;
  griddep_launch_dependents();
  griddep_wait();
  if (tid < 8) {
    const int h = h0 + tid;
    const float* ml = a.part_ml + (int64_t)q * nsplit * 128;
    float M = a.sink ? a.sink[h] * kLog2e : -INFINITY;
    for (int j = 0; j < nsplit; ++j) M = fmaxf(M, ml[j * 128 + h]);
    float Z = a.sink ? ex2(a.sink[h] * kLog2e - M) : 0.f;
    for (int j = 0; j < nsplit; ++j) {
      const float mj = ml[j * 128 + h];
      if (mj != -INFINITY) Z += ex2(mj - M) * ml[j * 128 + 64 + h];
    }
    const float inv = 1.f / Z;
    for (int j = 0; j < nsplit; ++j) {
      const float mj = ml[j * 128 + h];
      coef[j][tid] = mj == -INFINITY ? 0.f : ex2(mj - M) * inv;
    }
    lse2[tid] = M + __log2f(Z);
  }
  __syncthreads();
  // 8 heads x 512 dims = 512 groups of 8 elements; 2 per thread
  for (int gidx = tid; gidx < 512; gidx += 256) {
    const int hl = gidx >> 6, d = (gidx & 63) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < nsplit; ++j) {
      const float w = coef[j][hl];
      if (w == 0.f) continue;
      const float4* src = reinterpret_cast<const float4*>(
          a.part_o + (((int64_t)q * nsplit + j) * kHeads + h0 + hl) * kDLat + d);
      const float4 x0 = src[0], x1 = src[1];
      acc[0] += w * x0.x; acc[1] += w * x0.y; acc[2] += w * x0.z; acc[3] += w * x0.w;
      acc[4] += w * x1.x; acc[5] += w * x1.y; acc[6] += w * x1.z; acc[7] += w * x1.w;
    }
    uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)q * kHeads + h0 + hl) * kDLat + d);
    *dst = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                      pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
  if (a.lse && tid < 8) a.lse[(int64_t)q * kHeads + h0 + tid] = lse2[tid] * 0.6931471805599453f;
}

}  // namespace

size_t attn_smem_bytes() { return 1024 + kQBytes + kKVBytes + kPBytes + sizeof(Aux); }

// CTAs per query: as many as keep every CTA of the launch in one wave (one CTA per SM),
// at most one tile each.
int attn_num_splits(int Q, int nsel, int num_sms) {
  const int ntiles = 1 + (nsel + 127) / 128;
  int nsplit = num_sms / (Q > 0 ? Q : 1);
  return nsplit < 1 ? 1 : (nsplit > ntiles ? ntiles : nsplit);
}

cudaError_t launch_attn(const AttnArgs& a, int nsplit, cudaStream_t s) {
  if (a.Q == 0) return cudaSuccess;
  const size_t smem = attn_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(sparse_attn_kernel, dim3((unsigned)nsplit, (unsigned)a.Q), dim3(kThreads), smem,
                 s, a);
  if (e != cudaSuccess || nsplit == 1) return e;
  return launch_pdl(attn_combine_kernel, dim3((unsigned)a.Q, kHeads / 8), dim3(256), 0, s, a,
                    nsplit);
}

}  // namespace csa2

// k_attn.cu -- CSA2 sparse MQA attention (64 heads x 512 dims, K = V) over the
// layer's sliding window plus the selected compressed rows, one softmax with a
// per-head sink logit in the denominator.
// [A] "四种层合并出来的是什么形状" (one CSR, one softmax, K = V, <= 640 rows, sink only in
// the denominator); [B] §4.1 (two sources, no de-duplication), §4.4 step 4 (window
// slots); [C] §5.5-5.6 (logical concatenation, no physical copy), A.19.3 (gather by
// int32 index, online softmax with running max and sum, fused sink);
// [E] Fig. 2d (out_h = sum e^{s_j} v_j / (e^{sink_h} + sum e^{s_j})).
//
// One CTA per query.  Entries are processed in tiles of 128 rows: tile 0 is the
// window (positions p-127..p), tiles 1..4 hold sel[0..511].  Per tile:
//   gather   128 rows (bf16, or FP8 dequantised to bf16) into a 128-byte-swizzled
//            shared tile [8 dim blocks][128 rows][128 B]
//   S^T      = KV[128 x 512] . Q^T[512 x 64]  -> TMEM (row = lane, head = column)
//   softmax  per head over the 128 rows (warp butterfly + 4-warp combine), lazy
//            rescaling: the running max moves only when it grows by > 8 (log2 units)
//   O^T     += V^T[512 x 128] . P^T[128 x 64] -> TMEM, four M=128 tiles; the same KV
//            tile is the A operand again, read MN-major
// The running max starts at the sink logit with running sum 1, which is exactly the
// sink's term of the denominator.
#include <cuda_fp8.h>

#include "common.cuh"

CSA2_DEFINE_FAULT_FLAG(attn)

namespace csa2 {
namespace {

constexpr int kThreads = 256;
constexpr int kQBytes = 8 * 64 * 128;     // 64 KiB
constexpr int kKVBytes = 8 * 128 * 128;   // 128 KiB
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
  int64_t rowsrc[128];
  uint64_t bar_s;
  uint64_t bar_o;
  uint32_t tmem_slot;
  int rescale;
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
    const int half = 32 >> step;      // values still held: 2 * half
    const int bit = 16 >> step;       // partner distance
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      if (i < half) {
        const float send = upper ? v[i] : v[i + half];
        const float keep = upper ? v[i + half] : v[i];
        const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, bit);
        v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
      }
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

__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + kQBytes;
  uint8_t* p_s = kv_s + kKVBytes;
  Aux& X = *reinterpret_cast<Aux*>(p_s + kPBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = blockIdx.x;
  const int b = a.q_seq[q];
  const int64_t p = a.q_pos[q];
  const float scale2 = a.scale * kLog2e;

  if (tid == 0) {
    mbar_init(smem_u32(&X.bar_s), 1);
    mbar_init(smem_u32(&X.bar_o), 1);
    X.rescale = 0;
    mbar_fence_init();
  }
  if (tid < 64) {
    if (a.sink) { X.m_run[tid] = a.sink[tid] * kLog2e; X.l_run[tid] = 1.f; }
    else { X.m_run[tid] = -INFINITY; X.l_run[tid] = 0.f; }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&X.tmem_slot), 512);
    tmem_relinquish();
  }
  // Q[64 heads][512] -> 8 dim blocks of [64 rows][128 B], swizzled
  {
    const uint8_t* qg = reinterpret_cast<const uint8_t*>(a.q + (int64_t)q * kHeads * kDLat);
    const uint32_t qb = smem_u32(q_s);
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int flat = i * kThreads + tid;
      const int h = flat >> 6, c = flat & 63;
      cp_async16(qb + (c >> 3) * 8192 + sw128_off(h, c & 7), qg + h * 1024 + c * 16);
    }
    cp_async_commit();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = X.tmem_slot;

  const int ntiles = 1 + (a.nsel + 127) / 128;
  bool first_pv = true;
  uint32_t phase = 0;
  const int64_t win_lo = p - (kRing - 1) < 0 ? 0 : p - (kRing - 1);
  const int row_bytes_swa = a.swa_dtype == 1 ? 528 : 1024;

  for (int t = 0; t < ntiles; ++t) {
    bool bad = false;  // a bounded wait gave up (fault already raised)
    // ---- row sources of this tile ----
    int valid = 0;
    if (tid < 128) {
      int64_t off = -1;
      if (t == 0) {
        const int64_t pos = win_lo + tid;
        if (pos <= p) {
          int64_t idx;
          if (a.swa_mode == 0) idx = (int64_t)b * kRing + (pos & (kRing - 1));
          else idx = a.lin_base[b] + (pos - a.lin_pos0[b]);
          if (idx >= 0 && idx < a.swa_rows) off = idx * row_bytes_swa;
          else raise_fault(kFaultBounds);
        }
      } else {
        const int i = (t - 1) * 128 + tid;
        if (i < a.nsel) {
          const int32_t r = a.sel[(int64_t)q * a.nsel + i];
          if (r >= 0) {
            const int64_t idx = a.row_base[b] + r;
            if (idx < a.plane_rows) off = idx * 1024;
            else raise_fault(kFaultBounds);
          }
        }
      }
      X.rowsrc[tid] = off;
      valid = off >= 0;
    }
    const int nvalid = __syncthreads_count(valid);
    if (nvalid == 0) continue;

    // ---- gather ----
    const uint32_t kvb = smem_u32(kv_s);
    if (t == 0 && a.swa_dtype == 1) {
      // FP8 rows: 16 codes per thread-step -> two 16-byte bf16 chunks
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int flat = i * kThreads + tid;
        const int r = flat >> 5, c16 = flat & 31;
        const int64_t off = X.rowsrc[r];
        const uint32_t d0 = kvb + (c16 >> 2) * 16384 + sw128_off(r, (2 * c16) & 7);
        const uint32_t d1 = kvb + (c16 >> 2) * 16384 + sw128_off(r, (2 * c16 + 1) & 7);
        if (off < 0) { st_shared_zero16(d0); st_shared_zero16(d1); continue; }
        const uint8_t* src = a.swa + off;
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
      const uint8_t* base = t == 0 ? a.swa : reinterpret_cast<const uint8_t*>(a.plane);
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const int flat = i * kThreads + tid;
        const int r = flat >> 6, c = flat & 63;
        const int64_t off = X.rowsrc[r];
        const uint32_t dst = kvb + (c >> 3) * 16384 + sw128_off(r, c & 7);
        if (off < 0) st_shared_zero16(dst);
        else cp_async16(dst, base + off + c * 16);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncthreads();

    // ---- S^T = KV . Q^T ----
    if (tid == 128) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
      const uint32_t qb = smem_u32(q_s);
#pragma unroll
      for (int db = 0; db < 8; ++db)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + kColS, sdesc_sw128(kvb + db * 16384 + kk * 32, 16, 1024),
                    sdesc_sw128(qb + db * 8192 + kk * 32, 16, 1024), idesc, (db | kk) != 0);
      umma_commit(smem_u32(&X.bar_s));
    }

    // ---- softmax over the tile's rows (warps 0..3, TMEM lanes 0..127) ----
    if (warp < 4) {
      if (!mbar_wait(smem_u32(&X.bar_s), phase & 1)) bad = true;
      tc_fence_after();
      const int r = warp * 32 + lane;
      const uint32_t lrow = (uint32_t)(warp * 32) << 16;
      float s[64];
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lrow + kColS, v0);
        tmem_ld32(tmem + lrow + kColS + 32, v1);
        tmem_ld_wait();
        const bool ok = X.rowsrc[r] >= 0;
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
        const float tm = fmaxf(fmaxf(X.red[0][tid], X.red[1][tid]), fmaxf(X.red[2][tid], X.red[3][tid]));
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
      // P = 2^(s - m) in bf16; the running sum uses the rounded values
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
      asm volatile("bar.sync 1, 128;" ::: "memory");  // everyone has read X.red (max)
      X.red[warp][2 * lane] = red[0];
      X.red[warp][2 * lane + 1] = red[1];
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (tid < 64)
        X.l_run[tid] = X.l_run[tid] * X.fac[tid] + (X.red[0][tid] + X.red[1][tid]) +
                       (X.red[2][tid] + X.red[3][tid]);
      if (X.rescale && !first_pv) {
        // O^T columns are heads: scale column h of every O tile by fac[h]
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
          for (int hb = 0; hb < 64; hb += 32) {
            uint32_t v[32];
            const uint32_t ta = tmem + lrow + kColO + 64 * mt + hb;
            tmem_ld32(ta, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * X.fac[hb + j]);
            tmem_st32(ta, v);
          }
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
    }
    __syncthreads();
    if (tid == 0) X.rescale = 0;

    // ---- O^T += V^T . P^T ----
    if (tid == 128) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 64, 1, 1);
      const uint32_t pb = smem_u32(p_s);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + kColO + 64 * mt,
                    sdesc_sw128(kvb + 2 * mt * 16384 + kk * 2048, 16384, 1024),
                    sdesc_sw128(pb + kk * 2048, 8192, 1024), idesc, (!first_pv || kk > 0) ? 1 : 0);
      umma_commit(smem_u32(&X.bar_o));
    }
    first_pv = false;
    if (!mbar_wait(smem_u32(&X.bar_o), phase & 1)) bad = true;
    tc_fence_after();
    ++phase;
    if (__syncthreads_or(bad)) break;  // uniform exit: the output is garbage, flagged
  }

  // ---- epilogue: O^T / l -> bf16 [64 heads][512] staged in the KV tile ----
  __syncthreads();
  {
    const int sub = warp & 3;
    const uint32_t lrow = (uint32_t)(sub * 32) << 16;
    uint16_t* stage = reinterpret_cast<uint16_t*>(kv_s);
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
          const float o = first_pv ? 0.f : __uint_as_float(v[j]) / X.l_run[hb + j];
          __nv_bfloat16 bv = __float2bfloat16_rn(o);
          stage[(hb + j) * kDLat + dim] = *reinterpret_cast<uint16_t*>(&bv);
        }
      }
    }
  }
  __syncthreads();
  {
    const uint4* src = reinterpret_cast<const uint4*>(kv_s);
    uint4* dst = reinterpret_cast<uint4*>(a.out + (int64_t)q * kHeads * kDLat);
#pragma unroll 4
    for (int i = tid; i < kHeads * kDLat * 2 / 16; i += kThreads) dst[i] = src[i];
  }
  if (a.lse && tid < 64)
    a.lse[(int64_t)q * kHeads + tid] = (X.m_run[tid] + log2f(X.l_run[tid])) * 0.6931471805599453f;

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t attn_smem_bytes() { return 1024 + kQBytes + kKVBytes + kPBytes + sizeof(Aux); }

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  if (a.Q == 0) return cudaSuccess;
  const size_t smem = attn_smem_bytes();
  cudaError_t e =
      cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  sparse_attn_kernel<<<a.Q, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace csa2

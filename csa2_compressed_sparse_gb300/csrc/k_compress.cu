// k_compress.cu -- the CSA2 compressor: softmax-gated pooling of m (1 or 2) tokens
// per row, RMSNorm over the 512 dims, partial RoPE on dims 448..511 at the group's
// first position, bf16 store; the odd tail is kept in the per-sequence fp32 state.
// Optionally each row's index K (wk projection of the latent before RoPE, k_norm, RoPE
// on its last 64 dims) goes to the index plane.
// [A] "特殊模块 · compressor" and "CSA2 的池化比 V4 简单一截"; [B] §4.1, §6.1-6.2;
// [C] §6.2 (tail state), §6.4 (ratio 1 degenerates to projection + norm).
//
// One warp per new token.  The warp of a token that closes a group (pos % m == m-1)
// emits that group's row; the group's earlier tokens come from this call's input
// or, for the first group of a sequence, from the state.  The warp of the first
// token of each sequence additionally stores the tokens of a group left incomplete
// at the end of the call into the state.  With m <= 2 that warp is also the only
// reader of the state, so state reads precede state writes within one warp.
//
// Lane layout: lane l owns channels [8l, 8l+8) and [256+8l, 256+8l+8), i.e. two
// 16-byte vectors per row (coalesced 1 KiB row accesses).  Lanes 24..31 hold the
// RoPE dims 448..511 in their second vector, four adjacent pairs each.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

CSA2_DEFINE_FAULT_FLAG(compress)

namespace csa2 {
namespace {

// 4 warps (one token each) per CTA: a compress CTA (128 threads, at most 128 registers)
// fits beside a score CTA of the indexer, which may run concurrently on another stream.
constexpr int kWarps = 4;

__device__ __forceinline__ void load8_bf16(const uint16_t* p, float (&v)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load8_f32(const float* p, float (&v)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8_f32(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void store8_bf16(uint16_t* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// Fetch channels (c0..c0+7) of the token at position `pos` of sequence b: from the
// input when it arrived in this call, else from the state slot pos % m.
__device__ __forceinline__ void fetch(const CompressArgs& a, int b, int64_t pos, int64_t s0,
                                      int64_t t0, int c0, float (&kv)[8], float (&sc)[8]) {
  if (pos >= s0) {
    int64_t t = t0 + (pos - s0);
    load8_bf16(a.kv + t * kDLat + c0, kv);
    if (a.score) load8_bf16(a.score + t * kDLat + c0, sc);
    else
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i] = 0.f;
  } else {
    int slot = (int)(pos % a.ratio);
    load8_f32(a.kv_state + ((int64_t)b * 2 + slot) * kDLat + c0, kv);
    load8_f32(a.score_state + ((int64_t)b * 2 + slot) * kDLat + c0, sc);
  }
}

// Index K of one row, by the warp that emits it: [A] indexer figure, key side (the bf16
// latent before RoPE -> wk [128, 512] -> k_norm -> RoPE on the last 64 dims -> the index
// plane).  r holds the lane's 16 normalized channels before RoPE.  Each lane multiplies
// its channels into all 128 outputs (one 16-byte load of each wk row per half), and a
// butterfly over the lanes sums every block of 32 outputs so that lane l ends with
// outputs l, 32 + l, 64 + l, 96 + l; then the RMSNorm over the 128 and the rotation of
// pairs (64 + 2i, 65 + 2i), whose halves sit in lanes 2i and 2i + 1.
__device__ __forceinline__ void emit_index_k(const CompressArgs& a, const float (&r)[2][8],
                                             const int (&c)[2], int lane, uint64_t p0,
                                             int64_t row, const uint64_t* turn_s) {
  float x[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) x[h][i] = __bfloat162float(__float2bfloat16_rn(r[h][i]));
  float k[4];
#pragma unroll 1
  for (int blk = 0; blk < 4; ++blk) {
    float v[32];
#pragma unroll
    for (int oo = 0; oo < 32; ++oo) {
      const uint16_t* wr = a.wk + (int64_t)(32 * blk + oo) * kDLat;
      float w0[8], w1[8];
      load8_bf16(wr + c[0], w0);
      load8_bf16(wr + c[1], w1);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(w0[i], x[0][i], acc);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(w1[i], x[1][i], acc);
      v[oo] = acc;
    }
#pragma unroll
    for (int off = 16, n = 16; off >= 1; off >>= 1, n >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < n; ++i) {
        const float send = upper ? v[i] : v[i + n];
        const float keep = upper ? v[i + n] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
      }
    }
    k[blk] = v[0];
  }
  float ss = k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const float rstd = 1.0f / sqrtf(ss / (float)kDIdx + a.eps);
#pragma unroll
  for (int blk = 0; blk < 4; ++blk)
    k[blk] *= rstd * (a.knorm_w ? a.knorm_w[32 * blk + lane] : 1.f);
#pragma unroll
  for (int blk = 2; blk < 4; ++blk) {
    const int pair = 16 * (blk - 2) + (lane >> 1);
    float fs, fc;
    sincosf(rope_angle(turn_s[pair], p0), &fs, &fc);
    const float other = __shfl_xor_sync(0xFFFFFFFFu, k[blk], 1);
    k[blk] = (lane & 1) ? other * fs + k[blk] * fc : k[blk] * fc - other * fs;
  }
  uint16_t* dst = a.index_plane + row * kDIdx;
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) dst[32 * blk + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(k[blk]));
}

__global__ void __launch_bounds__(kWarps * 32, 4) compress_kernel(CompressArgs a) {
  // cu_seqlens in shared memory (one coalesced read instead of a chain of dependent
  // global loads in the binary search below)
  extern __shared__ int32_t cu_s[];
  __shared__ uint64_t turn_s[32];
  griddep_launch_dependents();
  griddep_wait();
  for (int i = threadIdx.x; i <= a.B; i += blockDim.x) cu_s[i] = a.cu_seqlens[i];
  if (threadIdx.x < 32) turn_s[threadIdx.x] = rope_turn(a.inv_freq[threadIdx.x]);
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  // this token's own kv / score do not depend on its sequence: start them now
  float own_kv[2][8], own_sc[2][8];
  if (t < a.T) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      load8_bf16(a.kv + t * kDLat + (h ? 256 : 0) + 8 * lane, own_kv[h]);
      if (a.score) load8_bf16(a.score + t * kDLat + (h ? 256 : 0) + 8 * lane, own_sc[h]);
      else
#pragma unroll
        for (int i = 0; i < 8; ++i) own_sc[h][i] = 0.f;
    }
  }
  __syncthreads();
  if (t >= a.T) return;
  // sequence of token t: last b with cu_seqlens[b] <= t
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu_s[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int64_t t0 = cu_s[b];
  const int64_t t1 = cu_s[b + 1];
  const int64_t s0 = a.start_pos[b];
  const int64_t pos = s0 + (t - t0);
  const int m = a.ratio;
  const int c[2] = {8 * lane, 256 + 8 * lane};

  // ---- emit the row of a group that this token closes ----
  if (pos % m == m - 1) {
    const int64_t j = pos / m;
    float r[2][8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (m == 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) r[h][i] = own_kv[h][i];
      } else {
        float k0[8], q0[8];
        fetch(a, b, pos - 1, s0, t0, c[h], k0, q0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // per-channel softmax over the two slots
          const float k1 = own_kv[h][i], q1 = own_sc[h][i];
          float mx = fmaxf(q0[i], q1);
          float e0 = expf(q0[i] - mx), e1 = expf(q1 - mx);
          r[h][i] = (e0 * k0[i] + e1 * k1) / (e0 + e1);
        }
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += r[h][i] * r[h][i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    const float rstd = 1.0f / sqrtf(ss / (float)kDLat + a.eps);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float wv[8];
      if (a.norm_w) load8_f32(a.norm_w + c[h], wv);
      else
#pragma unroll
        for (int i = 0; i < 8; ++i) wv[i] = 1.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) r[h][i] = r[h][i] * rstd * wv[i];
    }
    const int64_t row = a.row_base[b] + j;
    const bool row_ok = row >= 0 && row < a.plane_rows;
    // the indexer's branch leaves before the main RoPE
    if (a.wk && row_ok) emit_index_k(a, r, c, lane, (uint64_t)(j * m), row, turn_s);
    if (lane >= 24) {  // dims 448 + 8(lane-24) .. +7: four rotation pairs
      const uint64_t p0 = (uint64_t)(j * m);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int pair = 4 * (lane - 24) + k;
        const float ang = rope_angle(turn_s[pair], p0);
        float fs, fc;
        sincosf(ang, &fs, &fc);
        const float x0 = r[1][2 * k], x1 = r[1][2 * k + 1];
        r[1][2 * k] = x0 * fc - x1 * fs;
        r[1][2 * k + 1] = x0 * fs + x1 * fc;
      }
    }
    if (!row_ok) {
      if (lane == 0) raise_fault(kFaultBounds);
    } else {
      store8_bf16(a.plane + row * kDLat + c[0], r[0]);
      store8_bf16(a.plane + row * kDLat + c[1], r[1]);
    }
  }

  // ---- first token of the sequence: keep an incomplete trailing group ----
  if (t == t0 && m > 1) {
    const int64_t last = s0 + (t1 - t0) - 1;
    if (last % m != m - 1) {
      for (int64_t p = (last / m) * m; p <= last; ++p) {
        if (p < s0) continue;  // already in the state from an earlier call
        const int64_t tp = t0 + (p - s0);
        const int slot = (int)(p % m);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float kv[8], sc[8];
          load8_bf16(a.kv + tp * kDLat + c[h], kv);
          if (a.score) load8_bf16(a.score + tp * kDLat + c[h], sc);
          else
#pragma unroll
            for (int i = 0; i < 8; ++i) sc[i] = 0.f;
          store8_f32(a.kv_state + ((int64_t)b * 2 + slot) * kDLat + c[h], kv);
          store8_f32(a.score_state + ((int64_t)b * 2 + slot) * kDLat + c[h], sc);
        }
      }
    }
  }
}

// E4M3 value of a code below 0x7F, from the format's fields.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e == 0 ? (float)m * (1.f / 512.f) : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// FP4 plane rows ([A] pool switch: nvfp4 rows of 288 B, E2M1 with an E4M3 scale per 16
// dims): one warp per row, lane l quantises dims 16 l .. 16 l + 15.  The scale is the
// smallest E4M3 value s with 6 s >= max |x| (0 for an all-zero group; 448 at most),
// found from the nearest code and one exact comparison; codes are E2M1(x / s).
__global__ void __launch_bounds__(256) plane_fp4_kernel(const uint16_t* rows, int64_t n,
                                                        uint8_t* out) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= n) return;
  float v[16];
  load8_bf16(rows + r * kDLat + 16 * lane, *reinterpret_cast<float(*)[8]>(v));
  load8_bf16(rows + r * kDLat + 16 * lane + 8, *reinterpret_cast<float(*)[8]>(v + 8));
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  uint32_t sc = 0;
  if (amax > 0.f) {
    sc = (uint32_t)__nv_cvt_float_to_fp8(amax / 6.f, __NV_SATFINITE, __NV_E4M3);
    if (6.f * e4m3_value(sc) < amax && sc < 0x7Eu) ++sc;  // 6 * value is exact in fp32
  }
  const float s = e4m3_value(sc);
  uint32_t w[2] = {0u, 0u};
  if (sc != 0) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint32_t two = (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(v[i] / s, v[i + 1] / s),
                                                              __NV_E2M1, cudaRoundNearest);
      w[i >> 3] |= (two & 0xFFu) << (8 * ((i & 7) >> 1));
    }
  }
  uint8_t* o = out + r * 288;
  *reinterpret_cast<uint2*>(o + 8 * lane) = make_uint2(w[0], w[1]);
  o[256 + lane] = (uint8_t)sc;
}

}  // namespace

cudaError_t launch_plane_fp4(const uint16_t* rows, int64_t n, uint8_t* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(plane_fp4_kernel, dim3((unsigned)((n + 7) / 8)), dim3(256), 0, s, rows, n,
                    out);
}

// Self-test of the bounded waits: thread 0 waits for the first phase of a fresh
// mbarrier that nothing arrives on (no copy or MMA is attached to it), so the wait runs
// out after limit_ns, records the timeout in the fault flag and the kernel returns.
__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
    mbar_wait(smem_u32(&bar), 0, limit_ns);
  }
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  const int grid = (a.T + kWarps - 1) / kWarps;
  return launch_pdl(compress_kernel, dim3(grid), dim3(kWarps * 32),
                    (size_t)(a.B + 1) * sizeof(int32_t), s, a);
}

}  // namespace csa2

// k_compress.cu -- the CSA2 compressor: softmax-gated pooling of m (1 or 2) tokens
// per row, RMSNorm over the 512 dims, partial RoPE on dims 448..511 at the group's
// first position, bf16 store; the odd tail is kept in the per-sequence fp32 state.
// Optionally each row's index K (wk projection of the latent before RoPE, k_norm, RoPE
// on its last 64 dims) goes to the index plane.
// [A] "特殊模块 · compressor" and "CSA2 的池化比 V4 简单一截"; [B] §4.1, §6.1-6.2;
// [C] §6.2 (tail state), §6.4 (ratio 1 degenerates to projection + norm).
//
// The per-token work (one warp per token) is in compress_dev.cuh.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "compress_dev.cuh"

CSA2_DEFINE_FAULT_FLAG(compress)

namespace csa2 {
namespace {

// 4 warps (one token each) per CTA: a compress CTA (128 threads, at most 128 registers)
// fits beside a score CTA of the indexer, which may run concurrently on another stream.
constexpr int kWarps = 4;

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
  if (t < a.T) cdev::load_own(a, t, lane, own_kv, own_sc);
  __syncthreads();
  if (t >= a.T) return;
  // sequence of token t: last b with cu_seqlens[b] <= t
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu_s[mid] <= t) lo = mid; else hi = mid - 1;
  }
  cdev::token(a, t, lo, cu_s[lo], cu_s[lo + 1], own_kv, own_sc, lane, turn_s);
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
  cdev::load8_bf16(rows + r * kDLat + 16 * lane, *reinterpret_cast<float(*)[8]>(v));
  cdev::load8_bf16(rows + r * kDLat + 16 * lane + 8, *reinterpret_cast<float(*)[8]>(v + 8));
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

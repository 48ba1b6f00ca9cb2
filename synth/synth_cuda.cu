/*
 * synth_cuda.cu -- device side of the seeded input generator (see synth.h).
 * Same definitions as synth.c, written into caller-owned device buffers on the
 * caller's stream, so multi-GB inputs never cross the host link.  Each function
 * returns 0 on success or the cudaError_t of the launch.
 */
#include <cuda_runtime.h>

#include "synth.h"

#define SCALE_STREAM_OFFSET 0x100000ULL

namespace {

constexpr int kThreads = 256;

__global__ void k_normal_bf16(uint16_t* out, int64_t n, uint64_t base, uint64_t offset) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = synth_bf16(synth_normal(base, offset + (uint64_t)i));
}

__global__ void k_normal_f32(float* out, int64_t n, uint64_t base, uint64_t offset) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = synth_normal(base, offset + (uint64_t)i);
}

__global__ void k_rows_bf16(uint16_t* out, uint64_t b, int64_t j0, int64_t nrows, int64_t D,
                            uint64_t base) {
  int64_t n = nrows * D;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / D, d = i - r * D;
    out[i] = synth_bf16(
        synth_normal(base, synth_row_elem(b, (uint64_t)(j0 + r), (uint64_t)D, (uint64_t)d)));
  }
}

__global__ void k_rows_fp8s128(uint8_t* out, uint64_t b, int64_t j0, int64_t nrows, uint64_t base,
                               uint64_t sbase) {
  int64_t n = nrows * 516; /* 512 codes + 4 scales per row */
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / 516, c = i - r * 516;
    uint64_t j = (uint64_t)(j0 + r);
    uint8_t* row = out + r * 528;
    if (c < 512) {
      row[c] = synth_e4m3(64.0f * synth_normal(base, synth_row_elem(b, j, 512, (uint64_t)c)));
    } else {
      int k = (int)(c - 512);
      float s = (0.75f + 0.5f * synth_uniform(sbase, synth_row_elem(b, j, 4, (uint64_t)k))) *
                0.015625f;
      *reinterpret_cast<float*>(row + 512 + 4 * k) = s;
    }
  }
}

int grid_for(int64_t n) {
  int64_t g = (n + kThreads - 1) / kThreads;
  if (g > 152 * 32) g = 152 * 32;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

extern "C" {

int synth_fill_normal_bf16_cuda(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream,
                                uint64_t offset, void* cuda_stream) {
  if (n <= 0) return 0;
  k_normal_bf16<<<grid_for(n), kThreads, 0, (cudaStream_t)cuda_stream>>>(
      out, n, synth_base(seed, stream), offset);
  return (int)cudaGetLastError();
}

int synth_fill_normal_f32_cuda(float* out, int64_t n, uint64_t seed, uint64_t stream,
                               uint64_t offset, void* cuda_stream) {
  if (n <= 0) return 0;
  k_normal_f32<<<grid_for(n), kThreads, 0, (cudaStream_t)cuda_stream>>>(
      out, n, synth_base(seed, stream), offset);
  return (int)cudaGetLastError();
}

int synth_fill_rows_bf16_cuda(uint16_t* out, uint64_t b, int64_t j0, int64_t nrows, int64_t D,
                              uint64_t seed, uint64_t stream, void* cuda_stream) {
  if (nrows <= 0) return 0;
  k_rows_bf16<<<grid_for(nrows * D), kThreads, 0, (cudaStream_t)cuda_stream>>>(
      out, b, j0, nrows, D, synth_base(seed, stream));
  return (int)cudaGetLastError();
}

int synth_fill_rows_fp8s128_cuda(uint8_t* out, uint64_t b, int64_t j0, int64_t nrows,
                                 uint64_t seed, uint64_t stream, void* cuda_stream) {
  if (nrows <= 0) return 0;
  k_rows_fp8s128<<<grid_for(nrows * 516), kThreads, 0, (cudaStream_t)cuda_stream>>>(
      out, b, j0, nrows, synth_base(seed, stream),
      synth_base(seed, stream + SCALE_STREAM_OFFSET));
  return (int)cudaGetLastError();
}

}  // extern "C"

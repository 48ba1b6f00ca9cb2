// noalloc.cu -- csa2_index_topk for callers that cannot hand the library a workspace.
//
// Some callers have no way to obtain device memory for a workspace: a plugin that
// an inference runtime drives through a fixed "inputs in, outputs out" interface
// with no scratch slot, an engine that reserves every byte of HBM for its own pool
// at start-up and forbids any other allocation, or a latency-critical path where the
// implicit device synchronisation of cudaMalloc/cudaFree cannot be tolerated.  For
// them this file keeps the indexer's scratch in a fixed device array that is part of
// the library image, so the call itself allocates nothing.
//
// The array holds kScratchBytes on every GPU that loads the library, until the
// process exits.  All calls on a device share it and it keeps whatever the previous
// call left there; nothing in it needs to start at zero, because every entry the
// indexer and the top-k read is written earlier in the same call.  Two calls whose
// kernels overlap on the GPU (different streams, no ordering between them) race on
// the array and produce wrong results: order them on one stream or with events.
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/csa2.h"
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB per device

static __device__ __align__(256) uint8_t g_index_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.  A device
// reset (cudaDeviceReset) or a re-created primary context reloads the library's module,
// and the array may then sit elsewhere, so the address is looked up again whenever the
// current context is not the one it came from.
CUcontext g_scratch_ctx[kMaxDevices] = {};
void* g_scratch_ptr[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 ctx_getter() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  return fn;
}

// Device address of g_index_scratch in the current device's current context (the
// host-side name of the array is only a stand-in and must not reach a kernel).  On
// failure writes the reason to msg and returns CSA2_ECUDA, leaving no CUDA error pending.
csa2_status scratch_on_current_device(void** out, char* msg, size_t msg_len) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    snprintf(msg, msg_len, "csa2_index_topk_noalloc: cudaGetDevice failed: %s",
             cudaGetErrorString(e));
    return CSA2_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, msg_len, "csa2_index_topk_noalloc: device %d is beyond the %d devices this "
             "entry point serves", dev, kMaxDevices);
    return CSA2_ECUDA;
  }
  // cudaFree(0) is not called: with no context yet, cudaGetSymbolAddress creates the
  // primary context itself; the context is read after it.
  std::lock_guard<std::mutex> lock(g_mu);
  CUcontext ctx = nullptr;
  PFN_cuCtxGetCurrent_v4000 get = ctx_getter();
  if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  if (!g_scratch_ptr[dev] || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_index_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // a failed lookup must not surface in the caller's next check
      snprintf(msg, msg_len,
               "csa2_index_topk_noalloc: no device address for the scratch array on device %d: %s",
               dev, e != cudaSuccess ? cudaGetErrorString(e) : "null address");
      g_scratch_ptr[dev] = nullptr;
      return CSA2_ECUDA;
    }
    if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;  // the lookup may have made it
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return CSA2_OK;
}

}  // namespace

extern "C" {

csa2_status csa2_index_topk_noalloc(const csa2_bf16* iq, const float* w, int Q, int H,
                                    const csa2_bf16* index_k, int64_t index_rows,
                                    const int64_t* row_base, const int32_t* q_seq,
                                    const int64_t* q_pos, int ratio, const int32_t* cand, int ncb,
                                    int k, int relu, int64_t max_scored, int32_t* sel,
                                    float* sel_scores, float* scores_out, csa2_stream stream) {
  // invalid arguments give 0 here and are reported by csa2_index_topk below
  const size_t need = csa2_index_topk_workspace_size(Q, H, max_scored, k);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "csa2_index_topk_noalloc: Q = %d with max_scored = %lld needs %zu bytes of scratch, "
             "more than the fixed %zu-byte device array; use csa2_index_topk with a workspace",
             Q, (long long)max_scored, need, kScratchBytes);
    csa2::set_last_error(msg);
    return CSA2_ENOSPACE;
  }
  void* p = nullptr;
  char msg[256];
  if (scratch_on_current_device(&p, msg, sizeof(msg)) != CSA2_OK) {
    csa2::set_last_error(msg);
    return CSA2_ECUDA;
  }
  return csa2_index_topk(iq, w, Q, H, index_k, index_rows, row_base, q_seq, q_pos, ratio, cand,
                         ncb, k, relu, max_scored, sel, sel_scores, scores_out, p, kScratchBytes,
                         stream);
}

}  // extern "C"

// k_topk.cu -- exact top-k per row by CTA-level radix select.
// [A] "特殊模块 · indexer" Fig. 3b (top_k_per_row: k = 512, ascending, -1 padded) and
// "visible 是每行自己的前缀长度" (-1 means fewer than k rows were scored).
//
// Scores are handled as order-preserving uint32 keys (score_key); key 0 marks a
// position that was not scored.  For one row segment of n keys cached in shared
// memory the CTA finds the threshold key T of the k-th largest entry with three
// histogram passes (key bits 31..21, 20..10, 9..0), then compacts, in position
// order, every key > T and the first (k - #greater) keys == T.  Ties therefore go
// to the lower position, and the output is ascending.
//
// Rows longer than one chunk are split: every chunk CTA writes its own exact top-k
// (key, position) list, and a merge CTA selects the top-k of the concatenated
// lists.  The true top-k is a subset of the union of the per-chunk top-k sets under
// the same total order (key desc, position asc), so the merge is exact.
#include "common.cuh"

CSA2_DEFINE_FAULT_FLAG(topk)

namespace csa2 {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kChunk = 16384;        // keys per chunk CTA (64 KiB of shared memory)
constexpr int kMaxChunks = 96;       // merge holds kMaxChunks * k keys (<= 192 KiB)

namespace {

struct SelectSmem {
  uint32_t hist[2048];
  int warp_a[kTopkWarps];
  int warp_b[kTopkWarps];
  int found_bin;
  int found_above;
  int keff;
};

// Block-wide: among bins (descending), find the bin where the running count from the
// top crosses `need`.  Writes found_bin and found_above (= count strictly above).
__device__ void find_crossing(SelectSmem& S, int nbins, int need) {
  const int tid = threadIdx.x;
  const int per = nbins / kTopkThreads;  // 4 or 2
  // thread tid owns bins nbins-1-per*tid-j, j = 0..per-1 (descending)
  int local = 0;
  for (int j = 0; j < per; ++j) local += (int)S.hist[nbins - 1 - per * tid - j];
  // exclusive scan of `local` over the block in tid order
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) S.warp_a[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += S.warp_a[w];
  int above = wbase + incl - local;
  for (int j = 0; j < per; ++j) {
    int bin = nbins - 1 - per * tid - j;
    int c = (int)S.hist[bin];
    if (above < need && need <= above + c) {
      S.found_bin = bin;
      S.found_above = above;
    }
    above += c;
  }
  __syncthreads();
}

// Exact top-k of keys[0..n) (shared memory).  Writes the selected positions in
// ascending order to out[0..keff) (shared memory) and returns keff.
__device__ int select_topk(const uint32_t* keys, int n, int k, int* out, SelectSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 2048; i += kTopkThreads) S.hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kTopkThreads) atomicAdd(&S.hist[keys[i] >> 21], 1u);
  __syncthreads();
  const int nvalid = n - (int)S.hist[0];  // only key 0 falls in bin 0
  const int keff = nvalid < k ? nvalid : k;
  if (keff <= 0) return 0;
  // pass 1: bits 31..21
  find_crossing(S, 2048, keff);
  const uint32_t b1 = (uint32_t)S.found_bin;
  int above = S.found_above;
  // pass 2: bits 20..10 among keys in bin b1
  for (int i = tid; i < 2048; i += kTopkThreads) S.hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kTopkThreads) {
    uint32_t kk = keys[i];
    if ((kk >> 21) == b1) atomicAdd(&S.hist[(kk >> 10) & 2047u], 1u);
  }
  __syncthreads();
  find_crossing(S, 2048, keff - above);
  const uint32_t b2 = (uint32_t)S.found_bin;
  above += S.found_above;
  // pass 3: bits 9..0 among keys with prefix (b1, b2)
  for (int i = tid; i < 1024; i += kTopkThreads) S.hist[i] = 0;
  __syncthreads();
  const uint32_t pre = (b1 << 11) | b2;
  for (int i = tid; i < n; i += kTopkThreads) {
    uint32_t kk = keys[i];
    if ((kk >> 10) == pre) atomicAdd(&S.hist[kk & 1023u], 1u);
  }
  __syncthreads();
  find_crossing(S, 1024, keff - above);
  const uint32_t T = (pre << 10) | (uint32_t)S.found_bin;
  above += S.found_above;
  const int need_eq = keff - above;  // >= 1
  // compaction in position order: warp w owns the contiguous segment [w*seg, ...)
  const int seg = ((n + kTopkWarps * 32 - 1) / (kTopkWarps * 32)) * 32;
  const int s0 = warp * seg, s1 = min(n, s0 + seg);
  int n_gt = 0, n_eq = 0;
  for (int i = s0 + lane; i < s1; i += 32) {
    uint32_t kk = keys[i];
    n_gt += kk > T;
    n_eq += kk == T;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n_gt += __shfl_xor_sync(0xFFFFFFFFu, n_gt, o);
    n_eq += __shfl_xor_sync(0xFFFFFFFFu, n_eq, o);
  }
  if (lane == 0) { S.warp_a[warp] = n_gt; S.warp_b[warp] = n_eq; }
  __syncthreads();
  int eq_before = 0, sel_before = 0;
  for (int w = 0; w < warp; ++w) {
    int take = min(max(need_eq - eq_before, 0), S.warp_b[w]);
    sel_before += S.warp_a[w] + take;
    eq_before += S.warp_b[w];
  }
  int take_eq = min(max(need_eq - eq_before, 0), n_eq);
  int off = sel_before;
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = s0; base < s1; base += 32) {
    int i = base + lane;
    uint32_t kk = i < s1 ? keys[i] : 0u;
    uint32_t gt = __ballot_sync(0xFFFFFFFFu, i < s1 && kk > T);
    uint32_t eq = __ballot_sync(0xFFFFFFFFu, i < s1 && kk == T);
    // keep the first take_eq equal keys of the segment
    uint32_t eq_keep = 0;
    if (take_eq > 0) {
      int cnt = __popc(eq);
      if (cnt <= take_eq) eq_keep = eq;
      else {
        uint32_t m = eq;
        for (int r = 0; r < take_eq; ++r) { uint32_t low = m & (~m + 1u); eq_keep |= low; m ^= low; }
      }
      take_eq -= __popc(eq_keep);
    }
    uint32_t selm = gt | eq_keep;
    if (selm & (1u << lane)) out[off + __popc(selm & lt)] = i;
    off += __popc(selm);
  }
  __syncthreads();
  return keff;
}

__device__ __forceinline__ int32_t pos_to_row(const TopkArgs& a, int q, uint32_t pos) {
  if (!a.cand) return (int32_t)pos;
  int32_t blk = a.cand[(int64_t)q * a.ncb + (pos >> 3)];
  return blk * 8 + (int32_t)(pos & 7u);
}

// Final write of one row: positions pos_of(i) for i < keff, then -1.
template <typename PosFn, typename KeyFn>
__device__ void write_row(const TopkArgs& a, int q, int keff, const int* idx, PosFn pos_of,
                          KeyFn key_of) {
  for (int i = threadIdx.x; i < a.k; i += kTopkThreads) {
    int32_t r = -1;
    float s = 0.f;
    if (i < keff) {
      uint32_t p = pos_of(idx[i]);
      r = pos_to_row(a, q, p);
      s = key_score(key_of(idx[i]));
    }
    a.sel[(int64_t)q * a.k + i] = r;
    if (a.sel_scores) a.sel_scores[(int64_t)q * a.k + i] = s;
  }
}

template <bool kFromFloat>
__global__ void __launch_bounds__(kTopkThreads) topk_chunk_kernel(TopkArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw);
  int* out = reinterpret_cast<int*>(keys + kChunk);
  SelectSmem& S = *reinterpret_cast<SelectSmem*>(out + kMaxK);
  const int q = blockIdx.y, c = blockIdx.x;
  int n = a.n[q];
  if (n > a.ld) { if (threadIdx.x == 0) raise_fault(kFaultBounds); n = (int)a.ld; }
  const int begin = c * kChunk;
  const int len = max(0, min(kChunk, n - begin));
  const int64_t rowoff = (int64_t)q * a.ld + begin;
  for (int i = threadIdx.x; i < len; i += kTopkThreads)
    keys[i] = kFromFloat ? score_key(a.scores[rowoff + i]) : a.keys[rowoff + i];
  __syncthreads();
  const int keff = select_topk(keys, len, a.k, out, S);
  if (a.nchunk == 1) {
    write_row(a, q, keff, out, [&](int i) { return (uint32_t)(begin + i); },
              [&](int i) { return keys[i]; });
  } else {
    uint64_t* part = a.part + ((int64_t)q * a.nchunk + c) * a.k;
    for (int i = threadIdx.x; i < a.k; i += kTopkThreads) {
      uint64_t v = 0;
      if (i < keff) v = ((uint64_t)keys[out[i]] << 32) | (uint32_t)(begin + out[i]);
      part[i] = v;
    }
  }
}

__global__ void __launch_bounds__(kTopkThreads) topk_merge_kernel(TopkArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int ncand = a.nchunk * a.k;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw);
  int* out = reinterpret_cast<int*>(keys + ncand);
  SelectSmem& S = *reinterpret_cast<SelectSmem*>(out + kMaxK);
  const int q = blockIdx.x;
  const uint64_t* part = a.part + (int64_t)q * ncand;
  for (int i = threadIdx.x; i < ncand; i += kTopkThreads) keys[i] = (uint32_t)(part[i] >> 32);
  __syncthreads();
  // candidates are in chunk order and ascending within a chunk: index order is
  // position order, so the select's tie rule stays "lower position".
  const int keff = select_topk(keys, ncand, a.k, out, S);
  write_row(a, q, keff, out, [&](int i) { return (uint32_t)(part[i] & 0xFFFFFFFFu); },
            [&](int i) { return keys[i]; });
}

}  // namespace

int topk_num_chunks(int64_t ld) { return (int)((ld + kChunk - 1) / kChunk); }
int topk_max_chunks() { return kMaxChunks; }

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  if (a.Q == 0) return cudaSuccess;
  const size_t sel_smem = sizeof(SelectSmem) + kMaxK * sizeof(int);
  const size_t smem1 = (size_t)kChunk * 4 + sel_smem;
  dim3 grid(a.nchunk, a.Q);
  cudaError_t e;
  if (a.scores) {
    e = cudaFuncSetAttribute(topk_chunk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem1);
    if (e != cudaSuccess) return e;
    topk_chunk_kernel<true><<<grid, kTopkThreads, smem1, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(topk_chunk_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    if (e != cudaSuccess) return e;
    topk_chunk_kernel<false><<<grid, kTopkThreads, smem1, s>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || a.nchunk == 1) return e;
  const size_t smem2 = (size_t)a.nchunk * a.k * 4 + sel_smem;
  e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem2);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<a.Q, kTopkThreads, smem2, s>>>(a);
  return cudaGetLastError();
}

}  // namespace csa2

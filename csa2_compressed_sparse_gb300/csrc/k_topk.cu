// k_topk.cu -- exact top-k per row.
// [A] "特殊模块 · indexer" Fig. 3b (top_k_per_row: k = 512, ascending, -1 padded) and
// "visible 是每行自己的前缀长度" (-1 means fewer than k rows were scored).
//
// Scores are handled as order-preserving uint32 keys (score_key); key 0 marks a
// position that was not scored.  One CTA selects from a row segment of up to 32768
// positions:
//   1. sample: the segment is staged in shared memory by one bulk copy (a TMA copy has
//      the whole row in flight at once); meanwhile a histogram of the top 11 key bits
//      over an even sample of 2048 keys, read from global memory, gives a threshold bin
//      expected to hold about 2k + 64 (refined by the next 11 bits when the sample
//      crowds into that bin);
//   2. filter: one pass keeps the (key, position) pairs at or above the threshold (a
//      few times k of them); only a segment that kept fewer than k counts its scored
//      positions;
//   3. select: three histogram passes (key bits 31..21, 20..10, 9..0) over the kept
//      pairs give the k-th largest key T and how many keys equal to T are needed;
//   4. output: winners are marked in a position bitmap (keys > T; the lowest
//      positions among keys == T), which is scanned in order, so ties go to the lower
//      position and the output is ascending.
// If the sample misleads (fewer than k kept, or more than the buffer holds), steps 3
// and 4 run over the whole segment instead; the result is the same.
//
// A row of 32769..65536 positions (a prefill chunk's rows) runs on one CTA as well, with
// the same steps reading the row straight from global memory (the segment would not fit
// in shared memory; the filter keeps four 16-byte loads in flight per thread).
// Longer rows are split into chunks of 32768: every chunk CTA writes its exact top-k
// (key, position) list, and the chunk CTA that finishes last (a per-row arrival
// counter) selects the top-k of the concatenated lists.  The true top-k is a subset of
// the union of the per-chunk top-k sets under the same total order (key desc,
// position asc), so the merge is exact.
//
// Block mode (the candidate pool of a FULL layer, [A] Fig. 3b second stage): the items
// are blocks of 8 positions.  Each chunk CTA builds its blocks' keys from the row's
// position keys (the largest key of the block; the newest block pinned to ~0, above
// every score key, +inf included) in shared memory and selects among them in the same
// way; the output holds block ids.  It runs in the same launch as the row selection, on
// CTAs of its own.
#include "common.cuh"
#include "compress_dev.cuh"

CSA2_DEFINE_FAULT_FLAG(topk)

namespace csa2 {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kChunkLen = 32768;   // positions per CTA
constexpr int kMaxChunks = 48;     // chunks per row; the merge holds chunks * k <= kChunkLen pairs
constexpr int kCandCap = 8192;     // kept (key, index) pairs
constexpr int kWarpCap = kCandCap / (kTopkThreads / 32);  // per-warp region
constexpr int kLongLen = 65536;    // a row of up to this many positions: one CTA reading it
                                   // straight from global memory (no staging, no merge)
constexpr int kLongWords = kLongLen / 32;
constexpr int kSample = 2048;      // keys sampled for the threshold

namespace {

struct SelectSmem {
  uint32_t row[kChunkLen + 4];  // the segment's keys (shifted so its aligned part is)
  uint32_t hist[2048];
  uint32_t hist_kept[2048];  // top 11 key bits of the kept pairs (the first radix pass)
  uint32_t ckey[kCandCap];
  uint32_t cidx[kCandCap];
  uint32_t selmap[kLongWords];  // positions with key > T
  uint32_t eqmap[kLongWords];   // positions with key == T
  int wcnt[kTopkThreads / 32];  // kept pairs per warp region
  int ncand;
  int nvalid;
  int warp_a[kTopkWarps];
  int warp_b[kTopkWarps];
  int found_bin;
  int found_above;
  int last;
  uint64_t bar;  // bulk copy of the segment
};

// Block-wide: among bins of `hist` (descending), find the bin where the running count
// from the top crosses `need`.  Writes found_bin and found_above (= count strictly
// above).  If the total is below `need`, found_bin is 0 and found_above the total.
__device__ void find_crossing(SelectSmem& S, const uint32_t* hist, int nbins, int need) {
  const int tid = threadIdx.x;
  const int per = nbins / kTopkThreads;  // 2 or 1
  int local = 0;
  for (int j = 0; j < per; ++j) local += (int)hist[nbins - 1 - per * tid - j];
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (tid == 0) { S.found_bin = 0; S.found_above = 0; }
  if (lane == 31) S.warp_a[warp] = incl;
  __syncthreads();
  // every warp scans the warp totals itself
  const int wt = lane < kTopkWarps ? S.warp_a[lane] : 0;
  int wi = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xFFFFFFFFu, wi, o);
    if (lane >= o) wi += v;
  }
  const int wbase = __shfl_sync(0xFFFFFFFFu, wi - wt, warp);
  const int total = __shfl_sync(0xFFFFFFFFu, wi, 31);
  int above = wbase + incl - local;
  for (int j = 0; j < per; ++j) {
    int bin = nbins - 1 - per * tid - j;
    int c = (int)hist[bin];
    if (above < need && need <= above + c) {
      S.found_bin = bin;
      S.found_above = above;
    }
    above += c;
  }
  if (tid == 0 && total < need) S.found_above = total;
  __syncthreads();
}

// Warp-aggregated histogram increment: lanes with the same bin add once.  Called by
// all 32 lanes of a warp together; lanes with valid == false add nothing.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool valid) {
  const uint32_t m = __match_any_sync(0xFFFFFFFFu, valid ? bin : 0xFFFFFFFFu);
  const int lane = threadIdx.x & 31;
  if (valid && lane == __ffs(m) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(m));
}

__device__ __forceinline__ void clear_hist(SelectSmem& S, int nbins) {
  for (int i = threadIdx.x; i < nbins; i += kTopkThreads) S.hist[i] = 0;
}

// Keys of a row segment: workspace keys or raw fp32 scores in global memory, or keys
// staged in shared memory (the select always runs on the staged copy).
enum SrcKind { kSrcKeys = 0, kSrcScores = 1, kSrcSmem = 3 };

template <int kKind>
struct RowSrc {
  const void* base;
  bool aligned;  // 16-byte aligned base
  __device__ __forceinline__ uint32_t operator()(int i) const {
    if (kKind == kSrcSmem) return static_cast<const uint32_t*>(base)[i];
    if (kKind == kSrcScores) return score_key(__ldcg(static_cast<const float*>(base) + i));
    return __ldcg(static_cast<const uint32_t*>(base) + i);
  }
  // keys 4g .. 4g+3 (0 past n), with 16-byte loads when aligned
  __device__ __forceinline__ uint4 load4(int g, int n) const {
    const int i = 4 * g;
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (i >= n) return r;
    if (aligned && i + 4 <= n) {
      if (kKind == kSrcSmem)
        return *reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(base) + i);
      r = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint32_t*>(base) + i));
      if (kKind == kSrcScores)
        r = make_uint4(score_key(__uint_as_float(r.x)), score_key(__uint_as_float(r.y)),
                       score_key(__uint_as_float(r.z)), score_key(__uint_as_float(r.w)));
      return r;
    }
    r.x = (*this)(i);
    if (i + 1 < n) r.y = (*this)(i + 1);
    if (i + 2 < n) r.z = (*this)(i + 2);
    if (i + 3 < n) r.w = (*this)(i + 3);
    return r;
  }
};

// The select's counters, histograms and position bitmaps (nw words) set to zero; the
// caller makes them visible with a barrier.
__device__ __forceinline__ void clear_select(SelectSmem& S, int nw) {
  const int tid = threadIdx.x;
  clear_hist(S, 2048);
  for (int i = tid; i < 2048; i += kTopkThreads) S.hist_kept[i] = 0;
  if (tid == 0) { S.ncand = 0; S.nvalid = 0; }
  if (tid < kTopkWarps) S.wcnt[tid] = 0;
  for (int w = tid; w < nw; w += kTopkThreads) { S.selmap[w] = 0; S.eqmap[w] = 0; }
}

// Where the threshold's sample is read: the staged keys, or the row in global memory
// (keys, or raw scores converted on load) while its staged copy lands.
struct SampleSrc {
  const uint32_t* s;
  const uint32_t* gk;
  const float* gs;
  __device__ __forceinline__ uint32_t operator()(int i) const {
    if (s) return s[i];
    if (gs) return score_key(__ldcg(gs + i));
    return __ldcg(gk + i);
  }
};

// Exact top-k of src[0..n): emit(o, i) is called once for each selected index i, with
// o = its place in ascending order (0 .. keff - 1), by some thread of the CTA.  Returns
// keff = min(k, #scored).  dense: every key of src[0..n) is nonzero.  src is the staged
// copy in shared memory (n <= kChunkLen) or the row in global memory (n <= kLongLen).
// The threshold's sample is read from ssrc (the same keys: the staged copy, or the row
// in global memory while its copy lands); ready() is called by every thread, followed by
// a barrier, before src is first read (it waits for the staged copy).
template <int kSrc, typename Ready, typename Emit>
__device__ int select_topk(const RowSrc<kSrc>& src, const SampleSrc& ssrc, int n, int k,
                           bool dense, SelectSmem& S, bool precleared, Ready ready, Emit emit) {
  constexpr bool kStaged = kSrc == kSrcSmem;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = (n + 31) >> 5;
  // ---- 1. clear (done by the caller, before its dependency wait, when precleared) ----
  // thread (warp w, lane l) handles the 4-key groups w * 32 + l + u * kTopkThreads,
  // u < kU (n <= kChunkLen staged, kLongLen from global memory)
  constexpr int kU = (kStaged ? kChunkLen : kLongLen) / (4 * kTopkThreads);
  static_assert(kU <= 32, "one bit per group step");
  if (!precleared) {
    clear_select(S, nw);
    __syncthreads();
  }
  // ---- 2. threshold from an even sample of 2048 keys ----
  const int ns = n < kSample ? n : kSample;
  // sample s2 reads key (2 s2 + 1) n / (2 ns): s2 itself when the segment is no longer
  // than the sample, else a shift (2 ns = 4096; (2 s2 + 1) n < 2^32 for n <= kLongLen)
  static_assert(2 * kSample == 4096 && (uint64_t)(2 * kSample) * kLongLen < (1ull << 32),
                "sample index");
  auto sample_at = [&](int s2) {
    return ns == n ? s2 : (int)(((uint32_t)(2 * s2 + 1) * (uint32_t)n) >> 12);
  };
  // each thread's samples tid + j * kTopkThreads: all loads in flight before the first
  // use, and kept in registers for the refinement below (no second read of the row)
  static_assert(kSample % kTopkThreads == 0, "samples per thread");
  constexpr int kSampPer = kSample / kTopkThreads;
  uint32_t skey[kSampPer];
#pragma unroll
  for (int j = 0; j < kSampPer; ++j) {
    const int s2 = tid + j * kTopkThreads;
    skey[j] = s2 < ns ? ssrc(sample_at(s2)) : 0u;
  }
#pragma unroll
  for (int j = 0; j < kSampPer; ++j)
    if (skey[j]) atomicAdd(&S.hist[skey[j] >> 21], 1u);
  __syncthreads();
  // sample keys wanted above the threshold: about (2k + 64) / n of the sample
  const int want = (int)(((uint32_t)(2 * k + 64) * (uint32_t)ns + n - 1) / (uint32_t)(n > 0 ? n : 1));
  find_crossing(S, S.hist, 2048, want);
  uint32_t thr = want >= ns ? 1u : max((uint32_t)S.found_bin << 21, 1u);
  if (want < ns) {
    // A crowded threshold bin (keys bunched in one quarter octave, as block maxima
    // are) would keep far more than the buffer holds: refine it by the sample's next
    // 11 key bits.
    const uint32_t bin = (uint32_t)S.found_bin;
    const int above = S.found_above;
    if (above + (int)S.hist[bin] > 2 * want + 64) {
      __syncthreads();  // every thread has read hist[bin]
      clear_hist(S, 2048);
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kSampPer; ++j)
        if (skey[j] && (skey[j] >> 21) == bin) atomicAdd(&S.hist[(skey[j] >> 10) & 2047u], 1u);
      __syncthreads();
      find_crossing(S, S.hist, 2048, want - above);
      thr = max((bin << 21) | ((uint32_t)S.found_bin << 10), 1u);
    }
  }
  ready();  // the staged copy of the segment has landed
  // keys past n up to whole 4096-key steps of the filter read as unscored (0), so the
  // filter's loads need no bounds (nu * 4096 <= kChunkLen: inside the staging buffer);
  // loads from global memory are bounded at n instead
  const int nu = (n + 4 * kTopkThreads - 1) / (4 * kTopkThreads);  // <= kU, CTA-uniform
  if constexpr (kStaged) {
    uint32_t* rb = const_cast<uint32_t*>(static_cast<const uint32_t*>(src.base));
    for (int i = n + tid; i < nu * 4 * kTopkThreads; i += kTopkThreads) rb[i] = 0u;
  }
  __syncthreads();  // ... for every thread; and every thread has read the sample's histogram
  // ---- 3. filter: keep keys >= thr, count scored positions ----
  // Warp w's lanes take the 4-key groups w * 32 + lane + u * kTopkThreads.  First pass:
  // each lane counts its kept keys (and which of its groups hold one); one warp-wide
  // exclusive sum gives each lane its first slot in the warp's region [w * kWarpCap, ...),
  // so no atomic is needed for the slots; the second pass re-reads only the groups that
  // hold kept keys and stores them.  A dense segment (every position scored) needs no
  // count.  The sample's histogram is cleared here for the radix passes.
  clear_hist(S, 2048);
  uint32_t* wkey = S.ckey + warp * kWarpCap;
  uint32_t* widx = S.cidx + warp * kWarpCap;
  int mine = 0;
  uint32_t hit = 0;  // bit u: group u holds a kept key (thr >= 1: never an unscored one)
  auto count = [&](const uint4& vv, int u) {
    const int cnt = (vv.x >= thr) + (vv.y >= thr) + (vv.z >= thr) + (vv.w >= thr);
    mine += cnt;
    hit |= (cnt ? 1u : 0u) << u;
  };
  if constexpr (!kStaged) {  // from global memory: four 16-byte loads in flight, bounded
#pragma unroll
    for (int u0 = 0; u0 < kU; u0 += 4) {
      if (u0 < nu) {
        uint4 vv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          vv[j] = u0 + j < nu ? src.load4(warp * 32 + (u0 + j) * kTopkThreads + lane, n)
                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) count(vv[j], u0 + j);
      }
    }
  } else if (src.aligned) {  // plain 16-byte shared loads, four in flight
    const uint32_t gaddr = smem_u32(src.base) + 16u * (uint32_t)(warp * 32 + lane);
#pragma unroll
    for (int u0 = 0; u0 < kU; u0 += 4) {
      if (u0 < nu) {
        uint4 vv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          vv[j] = u0 + j < nu ? ld_shared16(gaddr + 16u * kTopkThreads * (uint32_t)(u0 + j))
                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) count(vv[j], u0 + j);
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (u < nu) count(src.load4(warp * 32 + u * kTopkThreads + lane, n), u);
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  const int wpos = __shfl_sync(0xFFFFFFFFu, incl, 31);
  int slot = incl - mine;
  while (hit) {
    const int u = __ffs(hit) - 1;
    hit &= hit - 1u;
    const int g = warp * 32 + u * kTopkThreads + lane;
    const uint4 vv = src.load4(g, n);
    const uint32_t kk[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (kk[jj] >= thr) {
        if (slot < kWarpCap) { wkey[slot] = kk[jj]; widx[slot] = (uint32_t)(4 * g + jj); }
        ++slot;
      }
    }
  }
  if (lane == 0) S.wcnt[warp] = wpos;
  if (lane == 0) atomicAdd(&S.ncand, wpos > kWarpCap ? kCandCap + 1 : wpos);  // full: no fast path
  __syncthreads();
  const int nc = S.ncand;
  // keff = min(k, #scored): a dense segment has n scored positions; otherwise, with at
  // least k kept keys (all scored), keff = k, and only a segment that kept fewer needs
  // its scored positions counted
  int nvalid = dense ? n : nc;
  if (!dense && nc < k) {
    int nv = 0;
    for (int i = tid; i < n; i += kTopkThreads) nv += src(i) != 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xFFFFFFFFu, nv, o);
    if (lane == 0) atomicAdd(&S.nvalid, nv);
    __syncthreads();
    nvalid = S.nvalid;
  }
  const int keff = nvalid < k ? nvalid : k;
  if (keff <= 0) return 0;
  const bool fast = nc >= keff && nc <= kCandCap;  // the kept pairs hold the top-k
  // ---- 4. radix select over the kept pairs (or the whole segment) ----
  // fn(key, valid) is called by the 32 lanes of a warp together (warp-uniform loops).
  const int my_cnt = S.wcnt[warp];
  auto for_keys = [&](auto&& fn) {
    if (fast) {  // each warp walks its own region
      for (int j0 = 0; j0 < my_cnt; j0 += 32) {
        const int jx = j0 + lane;
        const bool ok = jx < my_cnt;
        fn(ok ? wkey[jx] : 0u, ok);
      }
    } else {
      for (int i0 = warp * 32; i0 < n; i0 += kTopkThreads) {
        const int ix = i0 + lane;
        const bool ok = ix < n;
        fn(ok ? src(ix) : 0u, ok);
      }
    }
  };
  // Pass 1 (key bits 31..21) counts the kept pairs into hist_kept (clear since the start),
  // or the whole segment's keys into hist (cleared by the filter).  Pass 2 counts into the
  // other histogram, pass 3 into pass 1's again, cleared while pass 2 runs (its crossing
  // has been read: find_crossing ends with a barrier).  Passes 1 and 2 over the kept pairs
  // and pass 3 count with plain atomics (few keys per bin).
  uint32_t* h1 = fast ? S.hist_kept : S.hist;
  uint32_t* h2 = fast ? S.hist : S.hist_kept;
  if (fast) {
    for_keys([&](uint32_t key, bool ok) {
      if (ok && key != 0u) atomicAdd(&h1[key >> 21], 1u);
    });
  } else {  // hist_kept (clear since the start) is pass 2's
    for_keys([&](uint32_t key, bool ok) { hist_add(h1, key >> 21, ok && key != 0u); });
  }
  __syncthreads();
  find_crossing(S, h1, 2048, keff);
  const uint32_t b1 = (uint32_t)S.found_bin;
  int above = S.found_above;
  uint32_t* h3 = h1;
  for (int i = threadIdx.x; i < 1024; i += kTopkThreads) h3[i] = 0;
  for_keys([&](uint32_t key, bool ok) {
    if (ok && key != 0u && (key >> 21) == b1) atomicAdd(&h2[(key >> 10) & 2047u], 1u);
  });
  __syncthreads();
  find_crossing(S, h2, 2048, keff - above);
  const uint32_t pre = (b1 << 11) | (uint32_t)S.found_bin;
  above += S.found_above;
  for_keys([&](uint32_t key, bool ok) {
    if (ok && key != 0u && (key >> 10) == pre) atomicAdd(&h3[key & 1023u], 1u);
  });
  __syncthreads();
  find_crossing(S, h3, 1024, keff - above);
  const uint32_t T = (pre << 10) | (uint32_t)S.found_bin;
  above += S.found_above;
  const int need_eq = keff - above;  // >= 1
  // ---- 5. mark winners by position, then scan the bitmaps in order ----
  if (fast) {
    for (int j = lane; j < my_cnt; j += 32) {
      const uint32_t key = wkey[j], idx = widx[j];
      if (key > T) atomicOr(&S.selmap[idx >> 5], 1u << (idx & 31));
      else if (key == T) atomicOr(&S.eqmap[idx >> 5], 1u << (idx & 31));
    }
  } else {
    for (int i0 = warp * 32; i0 < nw * 32; i0 += kTopkThreads) {  // one word per warp step
      const int i = i0 + lane;
      const uint32_t key = i < n ? src(i) : 0u;
      const uint32_t gt = __ballot_sync(0xFFFFFFFFu, key && key > T);
      const uint32_t eq = __ballot_sync(0xFFFFFFFFu, key && key == T);
      if (lane == 0) { S.selmap[i0 >> 5] = gt; S.eqmap[i0 >> 5] = eq; }
    }
  }
  __syncthreads();
  // thread t owns words [t*wpt, (t+1)*wpt); equal keys are taken in position order
  const int wpt = (nw + kTopkThreads - 1) / kTopkThreads;
  const int w0 = tid * wpt, w1 = min(nw, w0 + wpt);
  int c_eq = 0, c_gt = 0;
  for (int w = w0; w < w1; ++w) { c_eq += __popc(S.eqmap[w]); c_gt += __popc(S.selmap[w]); }
  // one block-wide scan of both counts: winners before this thread's words are the
  // keys > T before them plus the first need_eq keys == T, min(need_eq, eq_before)
  int eq_incl = c_eq, gt_incl = c_gt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ve = __shfl_up_sync(0xFFFFFFFFu, eq_incl, o);
    const int vg = __shfl_up_sync(0xFFFFFFFFu, gt_incl, o);
    if (lane >= o) { eq_incl += ve; gt_incl += vg; }
  }
  if (lane == 31) { S.warp_a[warp] = eq_incl; S.warp_b[warp] = gt_incl; }
  __syncthreads();
  const int we = lane < kTopkWarps ? S.warp_a[lane] : 0;
  const int wg = lane < kTopkWarps ? S.warp_b[lane] : 0;
  int we_incl = we, wg_incl = wg;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ve = __shfl_up_sync(0xFFFFFFFFu, we_incl, o);
    const int vg = __shfl_up_sync(0xFFFFFFFFu, wg_incl, o);
    if (lane >= o) { we_incl += ve; wg_incl += vg; }
  }
  const int eq_before = __shfl_sync(0xFFFFFFFFu, we_incl - we, warp) + eq_incl - c_eq;
  const int gt_before = __shfl_sync(0xFFFFFFFFu, wg_incl - wg, warp) + gt_incl - c_gt;
  int take_eq = min(max(need_eq - eq_before, 0), c_eq);
  int o = gt_before + min(need_eq, eq_before);
  for (int w = w0; w < w1; ++w) {
    uint32_t bits = S.selmap[w];
    uint32_t eqb = S.eqmap[w];
    while (take_eq > 0 && eqb) {  // lowest positions first
      const uint32_t low = eqb & (~eqb + 1u);
      bits |= low;
      eqb ^= low;
      --take_eq;
    }
    while (bits) {
      const int b = __ffs(bits) - 1;
      emit(o++, w * 32 + b);
      bits &= bits - 1u;
    }
  }
  __syncthreads();
  return keff;
}

// ccache: the row's candidate block ids in shared memory, or null (read from global).
__device__ __forceinline__ int32_t pos_to_row(const TopkArgs& a, int q, uint32_t pos,
                                              const int32_t* ccache = nullptr) {
  if (!a.cand) return (int32_t)pos;
  int32_t blk = ccache ? ccache[pos >> 3] : a.cand[(int64_t)q * a.ncb + (pos >> 3)];
  return blk * 8 + (int32_t)(pos & 7u);
}

// Entries keff .. k - 1 of row q: -1 (score 0).
__device__ void pad_row(const TopkArgs& a, int q, int keff) {
  for (int i = keff + (int)threadIdx.x; i < a.k; i += kTopkThreads) {
    a.sel[(int64_t)q * a.k + i] = -1;
    if (a.sel_scores) a.sel_scores[(int64_t)q * a.k + i] = 0.f;
  }
}

// Chunk blockIdx.x of row blockIdx.y of the selection described by `a`.
template <int kKind>
__device__ __forceinline__ void topk_row(const TopkArgs& a, int c) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelectSmem& S = *reinterpret_cast<SelectSmem*>(smem_raw);
  const int q = blockIdx.y;
  if (!a.blocks && threadIdx.x == 0) {  // the staging copy's barrier (shared memory only)
    mbar_init(smem_u32(&S.bar), 1);
    mbar_fence_init();
  }
  // the select's state, for a segment of up to kLongLen items (shared memory only, so
  // before the wait; a barrier below makes it visible)
  clear_select(S, kLongWords);
  // positions of this row: from the query's position when the call gives it (a call
  // input, read before the dependency wait), else from the count array
  int n;
  if (a.q_pos) {
    const int64_t p1 = a.q_pos[q] + 1;  // ratio 1 or 2
    const int64_t v = a.cand ? (int64_t)a.ncb * 8 : (a.ratio == 2 ? p1 >> 1 : p1);
    n = (int)(v < a.ld ? v : a.ld);
    griddep_wait();
  } else {
    griddep_wait();
    n = a.n[q];
  }
  if (n > a.ld) { if (threadIdx.x == 0) raise_fault(kFaultBounds); n = (int)a.ld; }
  const int items = a.blocks ? (n + 7) >> 3 : n;  // positions, or blocks of 8 positions
  const int begin = c * a.chunk;
  const int len = max(0, min(a.chunk, items - begin));
  const int tid = threadIdx.x;
  int32_t* sel_q = a.sel + (int64_t)q * a.k;
  float* sc_q = a.sel_scores ? a.sel_scores + (int64_t)q * a.k : nullptr;
  if (!a.blocks && len > kChunkLen) {
    // A whole row of up to kLongLen positions (one chunk) on one CTA, read straight from
    // global memory: no staging copy (it would not fit) and no merge of two chunk lists.
    const int64_t rowoff = (int64_t)q * a.ld;
    const bool dense_g = a.cand == nullptr;
    __syncthreads();  // the cleared select state is visible
    int keff;
    if constexpr (kKind == kSrcScores) {
      const float* g = a.scores + rowoff;
      const RowSrc<kSrcScores> gsrc{g, (reinterpret_cast<uintptr_t>(g) & 15u) == 0};
      keff = select_topk(gsrc, SampleSrc{nullptr, nullptr, g}, len, a.k, dense_g, S, true,
                         [] {}, [&](int o, int i) {
                           sel_q[o] = pos_to_row(a, q, (uint32_t)i);
                           if (sc_q) sc_q[o] = key_score(gsrc(i));
                         });
    } else {
      const uint32_t* g = a.keys + rowoff;
      const RowSrc<kSrcKeys> gsrc{g, (reinterpret_cast<uintptr_t>(g) & 15u) == 0};
      keff = select_topk(gsrc, SampleSrc{nullptr, g, nullptr}, len, a.k, dense_g, S, true,
                         [] {}, [&](int o, int i) {
                           sel_q[o] = pos_to_row(a, q, (uint32_t)i);
                           if (sc_q) sc_q[o] = key_score(gsrc(i));
                         });
    }
    pad_row(a, q, keff);
    return;
  }
  uint32_t* rowbuf = S.row;
  int pad = 0, head = 0, body = 0;
  SampleSrc ssrc{nullptr, nullptr, nullptr};
  if (a.blocks) {
    // Block keys of this chunk straight from the row's position keys (8 keys = two
    // 16-byte loads per block; rows start 16-byte aligned): the largest key of the
    // block's positions < n, the newest block pinned above every key.
    // Four blocks per thread and step, all loads in flight before the first use.
    const uint32_t* g = a.keys + (int64_t)q * a.ld;
    constexpr int kU = 4;
    for (int j0 = tid; j0 < len; j0 += kU * kTopkThreads) {
      uint4 x[kU], y[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u * kTopkThreads;
        const int p0 = 8 * (begin + j);
        x[u] = y[u] = make_uint4(0u, 0u, 0u, 0u);
        if (j < len && p0 + 8 <= n) {
          x[u] = __ldcg(reinterpret_cast<const uint4*>(g + p0));
          y[u] = __ldcg(reinterpret_cast<const uint4*>(g + p0 + 4));
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u * kTopkThreads;
        if (j >= len) break;
        const int b = begin + j;
        // only the newest block can be partial, and it is pinned
        const uint32_t m = max(max(max(x[u].x, x[u].y), max(x[u].z, x[u].w)),
                               max(max(y[u].x, y[u].y), max(y[u].z, y[u].w)));
        rowbuf[j] = b == items - 1 ? 0xFFFFFFFFu : m;
      }
    }
  } else {
    // The segment into shared memory: one bulk copy of its 16-byte aligned interior (a
    // TMA copy has the whole row in flight at once), the ragged ends (at most 3 keys
    // each) by plain loads; scores become keys in place.
    const int64_t rowoff = (int64_t)q * a.ld + begin;
    const uint32_t* g = kKind == kSrcScores
                            ? reinterpret_cast<const uint32_t*>(a.scores + rowoff)
                            : a.keys + rowoff;
    head = (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(g) & 15u)) & 15u) >> 2);
    head = min(head, len);
    body = ((len - head) >> 2) << 2;
    if (kKind == kSrcScores) ssrc.gs = a.scores + rowoff;
    else ssrc.gk = g;
    pad = (4 - head) & 3;  // row[pad + head] is 16-byte aligned
    rowbuf = S.row + pad;
    __syncthreads();  // the barrier's initialisation is visible
    if (tid == 0 && body > 0) {
      mbar_arrive_expect_tx(smem_u32(&S.bar), (uint32_t)body * 4u);
      bulk_copy_g2s(smem_u32(rowbuf + head), g + head, (uint32_t)body * 4u, smem_u32(&S.bar));
    }
    // the copy (and the ragged ends, in ready()) are waited for inside the select, after
    // the threshold's sample, which reads the row from global memory meanwhile
  }
  __syncthreads();
  RowSrc<kSrcSmem> src{rowbuf, pad == 0};
  if (a.blocks) ssrc.s = rowbuf;  // block keys exist only in shared memory
  auto ready = [&]() {
    if (a.blocks) return;
    const int64_t rowoff = (int64_t)q * a.ld + begin;
    const uint32_t* g = kKind == kSrcScores
                            ? reinterpret_cast<const uint32_t*>(a.scores + rowoff)
                            : a.keys + rowoff;
    if (tid < head) rowbuf[tid] = __ldcg(g + tid);
    if (head + body + tid < len) rowbuf[head + body + tid] = __ldcg(g + head + body + tid);
    if (body > 0) mbar_wait(smem_u32(&S.bar), 0);
    if (kKind == kSrcScores) {
      __syncthreads();
      for (int i = tid; i < len; i += kTopkThreads)
        rowbuf[i] = score_key(__uint_as_float(rowbuf[i]));
    }
  };
  // every position below n is scored unless the row maps candidate blocks (REINDEX);
  // every block below the row's count has a key
  const bool dense = a.blocks || a.cand == nullptr;
  if (a.nchunk == 1) {
    // REINDEX: the row's candidate block ids (up to two per thread) are loaded now (after
    // the wait: a preceding call may have written them) and stored, once the threshold is
    // known, at the free end of the staging buffer, so the ordered output maps positions
    // to rows from shared memory
    const int nu_end = pad + ((len + 4 * kTopkThreads - 1) / (4 * kTopkThreads)) * 4 * kTopkThreads;
    const bool cache = a.cand && !a.blocks && a.ncb <= 2 * kTopkThreads &&
                       nu_end + a.ncb <= kChunkLen + 4;
    int32_t* cc = reinterpret_cast<int32_t*>(S.row + (kChunkLen + 4 - a.ncb));
    int32_t cv0 = 0, cv1 = 0;
    if (cache) {
      const int32_t* cg = a.cand + (int64_t)q * a.ncb;
      if (tid < a.ncb) cv0 = __ldg(cg + tid);
      if (tid + kTopkThreads < a.ncb) cv1 = __ldg(cg + tid + kTopkThreads);
    }
    auto ready_c = [&]() {
      ready();
      if (cache) {
        if (tid < a.ncb) cc[tid] = cv0;
        if (tid + kTopkThreads < a.ncb) cc[tid + kTopkThreads] = cv1;
      }
    };
    const int32_t* ccache = cache ? cc : nullptr;  // read after the select's barriers
    const int keff = select_topk(src, ssrc, len, a.k, dense, S, true, ready_c, [&](int o, int i) {
      sel_q[o] = pos_to_row(a, q, (uint32_t)(begin + i), ccache);
      if (sc_q) sc_q[o] = key_score(src(i));
    });
    pad_row(a, q, keff);
    return;
  }
  // partial list of this chunk, then the last chunk CTA of the row merges
  uint64_t* part = a.part + ((int64_t)q * a.nchunk + c) * a.k;
  const int keff = select_topk(src, ssrc, len, a.k, dense, S, true, ready, [&](int o, int i) {
    part[o] = ((uint64_t)src(i) << 32) | (uint32_t)(begin + i);
  });
  for (int i = keff + (int)threadIdx.x; i < a.k; i += kTopkThreads) part[i] = 0;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) S.last = atomicAdd(&a.count[q], 1) == a.nchunk - 1;
  __syncthreads();
  if (!S.last) return;
  __threadfence();
  // candidates are in chunk order and ascending within a chunk: index order is
  // position order, so the select's tie rule stays "lower position".
  // The lists' keys go to shared memory (the segment's buffer is free again: the
  // select reads them several times); positions are fetched for the winners only.
  const int ncand = a.nchunk * a.k;  // <= kChunkLen
  const uint64_t* row = a.part + (int64_t)q * ncand;
  uint32_t* mk = S.row;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    const uint4* r4 = reinterpret_cast<const uint4*>(row);
    const int npair2 = ncand >> 1;
    constexpr int kU = 4;
    for (int i0 = tid; i0 < npair2; i0 += kU * kTopkThreads) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kTopkThreads;
        v[u] = i < npair2 ? __ldcg(r4 + i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kTopkThreads;
        if (i < npair2) { mk[2 * i] = v[u].y; mk[2 * i + 1] = v[u].w; }
      }
    }
    if ((ncand & 1) && tid == 0) mk[ncand - 1] = (uint32_t)(__ldcg(row + ncand - 1) >> 32);
  } else {
    for (int i = tid; i < ncand; i += kTopkThreads) mk[i] = (uint32_t)(__ldcg(row + i) >> 32);
  }
  __syncthreads();
  RowSrc<kSrcSmem> msrc{mk, true};
  const SampleSrc mss{mk, nullptr, nullptr};
  const int keff2 = select_topk(msrc, mss, ncand, a.k, false, S, false, [] {}, [&](int o, int i) {
    sel_q[o] = pos_to_row(a, q, (uint32_t)(__ldcg(row + i) & 0xFFFFFFFFu));
    if (sc_q) sc_q[o] = key_score(mk[i]);
  });
  pad_row(a, q, keff2);
  if (threadIdx.x == 0) a.count[q] = 0;  // ready for the next call
}

// The compressor's tokens on CTA `cta` of the compressor rows of a top-k launch
// (csa2_compress_index_topk): warp w takes token cta * 32 + w, with the same per-token
// work as the compressor kernel (compress_dev.cuh).  The compressor writes only the main
// plane and its states, which no selection reads, so these CTAs run beside the selection
// CTAs on SMs the selection leaves idle.  Kept out of line, apart from the selection's
// code.  The token's own channels and its sequence come from the call's inputs, so they
// are read before the dependency wait; the states and the plane after it.
__device__ __noinline__ void compress_cta(const CompressArgs& c, int64_t cta) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint64_t* turn_s = reinterpret_cast<uint64_t*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 32) turn_s[threadIdx.x] = rope_turn(c.inv_freq[threadIdx.x]);
  __syncthreads();
  const int64_t t = cta * kTopkWarps + warp;
  if (t >= c.T) return;  // nothing to read or write
  float own_kv[2][8], own_sc[2][8];
  cdev::load_own(c, t, lane, own_kv, own_sc);
  const int b = cdev::warp_find_seq(c.cu_seqlens, c.B, t, lane);
  const int64_t t0 = __ldg(c.cu_seqlens + b), t1 = __ldg(c.cu_seqlens + b + 1);
  griddep_wait();  // the previous step's readers of the plane and states are done
  cdev::token<false>(c, t, b, t0, t1, own_kv, own_sc, lane, turn_s);
}

// One launch runs one or two independent selections over the same queries, e.g. the
// top rows and the top candidate blocks of a FULL layer side by side: blockIdx.x below
// a0.nchunk is a chunk of a0, the rest are chunks of a1 (blockIdx.y = query).  Rows
// blockIdx.y >= Q (if any) run the compressor's tokens, just as many CTAs as they need.
template <int kKind>
__global__ void __launch_bounds__(kTopkThreads, 1)
    topk_kernel(TopkArgs a0, TopkArgs a1, CompressArgs comp) {
  griddep_launch_dependents();
  const int c = blockIdx.x;
  if ((int)blockIdx.y >= a0.Q) {
    const int64_t cta = (int64_t)(blockIdx.y - a0.Q) * gridDim.x + c;
    if (cta * kTopkWarps >= comp.T) return;
    compress_cta(comp, cta);  // waits for the preceding kernel after reading its inputs
    return;
  }
  if (c < a0.nchunk) topk_row<kKind>(a0, c);
  else topk_row<kKind>(a1, c - a0.nchunk);
}

}  // namespace

// Items per chunk CTA of the staged select (the candidate pool's blocks): the whole row
// up to 32768, else chunks of 32768 (rows up to 48 x 32768 = 1,572,864 items).
int topk_chunk_len(int64_t ld) { return ld <= kChunkLen ? (int)ld : kChunkLen; }
int topk_num_chunks(int64_t ld) {
  const int64_t c = topk_chunk_len(ld);
  return (int)((ld + c - 1) / c);
}
int64_t topk_max_len() { return (int64_t)kChunkLen * kMaxChunks; }
bool topk_fits(int64_t ld, int k) {
  return ld >= 1 && ld <= topk_max_len() && k >= 1 &&
         (topk_num_chunks(ld) == 1 || (int64_t)topk_num_chunks(ld) * k <= kChunkLen);
}
// Positions per chunk CTA of a row selection: the whole row up to 65536 (one CTA reading
// it from global memory), else chunks of 32768 merged by the last chunk CTA.
int topk_row_chunk_len(int64_t ld) { return ld <= kLongLen ? (int)ld : kChunkLen; }
int topk_row_num_chunks(int64_t ld) {
  const int64_t c = topk_row_chunk_len(ld);
  return (int)((ld + c - 1) / c);
}
bool topk_row_fits(int64_t ld, int k) {
  return ld >= 1 && ld <= topk_max_len() && k >= 1 &&
         (topk_row_num_chunks(ld) == 1 || (int64_t)topk_row_num_chunks(ld) * k <= kChunkLen);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, const TopkArgs* b,
                        const CompressArgs* comp) {
  if (a.Q == 0) return cudaSuccess;
  if (b && (b->Q != a.Q || (b->scores != nullptr) != (a.scores != nullptr)))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(SelectSmem);
  auto kern = a.scores ? topk_kernel<kSrcScores> : topk_kernel<kSrcKeys>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int nx = a.nchunk + (b ? b->nchunk : 0);
  // compressor rows: 32 tokens (one per warp) per CTA, nx CTAs per row
  const int64_t per_row = (int64_t)kTopkWarps * nx;
  const int ncomp = comp && comp->T > 0 ? (int)((comp->T + per_row - 1) / per_row) : 0;
  const CompressArgs c = ncomp ? *comp : CompressArgs{};
  return launch_pdl(kern, dim3(nx, a.Q + ncomp), dim3(kTopkThreads), smem, s, a, b ? *b : a, c);
}

}  // namespace csa2

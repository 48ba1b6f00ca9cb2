// common.cuh -- argument blocks shared by the C-ABI layer and the kernels, plus the
// per-translation-unit fault flag helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "ptx.cuh"

namespace csa2 {

constexpr int kDLat = 512;   // latent width (K = V)
constexpr int kDIdx = 128;   // indexer head width
constexpr int kHeads = 64;   // attention query heads
constexpr int kRing = 128;   // sliding-window slots
constexpr int kRopeDim0 = 448;
constexpr int kMaxK = 512;   // largest top-k

struct CompressArgs {
  const uint16_t* kv;
  const uint16_t* score;
  int T;
  const int32_t* cu_seqlens;
  int B;
  const int64_t* start_pos;
  int ratio;
  float* kv_state;
  float* score_state;
  uint16_t* plane;
  int64_t plane_rows;
  const int64_t* row_base;
  const float* norm_w;
  float eps;
  const float* inv_freq;
  // index K of each row (null wk: none): wk [128][512] bf16, knorm_w [128] (null: ones),
  // index_plane [plane_rows][128] bf16
  const uint16_t* wk;
  const float* knorm_w;
  uint16_t* index_plane;
};

// A query group of the indexer: queries q0 .. q0 + nq - 1 of sequence seq (row_base rb)
// own the work tiles tile0 .. tile1 - 1.
struct __align__(16) GroupRec {
  int32_t q0, nq, seq, pad0;
  int64_t tile0, tile1;
  int64_t rb, pad1;
};
// A score CTA's work: tiles it_lo .. it_hi - 1, starting in group g_first.
struct __align__(16) CtaRec {
  int32_t g_first, pad0;
  int64_t it_lo, it_hi, pad1;
};
constexpr int kMaxIndexCtas = 1024;

struct IndexArgs {
  const uint16_t* iq;   // [Q][H][128]
  const float* w;       // [Q][H]
  int Q, H;
  const uint16_t* index_k;
  int64_t index_rows;
  const int64_t* row_base;
  const int32_t* q_seq;
  const int64_t* q_pos;
  int ratio;
  const int32_t* cand;  // [Q][ncb] or null
  int ncb;
  int relu;
  int64_t ld;           // max_scored: positions per query (row stride of scores_out)
  int64_t ldk;          // row stride of keys (ld rounded up to a multiple of 4)
  float* scores_out;    // optional [Q][ld]
  // workspace views
  uint32_t* keys;       // [Q][ldk]
  int32_t* n_scored;    // [Q]
  struct GroupRec* grp;  // [Q]  query groups (written by the prep kernel)
  struct CtaRec* cta;    // [nctas] each score CTA's tile range and first group
  int nctas;             // score kernel CTAs (<= kMaxIndexCtas)
  int32_t* n_groups;     // [2]  groups, largest group size
  int32_t* topk_count;  // [Q]  zeroed by the prep kernel for the top-k merge
  int group_max;        // queries per group (FULL: 256 / H; REINDEX: 1)
  int32_t* pool_count;  // [Q]  or null: zeroed by the prep kernel for the candidate
                        //      pool's top-k merge
  // FP8 index plane (null: index_k is bf16): blocks of 8 rows, 8 x 128 E4M3 codes then
  // 8 fp32 scales (1056 bytes); row_base values are multiples of 8
  const uint8_t* plane8;
  const uint8_t* plane4;  // MXFP4 index plane (blocks of 8 rows, 544 bytes), or null
  uint8_t* q8;          // [Q*H][128] E4M3 codes of the quantised queries (workspace)
  float* qscale;        // [Q*H] their power-of-two scales (workspace)
};

struct TopkArgs {
  const uint32_t* keys;   // [Q][ld] order-preserving keys (0 = not scored), or
  const float* scores;    // [Q][ld] raw fp32 scores (converted on load)
  const int32_t* n;       // [Q] positions per row
  int Q;
  int64_t ld;
  int k;
  const int32_t* cand;    // [Q][ncb] position -> row map for REINDEX, else null
  int ncb;
  int32_t* sel;           // [Q][k]
  float* sel_scores;      // [Q][k] or null
  uint64_t* part;         // [Q][nchunk][k] (key << 32 | position) partial results
  int32_t* count;         // [Q] chunk arrivals (zero before the call; reset by the merge)
  int nchunk;             // chunks per row (1 = single pass)
  int chunk;              // positions (blocks) per chunk
  int blocks;             // 1: select blocks of 8 positions of `keys` instead (candidate
                          //    pool): a block's key is the largest key of its positions
                          //    < n[q], the newest block ceil(n[q] / 8) - 1 is pinned to
                          //    ~0, and the output holds block ids
  const int64_t* q_pos;   // or null: n[q] = min(ld, cand ? ncb * 8 : (q_pos[q] + 1) / ratio),
  int ratio;              //    the index call's scored count, known before its prep ends
};

struct AttnArgs {
  const uint16_t* q;
  int Q;
  const int32_t* q_seq;
  const int64_t* q_pos;
  int swa_mode, swa_dtype;
  const uint8_t* swa;
  int64_t swa_rows;
  const int64_t* lin_base;
  const int64_t* lin_pos0;
  const uint16_t* plane;
  int64_t plane_rows;
  const int64_t* row_base;
  const int32_t* sel;
  int nsel;
  const float* sink;
  float scale;
  uint16_t* out;
  float* lse;
  int cluster;     // nsplit == 2: the two CTAs of a query form a cluster and merge in place
  const float* inv_freq;  // [32] or null: rotate the output's dims 448..511 back by q_pos
  int plane_dtype;        // 0: bf16 plane rows [512]; 1: FP4 rows of 288 bytes (E2M1 codes,
                          //    low nibble first, then 32 E4M3 scales, one per 16 dims)
  int stream_rows;        // 1: the call reads fewer rows than the plane holds, so a row is
                          //    read about once: gathered bf16 rows are evicted from L2 first
  int persist;            // > 0 (one CTA per query, more queries than SMs): that many CTAs,
                          //    each carrying on from query to query
};

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s);
// One CTA whose bounded wait runs out after limit_ns (test of the timeout path).
cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_index(const IndexArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_plane_fp4_index(const uint16_t* k, int64_t n, uint8_t* plane, cudaStream_t s);
// bf16 plane rows [n][512] -> FP4 rows [n][288].
cudaError_t launch_plane_fp4(const uint16_t* rows, int64_t n, uint8_t* out, cudaStream_t s);
// bf16 index rows [n][128] -> FP8 plane (ceil(n / 8) blocks of 1056 bytes).
cudaError_t launch_plane_fp8(const uint16_t* k, int64_t n, uint8_t* plane, cudaStream_t s);
// One launch for selection `a` and, when b != null, a second selection over the same
// queries that runs beside it; when comp != null (comp->T > 0) further CTAs of the same
// launch run the compressor's tokens (csa2_compress_index_topk).
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, const TopkArgs* b = nullptr,
                        const CompressArgs* comp = nullptr);
int attn_num_splits(int Q, int nsel, int num_sms);

// 2-D tensor map over `rows` bf16 rows of `cols` elements (row stride cols * 2 bytes),
// boxes of box_cols x box_rows, 128-byte swizzle, out-of-range elements read as zero.
// A tensor map over bytes: rank 2 or 3, dims[0] contiguous, strides[i] = byte stride of
// dims[i + 1]; 128-byte swizzle (box[0] must be 128).
bool encode_bytes(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                  const uint64_t* strides, const uint32_t* box);
bool encode_rows_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint32_t cols,
                      uint32_t box_cols, uint32_t box_rows);
cudaError_t launch_attn(const AttnArgs& a, int nsplit, cudaStream_t s);

int topk_chunk_len(int64_t ld);
int topk_num_chunks(int64_t ld);
int64_t topk_max_len();
// Can one call select the top-k of rows of ld items?  (the chunk merge holds chunks * k
// pairs)  topk_chunk_len / topk_num_chunks / topk_fits: the staged select of the
// candidate pool's blocks; topk_row_*: the row selection, whose rows of up to 65536
// positions run on one CTA.
bool topk_fits(int64_t ld, int k);
int topk_row_chunk_len(int64_t ld);
int topk_row_num_chunks(int64_t ld);
bool topk_row_fits(int64_t ld, int k);

// Replace the calling thread's csa2_last_error() text.
void set_last_error(const char* msg);

// Fault flags of each translation unit (read and cleared, host side).
int take_fault_compress();
int take_fault_index();
int take_fault_topk();
int take_fault_attn();

// Order-preserving map of fp32 scores to uint32 keys: NaN ranks as -inf, -0 as +0,
// and every key of a real score is >= 1 so that 0 can mark "not scored".
// RoPE phase of position p for frequency theta: theta / (2 pi) is kept as a 64-bit binary
// fraction of a turn (its fractional part only), so (p * turn) mod 2^64 is the phase of
// p exactly in integer arithmetic; read as a signed fraction it is an angle in [-pi, pi).
__device__ __forceinline__ uint64_t rope_turn(float theta) {
  double tr = (double)theta * 0.15915494309189535;
  tr -= floor(tr);
  const double sc = tr * 18446744073709551616.0;  // 2^64
  return sc >= 18446744073709551615.0 ? ~0ull : (uint64_t)sc;
}
__device__ __forceinline__ float rope_angle(uint64_t turn, uint64_t p) {
  return (float)(int64_t)(p * turn) * 3.4061215800865545e-19f;  // 2 pi / 2^64
}

__host__ __device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u;
#ifdef __CUDA_ARCH__
  u = __float_as_uint(f);
#else
  memcpy(&u, &f, 4);
#endif
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) u = 0xFF800000u;  // NaN -> -inf
  if (u == 0x80000000u) u = 0u;                           // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
#ifdef __CUDA_ARCH__
  return __uint_as_float(u);
#else
  float f;
  memcpy(&f, &u, 4);
  return f;
#endif
}

}  // namespace csa2

// Host reader of this translation unit's fault flag.
#define CSA2_DEFINE_FAULT_FLAG(NAME)                                     \
  namespace csa2 {                                                       \
  int take_fault_##NAME() {                                              \
    int v = 0, z = 0;                                                    \
    if (cudaMemcpyFromSymbol(&v, g_fault, sizeof(int)) != cudaSuccess)   \
      return 0;                                                          \
    if (v) cudaMemcpyToSymbol(g_fault, &z, sizeof(int));                 \
    return v;                                                            \
  }                                                                      \
  }

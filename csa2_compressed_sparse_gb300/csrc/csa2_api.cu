// csa2_api.cu -- the extern "C" entry points declared in include/csa2.h: argument
// validation on the host, workspace layout, kernel dispatch and error reporting.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/csa2.h"
#include "common.cuh"

namespace {

thread_local std::string g_last_error;

csa2_status fail(csa2_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

csa2_status cuda_fail(cudaError_t e, const char* where) {
  return fail(CSA2_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, ...)                         \
  do {                                             \
    if (!(cond)) return fail(CSA2_EINVAL, __VA_ARGS__); \
  } while (0)

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of csa2_index_topk.
struct IndexWs {
  size_t keys, n_scored, grp, cta, n_groups, count, part, total;
  int nchunk;
  // candidate pool (nbk > 0): merge counters and partial lists of the block selection
  size_t pcount, ppart;
  // FP8 plane (qrows > 0): the quantised queries and their scales
  size_t q8, qscale;
  int64_t nb_max;
  int pnchunk;
};

// Blocks of 8 positions in a row of ld positions.
int64_t pool_blocks(int64_t ld) { return (ld + 7) / 8; }

// Chunks of the candidate-block selection.  A chunk CTA reads 8 position keys per block;
// when few queries have long rows (a long-context decode batch) most SMs would idle
// while a handful of CTAs each stream 1 MiB, so the rows are cut into chunks of 8192
// blocks (256 KiB of keys) as long as the merge holds their lists and the chunks fit
// twice over on the SMs; otherwise chunks of up to 32768 blocks.  sms == 0 gives the
// most chunks any call can use (for the workspace size).
int pool_chunks(int64_t nb, int nbk, int Q, int sms) {
  const int big = csa2::topk_num_chunks(nb);
  const int64_t small = (nb + 8191) / 8192;
  if (small > big && small * nbk <= 32768 && (sms == 0 || (int64_t)Q * small <= 2 * sms))
    return (int)small;
  return big;
}

IndexWs index_ws_layout(int Q, int64_t ld, int k, int nbk = 0, int64_t qrows = 0) {
  IndexWs w{};
  size_t o = 0;
  w.keys = o; o = up256(o + (size_t)Q * (size_t)((ld + 3) & ~int64_t(3)) * 4);
  w.n_scored = o; o = up256(o + (size_t)Q * 4);
  w.grp = o; o = up256(o + (size_t)Q * sizeof(csa2::GroupRec));
  w.cta = o; o = up256(o + (size_t)csa2::kMaxIndexCtas * sizeof(csa2::CtaRec));
  w.n_groups = o; o = up256(o + 8);
  w.count = o; o = up256(o + (size_t)Q * 4);
  w.nchunk = csa2::topk_row_num_chunks(ld);
  w.part = o;
  if (w.nchunk > 1) o = up256(o + (size_t)Q * w.nchunk * k * 8);
  if (nbk > 0) {
    w.nb_max = pool_blocks(ld);
    w.pnchunk = pool_chunks(w.nb_max, nbk, Q, 0);
    w.pcount = o; o = up256(o + (size_t)Q * 4);
    w.ppart = o;
    if (w.pnchunk > 1) o = up256(o + (size_t)Q * w.pnchunk * nbk * 8);
  }
  if (qrows > 0) {
    w.q8 = o; o = up256(o + (size_t)qrows * 128);
    w.qscale = o; o = up256(o + (size_t)qrows * 4);
  }
  w.total = o;
  return w;
}

// csa2_topk_scores: per-row arrival counters, then the partial lists.
size_t topk_ws_bytes(int Q, int64_t ld, int k) {
  const int nchunk = csa2::topk_row_num_chunks(ld);
  return nchunk > 1 ? up256((size_t)Q * 4) + up256((size_t)Q * nchunk * k * 8) : 0;
}


csa2_status attn_common(const char* name, const csa2_bf16* q, int Q, const int32_t* q_seq,
                        const int64_t* q_pos, const csa2_swa* swa, const void* plane,
                        int64_t plane_rows, const int64_t* row_base, const int32_t* sel, int nsel,
                        const float* sink, float scale, csa2_bf16* out, float* lse, void* ws,
                        size_t ws_bytes, const float* inv_freq, int plane_dtype, csa2_stream stream) {
  REQUIRE(Q >= 0 && Q <= 65535, "%s: Q must be in [0, 65535] (got %d)", name, Q);
  if (Q == 0) return CSA2_OK;
  REQUIRE(q && q_seq && q_pos && swa && out, "%s: q, q_seq, q_pos, swa and out are required", name);
  REQUIRE(aligned16(q) && aligned16(out), "%s: q and out must be 16-byte aligned", name);
  REQUIRE(nsel >= 0 && nsel <= 512, "%s: nsel must be in [0, 512] (got %d)", name, nsel);
  REQUIRE(nsel == 0 || (sel && plane && row_base), "%s: sel, plane and row_base are required when nsel > 0", name);
  REQUIRE(plane == nullptr || aligned16(plane), "%s: plane must be 16-byte aligned", name);
  REQUIRE(swa->mode == CSA2_SWA_RING || swa->mode == CSA2_SWA_LINEAR, "%s: bad swa.mode %d", name, swa->mode);
  REQUIRE(swa->dtype == CSA2_SWA_BF16 || swa->dtype == CSA2_SWA_FP8_S128 ||
              swa->dtype == CSA2_SWA_FP8_E8M0,
          "%s: bad swa.dtype %d", name, swa->dtype);
  REQUIRE(swa->data && aligned16(swa->data), "%s: swa.data must be a 16-byte aligned pointer", name);
  REQUIRE(swa->n_rows >= 0, "%s: swa.n_rows must be >= 0", name);
  REQUIRE(swa->mode == CSA2_SWA_RING || (swa->lin_base && swa->lin_pos0),
          "%s: LINEAR windows need lin_base and lin_pos0", name);
  REQUIRE(std::isfinite(scale), "%s: scale must be finite", name);
  REQUIRE(plane_rows >= 0 && plane_rows < ((int64_t)1 << 31),
          "%s: plane_rows must be in [0, 2^31)", name);
  REQUIRE(swa->n_rows < ((int64_t)1 << 31), "%s: swa.n_rows must be < 2^31", name);
  csa2::AttnArgs a{};
  a.q = q; a.Q = Q; a.q_seq = q_seq; a.q_pos = q_pos;
  a.swa_mode = swa->mode; a.swa_dtype = swa->dtype;
  a.swa = static_cast<const uint8_t*>(swa->data); a.swa_rows = swa->n_rows;
  a.lin_base = swa->lin_base; a.lin_pos0 = swa->lin_pos0;
  a.plane = static_cast<const uint16_t*>(plane); a.plane_rows = plane_rows; a.row_base = row_base;
  a.plane_dtype = plane_dtype;
  a.sel = sel; a.nsel = nsel; a.sink = sink; a.scale = scale; a.out = out; a.lse = lse;
  a.inv_freq = inv_freq;
  // rows read about once (a decode batch) are streamed through L2; a prefill chunk's
  // queries share the plane's rows, which stay
  a.stream_rows = (int64_t)Q * (128 + nsel) <= plane_rows ? 1 : 0;
  REQUIRE(ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) == 0,
          "%s: ws must be 256-byte aligned", name);
  const int sms = num_sms();
  if (sms <= 0) return fail(CSA2_ECUDA, "%s: no CUDA device", name);
  (void)ws_bytes;  // the attention needs no workspace (see csa2_attn_workspace_size)
  const int nsplit = csa2::attn_num_splits(Q, nsel, sms);
  // more queries than SMs: one CTA per SM walks its queries, overlapping a query's output
  // and the next query's set-up with the gathers
  a.persist = nsplit == 1 && Q > sms ? sms : 0;
  cudaError_t e = csa2::launch_attn(a, nsplit, stream);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return CSA2_OK;
}

}  // namespace

namespace csa2 {
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace csa2

extern "C" {

const char* csa2_last_error(void) { return g_last_error.c_str(); }

const char* csa2_version(void) { return "csa2 0.1 sm_103a"; }

csa2_status csa2_device_status(csa2_stream stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_device_status");
  int f = 0;
  for (int v : {csa2::take_fault_compress(), csa2::take_fault_index(), csa2::take_fault_topk(),
                csa2::take_fault_attn()})
    if (!f) f = v;
  if (f == csa2::kFaultTimeout) return fail(CSA2_ETIMEOUT, "a kernel gave up a bounded wait");
  if (f == csa2::kFaultBounds) return fail(CSA2_EBOUNDS, "a kernel met an index outside its buffer");
  return CSA2_OK;
}

csa2_status csa2_selftest_wait_timeout(int64_t limit_ns, csa2_stream stream) {
  REQUIRE(limit_ns >= 1000 && limit_ns <= 1000000000,
          "csa2_selftest_wait_timeout: limit_ns must be in [1e3, 1e9] (got %lld)",
          (long long)limit_ns);
  cudaError_t e = csa2::launch_wait_timeout((uint64_t)limit_ns, stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_selftest_wait_timeout");
  return CSA2_OK;
}

namespace {

// Checks of the compressor's arguments (csa2_compress and the calls that include it);
// fills *a (a->T == 0: nothing to compress).
csa2_status compress_args(const char* name, const csa2_bf16* kv, const csa2_bf16* score, int T,
                          const int32_t* cu_seqlens, int B, const int64_t* start_pos, int ratio,
                          float* kv_state, float* score_state, csa2_bf16* plane,
                          int64_t plane_rows, const int64_t* row_base, const float* norm_w,
                          float eps, const float* inv_freq, csa2::CompressArgs* a) {
  *a = csa2::CompressArgs{};
  REQUIRE(ratio == 1 || ratio == 2, "%s: ratio must be 1 or 2 (got %d)", name, ratio);
  REQUIRE(B >= 1 && B <= 8192, "%s: B must be in [1, 8192] (got %d)", name, B);
  REQUIRE(T >= 0, "%s: T must be >= 0 (got %d)", name, T);
  if (T == 0) return CSA2_OK;
  REQUIRE(kv && cu_seqlens && start_pos && plane && row_base && inv_freq,
          "%s: kv, cu_seqlens, start_pos, plane, row_base and inv_freq are required", name);
  REQUIRE(ratio == 1 || (score && kv_state && score_state),
          "%s: ratio 2 needs score, kv_state and score_state", name);
  REQUIRE(aligned16(kv) && aligned16(plane) && (!score || aligned16(score)) &&
              (!kv_state || aligned16(kv_state)) && (!score_state || aligned16(score_state)) &&
              (!norm_w || aligned16(norm_w)),
          "%s: kv, score, plane, states and norm_w must be 16-byte aligned", name);
  REQUIRE(eps >= 0.f && std::isfinite(eps), "%s: eps must be finite and >= 0", name);
  REQUIRE(plane_rows >= 0, "%s: plane_rows must be >= 0", name);
  *a = csa2::CompressArgs{kv, score, T, cu_seqlens, B, start_pos, ratio, kv_state, score_state,
                          plane, plane_rows, row_base, norm_w, eps, inv_freq,
                          nullptr, nullptr, nullptr};
  return CSA2_OK;
}

}  // namespace

csa2_status csa2_compress(const csa2_bf16* kv, const csa2_bf16* score, int T,
                          const int32_t* cu_seqlens, int B, const int64_t* start_pos, int ratio,
                          float* kv_state, float* score_state, csa2_bf16* plane,
                          int64_t plane_rows, const int64_t* row_base, const float* norm_w,
                          float eps, const float* inv_freq, csa2_stream stream) {
  csa2::CompressArgs a;
  const csa2_status st = compress_args("csa2_compress", kv, score, T, cu_seqlens, B, start_pos,
                                       ratio, kv_state, score_state, plane, plane_rows, row_base,
                                       norm_w, eps, inv_freq, &a);
  if (st != CSA2_OK || a.T == 0) return st;
  cudaError_t e = csa2::launch_compress(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_compress");
  return CSA2_OK;
}

csa2_status csa2_compress_index(const csa2_bf16* kv, const csa2_bf16* score, int T,
                                const int32_t* cu_seqlens, int B, const int64_t* start_pos,
                                int ratio, float* kv_state, float* score_state, csa2_bf16* plane,
                                int64_t plane_rows, const int64_t* row_base, const float* norm_w,
                                float eps, const float* inv_freq, const csa2_bf16* wk,
                                const float* knorm_w, csa2_bf16* index_plane,
                                csa2_stream stream) {
  REQUIRE(T <= 0 || (wk && index_plane), "csa2_compress_index: wk and index_plane are required");
  REQUIRE(!wk || (aligned16(wk) && aligned16(index_plane)),
          "csa2_compress_index: wk and index_plane must be 16-byte aligned");
  // the plain compressor's checks next
  csa2::CompressArgs a;
  const csa2_status st = compress_args("csa2_compress", kv, score, T, cu_seqlens, B, start_pos,
                                       ratio, kv_state, score_state, plane, plane_rows, row_base,
                                       norm_w, eps, inv_freq, &a);
  if (st != CSA2_OK || a.T == 0) return st;
  a.wk = reinterpret_cast<const uint16_t*>(wk);
  a.knorm_w = knorm_w;
  a.index_plane = reinterpret_cast<uint16_t*>(index_plane);
  cudaError_t e = csa2::launch_compress(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_compress_index");
  return CSA2_OK;
}

size_t csa2_index_topk_workspace_size(int Q, int H, int64_t max_scored, int k) {
  (void)H;
  if (Q < 0 || max_scored < 1 || k < 1 || k > 512) return 0;
  return index_ws_layout(Q, max_scored, k).total;
}

namespace {

// plane_fmt: 1 = FP8 blocks (plane), 2 = MXFP4 blocks (plane); 0 = bf16 rows (index_k)
csa2_status index_topk_impl(const csa2_bf16* iq, const float* w, int Q, int H,
                            const csa2_bf16* index_k, const uint8_t* plane, int plane_fmt,
                            int64_t index_rows,
                            const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos,
                            int ratio, const int32_t* cand, int ncb, int k, int relu,
                            int64_t max_scored, int32_t* sel, float* sel_scores,
                            float* scores_out, int nbk, int32_t* pool, void* ws, size_t ws_bytes,
                            csa2_stream stream, const csa2::CompressArgs* comp = nullptr) {
  REQUIRE(Q >= 0, "csa2_index_topk: Q must be >= 0 (got %d)", Q);
  REQUIRE(H == 32 || H == 64, "csa2_index_topk: H must be 32 or 64 (got %d)", H);
  REQUIRE(ratio == 1 || ratio == 2, "csa2_index_topk: ratio must be 1 or 2 (got %d)", ratio);
  REQUIRE(k >= 1 && k <= 512, "csa2_index_topk: k must be in [1, 512] (got %d)", k);
  REQUIRE(max_scored >= 1, "csa2_index_topk: max_scored must be >= 1");
  if (cand) {
    REQUIRE(ncb >= 1, "csa2_index_topk: ncb must be >= 1 with a candidate pool");
    REQUIRE((int64_t)ncb * 8 >= k,
            "csa2_index_topk: candidate pool of %d blocks x 8 rows cannot hold top-%d", ncb, k);
    REQUIRE(max_scored == (int64_t)ncb * 8, "csa2_index_topk: REINDEX needs max_scored == ncb * 8");
  }
  REQUIRE(max_scored <= csa2::topk_max_len(),
          "csa2_index_topk: max_scored %lld exceeds the supported %lld positions",
          (long long)max_scored, (long long)csa2::topk_max_len());
  if (Q == 0) {  // nothing to score: the compressor's tokens (if any) run on their own
    if (comp && comp->T > 0) {
      cudaError_t e = csa2::launch_compress(*comp, stream);
      if (e != cudaSuccess) return cuda_fail(e, "csa2_compress_index_topk (compress)");
    }
    return CSA2_OK;
  }
  REQUIRE(iq && w && (plane_fmt ? plane != nullptr : index_k != nullptr) && row_base && q_seq &&
              q_pos && sel && ws,
          "csa2_index_topk: iq, w, the index plane, row_base, q_seq, q_pos, sel and ws are required");
  REQUIRE(aligned16(iq) && aligned16(plane_fmt ? (const void*)plane : (const void*)index_k),
          "csa2_index_topk: iq and the index plane must be 16-byte aligned");
  REQUIRE(index_rows >= 1 && index_rows < (int64_t)1 << 31, "csa2_index_topk: index_rows out of range");
  REQUIRE((int64_t)Q * H < (int64_t)1 << 31, "csa2_index_topk: Q * H out of range");
  REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, "csa2_index_topk: ws must be 256-byte aligned");
  const IndexWs L = index_ws_layout(Q, max_scored, k, nbk, plane_fmt == 1 ? (int64_t)Q * H : 0);
  if (ws_bytes < L.total)
    return fail(CSA2_ENOSPACE, "csa2_index_topk: workspace %zu bytes < required %zu", ws_bytes, L.total);
  uint8_t* base = static_cast<uint8_t*>(ws);
  csa2::IndexArgs a{};
  a.iq = iq; a.w = w; a.Q = Q; a.H = H; a.index_k = index_k; a.index_rows = index_rows;
  a.row_base = row_base; a.q_seq = q_seq; a.q_pos = q_pos; a.ratio = ratio; a.cand = cand;
  a.ncb = cand ? ncb : 0; a.relu = relu ? 1 : 0; a.ld = max_scored; a.scores_out = scores_out;
  a.ldk = (max_scored + 3) & ~int64_t(3);
  a.keys = reinterpret_cast<uint32_t*>(base + L.keys);
  a.n_scored = reinterpret_cast<int32_t*>(base + L.n_scored);
  a.grp = reinterpret_cast<csa2::GroupRec*>(base + L.grp);
  a.cta = reinterpret_cast<csa2::CtaRec*>(base + L.cta);
  a.n_groups = reinterpret_cast<int32_t*>(base + L.n_groups);
  a.topk_count = reinterpret_cast<int32_t*>(base + L.count);
  a.group_max = cand ? 1 : 256 / H;
  if (nbk > 0) a.pool_count = reinterpret_cast<int32_t*>(base + L.pcount);
  if (plane_fmt == 1) {
    a.index_k = nullptr;
    a.plane8 = plane;
    a.q8 = base + L.q8;
    a.qscale = reinterpret_cast<float*>(base + L.qscale);
  } else if (plane_fmt == 2) {
    a.index_k = nullptr;
    a.plane4 = plane;
  }
  const int sms = num_sms();
  if (sms <= 0) return fail(CSA2_ECUDA, "csa2_index_topk: no CUDA device");
  cudaError_t e = csa2::launch_index(a, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_index_topk (scores)");
  csa2::TopkArgs t{};
  t.keys = a.keys; t.scores = nullptr; t.n = a.n_scored; t.Q = Q; t.ld = a.ldk; t.k = k;
  t.cand = cand; t.ncb = a.ncb; t.sel = sel; t.sel_scores = sel_scores;
  t.part = reinterpret_cast<uint64_t*>(base + L.part); t.nchunk = L.nchunk;
  t.count = a.topk_count;
  t.chunk = csa2::topk_row_chunk_len(max_scored);
  t.q_pos = q_pos;
  t.ratio = ratio;
  // n_scored <= max_scored <= ldk: the chunking of max_scored covers every row
  csa2::TopkArgs p{};
  if (nbk > 0) {  // the candidate blocks, from the same keys, in the same launch
    p = t;
    p.sel_scores = nullptr;
    p.k = nbk; p.sel = pool; p.blocks = 1;
    p.part = reinterpret_cast<uint64_t*>(base + L.ppart);
    p.nchunk = pool_chunks(L.nb_max, nbk, Q, sms);
    p.count = a.pool_count;
    p.chunk = (int)((L.nb_max + p.nchunk - 1) / p.nchunk);
  }
  // the block selection's CTAs (the longer ones) first
  e = nbk > 0 ? csa2::launch_topk(p, stream, &t, comp) : csa2::launch_topk(t, stream, nullptr, comp);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_index_topk (top-k)");
  return CSA2_OK;
}

}  // namespace

csa2_status csa2_index_topk(const csa2_bf16* iq, const float* w, int Q, int H,
                            const csa2_bf16* index_k, int64_t index_rows,
                            const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos,
                            int ratio, const int32_t* cand, int ncb, int k, int relu,
                            int64_t max_scored, int32_t* sel, float* sel_scores,
                            float* scores_out, void* ws, size_t ws_bytes, csa2_stream stream) {
  return index_topk_impl(iq, w, Q, H, index_k, nullptr, 0, index_rows, row_base, q_seq, q_pos,
                         ratio, cand, ncb, k, relu, max_scored, sel, sel_scores, scores_out, 0,
                         nullptr, ws, ws_bytes, stream);
}

csa2_status csa2_compress_index_topk(
    const csa2_bf16* kv, const csa2_bf16* score, int T, const int32_t* cu_seqlens, int B,
    const int64_t* start_pos, float* kv_state, float* score_state, csa2_bf16* plane,
    int64_t plane_rows, const float* norm_w, float eps, const float* inv_freq,
    const csa2_bf16* iq, const float* w, int Q, int H, const csa2_bf16* index_k,
    int64_t index_rows, const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos,
    int ratio, const int32_t* cand, int ncb, int k, int relu, int64_t max_scored, int32_t* sel,
    float* sel_scores, float* scores_out, void* ws, size_t ws_bytes, csa2_stream stream) {
  csa2::CompressArgs c;
  const csa2_status st = compress_args("csa2_compress_index_topk", kv, score, T, cu_seqlens, B,
                                       start_pos, ratio, kv_state, score_state, plane,
                                       plane_rows, row_base, norm_w, eps, inv_freq, &c);
  if (st != CSA2_OK) return st;
  return index_topk_impl(iq, w, Q, H, index_k, nullptr, 0, index_rows, row_base, q_seq, q_pos,
                         ratio, cand, ncb, k, relu, max_scored, sel, sel_scores, scores_out, 0,
                         nullptr, ws, ws_bytes, stream, c.T > 0 ? &c : nullptr);
}

size_t csa2_index_topk_pool_workspace_size(int Q, int H, int64_t max_scored, int k, int nbk) {
  (void)H;
  if (Q < 0 || max_scored < 1 || k < 1 || k > 512 || nbk < 1 || nbk > 2048) return 0;
  return index_ws_layout(Q, max_scored, k, nbk).total;
}

csa2_status csa2_index_topk_pool(const csa2_bf16* iq, const float* w, int Q, int H,
                                 const csa2_bf16* index_k, int64_t index_rows,
                                 const int64_t* row_base, const int32_t* q_seq,
                                 const int64_t* q_pos, int ratio, int k, int relu,
                                 int64_t max_scored, int32_t* sel, float* sel_scores,
                                 float* scores_out, int nbk, int32_t* pool, void* ws,
                                 size_t ws_bytes, csa2_stream stream) {
  REQUIRE(nbk >= 1 && nbk <= 2048, "csa2_index_topk_pool: nbk must be in [1, 2048] (got %d)", nbk);
  REQUIRE(max_scored >= 1 && csa2::topk_fits(pool_blocks(max_scored), nbk),
          "csa2_index_topk_pool: %lld blocks per row with nbk = %d exceed the block selection",
          (long long)pool_blocks(max_scored), nbk);
  REQUIRE(Q == 0 || pool, "csa2_index_topk_pool: pool is required");
  return index_topk_impl(iq, w, Q, H, index_k, nullptr, 0, index_rows, row_base, q_seq, q_pos,
                         ratio, nullptr, 0, k, relu, max_scored, sel, sel_scores, scores_out,
                         nbk, pool, ws, ws_bytes, stream);
}

size_t csa2_index_topk_fp8_workspace_size(int Q, int H, int64_t max_scored, int k) {
  if (Q < 0 || (H != 32 && H != 64) || max_scored < 1 || k < 1 || k > 512) return 0;
  return index_ws_layout(Q, max_scored, k, 0, (int64_t)Q * H).total;
}

csa2_status csa2_index_topk_fp8(const csa2_bf16* iq, const float* w, int Q, int H,
                                const uint8_t* plane, int64_t index_rows,
                                const int64_t* row_base, const int32_t* q_seq,
                                const int64_t* q_pos, int ratio, const int32_t* cand, int ncb,
                                int k, int relu, int64_t max_scored, int32_t* sel,
                                float* sel_scores, float* scores_out, void* ws, size_t ws_bytes,
                                csa2_stream stream) {
  REQUIRE(Q == 0 || plane, "csa2_index_topk_fp8: plane is required");
  return index_topk_impl(iq, w, Q, H, nullptr, plane, 1, index_rows, row_base, q_seq, q_pos,
                         ratio, cand, ncb, k, relu, max_scored, sel, sel_scores, scores_out, 0,
                         nullptr, ws, ws_bytes, stream);
}

size_t csa2_index_topk_fp4_workspace_size(int Q, int H, int64_t max_scored, int k) {
  if (Q < 0 || (H != 32 && H != 64) || max_scored < 1 || k < 1 || k > 512) return 0;
  return index_ws_layout(Q, max_scored, k).total;
}

csa2_status csa2_index_topk_fp4(const csa2_bf16* iq, const float* w, int Q, int H,
                                const uint8_t* plane, int64_t index_rows,
                                const int64_t* row_base, const int32_t* q_seq,
                                const int64_t* q_pos, int ratio, const int32_t* cand, int ncb,
                                int k, int relu, int64_t max_scored, int32_t* sel,
                                float* sel_scores, float* scores_out, void* ws, size_t ws_bytes,
                                csa2_stream stream) {
  REQUIRE(Q == 0 || plane, "csa2_index_topk_fp4: plane is required");
  return index_topk_impl(iq, w, Q, H, nullptr, plane, 2, index_rows, row_base, q_seq, q_pos,
                         ratio, cand, ncb, k, relu, max_scored, sel, sel_scores, scores_out, 0,
                         nullptr, ws, ws_bytes, stream);
}

size_t csa2_index_plane_fp4_bytes(int64_t rows) {
  return rows <= 0 ? 0 : (size_t)((rows + 7) / 8) * 544;
}

csa2_status csa2_index_plane_fp4(const csa2_bf16* index_k, int64_t rows, uint8_t* plane,
                                 csa2_stream stream) {
  REQUIRE(rows >= 0 && rows < (int64_t)1 << 34, "csa2_index_plane_fp4: rows out of range");
  if (rows == 0) return CSA2_OK;
  REQUIRE(index_k && plane, "csa2_index_plane_fp4: index_k and plane are required");
  REQUIRE(aligned16(index_k) && aligned16(plane),
          "csa2_index_plane_fp4: index_k and plane must be 16-byte aligned");
  cudaError_t e = csa2::launch_plane_fp4_index(reinterpret_cast<const uint16_t*>(index_k), rows,
                                               plane, stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_index_plane_fp4");
  return CSA2_OK;
}

size_t csa2_index_plane_fp8_bytes(int64_t rows) {
  return rows <= 0 ? 0 : (size_t)((rows + 7) / 8) * 1056;
}

csa2_status csa2_index_plane_fp8(const csa2_bf16* index_k, int64_t rows, uint8_t* plane,
                                 csa2_stream stream) {
  REQUIRE(rows >= 0 && rows < (int64_t)1 << 34, "csa2_index_plane_fp8: rows out of range");
  if (rows == 0) return CSA2_OK;
  REQUIRE(index_k && plane, "csa2_index_plane_fp8: index_k and plane are required");
  REQUIRE(aligned16(index_k) && aligned16(plane),
          "csa2_index_plane_fp8: index_k and plane must be 16-byte aligned");
  cudaError_t e = csa2::launch_plane_fp8(reinterpret_cast<const uint16_t*>(index_k), rows, plane,
                                         stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_index_plane_fp8");
  return CSA2_OK;
}

size_t csa2_topk_workspace_size(int Q, int64_t ld, int k) {
  if (Q < 0 || ld < 1 || k < 1 || k > 2048 || !csa2::topk_row_fits(ld, k)) return 0;
  return topk_ws_bytes(Q, ld, k);
}

csa2_status csa2_topk_scores(const float* scores, const int32_t* n, int Q, int64_t ld, int k,
                             int32_t* sel, float* sel_scores, void* ws, size_t ws_bytes,
                             csa2_stream stream) {
  REQUIRE(Q >= 0, "csa2_topk_scores: Q must be >= 0");
  REQUIRE(k >= 1 && k <= 2048, "csa2_topk_scores: k must be in [1, 2048] (got %d)", k);
  REQUIRE(ld >= 1, "csa2_topk_scores: ld must be >= 1");
  REQUIRE(ld <= csa2::topk_max_len(),
          "csa2_topk_scores: ld %lld exceeds the supported %lld positions", (long long)ld,
          (long long)csa2::topk_max_len());
  REQUIRE(csa2::topk_row_fits(ld, k),
          "csa2_topk_scores: rows of %lld positions with k = %d exceed the chunk merge "
          "(chunks of 32768 positions x k must be <= 32768)", (long long)ld, k);
  if (Q == 0) return CSA2_OK;
  REQUIRE(scores && n && sel, "csa2_topk_scores: scores, n and sel are required");
  const size_t need = topk_ws_bytes(Q, ld, k);
  if (need) {
    REQUIRE(ws && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0,
            "csa2_topk_scores: ws must be a 256-byte aligned pointer");
    if (ws_bytes < need)
      return fail(CSA2_ENOSPACE, "csa2_topk_scores: workspace %zu bytes < required %zu", ws_bytes, need);
  }
  csa2::TopkArgs t{};
  t.keys = nullptr; t.scores = scores; t.n = n; t.Q = Q; t.ld = ld; t.k = k; t.cand = nullptr;
  t.ncb = 0; t.sel = sel; t.sel_scores = sel_scores;
  t.nchunk = csa2::topk_row_num_chunks(ld);
  t.chunk = csa2::topk_row_chunk_len(ld);
  if (t.nchunk > 1) {
    t.count = static_cast<int32_t*>(ws);
    t.part = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + up256((size_t)Q * 4));
    cudaError_t z = cudaMemsetAsync(t.count, 0, (size_t)Q * 4, stream);
    if (z != cudaSuccess) return cuda_fail(z, "csa2_topk_scores");
  }
  cudaError_t e = csa2::launch_topk(t, stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_topk_scores");
  return CSA2_OK;
}

size_t csa2_attn_workspace_size(int Q, int nsel) {
  (void)Q;
  (void)nsel;
  return 0;  // one or two CTAs per query, merging in distributed shared memory
}

csa2_status csa2_sparse_attn(const csa2_bf16* q, int Q, const int32_t* q_seq,
                             const int64_t* q_pos, const csa2_swa* swa, const csa2_bf16* plane,
                             int64_t plane_rows, const int64_t* row_base, const int32_t* sel,
                             int nsel, const float* sink, float scale, csa2_bf16* out, float* lse,
                             void* ws, size_t ws_bytes, csa2_stream stream) {
  return attn_common("csa2_sparse_attn", q, Q, q_seq, q_pos, swa, plane, plane_rows, row_base,
                     sel, nsel, sink, scale, out, lse, ws, ws_bytes, nullptr, 0, stream);
}

csa2_status csa2_reuse_attn(const csa2_bf16* q, int Q, const int32_t* q_seq,
                            const int64_t* q_pos, const csa2_swa* swa, const csa2_bf16* plane,
                            int64_t plane_rows, const int64_t* row_base, const int32_t* sel,
                            int nsel, const float* sink, float scale, csa2_bf16* out, float* lse,
                            void* ws, size_t ws_bytes, csa2_stream stream) {
  return attn_common("csa2_reuse_attn", q, Q, q_seq, q_pos, swa, plane, plane_rows, row_base,
                     sel, nsel, sink, scale, out, lse, ws, ws_bytes, nullptr, 0, stream);
}

csa2_status csa2_sparse_attn_rope(const csa2_bf16* q, int Q, const int32_t* q_seq,
                                  const int64_t* q_pos, const csa2_swa* swa,
                                  const csa2_bf16* plane, int64_t plane_rows,
                                  const int64_t* row_base, const int32_t* sel, int nsel,
                                  const float* sink, float scale, csa2_bf16* out, float* lse,
                                  void* ws, size_t ws_bytes, const float* inv_freq,
                                  csa2_stream stream) {
  REQUIRE(inv_freq != nullptr, "csa2_sparse_attn_rope: inv_freq is required");
  return attn_common("csa2_sparse_attn_rope", q, Q, q_seq, q_pos, swa, plane, plane_rows,
                     row_base, sel, nsel, sink, scale, out, lse, ws, ws_bytes, inv_freq, 0,
                     stream);
}

csa2_status csa2_reuse_attn_rope(const csa2_bf16* q, int Q, const int32_t* q_seq,
                                 const int64_t* q_pos, const csa2_swa* swa,
                                 const csa2_bf16* plane, int64_t plane_rows,
                                 const int64_t* row_base, const int32_t* sel, int nsel,
                                 const float* sink, float scale, csa2_bf16* out, float* lse,
                                 void* ws, size_t ws_bytes, const float* inv_freq,
                                 csa2_stream stream) {
  REQUIRE(inv_freq != nullptr, "csa2_reuse_attn_rope: inv_freq is required");
  return attn_common("csa2_reuse_attn_rope", q, Q, q_seq, q_pos, swa, plane, plane_rows,
                     row_base, sel, nsel, sink, scale, out, lse, ws, ws_bytes, inv_freq, 0,
                     stream);
}

csa2_status csa2_sparse_attn_fp4(const csa2_bf16* q, int Q, const int32_t* q_seq,
                                 const int64_t* q_pos, const csa2_swa* swa, const uint8_t* plane,
                                 int64_t plane_rows, const int64_t* row_base, const int32_t* sel,
                                 int nsel, const float* sink, float scale, csa2_bf16* out,
                                 float* lse, void* ws, size_t ws_bytes, const float* inv_freq,
                                 csa2_stream stream) {
  return attn_common("csa2_sparse_attn_fp4", q, Q, q_seq, q_pos, swa, plane, plane_rows,
                     row_base, sel, nsel, sink, scale, out, lse, ws, ws_bytes, inv_freq, 1,
                     stream);
}

size_t csa2_plane_fp4_bytes(int64_t rows) { return rows <= 0 ? 0 : (size_t)rows * 288; }

csa2_status csa2_plane_fp4(const csa2_bf16* plane, int64_t rows, uint8_t* out,
                           csa2_stream stream) {
  REQUIRE(rows >= 0 && rows < (int64_t)1 << 31, "csa2_plane_fp4: rows out of range");
  if (rows == 0) return CSA2_OK;
  REQUIRE(plane && out, "csa2_plane_fp4: plane and out are required");
  REQUIRE(aligned16(plane) && aligned16(out), "csa2_plane_fp4: plane and out must be 16-byte aligned");
  cudaError_t e =
      csa2::launch_plane_fp4(reinterpret_cast<const uint16_t*>(plane), rows, out, stream);
  if (e != cudaSuccess) return cuda_fail(e, "csa2_plane_fp4");
  return CSA2_OK;
}

}  // extern "C"

namespace csa2 {

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_bytes(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                  const uint64_t* strides, const uint32_t* box) {
  auto fn = tensor_map_encoder();
  if (!fn || !base || rank < 2 || rank > 3) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    if (dims[i] == 0) return false;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d,
                  st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_rows_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint32_t cols,
                      uint32_t box_cols, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn || !base || rows == 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace csa2

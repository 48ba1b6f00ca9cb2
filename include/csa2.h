/*
 * csa2.h -- C ABI of the CSA2 compressed-sparse attention step on one GB300 (sm_103a).
 *
 * The step, as the source pages state it (DeepSeek-V4.1-Flash CSA2 attention):
 *   compress     -> pool each group of m (1 or 2) new tokens into one 512-d row
 *   index_topk   -> lightning-indexer scores over the visible rows (or over a
 *                   candidate pool), then the 512 best rows
 *   sparse_attn  -> 64-head single-KV-head attention over the 128-position window
 *                   plus the selected rows, one softmax with a per-head sink
 *   reuse_attn   -> the same attention with a selection taken from another layer
 *
 * Conventions (every entry point):
 *   - Every pointer argument is a DEVICE pointer unless its comment says HOST.  The
 *     caller owns every buffer; the library allocates no device memory.  Scratch
 *     memory is caller-provided through the *_workspace_size queries.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No call synchronises except csa2_device_status().  Kernels are
 *     launched as programmatic dependents: a call may start while the preceding kernel
 *     of this library on the stream drains, and reads only its own inputs (queries,
 *     positions, window rows) before that kernel has finished; whatever that kernel
 *     produces (a selection, keys) is read after it, and workspace is written after it.
 *     Inputs written by other kernels must be complete in stream order, as usual.
 *   - Argument errors are detected on the host before anything is launched and
 *     return CSA2_EINVAL.  CUDA launch failures return CSA2_ECUDA.  The text of the
 *     last failure on the calling thread is available from csa2_last_error().
 *   - Data-dependent faults found by the kernels (an index outside its buffer, a
 *     wait that ran past its time limit) skip the offending access and raise a
 *     device-side flag; csa2_device_status() reports and clears it.
 *   - Row ids in `sel`/`cand` are sequence-local; -1 marks an empty entry.  bf16
 *     tensors are raw 16-bit patterns (csa2_bf16).  Layouts are row-major, dense.
 *   - Base addresses must be 16-byte aligned; the library checks this.
 *
 * Page references ("section" names are the pages' own headings):
 *   [A] "DeepSeek-V4.1-Flash 架构解剖" (perryzhang01.github.io, v41_flash_anatomy)
 *   [B] "DeepSeek-V4.1-Flash 结构说明" (treert.github.io, ds-v4-1-flash-structure)
 *   [C] "万字长文解析DeekSeekV4.1flash" (yuyanqi.com)
 *   [E] "DeepSeek-V4-Pro 架构解剖" (perryzhang01.github.io, v4_pro_anatomy)
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA2_OK = 0,
  CSA2_EINVAL = 1,   /* invalid argument; nothing was enqueued */
  CSA2_ECUDA = 2,    /* a CUDA runtime call failed */
  CSA2_ETIMEOUT = 3, /* a kernel gave up a bounded wait (from csa2_device_status) */
  CSA2_EBOUNDS = 4,  /* a kernel met an index outside its buffer (from csa2_device_status) */
  CSA2_ENOSPACE = 5  /* the workspace is smaller than the size query returned */
} csa2_status;

typedef struct CUstream_st* csa2_stream; /* same type as cudaStream_t */
typedef uint16_t csa2_bf16;              /* bfloat16 bit pattern */

/* Message of the last failing call on this thread ("" if none).  The string is
 * owned by the library and stays valid until the next call on this thread. */
const char* csa2_last_error(void);

/* Library version string, e.g. "csa2 0.1 sm_103a". */
const char* csa2_version(void);

/* Synchronises `stream`, then reports and clears the device-side fault flag raised
 * by any kernel of this library since the previous call: CSA2_OK, CSA2_ETIMEOUT or
 * CSA2_EBOUNDS (the first fault wins).  CSA2_ECUDA if the synchronisation failed. */
csa2_status csa2_device_status(csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_selftest_wait_timeout -- test export; the pages have no counterpart.
 *
 * Every wait inside the library's kernels (on an mbarrier: a copy landing, an MMA
 * completing, a partner warp) is bounded: when it runs out the kernel records
 * CSA2_ETIMEOUT in the device fault flag and unwinds instead of hanging the GPU.  This
 * call exercises that path on purpose: it launches one CTA whose thread waits for an
 * mbarrier phase that nothing completes (no copy or MMA is attached to it), with the
 * limit limit_ns nanoseconds (1e3 .. 1e9).  The wait runs out, the kernel returns, and
 * the next csa2_device_status() reports CSA2_ETIMEOUT (and clears the flag).  The
 * context stays usable. */
csa2_status csa2_selftest_wait_timeout(int64_t limit_ns, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_compress -- [A] "特殊模块 · compressor", "CSA2 的池化比 V4 简单一截";
 * [B] §4.1 (odd tail), §6.1-6.2 (partial RoPE at the group head); [C] §6.2, §6.4.
 *
 * New tokens of B sequences arrive as a ragged batch: tokens cu_seqlens[b] ..
 * cu_seqlens[b+1]-1 of kv/score belong to sequence b and sit at absolute positions
 * start_pos[b], start_pos[b]+1, ...  For every group j whose last token
 * (j*ratio + ratio - 1) arrives in this call the library writes plane row
 * row_base[b] + j:
 *     r[d] = sum_i softmax_i(score_i[d]) * kv_i[d]          (i over the group's tokens)
 *     y    = r * rsqrt(mean(r^2) + eps) * norm_w             (RMSNorm over 512 dims)
 *     y[448+2i], y[449+2i] rotated by angle (j*ratio) * inv_freq[i], i = 0..31
 * in fp32, stored as bf16 (round to nearest even).  Tokens of a group that is still
 * incomplete at the end of the call are stored in kv_state/score_state slot
 * (position % ratio) of their sequence; tokens of a group that started in an
 * earlier call are read from there.  With ratio 1 every token is a group and the
 * states are not touched (they may be NULL).
 *   kv, score    [T][512] bf16 (score may be NULL when ratio == 1)
 *   cu_seqlens   [B+1] int32, non-decreasing, cu_seqlens[0] == 0, cu_seqlens[B] == T
 *   start_pos    [B] int64 >= 0
 *   ratio        1 or 2
 *   kv_state, score_state  [B][2][512] fp32, read and written
 *   plane        [plane_rows][512] bf16, rows written as above
 *   row_base     [B] int64; rows past plane_rows raise CSA2_EBOUNDS and are skipped
 *   norm_w       [512] fp32 RMSNorm weight, NULL = all ones
 *   inv_freq     [32] fp32 RoPE inverse frequencies (a YaRN table drops in here)
 * Limits: 1 <= B <= 8192, T >= 0. */
csa2_status csa2_compress(const csa2_bf16* kv, const csa2_bf16* score, int T,
                          const int32_t* cu_seqlens, int B, const int64_t* start_pos, int ratio,
                          float* kv_state, float* score_state, csa2_bf16* plane,
                          int64_t plane_rows, const int64_t* row_base, const float* norm_w,
                          float eps, const float* inv_freq, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_compress_index -- csa2_compress plus the index K of every row it writes, as a
 * FULL layer produces it.  [A] indexer figure, key side (the compressed latent before
 * RoPE, as bf16, through indexer.wk [128, 512], then k_norm, then RoPE, into the index
 * plane); [A] compressor figure (the two branches part after the RMSNorm); [C] A.6.2
 * (index K projected from the main latent).
 *
 * For each row written, with y its normalized latent before the main RoPE and p0 = j *
 * ratio its group-head position:
 *     x    = bf16(y)
 *     k[o] = sum_d wk[o][d] x[d]                         (o < 128, fp32 sums)
 *     k    = k * rsqrt(mean(k^2) + eps) * knorm_w        (RMSNorm over the 128 dims)
 *     k[64+2i], k[65+2i] rotated by angle p0 * inv_freq[i], i = 0..31
 * stored as bf16 to index_plane row row_base[b] + j (the same row as the main plane).
 *   wk           [128][512] bf16, 16-byte aligned
 *   knorm_w      [128] fp32, NULL = all ones
 *   index_plane  [plane_rows][128] bf16, 16-byte aligned
 * Everything else (arguments, main plane, states, limits, errors) as csa2_compress. */
csa2_status csa2_compress_index(const csa2_bf16* kv, const csa2_bf16* score, int T,
                                const int32_t* cu_seqlens, int B, const int64_t* start_pos,
                                int ratio, float* kv_state, float* score_state, csa2_bf16* plane,
                                int64_t plane_rows, const int64_t* row_base, const float* norm_w,
                                float eps, const float* inv_freq, const csa2_bf16* wk,
                                const float* knorm_w, csa2_bf16* index_plane, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_index_topk -- [A] "特殊模块 · indexer" Fig. 3b and "visible 是每行自己的前缀长度";
 * [A] Fig. 2c (candidate blocks); [C] A.15.2.
 *
 * For query q (sequence q_seq[q], position q_pos[q]) the visible rows are
 * c < n_vis = floor((q_pos[q] + 1) / ratio).  Each scored row c gets
 *     s(c) = alpha * sum_h w[q][h] * relu(<iq[q][h], index_k[row_base[b] + c]>),
 *     alpha = 128^-1/2 * H^-1/2   (relu dropped when relu == 0)
 * FULL mode (cand == NULL): every visible row is scored.
 * REINDEX mode: only rows 8*cand[q][i] + r (r < 8) that are visible; cand[q] holds
 * ncb block ids in ascending order, -1 padded.
 * The k_eff = min(k, #scored) highest scores are kept (ties: lower row id;
 * NaN ranks as -inf) and written as ascending row ids to sel[q][0..k_eff), the rest
 * of sel[q][0..k) set to -1.  sel_scores (optional) receives the matching scores
 * (0 for -1 entries).
 *   iq         [Q][H][128] bf16;  w [Q][H] fp32;  H = 32 or 64
 *   index_k    [index_rows][128] bf16;  row_base [..] int64;  q_seq [Q] int32;
 *   q_pos      [Q] int64
 *   max_scored bound on positions scored per query: FULL >= max n_vis (larger n_vis
 *              raises CSA2_EBOUNDS and is clipped); REINDEX must equal ncb * 8
 *   k          1..512;  REINDEX requires ncb * 8 >= k
 *   scores_out optional [Q][max_scored] fp32: the score of every position (FULL:
 *              position = row; REINDEX: position = 8 * i + r); unscored positions
 *              are not written.  For tests.
 *   ws         workspace of at least csa2_index_topk_workspace_size(Q, H,
 *              max_scored, k) bytes, 256-byte aligned; contents are scratch. */
size_t csa2_index_topk_workspace_size(int Q, int H, int64_t max_scored, int k);
csa2_status csa2_index_topk(const csa2_bf16* iq, const float* w, int Q, int H,
                            const csa2_bf16* index_k, int64_t index_rows,
                            const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos,
                            int ratio, const int32_t* cand, int ncb, int k, int relu,
                            int64_t max_scored, int32_t* sel, float* sel_scores,
                            float* scores_out, void* ws, size_t ws_bytes, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_compress_index_topk -- csa2_compress and csa2_index_topk as one call: the first
 * two parts of the step ([A] "特殊模块 · compressor" and "特殊模块 · indexer" Fig. 3b,
 * as for the two calls).  The compressor writes only the main plane and its states,
 * which the indexer does not read (the index plane is an input), so the library runs
 * the compressor's tokens on extra CTAs of the top-k launch, beside the selection (on
 * SMs it leaves idle), instead of as a kernel of its own; the step is then one chain of
 * kernels on one stream.  The results are exactly those of
 * csa2_compress followed by csa2_index_topk with the same arguments (bit for bit: the
 * same per-token and per-row arithmetic), and a following csa2_sparse_attn on the
 * same stream sees the compressed rows.
 *   kv, score, T, cu_seqlens, B, start_pos, kv_state, score_state, plane, plane_rows,
 *   norm_w, eps, inv_freq   as csa2_compress (ratio and row_base are shared with the
 *                           indexer); T == 0 compresses nothing
 *   the remaining arguments as csa2_index_topk (bf16 index plane)
 * Errors: the compressor's argument checks first, then the indexer's; nothing is
 * enqueued when either fails.  With Q == 0 only the compressor runs. */
csa2_status csa2_compress_index_topk(
    const csa2_bf16* kv, const csa2_bf16* score, int T, const int32_t* cu_seqlens, int B,
    const int64_t* start_pos, float* kv_state, float* score_state, csa2_bf16* plane,
    int64_t plane_rows, const float* norm_w, float eps, const float* inv_freq,
    const csa2_bf16* iq, const float* w, int Q, int H, const csa2_bf16* index_k,
    int64_t index_rows, const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos,
    int ratio, const int32_t* cand, int ncb, int k, int relu, int64_t max_scored, int32_t* sel,
    float* sel_scores, float* scores_out, void* ws, size_t ws_bytes, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_index_topk_pool -- csa2_index_topk in FULL mode plus the candidate pool that a
 * FULL layer hands to the REINDEX layers after it.  [A] Fig. 3b (second stage of the
 * indexer: block maxima, newest block pinned to +inf, top-2048 blocks, ascending, -1
 * padded); [B] §5.2 (a block scores as its best row; the partial newest block is
 * always kept); [C] A.11 (2048 candidate blocks of 8 rows).
 *
 * sel / sel_scores / scores_out are those of csa2_index_topk with cand == NULL.  In
 * addition, for query q with n_vis visible rows, block j (rows 8j .. 8j+7, j <
 * ceil(n_vis / 8)) scores as the largest s(c) of its visible rows (NaN ranks as -inf;
 * +inf ranks below the pinned block), the newest block ceil(n_vis / 8) - 1 is pinned
 * above every score, and the min(nbk, ceil(n_vis / 8)) best blocks (ties: lower block
 * id) are written as ascending block ids to pool[q][0..), the rest of pool[q][0..nbk)
 * set to -1.  pool rows feed csa2_index_topk's `cand` (ncb = nbk) directly.
 *   nbk        1..2048, with ceil(max_scored / 8) blocks per row selectable
 *              (csa2_index_topk_pool_workspace_size returns 0 otherwise)
 *   pool       [Q][nbk] int32
 *   ws         workspace of csa2_index_topk_pool_workspace_size(Q, H, max_scored, k,
 *              nbk) bytes, 256-byte aligned; contents are scratch.
 * Other arguments and errors as csa2_index_topk (cand = NULL). */
size_t csa2_index_topk_pool_workspace_size(int Q, int H, int64_t max_scored, int k, int nbk);
csa2_status csa2_index_topk_pool(const csa2_bf16* iq, const float* w, int Q, int H,
                                 const csa2_bf16* index_k, int64_t index_rows,
                                 const int64_t* row_base, const int32_t* q_seq,
                                 const int64_t* q_pos, int ratio, int k, int relu,
                                 int64_t max_scored, int32_t* sel, float* sel_scores,
                                 float* scores_out, int nbk, int32_t* pool, void* ws,
                                 size_t ws_bytes, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_index_plane_fp8 -- the FP8 index plane.  [A] indexer figure (FP8 index rows of
 * 132 B: 128 E4M3 codes and one fp32 scale; blocks of 8 rows with the values first and
 * the scales at the block tail); [E] indexer compressor (row amax -> ue8m0 -> e4m3).
 *
 * Row r of index_k [rows][128] bf16 is quantised with the scale s = 2^e, the smallest
 * power of two with max_d |x_d| / s <= 448 (s = 1 for an all-zero row), into codes
 * E4M3(x_d / s) (nearest, ties to even).  Block b = r / 8 of the plane holds, at byte
 * 1056 * b, the codes of rows 8b .. 8b+7 (128 bytes each) and then their 8 scales as
 * fp32.  Rows of the last block past `rows` are zero with scale 1.
 *   plane  csa2_index_plane_fp8_bytes(rows) bytes, 16-byte aligned */
size_t csa2_index_plane_fp8_bytes(int64_t rows);
csa2_status csa2_index_plane_fp8(const csa2_bf16* index_k, int64_t rows, uint8_t* plane,
                                 csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_index_topk_fp8 -- csa2_index_topk on an FP8 index plane.  [A] indexer figure
 * (FP8 plane; the query quantised per (token, head), its fp32 scale folded into w).
 *
 * Each query row iq[q][h] is quantised like a plane row (scale sq_qh, codes cq); with
 * plane row c of sequence b = the row row_base[b] + c of the plane (codes ck_c, scale
 * sk_c),
 *     s(c) = alpha * sum_h w[q][h] * relu(sq_qh * sk_c * <E4M3(cq_qh), E4M3(ck_c)>)
 * on the tensor cores (E4M3 x E4M3 products, fp32 sums); everything else (visibility,
 * REINDEX, selection, outputs, errors) as csa2_index_topk.
 *   plane      csa2_index_plane_fp8 layout holding index_rows rows; every row_base[b]
 *              must be a multiple of 8 (each sequence starts on a block; a query of a
 *              sequence that does not raises CSA2_EBOUNDS)
 *   ws         csa2_index_topk_fp8_workspace_size(Q, H, max_scored, k) bytes */
size_t csa2_index_topk_fp8_workspace_size(int Q, int H, int64_t max_scored, int k);
csa2_status csa2_index_topk_fp8(const csa2_bf16* iq, const float* w, int Q, int H,
                                const uint8_t* plane, int64_t index_rows,
                                const int64_t* row_base, const int32_t* q_seq,
                                const int64_t* q_pos, int ratio, const int32_t* cand, int ncb,
                                int k, int relu, int64_t max_scored, int32_t* sel,
                                float* sel_scores, float* scores_out, void* ws, size_t ws_bytes,
                                csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_index_plane_fp4 -- the MXFP4 index plane.  [A] indexer figure (FP4 index rows of
 * 68 B: 64 B of values and 4 B of scales; planes paged in blocks of 8 rows); [A] indexer
 * K (E2M1 values with one E8M0 scale per 32 channels, pure powers of two).
 *
 * Quantises rows 0 .. rows-1 of a bf16 [rows][128] index plane.  Block b of the output
 * starts at byte 544 * b: 8 x 64 code bytes for rows 8b .. 8b+7 (byte i of a row holds
 * dim 2i in its low nibble and dim 2i+1 in its high nibble), then 8 x 4 scale bytes (byte
 * j of a row scales dims 32j .. 32j+31 by 2^(e - 127)).  A group's e is the smallest in
 * [0, 254] with max |x| <= 6 * 2^(e - 127), 127 for an all-zero group; its codes are the
 * E2M1 values nearest x / 2^(e - 127), ties to the even code.  Rows of the last block past
 * `rows` are zero with e = 127.  The values must stay below 3 * 2^125 in magnitude.
 *   index_k  device, [rows][128] bf16, 16-byte aligned
 *   plane    device, csa2_index_plane_fp4_bytes(rows) bytes, 16-byte aligned */
size_t csa2_index_plane_fp4_bytes(int64_t rows);
csa2_status csa2_index_plane_fp4(const csa2_bf16* index_k, int64_t rows, uint8_t* plane,
                                 csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_index_topk_fp4 -- csa2_index_topk on an MXFP4 index plane.  [A] indexer figure
 * (the FP4 plane); [A] Fig. 3b (the scores).
 *
 * K[c][d] is the decoded plane value (an E2M1 value times its group's power of two,
 * which bf16 holds exactly); the queries stay bf16 and the scores are those of
 * csa2_index_topk on these K rows, computed on the tensor cores in bf16 with fp32 sums.
 * Everything else (visibility, REINDEX, selection, outputs, errors) as csa2_index_topk.
 *   plane      csa2_index_plane_fp4 layout holding index_rows rows; every row_base[b]
 *              must be a multiple of 8 (each sequence starts on a block; a query of a
 *              sequence that does not raises CSA2_EBOUNDS); a REINDEX candidate block
 *              outside the plane raises CSA2_EBOUNDS
 *   ws         csa2_index_topk_fp4_workspace_size(Q, H, max_scored, k) bytes */
size_t csa2_index_topk_fp4_workspace_size(int Q, int H, int64_t max_scored, int k);
csa2_status csa2_index_topk_fp4(const csa2_bf16* iq, const float* w, int Q, int H,
                                const uint8_t* plane, int64_t index_rows,
                                const int64_t* row_base, const int32_t* q_seq,
                                const int64_t* q_pos, int ratio, const int32_t* cand, int ncb,
                                int k, int relu, int64_t max_scored, int32_t* sel,
                                float* sel_scores, float* scores_out, void* ws, size_t ws_bytes,
                                csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_index_topk_noalloc -- the paper has no counterpart: this is a library service.
 *
 * Same arguments and results as csa2_index_topk, minus the workspace.  It is for
 * callers that cannot provide device scratch memory: a plugin driven through a fixed
 * interface that passes only its inputs and outputs, an engine that owns all device
 * memory through its own pool and forbids other allocations, or a path that cannot
 * afford the device-wide synchronisation of cudaMalloc/cudaFree.  The scratch lives in
 * a fixed 64 MiB device array inside the library, present on every GPU that loads the
 * library until the process exits; the call itself allocates nothing.
 *   - Sizes needing more than 64 MiB (see csa2_index_topk_workspace_size) are refused
 *     with CSA2_ENOSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address with a host-side
 *     runtime call; make that first call before any stream capture.  The address is
 *     kept per device together with the CUDA context it came from; after a device reset
 *     or a re-created primary context the next call looks it up again (so, after a
 *     reset, make one call before capturing again).
 *   - A failed lookup returns CSA2_ECUDA with the CUDA error text in csa2_last_error()
 *     and leaves no error pending in cudaGetLastError().
 *   - All calls on a device share the array.  Calls whose kernels can overlap on the
 *     GPU (unordered streams) race and give wrong results: order them.
 *   - Nothing in the array needs to start at zero: each call writes every entry it
 *     reads, so stale contents of an earlier call are harmless. */
csa2_status csa2_index_topk_noalloc(const csa2_bf16* iq, const float* w, int Q, int H,
                                    const csa2_bf16* index_k, int64_t index_rows,
                                    const int64_t* row_base, const int32_t* q_seq,
                                    const int64_t* q_pos, int ratio, const int32_t* cand, int ncb,
                                    int k, int relu, int64_t max_scored, int32_t* sel,
                                    float* sel_scores, float* scores_out, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_topk_scores -- the selection step of csa2_index_topk on given scores.
 * [A] Fig. 3b (top_k_per_row: ascending, -1 padded).
 *
 * For row q of scores [Q][ld] fp32, the k_eff = min(k, n[q]) highest of
 * scores[q][0..n[q]) (ties: lower index; NaN ranks as -inf; -0 equals +0) are
 * written as ascending indices to sel[q][0..k_eff), -1 after.  sel_scores optional.
 *   n  [Q] int32, 0 <= n[q] <= ld;  k 1..2048.  A row of up to 65536 positions is
 *      selected by one CTA (no workspace); longer rows are cut into ceil(ld / 32768)
 *      chunks whose top-k lists are merged: chunks * k must be <= 32768
 *      (csa2_topk_workspace_size returns 0 otherwise)
 *   ws workspace of csa2_topk_workspace_size(Q, ld, k) bytes, 256-byte aligned. */
size_t csa2_topk_workspace_size(int Q, int64_t ld, int k);
csa2_status csa2_topk_scores(const float* scores, const int32_t* n, int Q, int64_t ld, int k,
                             int32_t* sel, float* sel_scores, void* ws, size_t ws_bytes,
                             csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_sparse_attn -- [A] "四种层合并出来的是什么形状" and Fig. 2a-2d; [B] §4.1, §4.4;
 * [C] §5.5-5.6, A.19.3; [E] Fig. 2d (sink in the denominator).
 *
 * Query q (sequence b = q_seq[q], position p = q_pos[q]) attends, with all 64 heads,
 * to the entry set
 *     window:   positions max(0, p-127) .. p of the layer's own sliding window
 *     selected: plane rows row_base[b] + sel[q][i] for sel[q][i] != -1
 * (the two parts are not de-duplicated, at most 128 + 512 entries).  Each entry's
 * 512-d vector x_j serves as key and value:
 *     s_j   = scale * <q[q][h], x_j>
 *     out_h = sum_j e^{s_j} x_j / (e^{sink[h]} + sum_j e^{s_j})
 *     lse_h = ln(e^{sink[h]} + sum_j e^{s_j})
 * computed with fp32 accumulation of bf16 operands; out is bf16 and still carries
 * the RoPE phase of the keys (the inverse rotation is not part of this call).
 *   q      [Q][64][512] bf16;  q_seq [Q] int32;  q_pos [Q] int64
 *   swa    window source (HOST struct, device pointers inside):
 *          RING:   data holds [B][128] rows, position pos in slot pos % 128
 *          LINEAR: data holds rows; position pos of sequence b is row
 *                  lin_base[b] + pos - lin_pos0[b]; the rows must cover every
 *                  window position max(0, p-127) .. p of each query, i.e.
 *                  lin_pos0[b] <= max(0, p-127).  A window position below lin_pos0[b]
 *                  raises CSA2_EBOUNDS and is skipped (it is never read from another
 *                  sequence's rows)
 *          BF16 rows are 512 bf16; FP8_S128 rows are 528 bytes: 512 E4M3 codes then
 *          four fp32 scales, value = code * scale[d / 128]; FP8_E8M0 rows are 528
 *          bytes: 512 E4M3 codes then 16 E8M0 scales, value = code * 2^(e[d / 32] - 127)
 *          ([A] pool switch: nvfp4 window rows of 512 FP8 and 16 E8M0)
 *          n_rows = rows in data, < 2^31 (indices beyond raise CSA2_EBOUNDS and are
 *          skipped)
 *   plane  [plane_rows][512] bf16, plane_rows < 2^31;  row_base int64;
 *          sel [Q][nsel] int32, nsel <= 512
 *          (sel may be NULL with nsel == 0: window only)
 *   sink   [64] fp32 or NULL (no sink term);  scale: softmax temperature (1/sqrt(512))
 *   out    [Q][64][512] bf16;  lse [Q][64] fp32 or NULL
 *   ws     optional workspace (256-byte aligned, NULL allowed) of
 *          csa2_attn_workspace_size(Q, nsel) bytes, which is 0: a query's entries run on
 *          one CTA, or on two that merge in distributed shared memory when 2 Q CTAs fit
 *          on the GPU at once; with more queries than SMs one CTA per SM walks its
 *          queries in turn.  The argument is kept so that callers that size and pass a
 *          workspace need no change. */
typedef enum { CSA2_SWA_RING = 0, CSA2_SWA_LINEAR = 1 } csa2_swa_mode;
typedef enum { CSA2_SWA_BF16 = 0, CSA2_SWA_FP8_S128 = 1, CSA2_SWA_FP8_E8M0 = 2 } csa2_swa_dtype;
typedef struct {
  int32_t mode;            /* csa2_swa_mode */
  int32_t dtype;           /* csa2_swa_dtype */
  const void* data;        /* device rows, see above */
  int64_t n_rows;          /* rows in data */
  const int64_t* lin_base; /* LINEAR only: device [B] */
  const int64_t* lin_pos0; /* LINEAR only: device [B] */
} csa2_swa;

size_t csa2_attn_workspace_size(int Q, int nsel);
csa2_status csa2_sparse_attn(const csa2_bf16* q, int Q, const int32_t* q_seq,
                             const int64_t* q_pos, const csa2_swa* swa, const csa2_bf16* plane,
                             int64_t plane_rows, const int64_t* row_base, const int32_t* sel,
                             int nsel, const float* sink, float scale, csa2_bf16* out, float* lse,
                             void* ws, size_t ws_bytes, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_reuse_attn -- [A] Fig. 2d (REUSE: no scoring kernel, the selection of the
 * group's first layer is replayed); [C] A.8.1.
 * Identical arguments and result to csa2_sparse_attn; `sel` is the stored selection
 * of the index-group start layer while q and swa are this layer's own. */
csa2_status csa2_reuse_attn(const csa2_bf16* q, int Q, const int32_t* q_seq,
                            const int64_t* q_pos, const csa2_swa* swa, const csa2_bf16* plane,
                            int64_t plane_rows, const int64_t* row_base, const int32_t* sel,
                            int nsel, const float* sink, float scale, csa2_bf16* out, float* lse,
                            void* ws, size_t ws_bytes, csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_sparse_attn_rope, csa2_reuse_attn_rope -- the same calls with the output's
 * inverse RoPE fused in: [A] "出来之后" (out -> inverse RoPE at the query's own
 * position, because K = V carries the rotation); [B] §6.1 (the output's last 64 dims
 * times the conjugate phase, apply_rotary_emb(o, freqs, inverse=True)); [C] A.12.1.
 * After the softmax-weighted sum, pair i of dims 448 + 2i, 449 + 2i of every head,
 * read as a complex number, is multiplied by e^{-i p theta_i}, p = q_pos[q],
 * theta_i = inv_freq[i] (the same 32-entry table as csa2_compress); the other 448 dims
 * are unchanged.  Arguments as csa2_sparse_attn / csa2_reuse_attn, plus
 *   inv_freq  [32] fp32 device, required (NULL is CSA2_EINVAL).
 * The rotation angle is computed from an exact 64-bit phase of p, so it holds for any
 * position the int64 q_pos can hold. */
csa2_status csa2_sparse_attn_rope(const csa2_bf16* q, int Q, const int32_t* q_seq,
                                  const int64_t* q_pos, const csa2_swa* swa,
                                  const csa2_bf16* plane, int64_t plane_rows,
                                  const int64_t* row_base, const int32_t* sel, int nsel,
                                  const float* sink, float scale, csa2_bf16* out, float* lse,
                                  void* ws, size_t ws_bytes, const float* inv_freq,
                                  csa2_stream stream);
csa2_status csa2_reuse_attn_rope(const csa2_bf16* q, int Q, const int32_t* q_seq,
                                 const int64_t* q_pos, const csa2_swa* swa,
                                 const csa2_bf16* plane, int64_t plane_rows,
                                 const int64_t* row_base, const int32_t* sel, int nsel,
                                 const float* sink, float scale, csa2_bf16* out, float* lse,
                                 void* ws, size_t ws_bytes, const float* inv_freq,
                                 csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_plane_fp4 -- the FP4 main plane.  [A] pool switch ("nvfp4": main plane rows of
 * 288 B, the 512 dims as E2M1 with an E4M3 scale per group of 16).
 *
 * Row r of plane [rows][512] bf16 becomes 288 bytes: bytes 0..255 the 512 E2M1 codes,
 * dim 2i in the low nibble of byte i and dim 2i + 1 in its high nibble; bytes 256..287
 * the 32 E4M3 scales, scale g for dims 16g .. 16g + 15.  A group's scale is the smallest
 * E4M3 value s with 6 s >= max |x| (0 for an all-zero group, 448 at most); its codes are
 * E2M1(x / s), nearest, ties to even, saturating at 6 (0 when s == 0).  The value of dim
 * d is E2M1(code) * E4M3(scale), which bf16 holds exactly.
 *   out  csa2_plane_fp4_bytes(rows) bytes, 16-byte aligned; plane 16-byte aligned */
size_t csa2_plane_fp4_bytes(int64_t rows);
csa2_status csa2_plane_fp4(const csa2_bf16* plane, int64_t rows, uint8_t* out,
                           csa2_stream stream);

/* ---------------------------------------------------------------------------------
 * csa2_sparse_attn_fp4 -- csa2_sparse_attn (or csa2_reuse_attn: the same computation)
 * reading the selected rows from an FP4 plane (csa2_plane_fp4 layout, plane_rows rows
 * of 288 bytes); the window is unchanged.  Each selected row is dequantised exactly to
 * bf16 before the dot products.  inv_freq: NULL, or the table of csa2_sparse_attn_rope
 * for the output's inverse RoPE.  [A] pool switch; the rest as csa2_sparse_attn. */
csa2_status csa2_sparse_attn_fp4(const csa2_bf16* q, int Q, const int32_t* q_seq,
                                 const int64_t* q_pos, const csa2_swa* swa, const uint8_t* plane,
                                 int64_t plane_rows, const int64_t* row_base, const int32_t* sel,
                                 int nsel, const float* sink, float scale, csa2_bf16* out,
                                 float* lse, void* ws, size_t ws_bytes, const float* inv_freq,
                                 csa2_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */

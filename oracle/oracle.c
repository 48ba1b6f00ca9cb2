/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle of the CSA2 attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code with the CUDA path.
 *
 * Arithmetic is IEEE double throughout; bf16 inputs are widened exactly, and the
 * only rounding to bf16 is the compressor's final store (one rounding, ties to
 * even).  Each function names the passage of the source pages it restates.
 * Pages:
 *   [A] "DeepSeek-V4.1-Flash 架构解剖" (perryzhang01.github.io, v41_flash_anatomy)
 *   [B] "DeepSeek-V4.1-Flash 结构说明" (treert.github.io, ds-v4-1-flash-structure)
 *   [C] "万字长文解析DeekSeekV4.1flash" (yuyanqi.com)
 *   [E] "DeepSeek-V4-Pro 架构解剖" (perryzhang01.github.io, v4_pro_anatomy)
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_LAT 512
#define D_IDX 128
#define N_HEADS 64
#define ROPE_DIM0 448
#define RING 128

/* ---- number formats ----------------------------------------------------------- */

static double bf16_val(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16, ties to even, in one rounding. */
uint16_t orc_f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  double m = frexp(a, &e); /* a = m * 2^e, 0.5 <= m < 1 */
  if (e - 1 < -126) {      /* subnormal: quantum 2^-133 */
    double qv = nearbyint(ldexp(a, 133));
    return sign | (uint16_t)qv; /* 128 is the smallest normal, encoded 0x0080 */
  }
  double s = nearbyint(ldexp(m, 8)); /* 8 significant bits: 128..256 */
  if (s == 256.0) { s = 128.0; e += 1; }
  int E = e - 1;
  if (E > 127) return sign | 0x7F80;
  return sign | (uint16_t)(((E + 127) << 7) | ((int)s - 128));
}

/* OCP FP8 E4M3 decode from the format's definition: bias 7, 3 mantissa bits,
 * exponent field 0 is subnormal (m/8 * 2^-6), S.1111.111 is NaN. */
double orc_e4m3_val(uint8_t c) {
  int sgn = c >> 7, ex = (c >> 3) & 15, mn = c & 7;
  double v;
  if (ex == 15 && mn == 7) return NAN;
  if (ex == 0) v = ldexp((double)mn / 8.0, -6);
  else v = ldexp(1.0 + (double)mn / 8.0, ex - 7);
  return sgn ? -v : v;
}

/* OCP FP8 E4M3 encode from the same definition: round to nearest, ties to the even
 * mantissa, finite values beyond the largest (448 = 1.75 * 2^8) saturate to it (the
 * format has no infinity).  Subnormals step by 2^-9 below 2^-6. */
uint8_t orc_e4m3_code(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (a < ldexp(1.0, -6)) {                       /* subnormal range (or zero) */
    double qv = nearbyint(ldexp(a, 9));            /* 0 .. 8; 8 is the smallest normal */
    return sign | (uint8_t)qv;
  }
  int e;
  double m = frexp(a, &e);                         /* a = m * 2^e, 0.5 <= m < 1 */
  int E = e - 1;                                   /* a = (2m) * 2^E, 1 <= 2m < 2 */
  double q = nearbyint((2.0 * m - 1.0) * 8.0);     /* mantissa steps of 1/8 */
  if (q == 8.0) { q = 0.0; E += 1; }
  if (E > 8 || (E == 8 && q > 6.0)) return sign | 0x7E;  /* saturate to 448 */
  return sign | (uint8_t)(((E + 7) << 3) | (int)q);
}

/* Power-of-two (E8M0) scale of a group with largest magnitude amax: the smallest
 * 2^e with amax / 2^e <= 448, so the group's codes use the top of the E4M3 range
 * without saturating.  amax == 0 gives 1.  [E] indexer compressor ("row amax ->
 * ue8m0 -> e4m3"). */
double orc_ue8m0_scale(double amax) {
  if (!(amax > 0.0)) return 1.0;
  int e;
  frexp(amax, &e);
  e -= 9;                                          /* below the answer */
  while (amax > 448.0 * ldexp(1.0, e)) e++;
  return ldexp(1.0, e);
}

/* OCP FP4 E2M1 from its definition: sign, 2 exponent bits (bias 1), 1 mantissa bit;
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7. */
double orc_e2m1_val(uint8_t c) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  return (c & 8) ? -mag[c & 7] : mag[c & 7];
}

/* Nearest E2M1 code, ties to the even code (mantissa bit 0), beyond 6 saturating to 6. */
uint8_t orc_e2m1_code(double x) {
  uint8_t sign = signbit(x) ? 8 : 0;
  double a = fabs(x);
  int best = 0;
  for (int c = 1; c < 8; c++) {
    double dc = fabs(orc_e2m1_val((uint8_t)c) - a), db = fabs(orc_e2m1_val((uint8_t)best) - a);
    if (dc < db || (dc == db && (c & 1) == 0)) best = c;
  }
  return sign | (uint8_t)best;
}

/* ---- visibility [A] "visible 是每行自己的前缀长度"; [B] §4.1 -------------------- */

/* Compressed row j covers positions j*m .. j*m+m-1 and becomes visible to the
 * query at position p once p has passed its last token.  Written as the count
 * of such rows, by enumeration. */
int64_t orc_n_visible(int64_t p, int m) {
  int64_t n = 0;
  while ((n + 1) * m - 1 <= p) n++;
  return n;
}

/* ---- compressor [A] "特殊模块 · compressor", "CSA2 的池化比 V4 简单一截";
 *      [C] §6.2, §6.4, A.15.1; [B] §4.1 (tail), §6.1-6.2 (RoPE) ---------------------
 *
 * Every new token at position t is appended to the tail slot t % m.  When the slot
 * is the last of its group (t % m == m-1) the group j = t / m is complete:
 *   r[d]  = sum_i softmax_i(score[i][d]) * kv[i][d]     (softmax over the m slots)
 *   y     = r / sqrt(mean(r^2) + eps) * norm_w          (RMSNorm over all 512 dims)
 *   y[448+2i], y[449+2i] rotated by angle (j*m) * inv_freq[i], i < 32
 * and y is stored to plane row row_base[b] + j as bf16.
 * State arrays are [B][m][512]; slot s holds the last token with t % m == s.
 * Returns the number of rows emitted in total. */
/* ---- index K of a compressed row [A] indexer figure, key side ("the compressed,
 *      pre-RoPE latent [512] BF16 -> indexer.wk [128, 512] -> k_norm -> RoPE -> the
 *      index plane"); [A] compressor figure (the two branches part after RMSNorm);
 *      [C] A.6.2 (index K projected from the main latent) -----------------------------
 *
 * x = bf16(y) is the row's normalized latent before RoPE, rounded to bf16 once;
 *   k[o] = sum_d wk[o][d] x[d]                     (o < 128)
 *   k    = k / sqrt(mean(k^2) + eps) * knorm_w     (RMSNorm over the 128 dims)
 *   k[64+2i], k[65+2i] rotated by angle p0 * inv_freq[i], i < 32 (the last 64 dims)
 * at the row's group-head position p0; stored as bf16 (and as double in k_f64). */
static void index_k_row(const double* y, double p0, const uint16_t* wk, const float* knorm_w,
                        double eps, const float* inv_freq, uint16_t* out, double* out_f64) {
  double x[D_LAT], k[D_IDX];
  for (int d = 0; d < D_LAT; d++) x[d] = bf16_val(orc_f64_to_bf16(y[d]));
  for (int o = 0; o < D_IDX; o++) {
    double acc = 0.0;
    for (int d = 0; d < D_LAT; d++) acc += bf16_val(wk[o * D_LAT + d]) * x[d];
    k[o] = acc;
  }
  double ms = 0.0;
  for (int o = 0; o < D_IDX; o++) ms += k[o] * k[o];
  double inv = 1.0 / sqrt(ms / D_IDX + eps);
  for (int o = 0; o < D_IDX; o++) k[o] = k[o] * inv * (knorm_w ? (double)knorm_w[o] : 1.0);
  for (int i = 0; i < 32; i++) {
    double ang = p0 * (double)inv_freq[i];
    double c = cos(ang), s = sin(ang);
    double a0 = k[64 + 2 * i], a1 = k[64 + 2 * i + 1];
    k[64 + 2 * i] = a0 * c - a1 * s;
    k[64 + 2 * i + 1] = a0 * s + a1 * c;
  }
  for (int o = 0; o < D_IDX; o++) {
    out[o] = orc_f64_to_bf16(k[o]);
    if (out_f64) out_f64[o] = k[o];
  }
}

/* orc_compress with, when wk != NULL, the row's index K written to index_plane (and
 * index_f64) at the same row. */
int64_t orc_compress_index(const uint16_t* kv, const uint16_t* score, const int32_t* cu_seqlens,
                           int B, const int64_t* start_pos, int m, double* kv_state,
                           double* score_state, uint16_t* plane, double* plane_f64,
                           const int64_t* row_base, const float* norm_w, double eps,
                           const float* inv_freq, const uint16_t* wk, const float* knorm_w,
                           uint16_t* index_plane, double* index_f64);

int64_t orc_compress(const uint16_t* kv, const uint16_t* score, const int32_t* cu_seqlens, int B,
                     const int64_t* start_pos, int m, double* kv_state, double* score_state,
                     uint16_t* plane, double* plane_f64, const int64_t* row_base,
                     const float* norm_w, double eps, const float* inv_freq) {
  return orc_compress_index(kv, score, cu_seqlens, B, start_pos, m, kv_state, score_state, plane,
                            plane_f64, row_base, norm_w, eps, inv_freq, NULL, NULL, NULL, NULL);
}

int64_t orc_compress_index(const uint16_t* kv, const uint16_t* score, const int32_t* cu_seqlens,
                           int B, const int64_t* start_pos, int m, double* kv_state,
                           double* score_state, uint16_t* plane, double* plane_f64,
                           const int64_t* row_base, const float* norm_w, double eps,
                           const float* inv_freq, const uint16_t* wk, const float* knorm_w,
                           uint16_t* index_plane, double* index_f64) {
  int64_t emitted = 0;
  for (int b = 0; b < B; b++) {
    double* ks = kv_state + (int64_t)b * m * D_LAT;
    double* ss = score_state + (int64_t)b * m * D_LAT;
    for (int64_t t = cu_seqlens[b]; t < cu_seqlens[b + 1]; t++) {
      int64_t pos = start_pos[b] + (t - cu_seqlens[b]);
      int slot = (int)(pos % m);
      for (int d = 0; d < D_LAT; d++) {
        ks[slot * D_LAT + d] = bf16_val(kv[t * D_LAT + d]);
        ss[slot * D_LAT + d] = score ? bf16_val(score[t * D_LAT + d]) : 0.0;
      }
      if (slot != m - 1) continue;
      int64_t j = pos / m;
      double y[D_LAT];
      for (int d = 0; d < D_LAT; d++) {
        double mx = -INFINITY;
        for (int i = 0; i < m; i++) mx = fmax(mx, ss[i * D_LAT + d]);
        double z = 0.0, acc = 0.0;
        for (int i = 0; i < m; i++) {
          double e = exp(ss[i * D_LAT + d] - mx);
          z += e;
          acc += e * ks[i * D_LAT + d];
        }
        y[d] = acc / z;
      }
      double ms = 0.0;
      for (int d = 0; d < D_LAT; d++) ms += y[d] * y[d];
      double inv = 1.0 / sqrt(ms / D_LAT + eps);
      for (int d = 0; d < D_LAT; d++) y[d] = y[d] * inv * (norm_w ? (double)norm_w[d] : 1.0);
      double p0 = (double)(j * m); /* group-head position */
      if (wk) /* the indexer's branch leaves before the main RoPE */
        index_k_row(y, p0, wk, knorm_w, eps, inv_freq, index_plane + (row_base[b] + j) * D_IDX,
                    index_f64 ? index_f64 + (row_base[b] + j) * D_IDX : NULL);
      for (int i = 0; i < 32; i++) {
        double ang = p0 * (double)inv_freq[i];
        double c = cos(ang), s = sin(ang);
        double a0 = y[ROPE_DIM0 + 2 * i], a1 = y[ROPE_DIM0 + 2 * i + 1];
        y[ROPE_DIM0 + 2 * i] = a0 * c - a1 * s;
        y[ROPE_DIM0 + 2 * i + 1] = a0 * s + a1 * c;
      }
      int64_t row = row_base[b] + j;
      for (int d = 0; d < D_LAT; d++) {
        plane[row * D_LAT + d] = orc_f64_to_bf16(y[d]);
        if (plane_f64) plane_f64[row * D_LAT + d] = y[d];
      }
      emitted++;
    }
  }
  return emitted;
}

/* ---- lightning indexer [A] "特殊模块 · indexer" Fig. 3b (score formula and
 *      weights_scale); [C] A.15.2 (ReLU per head, gather candidates first);
 *      [A] Fig. 2c (candidate blocks x 8 rows) -------------------------------------
 *
 * score[c] = alpha * sum_h w[h] * act(<iq[h], K[c]>),  alpha = 128^-1/2 * H^-1/2,
 * act = ReLU when relu != 0, identity otherwise.
 * FULL (cand == NULL): positions c < n_visible(p) are rows c.
 * REINDEX: position i*8 + r is row 8*cand[i] + r; it is scored only when
 * cand[i] >= 0 and that row is visible.
 * Outputs per query q: scores[q*ld + pos] and rows[q*ld + pos] (-1 = not scored). */
void orc_index_scores(const uint16_t* iq, const float* w, int Q, int H, const uint16_t* index_k,
                      const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos, int m,
                      const int32_t* cand, int ncb, int relu, double* scores, int64_t* rows,
                      int64_t ld) {
  double alpha = 1.0 / sqrt((double)D_IDX) / sqrt((double)H);
  for (int q = 0; q < Q; q++) {
    int64_t nvis = orc_n_visible(q_pos[q], m);
    const uint16_t* kb = index_k + row_base[q_seq[q]] * D_IDX;
    double qv[64 * D_IDX];
    for (int i = 0; i < H * D_IDX; i++) qv[i] = bf16_val(iq[(int64_t)q * H * D_IDX + i]);
    int64_t npos = cand ? (int64_t)ncb * 8 : nvis;
#pragma omp parallel for schedule(static)
    for (int64_t pos = 0; pos < ld; pos++) {
      int64_t row = -1;
      if (pos < npos) {
        if (!cand) row = pos;
        else {
          int32_t blk = cand[(int64_t)q * ncb + pos / 8];
          if (blk >= 0 && (int64_t)blk * 8 + pos % 8 < nvis) row = (int64_t)blk * 8 + pos % 8;
        }
      }
      rows[(int64_t)q * ld + pos] = row;
      if (row < 0) { scores[(int64_t)q * ld + pos] = 0.0; continue; }
      double kr[D_IDX];
      for (int d = 0; d < D_IDX; d++) kr[d] = bf16_val(kb[row * D_IDX + d]);
      double s = 0.0;
      for (int h = 0; h < H; h++) {
        double dot = 0.0;
        for (int d = 0; d < D_IDX; d++) dot += qv[h * D_IDX + d] * kr[d];
        if (relu && dot < 0.0) dot = 0.0;
        s += (double)w[(int64_t)q * H + h] * dot;
      }
      scores[(int64_t)q * ld + pos] = alpha * s;
    }
  }
}

/* ---- FP8 index plane [A] indexer figure (FP8: 132 B per row, blocks of 8 rows with
 *      the values first and the fp32 scales at the block tail; the query quantised per
 *      (token, head) with its fp32 scale folded into w); [E] indexer compressor
 *      ("row amax -> ue8m0 -> e4m3") -----------------------------------------------
 *
 * One row (128 bf16 values) -> scale = orc_ue8m0_scale(max |x|), codes = E4M3(x / scale).
 * Block b of the plane holds rows 8b .. 8b+7: 8 x 128 code bytes, then 8 fp32 scales
 * (1056 bytes).  n rows are written to ceil(n / 8) blocks; the rows of a partial last
 * block past n are zero with scale 1. */
void orc_index_plane_fp8(const uint16_t* k, int64_t n, uint8_t* plane) {
  int64_t nb = (n + 7) / 8;
  memset(plane, 0, (size_t)nb * 1056);
  for (int64_t r = 0; r < nb * 8; r++) {
    uint8_t* blk = plane + (r / 8) * 1056;
    float* sc = (float*)(blk + 1024);
    if (r >= n) { sc[r % 8] = 1.0f; continue; }
    double amax = 0.0;
    for (int d = 0; d < D_IDX; d++) {
      double v = fabs(bf16_val(k[r * D_IDX + d]));
      if (v > amax) amax = v;
    }
    double s = orc_ue8m0_scale(amax);
    for (int d = 0; d < D_IDX; d++)
      blk[(r % 8) * D_IDX + d] = orc_e4m3_code(bf16_val(k[r * D_IDX + d]) / s);
    sc[r % 8] = (float)s; /* a power of two: exact in fp32 */
  }
}

/* Index scores on the FP8 plane: the query of (q, h) is quantised like a plane row
 * (scale sq), the row c of sequence b is block (row_base[b] + c) / 8, slot
 * (row_base[b] + c) % 8 (row_base[b] is a multiple of 8), and
 *     s(c) = alpha * sum_h w[q][h] * relu(sq_h * sk_c * sum_d e4m3(qc_h,d) * e4m3(kc_c,d))
 * with the rest (visibility, REINDEX positions, alpha) as orc_index_scores. */
void orc_index_scores_fp8(const uint16_t* iq, const float* w, int Q, int H, const uint8_t* plane,
                          const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos,
                          int m, const int32_t* cand, int ncb, int relu, double* scores,
                          int64_t* rows, int64_t ld) {
  double alpha = 1.0 / sqrt((double)D_IDX) / sqrt((double)H);
  for (int q = 0; q < Q; q++) {
    int64_t nvis = orc_n_visible(q_pos[q], m);
    int64_t rb = row_base[q_seq[q]];
    double qv[64 * D_IDX], qs[64];
    for (int h = 0; h < H; h++) {
      const uint16_t* x = iq + ((int64_t)q * H + h) * D_IDX;
      double amax = 0.0;
      for (int d = 0; d < D_IDX; d++) if (fabs(bf16_val(x[d])) > amax) amax = fabs(bf16_val(x[d]));
      qs[h] = orc_ue8m0_scale(amax);
      for (int d = 0; d < D_IDX; d++) qv[h * D_IDX + d] = orc_e4m3_val(orc_e4m3_code(bf16_val(x[d]) / qs[h]));
    }
    int64_t npos = cand ? (int64_t)ncb * 8 : nvis;
#pragma omp parallel for schedule(static)
    for (int64_t pos = 0; pos < ld; pos++) {
      int64_t row = -1;
      if (pos < npos) {
        if (!cand) row = pos;
        else {
          int32_t blk = cand[(int64_t)q * ncb + pos / 8];
          if (blk >= 0 && (int64_t)blk * 8 + pos % 8 < nvis) row = (int64_t)blk * 8 + pos % 8;
        }
      }
      rows[(int64_t)q * ld + pos] = row;
      if (row < 0) { scores[(int64_t)q * ld + pos] = 0.0; continue; }
      const uint8_t* blk = plane + ((rb + row) / 8) * 1056;
      int slot = (int)((rb + row) % 8);
      float skf;
      memcpy(&skf, blk + 1024 + 4 * slot, 4);
      double sk = (double)skf;
      double kr[D_IDX];
      for (int d = 0; d < D_IDX; d++) kr[d] = orc_e4m3_val(blk[slot * D_IDX + d]);
      double s = 0.0;
      for (int h = 0; h < H; h++) {
        double dot = 0.0;
        for (int d = 0; d < D_IDX; d++) dot += qv[h * D_IDX + d] * kr[d];
        dot *= qs[h] * sk;
        if (relu && dot < 0.0) dot = 0.0;
        s += (double)w[(int64_t)q * H + h] * dot;
      }
      scores[(int64_t)q * ld + pos] = alpha * s;
    }
  }
}

/* ---- FP4 main plane [A] pool switch ("nvfp4": main plane rows of 288 B, the 512 dims
 *      as E2M1 with one E4M3 scale per group of 16) ---------------------------------
 *
 * Row layout: bytes 0..255 hold the 512 codes, element 2i in the low nibble of byte i
 * and element 2i + 1 in its high nibble; bytes 256..287 the 32 scales, scale g for
 * elements 16g .. 16g + 15.  A group's scale is the smallest E4M3 value s with 6 s >=
 * max |x| (0 for an all-zero group; the largest, 448, beyond), its codes E2M1(x / s)
 * (0 when s == 0); the value of element d is E2M1(code) * E4M3(scale). */
void orc_plane_fp4(const uint16_t* rows, int64_t n, uint8_t* out) {
  for (int64_t r = 0; r < n; r++) {
    uint8_t* o = out + r * 288;
    memset(o, 0, 288);
    for (int g = 0; g < 32; g++) {
      double amax = 0.0;
      for (int i = 0; i < 16; i++) {
        double v = fabs(bf16_val(rows[r * D_LAT + 16 * g + i]));
        if (v > amax) amax = v;
      }
      uint8_t sc = 0x7E;
      if (amax == 0.0) sc = 0;
      else
        for (int c = 0; c <= 0x7E; c++)
          if (6.0 * orc_e4m3_val((uint8_t)c) >= amax) { sc = (uint8_t)c; break; }
      o[256 + g] = sc;
      double s = orc_e4m3_val(sc);
      for (int i = 0; i < 16; i++) {
        int d = 16 * g + i;
        uint8_t code = s == 0.0 ? 0 : orc_e2m1_code(bf16_val(rows[r * D_LAT + d]) / s);
        o[d / 2] |= (uint8_t)(code << (4 * (d & 1)));
      }
    }
  }
}

static double fp4_plane_val(const uint8_t* row, int d) {
  uint8_t code = (row[d / 2] >> (4 * (d & 1))) & 15;
  return orc_e2m1_val(code) * orc_e4m3_val(row[256 + d / 16]);
}

/* ---- MXFP4 index plane [A] indexer figure (FP4 index rows of 68 B: 64 B of values and
 *      4 B of scales; planes paged in blocks of 8 rows); [A] indexer K (E2M1 with one
 *      E8M0 scale per 32 channels, pure powers of two) --------------------------------
 *
 * Block b holds rows 8b .. 8b+7: 8 x 64 code bytes (dim 2i in the low nibble of byte i),
 * then 8 x 4 E8M0 scale bytes (scale j of a row for dims 32j .. 32j+31): 544 bytes.  A
 * group's scale is the smallest 2^(e-127) with max |x| <= 6 * 2^(e-127) (e = 127 for an
 * all-zero group), its codes E2M1(x / 2^(e-127)).  Rows of a partial last block past n
 * are zero with e = 127. */
void orc_index_plane_fp4(const uint16_t* k, int64_t n, uint8_t* plane) {
  int64_t nb = (n + 7) / 8;
  memset(plane, 0, (size_t)nb * 544);
  for (int64_t r = 0; r < nb * 8; r++) {
    uint8_t* blk = plane + (r / 8) * 544;
    uint8_t* codes = blk + (r % 8) * 64;
    uint8_t* sc = blk + 512 + (r % 8) * 4;
    for (int j = 0; j < 4; j++) {
      if (r >= n) { sc[j] = 127; continue; }
      double amax = 0.0;
      for (int i = 0; i < 32; i++) {
        double v = fabs(bf16_val(k[r * D_IDX + 32 * j + i]));
        if (v > amax) amax = v;
      }
      int e = 127;
      if (amax > 0.0) {
        e = 0;
        while (e < 254 && amax > 6.0 * ldexp(1.0, e - 127)) e++;
      }
      sc[j] = (uint8_t)e;
      for (int i = 0; i < 32; i++) {
        int d = 32 * j + i;
        uint8_t c = orc_e2m1_code(bf16_val(k[r * D_IDX + d]) / ldexp(1.0, e - 127));
        codes[d / 2] |= (uint8_t)(c << (4 * (d & 1)));
      }
    }
  }
}

static double fp4_index_val(const uint8_t* plane, int64_t row, int d) {
  const uint8_t* blk = plane + (row / 8) * 544;
  uint8_t c = (blk[(row % 8) * 64 + d / 2] >> (4 * (d & 1))) & 15;
  int e = blk[512 + (row % 8) * 4 + d / 32];
  return orc_e2m1_val(c) * ldexp(1.0, e - 127);
}

/* Index scores on the MXFP4 plane: orc_index_scores with K[c][d] the decoded value of
 * row row_base[b] + c (row_base a multiple of 8); the query stays bf16. */
void orc_index_scores_fp4(const uint16_t* iq, const float* w, int Q, int H, const uint8_t* plane,
                          const int64_t* row_base, const int32_t* q_seq, const int64_t* q_pos,
                          int m, const int32_t* cand, int ncb, int relu, double* scores,
                          int64_t* rows, int64_t ld) {
  double alpha = 1.0 / sqrt((double)D_IDX) / sqrt((double)H);
  for (int q = 0; q < Q; q++) {
    int64_t nvis = orc_n_visible(q_pos[q], m);
    int64_t rb = row_base[q_seq[q]];
    double qv[64 * D_IDX];
    for (int i = 0; i < H * D_IDX; i++) qv[i] = bf16_val(iq[(int64_t)q * H * D_IDX + i]);
    int64_t npos = cand ? (int64_t)ncb * 8 : nvis;
#pragma omp parallel for schedule(static)
    for (int64_t pos = 0; pos < ld; pos++) {
      int64_t row = -1;
      if (pos < npos) {
        if (!cand) row = pos;
        else {
          int32_t blk = cand[(int64_t)q * ncb + pos / 8];
          if (blk >= 0 && (int64_t)blk * 8 + pos % 8 < nvis) row = (int64_t)blk * 8 + pos % 8;
        }
      }
      rows[(int64_t)q * ld + pos] = row;
      if (row < 0) { scores[(int64_t)q * ld + pos] = 0.0; continue; }
      double kr[D_IDX];
      for (int d = 0; d < D_IDX; d++) kr[d] = fp4_index_val(plane, rb + row, d);
      double s = 0.0;
      for (int h = 0; h < H; h++) {
        double dot = 0.0;
        for (int d = 0; d < D_IDX; d++) dot += qv[h * D_IDX + d] * kr[d];
        if (relu && dot < 0.0) dot = 0.0;
        s += (double)w[(int64_t)q * H + h] * dot;
      }
      scores[(int64_t)q * ld + pos] = alpha * s;
    }
  }
}

/* ---- top-k [A] Fig. 3b ("selected [rows, 512] 升序，-1 填充"), "visible 是每行
 *      自己的前缀长度" (-1 means the history is shorter than 512) ----------------------
 *
 * Keep k_eff = min(k, #scored) entries of highest score, ties to the lower row id,
 * NaN ranked as -inf; emit their row ids in ascending order, -1 padded to k. */
typedef struct { double s; int64_t row; } orc_pair;

static int cmp_rank(const void* a, const void* b) {
  const orc_pair* x = (const orc_pair*)a;
  const orc_pair* y = (const orc_pair*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->row < y->row) ? -1 : (x->row > y->row);
}

static int cmp_i64(const void* a, const void* b) {
  int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x < y) ? -1 : (x > y);
}

int orc_topk(const double* scores, const int64_t* rows, int64_t n, int k, int32_t* sel) {
  orc_pair* v = (orc_pair*)malloc(sizeof(orc_pair) * (n > 0 ? n : 1));
  int64_t nv = 0;
  for (int64_t i = 0; i < n; i++) {
    if (rows[i] < 0) continue;
    v[nv].s = isnan(scores[i]) ? -INFINITY : scores[i];
    v[nv].row = rows[i];
    nv++;
  }
  qsort(v, nv, sizeof(orc_pair), cmp_rank);
  int64_t keff = nv < k ? nv : k;
  int64_t* r = (int64_t*)malloc(sizeof(int64_t) * (keff > 0 ? keff : 1));
  for (int64_t i = 0; i < keff; i++) r[i] = v[i].row;
  qsort(r, keff, sizeof(int64_t), cmp_i64);
  for (int i = 0; i < k; i++) sel[i] = (i < keff) ? (int32_t)r[i] : -1;
  free(v);
  free(r);
  return (int)keff;
}

/* ---- sparse MQA attention with sink [A] "四种层合并出来的是什么形状", Fig. 2a-2d;
 *      [E] Fig. 2d (out_h formula with exp(sink_h) in the denominator);
 *      [B] §4.1 (640 positions, no de-duplication), §4.4 step 4 (window slots);
 *      [C] §5.5 (one softmax over the concatenated entries) ---------------------------
 *
 * For query q at position p in sequence b the entry set is the window positions
 * max(0, p-127) .. p (ring slot pos % 128, or the linear row for pos) followed by
 * the plane rows sel[q][i] != -1.  One KV vector per entry serves as key and value.
 *   s_j   = scale * <q_h, x_j>
 *   out_h = sum_j e^{s_j} x_j / (e^{sink_h} + sum_j e^{s_j})
 *   lse_h = log(e^{sink_h} + sum_j e^{s_j})
 * sink == NULL drops the sink term.  swa_mode 0 = ring [B][128][512],
 * 1 = linear rows lin_base[b] + (pos - lin_pos0[b]).  swa_dtype 0 = bf16,
 * 1 = 528-byte FP8 rows (512 E4M3 codes then 4 fp32 scales, one per 128 codes),
 * 2 = 528-byte FP8 rows with 16 E8M0 scales, one per 32 codes ([A] pool switch).
 * plane_dtype 0 = bf16 rows [.][512], 1 = FP4 rows of 288 B (orc_plane_fp4 layout). */
void orc_sparse_attn(const uint16_t* q, int Q, const int32_t* q_seq, const int64_t* q_pos,
                     int swa_mode, int swa_dtype, const void* swa, const int64_t* lin_base,
                     const int64_t* lin_pos0, int plane_dtype, const void* plane,
                     const int64_t* row_base, const int32_t* sel, int nsel, const float* sink,
                     double scale, double* out, double* lse) {
#pragma omp parallel for schedule(dynamic)
  for (int qi = 0; qi < Q; qi++) {
    int b = q_seq[qi];
    int64_t p = q_pos[qi];
    int64_t lo = p - (RING - 1) < 0 ? 0 : p - (RING - 1);
    int nwin = (int)(p - lo + 1);
    int nent = nwin;
    for (int i = 0; i < nsel; i++) nent += sel[(int64_t)qi * nsel + i] >= 0;
    double* x = (double*)malloc(sizeof(double) * (size_t)nent * D_LAT);
    int e = 0;
    for (int64_t pos = lo; pos <= p; pos++, e++) {
      if (swa_dtype == 0) {
        const uint16_t* src;
        if (swa_mode == 0) src = (const uint16_t*)swa + ((int64_t)b * RING + pos % RING) * D_LAT;
        else src = (const uint16_t*)swa + (lin_base[b] + (pos - lin_pos0[b])) * D_LAT;
        for (int d = 0; d < D_LAT; d++) x[(int64_t)e * D_LAT + d] = bf16_val(src[d]);
      } else {
        const uint8_t* src;
        if (swa_mode == 0) src = (const uint8_t*)swa + ((int64_t)b * RING + pos % RING) * 528;
        else src = (const uint8_t*)swa + (lin_base[b] + (pos - lin_pos0[b])) * 528;
        for (int d = 0; d < D_LAT; d++) {
          double sc;
          if (swa_dtype == 1) {
            float f;
            memcpy(&f, src + 512 + 4 * (d / 128), 4);
            sc = (double)f;
          } else { /* E8M0: 2^(e - 127), e = 255 is NaN */
            int ex = src[512 + d / 32];
            sc = ex == 255 ? NAN : ldexp(1.0, ex - 127);
          }
          x[(int64_t)e * D_LAT + d] = orc_e4m3_val(src[d]) * sc;
        }
      }
    }
    for (int i = 0; i < nsel; i++) {
      int32_t r = sel[(int64_t)qi * nsel + i];
      if (r < 0) continue;
      if (plane_dtype == 0) {
        const uint16_t* src = (const uint16_t*)plane + (row_base[b] + r) * D_LAT;
        for (int d = 0; d < D_LAT; d++) x[(int64_t)e * D_LAT + d] = bf16_val(src[d]);
      } else {
        const uint8_t* src = (const uint8_t*)plane + (row_base[b] + r) * 288;
        for (int d = 0; d < D_LAT; d++) x[(int64_t)e * D_LAT + d] = fp4_plane_val(src, d);
      }
      e++;
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)nent);
    for (int h = 0; h < N_HEADS; h++) {
      const uint16_t* qh = q + ((int64_t)qi * N_HEADS + h) * D_LAT;
      double qd[D_LAT];
      for (int d = 0; d < D_LAT; d++) qd[d] = bf16_val(qh[d]);
      double mx = sink ? (double)sink[h] : -INFINITY;
      for (int j = 0; j < nent; j++) {
        double dot = 0.0;
        for (int d = 0; d < D_LAT; d++) dot += qd[d] * x[(int64_t)j * D_LAT + d];
        s[j] = scale * dot;
        if (s[j] > mx) mx = s[j];
      }
      double z = sink ? exp((double)sink[h] - mx) : 0.0;
      double o[D_LAT];
      for (int d = 0; d < D_LAT; d++) o[d] = 0.0;
      for (int j = 0; j < nent; j++) {
        double pj = exp(s[j] - mx);
        z += pj;
        for (int d = 0; d < D_LAT; d++) o[d] += pj * x[(int64_t)j * D_LAT + d];
      }
      for (int d = 0; d < D_LAT; d++) out[((int64_t)qi * N_HEADS + h) * D_LAT + d] = o[d] / z;
      if (lse) lse[(int64_t)qi * N_HEADS + h] = mx + log(z);
    }
    free(s);
    free(x);
  }
}

/* ---- inverse RoPE of the attention output [A] "出来之后" (out -> inverse RoPE at the
 *      query's own position, because K = V carries the rotation); [B] §6.1 (the output's
 *      last 64 dims times the conjugate phase); [C] A.12.1 -----------------------------
 *
 * For query q at position p and every head, pair i of dims 448 + 2i, 449 + 2i, read as
 * a complex number, is multiplied by e^{-i p theta_i} with theta_i = inv_freq[i]:
 *   a0' = a0 cos(p theta_i) + a1 sin(p theta_i)
 *   a1' = a1 cos(p theta_i) - a0 sin(p theta_i)
 * The other 448 dims are unchanged.  out is [Q][64][512] double, rotated in place. */
void orc_inverse_rope(double* out, int Q, const int64_t* q_pos, const float* inv_freq) {
#pragma omp parallel for schedule(static)
  for (int qi = 0; qi < Q; qi++) {
    const double p = (double)q_pos[qi];
    for (int i = 0; i < 32; i++) {
      const double ang = p * (double)inv_freq[i];
      const double c = cos(ang), s = sin(ang);
      for (int h = 0; h < N_HEADS; h++) {
        double* o = out + ((int64_t)qi * N_HEADS + h) * D_LAT + ROPE_DIM0 + 2 * i;
        const double a0 = o[0], a1 = o[1];
        o[0] = a0 * c + a1 * s;
        o[1] = a1 * c - a0 * s;
      }
    }
  }
}

/* ---- candidate pool of the FULL layer [A] Fig. 3b (second stage: block maxima, newest
 *      block pinned to +inf, top-2048 blocks, ascending, -1 padded); [B] §5.2 (block
 *      score = the block's largest indexer score, the partial newest block is kept);
 *      [C] A.11 (2048 blocks of 8 positions) ----------------------------------------
 *
 * scores [ld] are one query's FULL logits, rows [ld] their row ids (-1 = not scored;
 * the scored rows are 0 .. n_vis - 1).  Block b holds rows 8b .. 8b + 7; its score is
 * the largest score of its scored rows, NaN counting as -inf and +inf clamped to the
 * largest finite value.  The newest block (the one holding row n_vis - 1) gets +inf.
 * Then the top nbk blocks by (score desc, block id asc), written ascending to cand
 * [nbk], -1 padded.  Returns the number of blocks selected. */
int orc_candidate_pool(const double* scores, const int64_t* rows, int64_t ld, int nbk,
                       int32_t* cand) {
  int64_t nvis = 0;
  for (int64_t i = 0; i < ld; i++)
    if (rows[i] >= 0 && rows[i] + 1 > nvis) nvis = rows[i] + 1;
  const int64_t nb = (nvis + 7) / 8;
  double* bs = (double*)malloc(sizeof(double) * (nb > 0 ? nb : 1));
  int64_t* ids = (int64_t*)malloc(sizeof(int64_t) * (nb > 0 ? nb : 1));
  for (int64_t b = 0; b < nb; b++) { bs[b] = -INFINITY; ids[b] = b; }
  for (int64_t i = 0; i < ld; i++) {
    if (rows[i] < 0) continue;
    double s = scores[i];
    if (isnan(s)) s = -INFINITY;
    if (s == INFINITY) s = DBL_MAX;
    const int64_t b = rows[i] / 8;
    if (s > bs[b]) bs[b] = s;
  }
  if (nb > 0) bs[nb - 1] = INFINITY;
  const int keff = orc_topk(bs, ids, nb, nbk, cand);
  free(bs);
  free(ids);
  return keff;
}

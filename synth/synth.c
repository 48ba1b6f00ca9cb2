/*
 * synth.c -- host side of the seeded input generator (see synth.h).
 * Every function fills a caller-owned host buffer; OpenMP splits the work.
 */
#include "synth.h"

#include <stddef.h>

#define SCALE_STREAM_OFFSET 0x100000ULL

void synth_fill_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream,
                            uint64_t offset) {
  uint64_t base = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = synth_bf16(synth_normal(base, offset + (uint64_t)i));
}

void synth_fill_normal_f32(float* out, int64_t n, uint64_t seed, uint64_t stream,
                           uint64_t offset) {
  uint64_t base = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = synth_normal(base, offset + (uint64_t)i);
}

void synth_fill_u64(uint64_t* out, int64_t n, uint64_t seed, uint64_t stream, uint64_t offset) {
  uint64_t base = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = synth_u64(base, offset + (uint64_t)i);
}

/* Rows j0 .. j0+nrows-1 of sequence b of a [rows, D] tensor, as bf16. */
void synth_fill_rows_bf16(uint16_t* out, uint64_t b, int64_t j0, int64_t nrows, int64_t D,
                          uint64_t seed, uint64_t stream) {
  uint64_t base = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; r++)
    for (int64_t d = 0; d < D; d++)
      out[r * D + d] = synth_bf16(
          synth_normal(base, synth_row_elem(b, (uint64_t)(j0 + r), (uint64_t)D, (uint64_t)d)));
}

/* Same rows as fp32 (the bf16 rounding is not applied). */
void synth_fill_rows_f32(float* out, uint64_t b, int64_t j0, int64_t nrows, int64_t D,
                         uint64_t seed, uint64_t stream) {
  uint64_t base = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; r++)
    for (int64_t d = 0; d < D; d++)
      out[r * D + d] =
          synth_normal(base, synth_row_elem(b, (uint64_t)(j0 + r), (uint64_t)D, (uint64_t)d));
}

/* Rows listed in rows[0..n-1] (any order, repeats allowed) of sequence b. */
void synth_fill_rowlist_bf16(uint16_t* out, uint64_t b, const int64_t* rows, int64_t n, int64_t D,
                             uint64_t seed, uint64_t stream) {
  uint64_t base = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; r++)
    for (int64_t d = 0; d < D; d++)
      out[r * D + d] = synth_bf16(
          synth_normal(base, synth_row_elem(b, (uint64_t)rows[r], (uint64_t)D, (uint64_t)d)));
}

/* FP8 rows of 528 bytes: 512 E4M3 codes of 64 * N(0,1), then four fp32 scales
 * in [0.75, 1.25) / 64, one per 128 consecutive codes. */
void synth_fill_rows_fp8s128(uint8_t* out, uint64_t b, int64_t j0, int64_t nrows, uint64_t seed,
                             uint64_t stream) {
  uint64_t base = synth_base(seed, stream);
  uint64_t sbase = synth_base(seed, stream + SCALE_STREAM_OFFSET);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; r++) {
    uint8_t* row = out + r * 528;
    uint64_t j = (uint64_t)(j0 + r);
    for (int d = 0; d < 512; d++)
      row[d] = synth_e4m3(64.0f * synth_normal(base, synth_row_elem(b, j, 512, (uint64_t)d)));
    for (int k = 0; k < 4; k++) {
      float s = (0.75f + 0.5f * synth_uniform(sbase, synth_row_elem(b, j, 4, (uint64_t)k))) *
                0.015625f;
      union { float f; uint8_t c[4]; } v;
      v.f = s;
      for (int t = 0; t < 4; t++) row[512 + 4 * k + t] = v.c[t];
    }
  }
}

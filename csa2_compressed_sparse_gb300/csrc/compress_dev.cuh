// compress_dev.cuh -- the per-token work of the CSA2 compressor, shared by the
// compressor kernel (k_compress.cu) and by the index score kernel, which runs it on a
// warp of its own when the compressor and the indexer are called together.
// [A] "特殊模块 · compressor" and "CSA2 的池化比 V4 简单一截"; [B] §4.1, §6.1-6.2;
// [C] §6.2 (tail state), §6.4 (ratio 1 degenerates to projection + norm).
//
// One warp per new token.  The warp of a token that closes a group (pos % m == m-1)
// emits that group's row; the group's earlier tokens come from this call's input
// or, for the first group of a sequence, from the state.  The warp of the first
// token of each sequence additionally stores the tokens of a group left incomplete
// at the end of the call into the state.  With m <= 2 that warp is also the only
// reader of the state, so state reads precede state writes within one warp.
//
// Lane layout: lane l owns channels [8l, 8l+8) and [256+8l, 256+8l+8), i.e. two
// 16-byte vectors per row (coalesced 1 KiB row accesses).  Lanes 24..31 hold the
// RoPE dims 448..511 in their second vector, four adjacent pairs each.
#pragma once

#include "common.cuh"

namespace csa2 {
namespace cdev {

__device__ __forceinline__ void load8_bf16(const uint16_t* p, float (&v)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load8_f32(const float* p, float (&v)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8_f32(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void store8_bf16(uint16_t* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// Fetch channels (c0..c0+7) of the token at position `pos` of sequence b: from the
// input when it arrived in this call, else from the state slot pos % m.
__device__ __forceinline__ void fetch(const CompressArgs& a, int b, int64_t pos, int64_t s0,
                                      int64_t t0, int c0, float (&kv)[8], float (&sc)[8]) {
  if (pos >= s0) {
    int64_t t = t0 + (pos - s0);
    load8_bf16(a.kv + t * kDLat + c0, kv);
    if (a.score) load8_bf16(a.score + t * kDLat + c0, sc);
    else
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i] = 0.f;
  } else {
    int slot = (int)(pos % a.ratio);
    load8_f32(a.kv_state + ((int64_t)b * 2 + slot) * kDLat + c0, kv);
    load8_f32(a.score_state + ((int64_t)b * 2 + slot) * kDLat + c0, sc);
  }
}

// Index K of one row, by the warp that emits it: [A] indexer figure, key side (the bf16
// latent before RoPE -> wk [128, 512] -> k_norm -> RoPE on the last 64 dims -> the index
// plane).  r holds the lane's 16 normalized channels before RoPE.  Each lane multiplies
// its channels into all 128 outputs (one 16-byte load of each wk row per half), and a
// butterfly over the lanes sums every block of 32 outputs so that lane l ends with
// outputs l, 32 + l, 64 + l, 96 + l; then the RMSNorm over the 128 and the rotation of
// pairs (64 + 2i, 65 + 2i), whose halves sit in lanes 2i and 2i + 1.
__device__ __forceinline__ void emit_index_k(const CompressArgs& a, const float (&r)[2][8],
                                             const int (&c)[2], int lane, uint64_t p0,
                                             int64_t row, const uint64_t* turn_s) {
  float x[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) x[h][i] = __bfloat162float(__float2bfloat16_rn(r[h][i]));
  float k[4];
#pragma unroll 1
  for (int blk = 0; blk < 4; ++blk) {
    float v[32];
#pragma unroll
    for (int oo = 0; oo < 32; ++oo) {
      const uint16_t* wr = a.wk + (int64_t)(32 * blk + oo) * kDLat;
      float w0[8], w1[8];
      load8_bf16(wr + c[0], w0);
      load8_bf16(wr + c[1], w1);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(w0[i], x[0][i], acc);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(w1[i], x[1][i], acc);
      v[oo] = acc;
    }
#pragma unroll
    for (int off = 16, n = 16; off >= 1; off >>= 1, n >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < n; ++i) {
        const float send = upper ? v[i] : v[i + n];
        const float keep = upper ? v[i + n] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
      }
    }
    k[blk] = v[0];
  }
  float ss = k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const float rstd = 1.0f / sqrtf(ss / (float)kDIdx + a.eps);
#pragma unroll
  for (int blk = 0; blk < 4; ++blk)
    k[blk] *= rstd * (a.knorm_w ? a.knorm_w[32 * blk + lane] : 1.f);
#pragma unroll
  for (int blk = 2; blk < 4; ++blk) {
    const int pair = 16 * (blk - 2) + (lane >> 1);
    float fs, fc;
    sincosf(rope_angle(turn_s[pair], p0), &fs, &fc);
    const float other = __shfl_xor_sync(0xFFFFFFFFu, k[blk], 1);
    k[blk] = (lane & 1) ? other * fs + k[blk] * fc : k[blk] * fc - other * fs;
  }
  uint16_t* dst = a.index_plane + row * kDIdx;
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) dst[32 * blk + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(k[blk]));
}

// This token's own kv / score channels (they do not depend on its sequence).
__device__ __forceinline__ void load_own(const CompressArgs& a, int64_t t, int lane,
                                         float (&own_kv)[2][8], float (&own_sc)[2][8]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    load8_bf16(a.kv + t * kDLat + (h ? 256 : 0) + 8 * lane, own_kv[h]);
    if (a.score) load8_bf16(a.score + t * kDLat + (h ? 256 : 0) + 8 * lane, own_sc[h]);
    else
#pragma unroll
      for (int i = 0; i < 8; ++i) own_sc[h][i] = 0.f;
  }
}

// Sequence of token t: the last b < B with cu[b] <= t (cu non-decreasing, cu[0] = 0),
// found by the 32 lanes of a warp together: each round probes 32 evenly spaced entries
// and keeps the span between the last probe at or below t and the next one, so B = 8192
// takes three rounds of loads.
__device__ __forceinline__ int warp_find_seq(const int32_t* cu, int B, int64_t t, int lane) {
  int lo = 0, hi = B - 1;
  while (hi > lo) {
    const int step = (hi - lo + 31) / 32;
    const int probe = min(hi, lo + step * (lane + 1));
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, (int64_t)__ldg(cu + probe) <= t);
    if (m == 0u) {
      hi = lo + step - 1;
    } else {
      lo = min(hi, lo + step * (32 - __clz((int)m)));
      hi = min(hi, lo + step - 1);
    }
  }
  return lo;
}

// Everything after the sequence lookup for token t of sequence b (tokens t0 .. t1 - 1 of
// the call), by one warp; turn_s holds the 32 RoPE turns (rope_turn of inv_freq).
// kIndexK = false leaves out the index K branch (callers whose a.wk is always null).
template <bool kIndexK = true>
__device__ __forceinline__ void token(const CompressArgs& a, int64_t t, int b, int64_t t0,
                                      int64_t t1, const float (&own_kv)[2][8],
                                      const float (&own_sc)[2][8], int lane,
                                      const uint64_t* turn_s) {
  const int64_t s0 = a.start_pos[b];
  const int64_t pos = s0 + (t - t0);
  const int m = a.ratio;
  const int c[2] = {8 * lane, 256 + 8 * lane};

  // ---- emit the row of a group that this token closes ----
  if (pos % m == m - 1) {
    const int64_t j = pos / m;
    float r[2][8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (m == 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) r[h][i] = own_kv[h][i];
      } else {
        float k0[8], q0[8];
        fetch(a, b, pos - 1, s0, t0, c[h], k0, q0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // per-channel softmax over the two slots
          const float k1 = own_kv[h][i], q1 = own_sc[h][i];
          float mx = fmaxf(q0[i], q1);
          float e0 = expf(q0[i] - mx), e1 = expf(q1 - mx);
          r[h][i] = (e0 * k0[i] + e1 * k1) / (e0 + e1);
        }
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += r[h][i] * r[h][i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    const float rstd = 1.0f / sqrtf(ss / (float)kDLat + a.eps);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float wv[8];
      if (a.norm_w) load8_f32(a.norm_w + c[h], wv);
      else
#pragma unroll
        for (int i = 0; i < 8; ++i) wv[i] = 1.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) r[h][i] = r[h][i] * rstd * wv[i];
    }
    const int64_t row = a.row_base[b] + j;
    const bool row_ok = row >= 0 && row < a.plane_rows;
    // the indexer's branch leaves before the main RoPE
    if (kIndexK && a.wk && row_ok) emit_index_k(a, r, c, lane, (uint64_t)(j * m), row, turn_s);
    if (lane >= 24) {  // dims 448 + 8(lane-24) .. +7: four rotation pairs
      const uint64_t p0 = (uint64_t)(j * m);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int pair = 4 * (lane - 24) + k;
        const float ang = rope_angle(turn_s[pair], p0);
        float fs, fc;
        sincosf(ang, &fs, &fc);
        const float x0 = r[1][2 * k], x1 = r[1][2 * k + 1];
        r[1][2 * k] = x0 * fc - x1 * fs;
        r[1][2 * k + 1] = x0 * fs + x1 * fc;
      }
    }
    if (!row_ok) {
      if (lane == 0) raise_fault(kFaultBounds);
    } else {
      store8_bf16(a.plane + row * kDLat + c[0], r[0]);
      store8_bf16(a.plane + row * kDLat + c[1], r[1]);
    }
  }

  // ---- first token of the sequence: keep an incomplete trailing group ----
  if (t == t0 && m > 1) {
    const int64_t last = s0 + (t1 - t0) - 1;
    if (last % m != m - 1) {
      for (int64_t p = (last / m) * m; p <= last; ++p) {
        if (p < s0) continue;  // already in the state from an earlier call
        const int64_t tp = t0 + (p - s0);
        const int slot = (int)(p % m);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float kv[8], sc[8];
          load8_bf16(a.kv + tp * kDLat + c[h], kv);
          if (a.score) load8_bf16(a.score + tp * kDLat + c[h], sc);
          else
#pragma unroll
            for (int i = 0; i < 8; ++i) sc[i] = 0.f;
          store8_f32(a.kv_state + ((int64_t)b * 2 + slot) * kDLat + c[h], kv);
          store8_f32(a.score_state + ((int64_t)b * 2 + slot) * kDLat + c[h], sc);
        }
      }
    }
  }
}

}  // namespace cdev
}  // namespace csa2

// common.cuh -- device-side definitions shared by the HyTopK kernels.
//
// Score arithmetic (identical in every kernel, so that the filter, the
// recovery path, the two-pass path and replay return the same bits for the
// same (query, key)):
//
//   dot_h  = sum_i q[t,h,i] * k[s,i]           raw elements (e4m3 codes or bf16)
//   acc    = sum_h wq[t,h] * max(dot_h, 0)     h = 0..H-1, fused multiply-add
//   score  = acc * k_scale[s]                  (k_scale = 1 for bf16)
//
// with wq[t,h] = w[t,h] * q_scale[t,h] (w for bf16). Because the scales are
// positive, ReLU(qs*ks*x) = qs*ks*ReLU(x), so this equals the indexer score
// I[t,s] = sum_h w[t,h] ReLU(q[t,h].k[s]) of the HyScale pages up to rounding.
// -0.0 is returned as +0.0.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "hytopk.h"

namespace hytopk {

constexpr int kTileKeys = 128;       // keys per scoring tile (one TMEM lane / thread each)
constexpr int kQueryPad = 512;       // query slots are padded to a multiple of this
constexpr int kMaxSamples = 8192;    // upper clamp of the sample count M
constexpr int kRecoveryCtas = 64;    // persistent CTAs of the recovery kernel (one row each)
constexpr int kTableCtas = 304;      // CTAs of the two-pass read-back (one row each, 2 per SM)
constexpr int kMaxTopK = 16384;

// Counters kept in the workspace (zeroed at the start of every call).
enum Counter : int {
  kCtrFilterWork = 0,
  kCtrFailed = 1,
  kCtrOverflow = 2,
  kCtrUnderK = 3,
  kCtrStatus = 4,
  kCtrRecoverWork = 5,
  kCtrCandLo = 6,  // 64-bit total candidates at [6,7]
  kCtrCount = 16
};

struct Problem {
  const void* q;
  const float* q_scale;
  const void* k;
  const float* k_scale;
  const float* w;
  const int32_t* positions;
  int n, L, H, d, k_top;
  int dt;   // key elements (and the packed query operand): 0 bf16, 1 e4m3
  int qdt;  // query elements as given: 0 bf16, 1 e4m3 (with q_scale)
};

// Workspace of hytopk_select, carved by the host.
struct SelectWs {
  int32_t* perm;        // [n_pad] slot -> query index, -1 for padding
  int32_t* qpos;        // [n_pad] slot -> position, -1 for padding / bad position
  float* wq;            // [n_pad, H] folded, halved head weights w * q_scale / 2
  void* qp;             // [n_pad, H, d] packed query elements
  float* thr;           // [n_pad] thresholds
  int32_t* cnt;         // [n_pad] candidate counts (may exceed C: overflow)
  uint64_t* cand;       // [n_pad, C] candidate keys
  int32_t* failed_list; // [n_pad]
  uint8_t* failed;      // [n_pad]
  uint32_t* counters;   // [kCtrCount]
  float* rowbuf;        // [kRecoveryCtas, L] full score rows (recovery)
  int32_t* plan;        // [nchunks + 1] filter work items per key chunk
  int n_pad, C;
};

// ---- the score ------------------------------------------------------------------

__device__ __forceinline__ float finish_score(float acc, float ks) {
  float s = acc * ks;
  return s == 0.0f ? 0.0f : s;
}

// 8 e4m3 codes -> 8 bf16 (exact: every e4m3 value is a bf16 value)
__device__ __forceinline__ uint4 e4m3x8_to_bf16(uint2 in) {
  const uint32_t w[2] = {in.x, in.y};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint16_t two = (uint16_t)(w[i] >> (16 * h));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
      const float f0 = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
      const float f1 = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
      uint32_t b2;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b2) : "f"(f1), "f"(f0));
      out[2 * i + h] = b2;
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// ---- ordered keys -------------------------------------------------------------------
// desc32(score): an unsigned key whose ascending order is descending score.
// cand_key(score, pos) = desc32 << 32 | pos: ascending order is score
// descending, then position ascending -- the output order of the selection.

__device__ __forceinline__ uint32_t desc32(float f) {
  uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
  uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ~asc;
}

__device__ __forceinline__ float desc32_score(uint32_t k) {
  uint32_t asc = ~k;
  uint32_t u = (asc & 0x80000000u) ? (asc & 0x7FFFFFFFu) : ~asc;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t cand_key(float score, int32_t pos) {
  return ((uint64_t)desc32(score) << 32) | (uint32_t)pos;
}

// ---- threshold parameters (HyScale explainer: HyTopK paragraph, worked example) ----

__host__ __device__ __forceinline__ int sample_count(int64_t ctx) {
  int64_t m = ctx / 128;
  m = m < 4096 ? 4096 : m;
  m = m > kMaxSamples ? kMaxSamples : m;
  return (int)(m < ctx ? m : ctx);
}

__host__ __device__ __forceinline__ int threshold_rank(int64_t ctx, int64_t k, int m) {
  int64_t r = (3 * k * (int64_t)m + ctx - 1) / ctx;
  return (int)(r < m ? r : m);
}

__host__ __device__ __forceinline__ int sample_position(int64_t ctx, int m, int j) {
  return (int)(((int64_t)j * ctx) / m);
}

// p_j = floor(j * ctx / M) without 64-bit division: with ctx = a*M + b,
// p_j = j*a + floor(j*b / M), and j*b < M^2 <= 2^26 fits 32 bits.
struct SampleStep {
  uint32_t a, b, m;
  __device__ __forceinline__ void init(int64_t ctx, int M) {
    m = (uint32_t)M;
    a = (uint32_t)(ctx / M);
    b = (uint32_t)(ctx - (int64_t)a * M);
  }
  __device__ __forceinline__ int at(int j) const {
    return (int)((uint32_t)j * a + ((uint32_t)j * b) / m);
  }
};

// The positions of samples j0, j0 + 128, j0 + 256, ... of one query, one per
// next() (the caller tells the samples past M apart), with no division per
// sample: with 128 b = dq M + dr, p(j + 128) = p(j) + 128 a + dq, plus one
// when the remainder of j b / M passes M.
struct SampleWalk {
  uint32_t p, rem, dp, dr, m;
  __device__ __forceinline__ void init(const SampleStep& st, int j0) {
    m = st.m;
    const uint32_t jb = (uint32_t)j0 * st.b, q0 = jb / m;
    p = (uint32_t)j0 * st.a + q0;
    rem = jb - q0 * m;
    const uint32_t tb = (uint32_t)kTileKeys * st.b, dq = tb / m;
    dp = (uint32_t)kTileKeys * st.a + dq;
    dr = tb - dq * m;
  }
  __device__ __forceinline__ int next() {
    const int s = (int)p;
    p += dp;
    rem += dr;
    if (rem >= m) {
      rem -= m;
      ++p;
    }
    return s;
  }
};

// Entries of the shared-memory sort buffer for k keys: the next power of two,
// at least 2 (so that what follows it stays 16-byte aligned).
__host__ __device__ __forceinline__ int sort_capacity(int k) {
  int P = 2;
  while (P < k) P <<= 1;
  return P;
}

// ---- small CTA utilities ---------------------------------------------------------

__device__ __forceinline__ void set_status(uint32_t* counters, uint32_t bits) {
  atomicOr(counters + kCtrStatus, bits);
}

}  // namespace hytopk

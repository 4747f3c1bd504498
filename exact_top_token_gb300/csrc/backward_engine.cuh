// backward_engine.cuh -- gradients of the indexer score at the selected
// entries: for every query t and stored index s = idx[t,j] with upstream
// gradient G = grad[t,j] (dLoss/dI[t,s]),
//   dw[t,h]   = sum_j G * max(0, x)
//   dq[t,h,:] = sum_j G * w[t,h] * [x > 0] * kd[s,:]
//   dk[s,:]  += G * sum_h w[t,h] * [x > 0] * qd[t,h,:]
// with qd = q * q_scale, kd = k * k_scale and x = qd[t,h] . kd[s].
//
// HyScale explainer, key-observation paragraph (the indexer's own loss reads
// only the scores at the selected entries) and selection-replay paragraph
// (during recomputation only those entries are rescored): this is that
// rescoring, fused with the gradient it exists for. The loss is not on the
// pages; its gradient at the entries is the input. The derivative of max(0,x)
// at x = 0 is taken as 0.
//
// Per query (one CTA per SM, queries blockIdx.x, +gridDim.x, ...) and per tile
// of 128 stored keys:
//   producers (warps 0-3): gather the 128 key rows into shared memory as bf16
//     (e4m3 codes convert exactly), 128-byte swizzle, 8 lanes per row;
//     at a query's start also its q rows (bf16) and its w and q_scale.
//   MMA issuer (warp 4), all kind::f16 with bf16 operands, fp32 accumulate:
//     X   [128 keys x H]  = Kt . Q^T            (keys K-major, q K-major)
//     DQ  [2H x d]       += Aq^T . Kt           (Aq MN-major, keys MN-major),
//         accumulated over the query's tiles
//     DK  [128 keys x d]  = Ak . Q              (Ak K-major, q MN-major)
//   epilogue (warps 8-15: two warpgroups, each for half of the heads and half
//     of the d columns; TMEM lane = key). The per-key factor c = G * k_scale
//     and the per-head factor v[h] = w[h] * q_scale[h] are each split once
//     into a bf16 high part and the bf16 of the remainder (~16 bits together);
//     from its row of X the thread writes Aq[key][h'] = [X[h] > 0] * c and
//     Ak[key][h'] = [X[h] > 0] * v[h] (high parts at h' = h, low parts at
//     h' = H + h: a mask, no arithmetic), so DQ[h] carries no w[h] and DK[key]
//     no G: they are applied in fp32 when DQ and DK are read out. It sums
//     c max(0, X[h]) over keys with warp butterflies (dw), adds G * DK into
//     dk[s] with vector reductions, and at the query's end writes
//     dq[t, h] = w[h] (DQ[h] + DQ[H + h]) and dw[t].
// The raw dot X uses the unscaled codes; scales are > 0, so [x > 0] =
// [X > 0] and max(0, x) = k_scale * q_scale * max(0, X).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc.cuh"

namespace hytopk {
namespace bwd {

constexpr int kGroups = 2;  // epilogue warpgroups; group g takes heads and d columns g / kGroups
constexpr int kEpiWarps = 4 * kGroups;
constexpr int kProducers = 128;
constexpr int kMmaWarp = 4;
constexpr int kTmemWarp = 5;
constexpr int kEpiFirstWarp = 8;
constexpr int kThreads = (kEpiFirstWarp + kEpiWarps) * 32;

struct BArgs {
  const void* q;
  const float* q_scale;
  const void* k;
  const float* k_scale;
  const float* w;
  const int32_t* idx;
  const float* grad;
  float* dq;
  float* dk;
  float* dw;
  int n, L, k_top;
  int q_e4m3;  // q rows are e4m3 codes with q_scale (keys may be bf16)
  uint32_t* status;
};

template <int D, int DT, int H>
struct Cfg {
  // heads as the engine sees them: H < 16 runs as 16 heads whose q rows and
  // weights beyond H are zero (N = 16 is the smallest MMA width here)
  static constexpr int HP = H < 16 ? 16 : H;
  static constexpr int ES = DT == 0 ? 2 : 1;  // input element bytes
  static constexpr int RB = D * 2;            // bf16 row bytes in shared memory
  static constexpr int DA = RB / 128;         // 128-byte atoms per bf16 row
  static constexpr int STAGES = D == 128 ? 2 : 3;
  static constexpr int KT = 128 * RB;        // bf16 key tile
  static constexpr int QT = HP * RB;         // bf16 q operand of one query
  static constexpr int AT = 128 * 256;       // Aq / Ak: 128 keys x 128 bf16
  static constexpr int RING_OFF = 0;
  static constexpr int Q_OFF = RING_OFF + STAGES * KT;
  static constexpr int AQ_OFF = Q_OFF + 2 * ((QT + 1023) / 1024 * 1024);
  static constexpr int AK_OFF = AQ_OFF + AT;
  // per query buffer: w [HP], q_scale [HP] (fp32), then w * q_scale split into
  // bf16 high / low parts packed two heads per word [HP/2] + [HP/2]
  static constexpr int WS_OFF = AK_OFF + AT;
  static constexpr int DWS_OFF = WS_OFF + 2 * 3 * HP * 4;  // dw partials [4][HP]
  // per epilogue warp: 32 rows x 32 fp32 (row stride 33) for coalescing dk additions
  static constexpr int TR_OFF = DWS_OFF + 4 * HP * 4;
  static constexpr int TR_FLOATS = 32 * 33;
  static constexpr int BAR_OFF = TR_OFF + kEpiWarps * TR_FLOATS * 4;
  // k_full[S], k_empty[S], q_full[2], q_empty[2], x_full[2], x_empty[2],
  // a_full, a_empty, dk_full[2], dk_empty[2], dq_full, dq_empty, epilogue meet
  static constexpr int NBARS = 2 * STAGES + 2 + 2 + 2 + 2 + 1 + 1 + 2 + 2 + 1 + 1 + 1;
  static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;
  // TMEM columns
  static constexpr int X_COL = 0;           // 2 buffers of HP
  static constexpr int DQ_COL = 128;        // d columns
  static constexpr int DK_COL = 256;        // 2 buffers of d
  static constexpr int CPRS = D * ES / 16;  // 16-byte source chunks per key row
  static_assert(H == 1 || H == 2 || H == 4 || H == 8 || H == 16 || H == 32 || H == 64, "H");
  static_assert(D == 64 || D == 128, "d");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Byte offset of bf16 element e of row r in a 128-byte-swizzled tile whose
// rows hold `rb` bytes, laid out as [atom][rows][128 B] (rows a multiple of 8).
__device__ __forceinline__ uint32_t sw_off(int r, int e, int rows) {
  const int atom = e >> 6;
  const int c = (e & 63) >> 3;
  return (uint32_t)(atom * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    ((c ^ (r & 7)) << 4) + (e & 7) * 2);
}

// Shared-memory descriptor with both byte offsets (SW128).
__device__ __forceinline__ uint64_t desc2(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// 16 e4m3 codes -> 16 bf16 (exact: every e4m3 value is a bf16 value).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 in, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint16_t two = (uint16_t)(w[i] >> (16 * p));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
      const float f0 = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
      const float f1 = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
      uint32_t b2;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b2) : "f"(f1), "f"(f0));
      out[2 * i + p] = b2;
    }
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// high bf16 part of v and the bf16 of the remainder, as raw bits
__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(l);
}

// The four epilogue warps meet on an mbarrier (count 128) rather than a named
// barrier, so that a wait that gives up cannot leave the others waiting
// forever.
__device__ __forceinline__ bool epi_meet(uint64_t* bar, uint32_t& phase, volatile int* abort_flag,
                                         uint32_t* status) {
  tc::mbar_arrive(bar);
  const bool ok = tc::mbar_wait(bar, phase, abort_flag, status);
  phase ^= 1u;
  return ok;
}

__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Sum N values over the 32 lanes of a warp; afterwards lane l holds the sums
// of the heads listed by butterfly_head (N/32 of them, or 1 shared by 32/N
// lanes when N < 32).
template <int N>
__device__ __forceinline__ void butterfly(float (&v)[N], int lane) {
  int cur = N;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (cur >= 2) {
      const int half = cur / 2;
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[half + i];
          const float keep = upper ? v[half + i] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      cur = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
}
// head (within the N summed) that lane `lane` holds in slot u after butterfly<N>
template <int N>
__device__ __forceinline__ int butterfly_head(int lane, int u) {
  if constexpr (N >= 32)
    return lane * (N / 32) + u;
  else
    return lane / (32 / N);
}

template <int D, int DT, int H>
__global__ void __launch_bounds__(kThreads, 1) k_backward(const BArgs a) {
  using C_ = Cfg<D, DT, H>;
  constexpr int STAGES = C_::STAGES, CPRS = C_::CPRS;
  constexpr int HP = C_::HP;  // heads in shared memory, TMEM and the MMAs (H: in global memory)
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  uint8_t* smem = tc::align1024(smem_dyn);
  uint8_t* ring = smem + C_::RING_OFF;
  uint8_t* aq = smem + C_::AQ_OFF;
  uint8_t* ak = smem + C_::AK_OFF;
  float* ws = reinterpret_cast<float*>(smem + C_::WS_OFF);     // [qb][w | q_scale | pairs]
  float* dws = reinterpret_cast<float*>(smem + C_::DWS_OFF);   // [4][HP]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C_::BAR_OFF);
  uint64_t* k_full = bars;
  uint64_t* k_empty = bars + STAGES;
  uint64_t* q_full = bars + 2 * STAGES;
  uint64_t* q_empty = q_full + 2;
  uint64_t* x_full = q_empty + 2;
  uint64_t* x_empty = x_full + 2;
  uint64_t* a_full = x_empty + 2;
  uint64_t* a_empty = a_full + 1;
  uint64_t* dk_full = a_empty + 1;
  uint64_t* dk_empty = dk_full + 2;
  uint64_t* dq_full = dk_empty + 2;
  uint64_t* dq_empty = dq_full + 1;
  uint64_t* meet = dq_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C_::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C_::MISC_OFF + 4);
  auto q_buf = [&](int qb) { return smem + C_::Q_OFF + qb * ((C_::QT + 1023) / 1024 * 1024); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ktiles = (a.k_top + 127) / 128;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(k_full + i, kProducers);
      tc::mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(q_full + i, kProducers);
      tc::mbar_init(q_empty + i, 1 + kEpiWarps);
      tc::mbar_init(x_full + i, 1);
      tc::mbar_init(x_empty + i, kEpiWarps);
      tc::mbar_init(dk_full + i, 1);
      tc::mbar_init(dk_empty + i, kEpiWarps);
    }
    tc::mbar_init(a_full, 32 * kEpiWarps);
    tc::mbar_init(a_empty, 1);
    tc::mbar_init(dq_full, 1);
    tc::mbar_init(dq_empty, kEpiWarps);
    tc::mbar_init(meet, 32 * kEpiWarps);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  // the rows h' >= 2H of Aq and Ak stay zero (M = 128 > 2H)
  for (int i = threadIdx.x; i < 2 * C_::AT / 16; i += kThreads)
    reinterpret_cast<uint4*>(aq)[i] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  if (warp == kTmemWarp) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int n_mine = a.n > (int)blockIdx.x ? (a.n - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int total = n_mine * ktiles;  // tiles of this CTA

  if (warp < 4) {
    // ---------------- producers ----------------
    // Lane l of warp w owns row 32w + l of every tile (its stored key); the
    // row copies go CPRS lanes per row, so each warp load instruction reads
    // 32 / CPRS whole rows. When a tile's row data fits twice in registers
    // (CPRS <= 8), the loads of tile g + 1 are issued before tile g is
    // converted and stored, so two tiles of loads are in flight per thread.
    const int tid = threadIdx.x;
    constexpr int RPP = 32 / CPRS;  // rows per warp instruction
    constexpr bool kTwoInFlight = CPRS <= 8;
    const int c = lane % CPRS;
    auto own_key = [&](int g) -> int {
      const int qi = g / ktiles, i = g - qi * ktiles;
      const int t = (int)blockIdx.x + qi * (int)gridDim.x;
      const int j = i * 128 + tid;
      int s = j < a.k_top ? __ldg(a.idx + (size_t)t * a.k_top + j) : -1;
      return s >= a.L ? -1 : s;
    };
    auto issue = [&](int s_own, uint4 (&v)[CPRS]) {
#pragma unroll
      for (int p = 0; p < CPRS; ++p) {
        const int sr = __shfl_sync(0xffffffffu, s_own, p * RPP + lane / CPRS);
        v[p] = sr >= 0 ? __ldg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.k) +
                                                               (size_t)sr * D * C_::ES) + c)
                       : make_uint4(0, 0, 0, 0);
      }
    };
    // the query's q rows (bf16, K-major = MN-major layout), w and q_scale
    auto load_query = [&](int qi) -> bool {
      const int t = (int)blockIdx.x + qi * (int)gridDim.x;
      const int qb = qi & 1;
      const bool ok = tc::mbar_wait(q_empty + qb, ((qi >> 1) & 1) ^ 1, abort_flag, a.status);
      if (!__all_sync(0xffffffffu, ok)) return false;
      uint8_t* qd = q_buf(qb);
      const bool q8 = DT == 1 || a.q_e4m3;  // q rows of e4m3 codes
      const int qes = q8 ? 1 : 2;
      const int qch = D * qes / 16;  // 16-byte source chunks per q row
      for (int f = tid; f < HP * qch; f += kProducers) {
        const int h = f / qch, cq = f - h * qch;
        // rows of padded heads (h >= H) are zero
        const uint8_t* row_src = static_cast<const uint8_t*>(a.q) + ((size_t)t * H + h) * D * qes;
        const uint4 v = h < H ? __ldg(reinterpret_cast<const uint4*>(row_src) + cq)
                              : make_uint4(0, 0, 0, 0);
        if (!q8) {
          *reinterpret_cast<uint4*>(qd + sw_off(h, cq * 8, HP)) = v;
        } else {
          uint4 lo, hi;
          e4m3x16_to_bf16(v, lo, hi);
          *reinterpret_cast<uint4*>(qd + sw_off(h, cq * 16, HP)) = lo;
          *reinterpret_cast<uint4*>(qd + sw_off(h, cq * 16 + 8, HP)) = hi;
        }
      }
      float* wsq = ws + qb * 3 * HP;
      uint32_t* pairs = reinterpret_cast<uint32_t*>(wsq + 2 * HP);
      for (int h = tid; h < HP; h += kProducers) {
        wsq[h] = h < H ? a.w[(size_t)t * H + h] : 0.0f;
        wsq[HP + h] = (q8 && h < H) ? a.q_scale[(size_t)t * H + h] : 1.0f;
      }
      auto head_factor = [&](int h) -> float {  // w * q_scale of head h, 0 if padded
        if (h >= H) return 0.0f;
        return a.w[(size_t)t * H + h] * (q8 ? a.q_scale[(size_t)t * H + h] : 1.0f);
      };
      for (int pr = tid; pr < HP / 2; pr += kProducers) {
        const int h = 2 * pr;
        uint16_t h0, l0, h1, l1;
        split_bf16(head_factor(h), h0, l0);
        split_bf16(head_factor(h + 1), h1, l1);
        pairs[pr] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        pairs[HP / 2 + pr] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(q_full + qb);
      return true;
    };
    // wait for tile g's stage, convert and store its rows, publish it
    auto store = [&](int g, const uint4 (&v)[CPRS]) -> bool {
      const int stage = g % STAGES;
      const bool ok =
          tc::mbar_wait(k_empty + stage, ((g / STAGES) & 1) ^ 1, abort_flag, a.status);
      if (!__all_sync(0xffffffffu, ok)) return false;
      uint8_t* dst = ring + stage * C_::KT;
#pragma unroll
      for (int p = 0; p < CPRS; ++p) {
        const int row = warp * 32 + p * RPP + lane / CPRS;
        if (DT == 0) {
          *reinterpret_cast<uint4*>(dst + sw_off(row, c * 8, 128)) = v[p];
        } else {
          uint4 lo, hi;
          e4m3x16_to_bf16(v[p], lo, hi);
          *reinterpret_cast<uint4*>(dst + sw_off(row, c * 16, 128)) = lo;
          *reinterpret_cast<uint4*>(dst + sw_off(row, c * 16 + 8, 128)) = hi;
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(k_full + stage);
      return true;
    };
    if constexpr (kTwoInFlight) {
      uint4 va[CPRS], vb[CPRS];
      int s_next = total > 1 ? own_key(1) : -1;
      if (total > 0) issue(own_key(0), va);
      // tiles in pairs so that the two register buffers alternate without copies
      for (int g = 0; g < total; g += 2) {
        if (g % ktiles == 0 && !load_query(g / ktiles)) break;
        if (g + 1 < total) issue(s_next, vb);
        if (g + 2 < total) s_next = own_key(g + 2);
        if (!store(g, va)) break;
        if (g + 1 >= total) break;
        if ((g + 1) % ktiles == 0 && !load_query((g + 1) / ktiles)) break;
        if (g + 2 < total) issue(s_next, va);
        if (g + 3 < total) s_next = own_key(g + 3);
        if (!store(g + 1, vb)) break;
      }
    } else {
      uint4 v[CPRS];
      for (int g = 0; g < total; ++g) {
        if (g % ktiles == 0 && !load_query(g / ktiles)) break;
        issue(own_key(g), v);
        if (!store(g, v)) break;
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t ID_X = tc::instr_desc(0, 128, HP);
      constexpr uint32_t ID_DQ = tc::instr_desc(0, 128, D) | (1u << 15) | (1u << 16);
      constexpr uint32_t ID_DK = tc::instr_desc(0, 128, D) | (1u << 16);
      const uint32_t ring_a = tc::smem_u32(ring), aq_a = tc::smem_u32(aq), ak_a = tc::smem_u32(ak);
      // forward X for tile g (keys of stage g % STAGES)
      auto forward = [&](int g) -> bool {
        const int qi = g / ktiles, i = g - qi * ktiles;
        const int stage = g % STAGES;
        if (i == 0 && !tc::mbar_wait(q_full + (qi & 1), (qi >> 1) & 1, abort_flag, a.status))
          return false;
        if (!tc::mbar_wait(k_full + stage, (g / STAGES) & 1, abort_flag, a.status)) return false;
        if (!tc::mbar_wait(x_empty + (g & 1), ((g >> 1) & 1) ^ 1, abort_flag, a.status))
          return false;
        tc::fence_after_sync();
        const uint32_t qa = tc::smem_u32(q_buf(qi & 1));
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {  // K = d, 16 per step, 32 bytes
          const uint32_t koff = (uint32_t)((j * 32) / 128), kin = (uint32_t)((j * 32) % 128);
          const uint64_t ad = desc2(ring_a + stage * C_::KT + koff * 128 * 128 + kin, 16, 1024);
          const uint64_t bd = desc2(qa + koff * HP * 128 + kin, 16, 1024);
          tc::mma<0>(tmem_base + C_::X_COL + (g & 1) * HP, ad, bd, ID_X, j > 0 ? 1u : 0u);
        }
        tc::mma_commit(x_full + (g & 1));
        return true;
      };
      // dq and dk for tile g, once the epilogue has written Aq / Ak
      auto grads = [&](int g) -> bool {
        const int qi = g / ktiles, i = g - qi * ktiles;
        const int stage = g % STAGES;
        if (!tc::mbar_wait(a_full, g & 1, abort_flag, a.status)) return false;
        if (i == 0 && !tc::mbar_wait(dq_empty, (qi & 1) ^ 1, abort_flag, a.status)) return false;
        if (!tc::mbar_wait(dk_empty + (g & 1), ((g >> 1) & 1) ^ 1, abort_flag, a.status))
          return false;
        tc::fence_after_sync();
        // DQ[h'][n] += sum_key Aq[key][h'] * Kt[key][n]: 8 steps of 16 keys
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint64_t ad = desc2(aq_a + s * 2048, 128 * 128, 1024);
          const uint64_t bd = desc2(ring_a + stage * C_::KT + s * 2048, 128 * 128, 1024);
          tc::mma<0>(tmem_base + C_::DQ_COL, ad, bd, ID_DQ, (i > 0 || s > 0) ? 1u : 0u);
        }
        // DK[key][n] = sum_h' Ak[key][h'] * Q[h' mod HP][n]: high then low halves
        const uint32_t qa = tc::smem_u32(q_buf(qi & 1));
#pragma unroll
        for (int s = 0; s < 2 * HP / 16; ++s) {
          const uint32_t koff = (uint32_t)((s * 32) / 128), kin = (uint32_t)((s * 32) % 128);
          const uint64_t ad = desc2(ak_a + koff * 128 * 128 + kin, 16, 1024);
          const uint64_t bd = desc2(qa + (s % (HP / 16)) * 2048, HP * 128, 1024);
          tc::mma<0>(tmem_base + C_::DK_COL + (g & 1) * D, ad, bd, ID_DK, s > 0 ? 1u : 0u);
        }
        tc::mma_commit(dk_full + (g & 1));
        tc::mma_commit(a_empty);
        tc::mma_commit(k_empty + stage);
        if (i == ktiles - 1) {
          tc::mma_commit(dq_full);
          tc::mma_commit(q_empty + (qi & 1));
        }
        return true;
      };
      // forward of tile g + 1 goes ahead of the gradients of tile g
      if (total > 0 && forward(0)) {
        for (int g = 0; g < total; ++g) {
          if (g + 1 < total && !forward(g + 1)) break;
          if (!grads(g)) break;
        }
      }
    }
  } else if (warp >= kEpiFirstWarp) {
    // ---------------- epilogue: TMEM lane = key ----------------
    const int e = warp - kEpiFirstWarp;
    const int gp = e / 4;                 // head / column group of this warp
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    constexpr int HG = HP / kGroups, DG = D / kGroups;
    constexpr int CH = HG < 32 ? HG : 32;       // X columns per TMEM load
    constexpr int NDW = HG >= 32 ? HG / 32 : 1;  // dw sums this lane keeps
    const int h0 = gp * HG, d0 = gp * DG;
    float dwacc[NDW];
    int s_prev = -1;
    float g_prev = 0.0f;
    uint32_t meet_phase = 0;
    bool ok = true;
    // this row's stored key, gradient and key scale for tile g (loaded a tile ahead)
    auto load_entry = [&](int g, int& s, float& G, float& ks) {
      const int qi = g / ktiles, i = g - qi * ktiles;
      const int t = (int)blockIdx.x + qi * (int)gridDim.x;
      const int j = i * 128 + row;
      s = j < a.k_top ? __ldg(a.idx + (size_t)t * a.k_top + j) : -1;
      if (s != -1 && (s < 0 || s >= a.L)) {
        if (a.status && gp == 0) atomicOr(a.status, HYTOPK_DEV_REPLAY_BAD_INDEX);
        s = -1;
      }
      G = s >= 0 ? __ldg(a.grad + (size_t)t * a.k_top + j) : 0.0f;
      ks = (s >= 0 && DT == 1) ? __ldg(a.k_scale + s) : 1.0f;
    };
    int s_next = -1;
    float G_next = 0.0f, ks_next = 1.0f;
    if (total > 0) load_entry(0, s_next, G_next, ks_next);
    for (int g = 0; g < total && ok; ++g) {
      const int qi = g / ktiles, i = g - qi * ktiles;
      const int t = (int)blockIdx.x + qi * (int)gridDim.x;
      const int qb = qi & 1;
      if (i == 0) {
#pragma unroll
        for (int u = 0; u < NDW; ++u) dwacc[u] = 0.0f;
        if (!__all_sync(0xffffffffu,
                        tc::mbar_wait(q_full + qb, (qi >> 1) & 1, abort_flag, a.status)))
          break;
      }
      const float* w_s = ws + qb * 3 * HP;
      const float* qs_s = w_s + HP;
      const uint32_t* vpair = reinterpret_cast<const uint32_t*>(w_s + 2 * HP);  // [hi HP/2][lo HP/2]
      const int s = s_next;
      const float G = G_next, ks = ks_next;
      if (g + 1 < total) load_entry(g + 1, s_next, G_next, ks_next);
      const float cdw = G * ks;  // the key's factor c (and its dw weight)
      uint32_t chh, cll;  // c split into bf16 high / low parts, repeated in both halves
      {
        uint16_t ch, cl;
        split_bf16(cdw, ch, cl);
        chh = (uint32_t)ch * 0x10001u;
        cll = (uint32_t)cl * 0x10001u;
      }
      // (a) wait for Aq / Ak to be free and X to be ready
      if (!__all_sync(0xffffffffu, tc::mbar_wait(a_empty, (g & 1) ^ 1, abort_flag, a.status)))
        break;
      if (!__all_sync(0xffffffffu,
                      tc::mbar_wait(x_full + (g & 1), (g >> 1) & 1, abort_flag, a.status)))
        break;
      tc::fence_after_sync();
      const uint32_t xaddr = tmem_base + lane_off + C_::X_COL + (g & 1) * HP;
#pragma unroll
      for (int cc = 0; cc < HG; cc += CH) {
        const int c0 = h0 + cc;
        float x[CH];
        if constexpr (CH == 32) {
          tc::tmem_ld32(xaddr + c0, x);
          tc::tmem_wait_ld(x);
        } else if constexpr (CH == 16) {
          tc::tmem_ld16(xaddr + c0, x);
          tc::tmem_wait_ld(x);
        } else {
          tc::tmem_ld8(xaddr + c0, x);
          tc::tmem_wait_ld(x);
        }
        // Aq / Ak rows: 8 heads per 16-byte chunk, high parts at h', low at HP + h'
#pragma unroll
        for (int h8 = 0; h8 < CH; h8 += 8) {
          uint32_t qh[4], ql[4], kh[4], kl[4];
          const uint4 vh = *reinterpret_cast<const uint4*>(vpair + (c0 + h8) / 2);
          const uint4 vl = *reinterpret_cast<const uint4*>(vpair + HP / 2 + (c0 + h8) / 2);
          const uint32_t vhs[4] = {vh.x, vh.y, vh.z, vh.w}, vls[4] = {vl.x, vl.y, vl.z, vl.w};
#pragma unroll
          for (int u = 0; u < 8; u += 2) {
            // [X > 0] of the two heads as a mask over their 16-bit halves
            const uint32_t m = (x[h8 + u] > 0.0f ? 0x0000FFFFu : 0u) |
                               (x[h8 + u + 1] > 0.0f ? 0xFFFF0000u : 0u);
            qh[u / 2] = chh & m;
            ql[u / 2] = cll & m;
            kh[u / 2] = vhs[u / 2] & m;
            kl[u / 2] = vls[u / 2] & m;
          }
          const int h = c0 + h8;
          *reinterpret_cast<uint4*>(aq + sw_off(row, h, 128)) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
          *reinterpret_cast<uint4*>(aq + sw_off(row, HP + h, 128)) = make_uint4(ql[0], ql[1], ql[2], ql[3]);
          *reinterpret_cast<uint4*>(ak + sw_off(row, h, 128)) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
          *reinterpret_cast<uint4*>(ak + sw_off(row, HP + h, 128)) = make_uint4(kl[0], kl[1], kl[2], kl[3]);
        }
        // dw: sum over the warp's 32 keys of G k_scale max(0, X)
#pragma unroll
        for (int u = 0; u < CH; ++u) x[u] = cdw * fmaxf(x[u], 0.0f);
        butterfly<CH>(x, lane);
        dwacc[cc / CH < NDW ? cc / CH : 0] += x[0];
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(x_empty + (g & 1));
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(a_full);
      // (c) the previous tile's DK rows into dk (deferred one tile), and at the
      // query's last tile this tile's too; this group adds columns [d0, d0 + DG)
      auto drain_dk = [&](int gg, int sk, float gk) -> bool {
        if (!__all_sync(0xffffffffu, tc::mbar_wait(dk_full + (gg & 1), (gg >> 1) & 1, abort_flag,
                                                   a.status)))
          return false;
        tc::fence_after_sync();
        const uint32_t daddr = tmem_base + lane_off + C_::DK_COL + (gg & 1) * D + d0;
        // Each lane holds its key's row; through the warp's staging block the
        // additions go out 4 rows x 128 bytes per instruction (8 lanes per row)
        // instead of 32 rows x 16 bytes, i.e. 4 cache lines instead of 32.
        float* tr = reinterpret_cast<float*>(smem + C_::TR_OFF) + e * C_::TR_FLOATS;
#pragma unroll
        for (int c0 = 0; c0 < DG; c0 += 32) {
          float v[32];
          tc::tmem_ld32(daddr + c0, v);
          tc::tmem_wait_ld(v);
#pragma unroll
          for (int u = 0; u < 32; ++u) tr[lane * 33 + u] = gk * v[u];
          __syncwarp();
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const int r = p * 4 + lane / 8, cc = (lane % 8) * 4;
            const int sr = __shfl_sync(0xffffffffu, sk, r);
            if (sr >= 0) {
              const float* src = tr + r * 33 + cc;
              red_add4(a.dk + (size_t)sr * D + d0 + c0 + cc, src[0], src[1], src[2], src[3]);
            }
          }
          __syncwarp();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(dk_empty + (gg & 1));
        return true;
      };
      if (i > 0 && !drain_dk(g - 1, s_prev, g_prev)) {
        ok = false;
        break;
      }
      s_prev = s;
      g_prev = G;
      if (i == ktiles - 1) {
        if (!drain_dk(g, s, G)) {
          ok = false;
          break;
        }
        // DQ: rows h' < HP are the high parts, HP <= h' < 2HP the low parts
        if (!__all_sync(0xffffffffu, tc::mbar_wait(dq_full, qi & 1, abort_flag, a.status))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        float* scratch = reinterpret_cast<float*>(ak);  // free: every MMA of the query is done
        const uint32_t qaddr = tmem_base + lane_off + C_::DQ_COL + d0;
        // TMEM loads are warp-collective: a warp loads if any of its rows is
        // needed, and each lane then keeps or drops its own row
        const bool warp_has_lo = quad * 32 < 2 * HP && quad * 32 + 32 > HP;
        const bool warp_has_hi = quad * 32 < HP;
        if (warp_has_lo) {
#pragma unroll
          for (int c0 = 0; c0 < DG; c0 += 32) {
            float v[32];
            tc::tmem_ld32(qaddr + c0, v);
            tc::tmem_wait_ld(v);
            if (row >= HP && row < 2 * HP) {
#pragma unroll
              for (int u = 0; u < 32; u += 4)
                *reinterpret_cast<float4*>(scratch + (row - HP) * D + d0 + c0 + u) =
                    make_float4(v[u], v[u + 1], v[u + 2], v[u + 3]);
            }
          }
        }
        // dw partials of the four lane quadrants for this group's heads
#pragma unroll
        for (int u = 0; u < NDW; ++u) {
          if constexpr (CH >= 32)
            dws[quad * HP + h0 + u * 32 + lane] = dwacc[u];
          else if (lane % (32 / CH) == 0)
            dws[quad * HP + h0 + butterfly_head<CH>(lane, 0)] = dwacc[u];
        }
        if (!__all_sync(0xffffffffu, epi_meet(meet, meet_phase, abort_flag, a.status))) {
          ok = false;
          break;
        }
        if (warp_has_hi) {
          float* dst = a.dq + ((size_t)t * H + (row < H ? row : 0)) * D + d0;
#pragma unroll
          for (int c0 = 0; c0 < DG; c0 += 32) {
            float v[32];
            tc::tmem_ld32(qaddr + c0, v);
            tc::tmem_wait_ld(v);
            if (row < H) {
              const float wh = w_s[row];
#pragma unroll
              for (int u = 0; u < 32; u += 4) {
                const float4 lo =
                    *reinterpret_cast<const float4*>(scratch + row * D + d0 + c0 + u);
                *reinterpret_cast<float4*>(dst + c0 + u) =
                    make_float4(wh * (v[u] + lo.x), wh * (v[u + 1] + lo.y),
                                wh * (v[u + 2] + lo.z), wh * (v[u + 3] + lo.w));
              }
            }
          }
        }
        if (gp == 0 && row < H) {
          const float dsum = (dws[row] + dws[HP + row]) + (dws[2 * HP + row] + dws[3 * HP + row]);
          a.dw[(size_t)t * H + row] = dsum * qs_s[row];
        }
        tc::fence_before_sync();
        // scratch and dw partials read: Ak may be rewritten
        if (!__all_sync(0xffffffffu, epi_meet(meet, meet_phase, abort_flag, a.status))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc::mbar_arrive(dq_empty);
          tc::mbar_arrive(q_empty + qb);
        }
      }
    }
    (void)ok;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTmemWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, 512);
  }
}

template <int D, int DT, int H>
inline int backward_smem_bytes() {
  return Cfg<D, DT, H>::SMEM;
}

}  // namespace bwd
}  // namespace hytopk

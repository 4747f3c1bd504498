// threshold_engine.cuh -- the sampled threshold of HyTopK: per query, score
// M evenly spaced sample keys on the tensor cores and take the r-th best
// sample score.
//
// HyScale explainer, HyTopK paragraph and worked example: M samples of the
// query's own context, spread evenly; the threshold is the sample score whose
// rank stands for about the 3k-th best key (r = ceil(3 k M / ctx)).
//
// The queries of a CTA flow through its roles without a CTA-wide barrier
// between them:
//   warps 0..3   producers: the query's q operand and folded weights into one
//                of two buffers, then its sample rows, gathered 128 at a time
//                with cp.async into a ring of stages
//   warp 12      TMEM allocator and MMA issuer (128 samples x max(H, 16))
//   warps 8..11  epilogue (TMEM lane = sample): the head reduction of the
//                filter (the accumulator handed back to the MMA issuer once
//                its last columns are in registers), then the sample's
//                ordered key desc32(score) stored into tensor memory, one
//                column per tile
//   warps 4..7   select: the r-th smallest key of the query's M keys, read
//                back from tensor memory (radix select over 2048 bins that
//                span the keys' own range, shared-memory histogram), while
//                the other roles already work on the next queries
// Two key buffers of 64 TMEM columns (M <= 8192 = 64 x 128) sit beside the
// two accumulators, so a query's keys are selected while the next query's are
// written. Scores are those of the filter, bit for bit (stream::HeadSum,
// finish_score).
#pragma once

#include "radix.cuh"
#include "stream_engine.cuh"

namespace hytopk {
namespace thr {

constexpr int kThreads = 416;   // 13 warps
constexpr int kProducers = 128; // warps 0..3
constexpr int kSelWarp0 = 4;    // warps 4..7 (lane quadrant = warp % 4)
constexpr int kEpiWarp0 = 8;    // warps 8..11
constexpr int kMmaWarp = 12;
constexpr int kSlots = 2;                          // TMEM accumulators
constexpr int kKeyCols = kMaxSamples / kTileKeys;  // key columns per buffer
constexpr int kSelBar = 2;                         // named barrier of the select warps
constexpr int kSelThreads = 128;
constexpr int kSelBins = 2048;                     // radix bins of the select
constexpr int kSelBinsPer = kSelBins / kSelThreads;  // bins prefix-summed per thread

struct TArgs {
  const void* k;
  const float* k_scale;
  int L, k_top;
  const int32_t* perm;  // slot -> query, -1 for padding
  const int32_t* qpos;  // slot -> position, -1 for padding / bad position
  const void* qp;       // packed q operand [n_pad, H, d] in the key element type
  const float* wq;      // halved folded weights [n_pad, H]
  float* thr;           // [n_pad] out
  const float* override_thr;
  int n_pad;
  uint32_t* status;
};

template <int D, int DT, int H>
struct TCfg {
  static constexpr int ES = DT == 0 ? 2 : 1;
  static constexpr int RB = D * ES;
  using Geo = tc::Geo<RB>;
  static constexpr int NQ = H < 16 ? 16 : H;  // MMA N (zero padded)
  static constexpr int CPR = RB / 16;         // 16-byte chunks per row
  static constexpr int QBYTES = NQ * RB;
  static constexpr int KT_BYTES = kTileKeys * RB;
  static constexpr int STAGES = RB == 256 ? 2 : (RB == 128 ? 4 : 8);  // a 64 KB ring
  static constexpr int ACC_COLS = kSlots * NQ;
  static constexpr int TMEM_COLS = ACC_COLS + 2 * kKeyCols <= 256 ? 256 : 512;
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = ((2 * QBYTES + 1023) / 1024) * 1024;
  static constexpr int W_OFF = RING_OFF + STAGES * KT_BYTES;  // [2][NQ] fp32
  static constexpr int HIST_OFF = W_OFF + 2 * NQ * 4;         // [kSelBins] u32
  static constexpr int SEL_OFF = HIST_OFF + kSelBins * 4;     // [16] u32
  static constexpr int BAR_OFF = SEL_OFF + 64;
  // full/empty stages, accumulators, q buffers, key buffers
  static constexpr int NBARS = 2 * STAGES + 2 * kSlots + 4 + 4;
  static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;        // TMEM base, abort flag
  static constexpr int END = MISC_OFF + 16;
  // more than 256 TMEM columns: shared memory sized so that one CTA holds an SM
  static constexpr int SMEM = 1024 + ((TMEM_COLS > 256 && END < 120 * 1024) ? 120 * 1024 : END);
  static_assert(END + 1024 <= 113 * 1024 || TMEM_COLS > 256 || RB == 256,
                "two CTAs per SM for the common shapes");
};

// A query's sampling parameters, the same for every role.
struct TQ {
  int t, ctx, M, r, ntiles;
  bool scored;
  SampleStep step;
};

__device__ __forceinline__ TQ thr_query(const TArgs& a, int slot) {
  TQ q{};
  q.t = __ldg(a.perm + slot);
  q.ctx = __ldg(a.qpos + slot) + 1;
  q.scored = q.t >= 0 && q.ctx > a.k_top && a.override_thr == nullptr;
  if (q.scored) {
    q.M = sample_count(q.ctx);
    q.r = threshold_rank(q.ctx, a.k_top, q.M);
    q.step.init(q.ctx, q.M);
    q.ntiles = (q.M + kTileKeys - 1) / kTileKeys;
  }
  return q;
}

// The kk-th smallest (1-based) of a query's M sample keys in the key buffer
// at kcol: sample j sits in column j / 128, TMEM lane j % 128 (the select
// warps cover the 128 lanes; thread st reads lane st). Radix select whose
// digit follows the keys' range: a first sweep finds their minimum and
// maximum, then each pass splits the current range [base, base + 2^width)
// into kSelBins bins of equal width, counts the keys in each (bin b kept at
// hist[(b % kSelBinsPer) * 128 + b / kSelBinsPer], so that each thread's
// prefix sum over its kSelBinsPer bins reads them without bank conflicts) and
// narrows the range to the bin holding the kk-th key -- until that bin is one
// key wide or holds the kk-th key alone. Scores spread over a few exponents
// fill the bins of the first pass evenly, so one pass and a sweep to fetch
// the lone key usually suffice. sh: 16 words of shared scratch. All 128
// select threads call it.
__device__ __forceinline__ uint32_t tmem_kth_smallest(uint32_t kcol, int M, uint32_t kk,
                                                      uint32_t* hist, uint32_t* sh) {
  const int st = (int)threadIdx.x - kSelWarp0 * 32, lane = st & 31, sw = st >> 5;
  const int ncols = (M + kTileKeys - 1) / kTileKeys;
  // f(key) for each of this lane's sample keys (padding rows past M skipped)
  auto sweep = [&](auto&& f) {
    for (int c0 = 0; c0 < ncols; c0 += 16) {
      uint32_t v[16];
      tc::tmem_ld16u(kcol + (uint32_t)c0, v);
      tc::tmem_wait_ld(v);
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if ((c0 + u) * kTileKeys + st < M) f(v[u]);
    }
  };
  uint32_t lo = 0xffffffffu, hi = 0u;
  sweep([&](uint32_t v) {
    lo = min(lo, v);
    hi = max(hi, v);
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    sh[sw] = lo;
    sh[4 + sw] = hi;
  }
  tc::bar_sync(kSelBar, kSelThreads);
  uint32_t base = min(min(sh[0], sh[1]), min(sh[2], sh[3]));
  const uint32_t top = max(max(sh[4], sh[5]), max(sh[6], sh[7]));
  int width = top == base ? 0 : 32 - __clz(top - base);  // keys in [base, base + 2^width)
  while (width > 0) {
    const int sft = width > 11 ? width - 11 : 0;
    for (int b = st; b < kSelBins; b += kSelThreads) hist[b] = 0u;
    tc::bar_sync(kSelBar, kSelThreads);
    sweep([&](uint32_t v) {
      const uint32_t off = v - base;
      if (v >= base && (width >= 32 || (off >> width) == 0u)) {
        const uint32_t bin = off >> sft;
        atomicAdd(hist + (bin % kSelBinsPer) * kSelThreads + bin / kSelBinsPer, 1u);
      }
    });
    tc::bar_sync(kSelBar, kSelThreads);
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < kSelBinsPer; ++j) local += hist[j * kSelThreads + st];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) sh[8 + sw] = incl;
    tc::bar_sync(kSelBar, kSelThreads);
    uint32_t run = incl - local;
    for (int w = 0; w < sw; ++w) run += sh[8 + w];
#pragma unroll
    for (int j = 0; j < kSelBinsPer; ++j) {
      const uint32_t c = hist[j * kSelThreads + st];
      if (run < kk && kk <= run + c) {
        sh[12] = (uint32_t)(st * kSelBinsPer + j);
        sh[13] = run;
        sh[14] = c;
      }
      run += c;
    }
    tc::bar_sync(kSelBar, kSelThreads);
    const uint32_t bstar = sh[12], before = sh[13], cnt = sh[14];
    kk -= before;
    base += bstar << sft;
    width = sft;
    if (width > 0 && cnt == 1u) {  // the kk-th key is alone in its bin: fetch it
      sweep([&](uint32_t v) {
        if (v >= base && ((v - base) >> width) == 0u) sh[15] = v;
      });
      tc::bar_sync(kSelBar, kSelThreads);
      base = sh[15];
      width = 0;
    }
  }
  // every thread is past its reads of sh and hist before they are reused
  tc::bar_sync(kSelBar, kSelThreads);
  return base;
}

template <int D, int DT, int H>
__global__ void __launch_bounds__(kThreads, 2) k_threshold(const TArgs a) {
  using C_ = TCfg<D, DT, H>;
  using Geo = typename C_::Geo;
  constexpr int NQ = C_::NQ, STAGES = C_::STAGES, CPR = C_::CPR, RB = C_::RB;
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  uint8_t* smem = tc::align1024(smem_dyn);
  uint8_t* qbuf = smem + C_::Q_OFF;
  uint8_t* ring = smem + C_::RING_OFF;
  float* wq_s = reinterpret_cast<float*>(smem + C_::W_OFF);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + C_::HIST_OFF);
  uint32_t* sel_sh = reinterpret_cast<uint32_t*>(smem + C_::SEL_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C_::BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + kSlots;
  uint64_t* q_full = acc_empty + kSlots;  // [2]
  uint64_t* q_empty = q_full + 2;         // [2]
  uint64_t* k_full = q_empty + 2;         // [2]
  uint64_t* k_empty = k_full + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C_::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C_::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(full + i, kProducers);
      tc::mbar_init(empty + i, 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      tc::mbar_init(acc_full + i, 1);
      tc::mbar_init(acc_empty + i, 4);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(q_full + i, kProducers);
      tc::mbar_init(q_empty + i, 1 + 4);  // the MMA commit and the 4 epilogue warps
      tc::mbar_init(k_full + i, 4);       // epilogue warps
      tc::mbar_init(k_empty + i, 4);      // select warps
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, C_::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 4) {
    // ---------------- producers ----------------
    // Per query: the operand rows and weights into buffer b, then the sample
    // rows. Warp w gathers rows 32w .. 32w+31 of each tile; lane l fetches the
    // key index of row 32w + l (two tiles ahead); the copies go CPR lanes per
    // row, so that each warp instruction reads 32 / CPR whole rows.
    const int tid = threadIdx.x;
    constexpr int RPP = 32 / CPR;
    int p_stage = 0, nq = 0;
    uint32_t p_phase = 0;
    for (int slot = blockIdx.x; slot < a.n_pad; slot += gridDim.x) {
      const TQ q = thr_query(a, slot);
      if (!q.scored) continue;
      const int b = nq & 1;
      const uint32_t par = (uint32_t)(nq >> 1) & 1u;
      ++nq;
      const bool okq = tc::mbar_wait(q_empty + b, par ^ 1u, abort_flag, a.status);
      if (!__all_sync(0xffffffffu, okq)) break;
      uint8_t* qb = qbuf + b * C_::QBYTES;
      const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(a.qp) + (size_t)slot * H * RB;
      for (int f = tid; f < NQ * CPR; f += kProducers) {
        const int row = f / CPR, c = f % CPR;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < H) v = *reinterpret_cast<const uint4*>(qsrc + (size_t)row * RB + c * 16);
        *reinterpret_cast<uint4*>(qb + Geo::chunk_offset(row, c, NQ)) = v;
      }
      for (int h = tid; h < NQ; h += kProducers)
        wq_s[b * NQ + h] = h < H ? __ldg(a.wq + (size_t)slot * H + h) : 0.0f;
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(q_full + b);
      SampleWalk walk;  // this lane's sample of each tile
      walk.init(q.step, tid);
      auto key_of = [&](int j) -> int {  // sample j = next tile's, -1 past M
        const int s = walk.next();
        return j < q.M ? s : -1;
      };
      int npend = 0;
      int s_next = key_of(tid), s_next2 = key_of(kTileKeys + tid);
      bool ok = true;
      for (int i = 0; i < q.ntiles; ++i) {
        const int s_own = s_next;
        s_next = s_next2;
        s_next2 = key_of((i + 2) * kTileKeys + tid);
        const bool okw = tc::mbar_wait(empty + p_stage, p_phase ^ 1u, abort_flag, a.status);
        if (!__all_sync(0xffffffffu, okw)) {
          ok = false;
          break;
        }
        uint8_t* dst = ring + p_stage * C_::KT_BYTES;
        const int c = lane % CPR;
#pragma unroll
        for (int pass = 0; pass < CPR; ++pass) {
          const int src_lane = pass * RPP + lane / CPR;
          const int s = __shfl_sync(0xffffffffu, s_own, src_lane);
          const int row = warp * 32 + src_lane;
          const uint8_t* src =
              reinterpret_cast<const uint8_t*>(a.k) + (s >= 0 ? (size_t)s * RB + c * 16 : 0);
          tc::cp_async16(dst + Geo::chunk_offset(row, c, kTileKeys), src, s >= 0);
        }
        tc::cp_async_commit();
        ++npend;
        if (npend == STAGES - 1) {
          tc::cp_async_wait<STAGES - 2>();
          tc::fence_proxy_async_smem();
          tc::mbar_arrive(full + (p_stage - (npend - 1) + STAGES) % STAGES);
          --npend;
        }
        if (++p_stage == STAGES) {
          p_stage = 0;
          p_phase ^= 1u;
        }
      }
      tc::cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      for (; npend > 0; --npend) tc::mbar_arrive(full + (p_stage - npend + STAGES) % STAGES);
      if (!ok) break;
    }
  } else if (warp < kEpiWarp0) {
    // ---------------- select ----------------
    const int st = (int)threadIdx.x - kSelWarp0 * 32;
    const int quad = warp & 3;
    int nq = 0;
    for (int slot = blockIdx.x; slot < a.n_pad; slot += gridDim.x) {
      const TQ q = thr_query(a, slot);
      if (q.t < 0) continue;
      if (!q.scored) {
        if (st == 0)
          a.thr[slot] = q.ctx <= a.k_top ? -__int_as_float(0x7f800000) : a.override_thr[q.t];
        continue;
      }
      const int b = nq & 1;
      const uint32_t par = (uint32_t)(nq >> 1) & 1u;
      ++nq;
      const bool ok = tc::mbar_wait(k_full + b, par, abort_flag, a.status);
      if (tc::bar_or(kSelBar, kSelThreads, !ok || *abort_flag != 0)) break;
      tc::fence_after_sync();
      const uint32_t kcol =
          tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(C_::ACC_COLS + b * kKeyCols);
      const uint32_t v = tmem_kth_smallest(kcol, q.M, (uint32_t)q.r, hist, sel_sh);
      if (st == 0) a.thr[slot] = desc32_score(v);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(k_empty + b);
    }
  } else if (warp < kMmaWarp) {
    // ---------------- epilogue: one sample per thread ----------------
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int e_slot = 0, nq = 0;
    uint32_t e_aphase = 0;
    auto scale_of = [&](int s) -> float {
      return DT == 1 ? ((s >= 0 && s < a.L) ? __ldg(a.k_scale + s) : 0.0f) : 1.0f;
    };
    for (int slot = blockIdx.x; slot < a.n_pad; slot += gridDim.x) {
      const TQ q = thr_query(a, slot);
      if (!q.scored) continue;
      const int b = nq & 1;
      const uint32_t par = (uint32_t)(nq >> 1) & 1u;
      ++nq;
      const bool ok1 = tc::mbar_wait(q_full + b, par, abort_flag, a.status);
      const bool ok2 = tc::mbar_wait(k_empty + b, par ^ 1u, abort_flag, a.status);
      if (!__all_sync(0xffffffffu, ok1 && ok2)) break;
      tc::fence_after_sync();
      const float* wq = wq_s + b * NQ;
      const uint32_t kcol = tmem_base + lane_off + (uint32_t)(C_::ACC_COLS + b * kKeyCols);
      SampleWalk walk;  // this thread's sample of each tile
      walk.init(q.step, row);
      auto key_of = [&](int j) -> int {  // sample j = next tile's, -1 past M
        const int s = walk.next();
        return j < q.M ? s : -1;
      };
      int s_next = key_of(row), s_next2 = key_of(kTileKeys + row);
      float ks_next = scale_of(s_next);
      bool ok = true;
      for (int i = 0; i < q.ntiles; ++i) {
        const float ks = ks_next;
        s_next = s_next2;
        ks_next = scale_of(s_next);
        s_next2 = key_of((i + 2) * kTileKeys + row);
        if (!tc::mbar_wait(acc_full + e_slot, e_aphase, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t taddr = tmem_base + lane_off + (uint32_t)(e_slot * NQ);
        stream::HeadSum<H> hs;
        hs.reset();
        float sc = 0.0f;
        // the accumulator goes back to the MMA issuer as soon as its last
        // columns are in registers, before they are reduced
        auto release = [&]() {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(acc_empty + e_slot);
          if (++e_slot == kSlots) {
            e_slot = 0;
            e_aphase ^= 1u;
          }
        };
        if constexpr (H >= 32) {
#pragma unroll
          for (int c0 = 0; c0 < H; c0 += 32) {
            float v[32];
            tc::tmem_ld32(taddr + c0, v);
            tc::tmem_wait_ld(v);
            if (c0 + 32 == H) release();
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(wq + c0 + h);
              hs.add_pair(c0 + h, v[h], v[h + 1], w4.x, w4.y);
              hs.add_pair(c0 + h + 2, v[h + 2], v[h + 3], w4.z, w4.w);
            }
          }
          sc = hs.total();
        } else {
          float v[16];
          tc::tmem_ld16(taddr, v);
          tc::tmem_wait_ld(v);
          release();
          if (H == 1) {
            sc = stream::single_head_score<H>(v[0], wq[0]);
          } else {
#pragma unroll
            for (int h = 0; h < (H < 16 ? H : 16); h += 2) hs.add_pair(h, v[h], v[h + 1], wq[h], wq[h + 1]);
            sc = hs.total();
          }
        }
        sc = finish_score(sc, ks);
        // rows past M (the last tile's padding) sort last
        tc::tmem_st1(kcol + (uint32_t)i, i * kTileKeys + row < q.M ? desc32(sc) : 0xffffffffu);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (!ok) break;
      if (lane == 0) {
        tc::mbar_arrive(k_full + b);
        tc::mbar_arrive(q_empty + b);
      }
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t IDESC = tc::instr_desc(DT, 128, NQ);
    const uint32_t r_addr = tc::smem_u32(ring);
    int m_stage = 0, m_slot = 0, nq = 0;
    uint32_t m_phase = 0, m_aphase = 0;
    for (int slot = blockIdx.x; slot < a.n_pad; slot += gridDim.x) {
      const TQ q = thr_query(a, slot);
      if (!q.scored) continue;
      const int b = nq & 1;
      const uint32_t par = (uint32_t)(nq >> 1) & 1u;
      ++nq;
      if (!tc::mbar_wait(q_full + b, par, abort_flag, a.status)) break;
      tc::fence_after_sync();
      const uint32_t q_addr = tc::smem_u32(qbuf + b * C_::QBYTES);
      bool ok = true;
      for (int i = 0; i < q.ntiles; ++i) {
        if (!tc::mbar_wait(full + m_stage, m_phase, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (!tc::mbar_wait(acc_empty + m_slot, m_aphase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d_tmem = tmem_base + (uint32_t)(m_slot * NQ);
#pragma unroll
        for (int j = 0; j < Geo::kSteps; ++j) {
          const uint64_t adesc = tc::smem_desc(
              r_addr + m_stage * C_::KT_BYTES + Geo::step_offset(j, kTileKeys), Geo::kSbo,
              Geo::kSwizzle);
          const uint64_t bdesc =
              tc::smem_desc(q_addr + Geo::step_offset(j, NQ), Geo::kSbo, Geo::kSwizzle);
          tc::mma<DT>(d_tmem, adesc, bdesc, IDESC, j > 0 ? 1u : 0u);
        }
        tc::mma_commit(acc_full + m_slot);
        tc::mma_commit(empty + m_stage);
        if (++m_stage == STAGES) {
          m_stage = 0;
          m_phase ^= 1u;
        }
        if (++m_slot == kSlots) {
          m_slot = 0;
          m_aphase ^= 1u;
        }
      }
      if (!ok) break;
      tc::mma_commit(q_empty + b);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, C_::TMEM_COLS);
  }
}

template <int D, int DT, int H>
cudaError_t threshold_go(const TArgs& a, int grid, cudaStream_t st) {
  constexpr int smem = TCfg<D, DT, H>::SMEM;
  auto fn = k_threshold<D, DT, H>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fn<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace thr
}  // namespace hytopk

// gather_engine.cuh -- the tensor-core scoring engine over gathered keys, one
// query at a time: selection replay and the recovery rescoring of failed
// queries (the sampled threshold has its own engine, threshold_engine.cuh,
// dispatched from here).
//
// HyScale explainer: the HyTopK paragraph (small recovery kernels rescore
// failed queries over their whole context) and the selection-replay
// paragraph (rescore only the k stored entries).
//
// Per query: the key rows it needs (stored indices or its whole prefix) are
// gathered 128 at a time with cp.async into swizzled shared memory; one
// elected thread multiplies each 128-key tile by the query's H x d operand
// (tcgen05, N = max(H, 16)); four epilogue warps (TMEM lane = key) reduce the
// heads with the same arithmetic as the streaming engine. The CTA then
// finishes the query together: nothing (replay) or an exact top-k of the
// rescored row (recovery).
//
// Paired replay (kReplayPair) serves two adjacent queries per item. Adjacent
// tokens select mostly the same keys (HyScale summary, "What the paper
// found"; explainer, limits paragraph), so the item gathers the union of the
// two stored index lists once (the first query's list, then the second
// query's other keys, matched through a shared-memory hash table) and one MMA
// with both queries' rows (N = 2H) scores every gathered key for both; each
// query keeps the scores of its own entries. Scores equal the single-query
// replay bit for bit.
//
//   warps 0..3  producers (cp.async gather, 128 threads)
//   warp 4      MMA issuer; warp 5 TMEM allocator
//   warps 8..11 epilogue
#pragma once

#include "radix.cuh"
#include "stream_engine.cuh"
#include "threshold_engine.cuh"

namespace hytopk {
namespace gather {

constexpr int kThreads = 384;
constexpr int kProducers = 128;
constexpr int kEpiFirstWarp = 8;
constexpr int kSlots = 2;  // TMEM accumulators

enum Mode { kThreshold = 0, kReplay = 1, kRecover = 2, kReplayPair = 3 };

// Paired replay: the hash table of the first query's keys (8 B per slot, at
// most half full) lives in the stage ring while the rows are built, so k is
// bounded by the ring.
constexpr int kMaxPairTopK = 2048;
__host__ __device__ constexpr int pair_table_slots(int k_top) {
  int ts = 1024;
  while (ts < 2 * k_top) ts *= 2;
  return ts;
}

template <int D, int DT, int H, int MODE>
struct Cfg {
  static constexpr int ES = DT == 0 ? 2 : 1;
  static constexpr int RB = D * ES;
  using Geo = tc::Geo<RB>;
  static constexpr bool PAIR = MODE == kReplayPair;
  static constexpr int QROWS = PAIR ? 2 * H : H;     // query rows of the operand
  static constexpr int NQ = QROWS < 16 ? 16 : QROWS; // MMA N (zero padded)
  static constexpr int CPR = RB / 16;                // 16-byte chunks per row
  static constexpr int STAGES =
      PAIR ? (RB == 256 ? 3 : (RB == 128 ? 4 : 8)) : (RB == 256 ? 3 : 4);
  static constexpr int KT_BYTES = 128 * RB;
  static constexpr int RING = STAGES * KT_BYTES;
  static constexpr int TMEM_COLS = (kSlots * NQ) < 32 ? 32 : (kSlots * NQ);
  static constexpr int Q_OFF = 0;
  static constexpr int U_OFF = ((NQ * RB + 1023) / 1024) * 1024;  // stage ring / post scratch
  static constexpr int NBARS = 2 * STAGES + 2 * kSlots;
  // host computes the union size (depends on k for recovery)
  static_assert(H >= 1 && H <= 128 && (H & (H - 1)) == 0, "H");
  static_assert(!PAIR || (H <= 64 && RING >= pair_table_slots(kMaxPairTopK) * 8 +
                                                 kMaxPairTopK * 4 + 8),
                "paired replay: 2H <= 128 columns, build scratch inside the ring");
};

struct GArgs {
  // the problem
  const void* k;
  const float* k_scale;
  int L, k_top, n;
  // threshold / recovery: packed slots
  const int32_t* perm;
  const int32_t* qpos;
  const void* qp;
  const float* wq;
  float* thr;
  const float* override_thr;
  int n_pad;
  // replay: original queries
  const void* q;
  const float* q_scale;
  int q_e4m3;  // replay: q rows are e4m3 codes (converted to the bf16 operand)
  const float* w;
  const int32_t* idx;
  float* out;
  // recovery
  uint32_t* counters;
  const int32_t* failed_list;
  float* rowbuf;
  int32_t* idx_out;
  float* scores_out;
  // layout
  int u_bytes;  // size of the stage-ring / post-processing union
  uint32_t* status;
};

// Paired replay: the rows of an item are the union of the two queries'
// entries, ordered so that whole warps serve one query where they can: first
// the first query's entries whose key the second query also holds (rja and
// rjb both set), then its other entries (rjb = -1), then the second query's
// entries whose key the first query does not hold (rja = -1, key in xkey).
// A first-query row's key is its stored index (unchecked, as in the
// single-query replay), read again from the list. The first query's keys
// are matched through an open-addressing table in the stage ring (buckets of
// four slots read with one 16-byte load, linear probing over buckets, at most
// half full); a repeated entry of the second query gets a row of its own. Second-query entries outside [0, L) are written here (-inf for -1, else NaN and a
// status bit). Whole CTA; returns the number of rows (k + second-only rows).
static __device__ __forceinline__ uint32_t pair_hash(int s, int ts) {
  return ((uint32_t)s * 0x9E3779B1u) >> (33 - __ffs(ts));
}

static __device__ __forceinline__ int build_pair_rows(const GArgs& a, int t, int tB,
                                                      uint8_t* scratch, int32_t* xkey,
                                                      int16_t* rja, int16_t* rjb, int* ucount) {
  constexpr int KPT = (kMaxPairTopK + kThreads - 1) / kThreads;  // entries per thread
  const int k = a.k_top;
  const int ts = pair_table_slots(k);
  const uint32_t nb = (uint32_t)ts / 4;  // buckets of 4 slots
  int32_t* tkey = reinterpret_cast<int32_t*>(scratch);
  int32_t* trow = tkey + ts;
  int32_t* pjb = trow + ts;   // [k] second-query entry paired with first-query entry j
  int* cnt = pjb + k;         // [2] rows taken from the front / from the back of [0, k)
  // both index lists in registers at once (entry j = threadIdx.x + i * kThreads)
  int sa[KPT], sb[KPT];
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int j = (int)threadIdx.x + i * kThreads;
    sa[i] = j < k ? __ldg(a.idx + (size_t)t * k + j) : -1;
    sb[i] = (j < k && tB >= 0) ? __ldg(a.idx + (size_t)tB * k + j) : -1;
  }
  for (int i = threadIdx.x; i < ts; i += kThreads) tkey[i] = -1;
  for (int j = threadIdx.x; j < k; j += kThreads) pjb[j] = -1;
  if (threadIdx.x == 0) {
    *ucount = 0;
    cnt[0] = cnt[1] = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const unsigned lanes_below = (1u << lane) - 1u;
  if (tB >= 0) {
    // the first query's keys -> one of its entries that holds the key
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const int j = (int)threadIdx.x + i * kThreads;
      const int s = sa[i];
      if (j >= k || s < 0 || s >= a.L) continue;
      // the first bucket (from the key's own) with a free slot; a slot lost to
      // another key sends the thread back to the same bucket. Ends: at most k
      // keys in 2k slots or more, and every failed claim fills a slot.
      uint32_t b = pair_hash(s, (int)nb);
      for (int round = 0; round < 2 * ts; ++round) {
        const int4 v = *reinterpret_cast<const int4*>(tkey + 4 * b);
        if (v.x == s || v.y == s || v.z == s || v.w == s) break;  // held by another entry
        const int e = v.x == -1 ? 0 : (v.y == -1 ? 1 : (v.z == -1 ? 2 : (v.w == -1 ? 3 : 4)));
        if (e == 4) {
          b = (b + 1) & (nb - 1);
          continue;
        }
        const int prev = tc::atom_cas_shared(tkey + 4 * b + e, -1, s);
        if (prev == -1) {
          trow[4 * b + e] = j;
          break;
        }
        if (prev == s) break;
      }
    }
    __syncthreads();
    // the second query's entries: paired with a first-query entry, or rows of their own
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const int j = (int)threadIdx.x + i * kThreads;
      const int s = sb[i];
      bool own = false;
      if (j < k) {
        if (s < 0 || s >= a.L) {
          float v = -__int_as_float(0x7f800000);
          if (s != -1) {
            v = __int_as_float(0x7fc00000);
            if (a.status) atomicOr(a.status, HYTOPK_DEV_REPLAY_BAD_INDEX);
          }
          a.out[(size_t)tB * k + j] = v;
        } else {
          // buckets from the key's own until the key or a free slot (absent)
          int row = -1;
          uint32_t b = pair_hash(s, (int)nb);
          for (uint32_t round = 0; round < nb; ++round) {
            const int4 v = *reinterpret_cast<const int4*>(tkey + 4 * b);
            const int e = v.x == s ? 0 : (v.y == s ? 1 : (v.z == s ? 2 : (v.w == s ? 3 : 4)));
            if (e < 4) {
              row = trow[4 * b + e];
              break;
            }
            if (v.x == -1 || v.y == -1 || v.z == -1 || v.w == -1) break;
            b = (b + 1) & (nb - 1);
          }
          own = row < 0 || tc::atom_cas_shared(pjb + row, -1, j) != -1;
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, own);
      if (m) {
        int u0 = 0;
        if (lane == 0) u0 = tc::atom_add_shared(ucount, __popc(m));
        u0 = __shfl_sync(0xffffffffu, u0, 0);
        if (own) {
          const int u = u0 + __popc(m & lanes_below);
          xkey[u] = s;
          rja[k + u] = -1;
          rjb[k + u] = (int16_t)j;
        }
      }
    }
    __syncthreads();
  }
  // the first query's entries: paired ones from the front, the others from the back
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int j = (int)threadIdx.x + i * kThreads;
    const bool in = j < k;
    const int jb = in ? pjb[j] : -1;
    const bool front = in && jb >= 0;
    const unsigned mf = __ballot_sync(0xffffffffu, front);
    const unsigned mb = __ballot_sync(0xffffffffu, in && !front);
    int f0 = 0, b0 = 0;
    if (lane == 0) {
      if (mf) f0 = tc::atom_add_shared(cnt, __popc(mf));
      if (mb) b0 = tc::atom_add_shared(cnt + 1, __popc(mb));
    }
    f0 = __shfl_sync(0xffffffffu, f0, 0);
    b0 = __shfl_sync(0xffffffffu, b0, 0);
    if (in) {
      const int r = front ? f0 + __popc(mf & lanes_below) : k - 1 - (b0 + __popc(mb & lanes_below));
      rja[r] = (int16_t)j;
      rjb[r] = (int16_t)jb;
    }
  }
  __syncthreads();
  const int n_rows = k + *ucount;
  __syncthreads();  // the table (in the stage ring) is free again after this
  return n_rows;
}

template <int D, int DT, int H, int MODE>
__global__ void __launch_bounds__(kThreads, 2) k_gather(const GArgs a) {
  using C_ = Cfg<D, DT, H, MODE>;
  using Geo = typename C_::Geo;
  constexpr int NQ = C_::NQ, STAGES = C_::STAGES, CPR = C_::CPR, RB = C_::RB;
  constexpr bool PAIR = C_::PAIR;
  constexpr bool REPLAY = MODE == kReplay || PAIR;
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  uint8_t* smem = tc::align1024(smem_dyn);
  uint8_t* qbuf = smem + C_::Q_OFF;
  uint8_t* ring = smem + C_::U_OFF;
  uint8_t* tail = ring + a.u_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tail);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = bars + 2 * STAGES + kSlots;
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + C_::NBARS);
  uint32_t* tmem_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  int* item_sh = reinterpret_cast<int*>(misc + 2);
  int* ucount = reinterpret_cast<int*>(misc + 3);                // paired: union size
  float* wq_s = reinterpret_cast<float*>(misc + 4);              // [H]
  RadixScratch& rsc = *reinterpret_cast<RadixScratch*>(ring);    // after the pipeline drains
  uint64_t* sel = reinterpret_cast<uint64_t*>(ring + sizeof(RadixScratch));
  // paired replay, after the ring: the keys of the second query's own rows,
  // then per row the entry of each query it serves (-1: none)
  int32_t* xkey = reinterpret_cast<int32_t*>(ring + C_::RING);  // [k]
  int16_t* rja = reinterpret_cast<int16_t*>(xkey + a.k_top);      // [2k]
  int16_t* rjb = rja + 2 * a.k_top;                               // [2k]

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
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tmem_slot, C_::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // pipeline state, continued across queries by each role
  int p_stage = 0, m_stage = 0, m_slot = 0, e_slot = 0;
  uint32_t p_phase = 0, m_phase = 0, m_aphase = 0, e_aphase = 0;

  const int n_items =
      MODE == kReplay ? a.n : (PAIR ? (a.n + 1) / 2 : 0);
  const uint32_t n_failed = MODE == kRecover ? a.counters[kCtrFailed] : 0u;
  const bool fallback = n_failed > HYTOPK_MAX_RECOVERY_ROWS;
  // past the limit every query goes through the table path of the fallback instead
  const int n_rec = MODE == kRecover ? (fallback ? 0 : (int)n_failed) : 0;

  for (int it = blockIdx.x;; it += gridDim.x) {
    // ---- pick the query (uniform across the CTA) ----
    int item;
    if (MODE == kRecover) {
      if (threadIdx.x == 0) *item_sh = (int)atomicAdd(a.counters + kCtrRecoverWork, 1u);
      __syncthreads();
      item = *item_sh;
      __syncthreads();
      if (item >= n_rec) break;
    } else {
      item = it;
      if (item >= n_items) break;
    }
    if (*abort_flag) break;
    int slot = -1, t = -1, ctx = 0, nrows = 0;
    int tB = -1;  // paired replay: the second query (t is the first)
    if (MODE == kReplay) {
      t = item;
      nrows = a.k_top;
    } else if (PAIR) {
      t = 2 * item;
      tB = t + 1 < a.n ? t + 1 : -1;
    } else {
      slot = a.failed_list[item];
      t = a.perm[slot];
      ctx = a.qpos[slot] + 1;
      if (t < 0) continue;
      nrows = ctx;
    }
    // key of row j of this query's list (replay: the stored index, unchecked;
    // paired replay: the union row, always inside [0, L))
    auto key_of = [&](int j) -> int {
      if (j >= nrows) return -1;
      if (MODE == kReplay) return __ldg(a.idx + (size_t)t * a.k_top + j);
      if (PAIR)
        return j < a.k_top ? __ldg(a.idx + (size_t)t * a.k_top + rja[j]) : xkey[j - a.k_top];
      return j;
    };

    // ---- the query operand (H rows of d, zero-padded to NQ) and weights ----
    {
      // e4m3 queries against bf16 keys (replay only; the other modes read the
      // packed operand): D-byte rows, 8 codes per 16-byte chunk of the operand
      const bool q8 = DT == 0 && REPLAY && a.q_e4m3;
      const int q_row_bytes = q8 ? D : RB;
      // paired replay: rows H..2H-1 are the second query's (zero if there is none)
      const uint8_t* qsrc =
          REPLAY ? reinterpret_cast<const uint8_t*>(a.q) + (size_t)t * H * q_row_bytes
                 : reinterpret_cast<const uint8_t*>(a.qp) + (size_t)slot * H * RB;
      const int q_rows = PAIR ? (tB >= 0 ? 2 * H : H) : H;
      for (int f = threadIdx.x; f < NQ * CPR; f += kThreads) {
        const int row = f / CPR, c = f % CPR;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < q_rows) {
          if (q8)
            v = e4m3x8_to_bf16(
                *reinterpret_cast<const uint2*>(qsrc + (size_t)row * q_row_bytes + c * 8));
          else
            v = *reinterpret_cast<const uint4*>(qsrc + (size_t)row * RB + c * 16);
        }
        *reinterpret_cast<uint4*>(qbuf + Geo::chunk_offset(row, c, NQ)) = v;
      }
      for (int h = threadIdx.x; h < C_::QROWS; h += kThreads) {
        float hw = 0.0f;  // halved folded weight, as in the prep kernel
        if (REPLAY) {
          // row h of the operand: head h of t, or head h - H of the second query
          if (h < q_rows) {
            float wv = a.w[(size_t)t * H + h];
            if (DT == 1 || a.q_e4m3) wv *= a.q_scale[(size_t)t * H + h];
            hw = 0.5f * wv;
          }
        } else {
          hw = a.wq[(size_t)slot * H + h];
        }
        wq_s[h] = hw;
      }
      tc::fence_proxy_async_smem();
      __syncthreads();
    }
    if constexpr (PAIR) nrows = build_pair_rows(a, t, tB, ring, xkey, rja, rjb, ucount);
    const int ntiles = (nrows + kTileKeys - 1) / kTileKeys;

    if (warp < 4) {
      // ---------------- producers: gather 128 key rows per tile ----------------
      // Warp w gathers rows 32w .. 32w+31 of each tile. Lane l fetches the key
      // index of row 32w + l (two tiles ahead); the copies go CPR lanes per row
      // (lane l moves 16-byte chunk l % CPR), so that each warp instruction
      // reads 32 / CPR whole rows.
      const int tid = threadIdx.x;
      constexpr int RPP = 32 / CPR;  // rows per warp instruction
      int npend = 0;
      int s_next = key_of(tid), s_next2 = key_of(kTileKeys + tid);
      for (int i = 0; i < ntiles; ++i) {
        int s_own = s_next;
        s_next = s_next2;
        s_next2 = key_of((i + 2) * kTileKeys + tid);
        if (s_own >= a.L) s_own = -1;  // stored indices outside [0, L) gather nothing
        // the warp leaves together (the copies below exchange keys by shuffles)
        const bool ok = tc::mbar_wait(empty + p_stage, p_phase ^ 1u, abort_flag, a.status);
        if (!__all_sync(0xffffffffu, ok)) break;
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
          const int st = (p_stage - (npend - 1) + STAGES) % STAGES;
          tc::mbar_arrive(full + st);
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
    } else if (warp == 4) {
      if (lane == 0) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t IDESC = tc::instr_desc(DT, 128, NQ);
        const uint32_t q_addr = tc::smem_u32(qbuf);
        const uint32_t r_addr = tc::smem_u32(ring);
        for (int i = 0; i < ntiles; ++i) {
          if (!tc::mbar_wait(full + m_stage, m_phase, abort_flag, a.status)) break;
          tc::fence_after_sync();
          if (!tc::mbar_wait(acc_empty + m_slot, m_aphase ^ 1u, abort_flag, a.status)) break;
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
      }
    } else if (warp >= kEpiFirstWarp) {
      // ---------------- epilogue: one key per thread ----------------
      const int quad = warp & 3;
      const int row = quad * 32 + lane;
      // keys two tiles ahead and key scales one tile ahead of their use
      auto scale_of = [&](int s) -> float {
        return DT == 1 ? ((s >= 0 && s < a.L) ? __ldg(a.k_scale + s) : 0.0f) : 1.0f;
      };
      int s_next = key_of(row), s_next2 = key_of(kTileKeys + row);
      float ks_next = scale_of(s_next);
      for (int i = 0; i < ntiles; ++i) {
        const int s = s_next;
        const float ks = ks_next;
        s_next = s_next2;
        ks_next = scale_of(s_next);
        s_next2 = key_of((i + 2) * kTileKeys + row);
        if (!tc::mbar_wait(acc_full + e_slot, e_aphase, abort_flag, a.status)) break;
        tc::fence_after_sync();
        const uint32_t taddr =
            tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(e_slot * NQ);
        const int j = i * kTileKeys + row;
        const bool valid = s >= 0 && s < a.L;
        stream::HeadSum<H> hs;
        hs.reset();
        float sc = 0.0f, scB = 0.0f;
        int ja = -1, jb = -1;  // paired replay: the entries this row serves
        if constexpr (PAIR) {
          // columns 0..H-1: the first query's heads, H..2H-1: the second's, with
          // the per-head arithmetic and order of the single-query replay; a warp
          // none of whose rows serves a query skips that query's columns
          if (j < nrows) {
            ja = rja[j];
            jb = rjb[j];
          }
          const bool need_a = __any_sync(0xffffffffu, ja >= 0);
          const bool need_b = __any_sync(0xffffffffu, jb >= 0);
          stream::HeadSum<H> hb;
          hb.reset();
          if constexpr (NQ >= 64) {
            if (need_a) {
#pragma unroll
              for (int c0 = 0; c0 < H; c0 += 32) {
                float v[32];
                tc::tmem_ld32(taddr + c0, v);
                tc::tmem_wait_ld(v);
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                  const float4 w4 = *reinterpret_cast<const float4*>(wq_s + c0 + h);
                  hs.add_pair(c0 + h, v[h], v[h + 1], w4.x, w4.y);
                  hs.add_pair(c0 + h + 2, v[h + 2], v[h + 3], w4.z, w4.w);
                }
              }
              sc = hs.total();
            }
            if (need_b) {
#pragma unroll
              for (int c0 = 0; c0 < H; c0 += 32) {
                float v[32];
                tc::tmem_ld32(taddr + H + c0, v);
                tc::tmem_wait_ld(v);
#pragma unroll
                for (int h = 0; h < 32; h += 4) {
                  const float4 w4 = *reinterpret_cast<const float4*>(wq_s + H + c0 + h);
                  hb.add_pair(c0 + h, v[h], v[h + 1], w4.x, w4.y);
                  hb.add_pair(c0 + h + 2, v[h + 2], v[h + 3], w4.z, w4.w);
                }
              }
              scB = hb.total();
            }
          } else if constexpr (NQ == 32) {  // H = 16: one load holds both queries
            float v[32];
            tc::tmem_ld32(taddr, v);
            tc::tmem_wait_ld(v);
#pragma unroll
            for (int h = 0; h < 16; h += 2) {
              hs.add_pair(h, v[h], v[h + 1], wq_s[h], wq_s[h + 1]);
              hb.add_pair(h, v[16 + h], v[17 + h], wq_s[16 + h], wq_s[17 + h]);
            }
            sc = hs.total();
            scB = hb.total();
          } else {  // H <= 8
            float v[16];
            tc::tmem_ld16(taddr, v);
            tc::tmem_wait_ld(v);
            if (H == 1) {
              sc = stream::single_head_score<H>(v[0], wq_s[0]);
              scB = stream::single_head_score<H>(v[1], wq_s[1]);
            } else {
#pragma unroll
              for (int h = 0; h < (H < 8 ? H : 8); h += 2) {
                hs.add_pair(h, v[h], v[h + 1], wq_s[h], wq_s[h + 1]);
                hb.add_pair(h, v[H + h], v[H + h + 1], wq_s[H + h], wq_s[H + h + 1]);
              }
              sc = hs.total();
              scB = hb.total();
            }
          }
          scB = finish_score(scB, ks);
        } else if (H >= 32) {
#pragma unroll
          for (int c0 = 0; c0 < H; c0 += 32) {
            float v[32];
            tc::tmem_ld32(taddr + c0, v);
            tc::tmem_wait_ld(v);
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
              const float4 w4 = *reinterpret_cast<const float4*>(wq_s + c0 + h);
              hs.add_pair(c0 + h, v[h], v[h + 1], w4.x, w4.y);
              hs.add_pair(c0 + h + 2, v[h + 2], v[h + 3], w4.z, w4.w);
            }
          }
          sc = hs.total();
        } else {
          float v[16];
          tc::tmem_ld16(taddr, v);
          tc::tmem_wait_ld(v);
          if (H == 1) {
            sc = stream::single_head_score<H>(v[0], wq_s[0]);
          } else {
#pragma unroll
            for (int h = 0; h < (H < 16 ? H : 16); h += 2)
              hs.add_pair(h, v[h], v[h + 1], wq_s[h], wq_s[h + 1]);
            sc = hs.total();
          }
        }
        sc = finish_score(sc, ks);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(acc_empty + e_slot);
        if (++e_slot == kSlots) {
          e_slot = 0;
          e_aphase ^= 1u;
        }
        if (j < nrows) {
          if (PAIR) {
            if (ja >= 0) {
              float v = sc;
              if (!valid) {
                if (s == -1) {
                  v = -__int_as_float(0x7f800000);
                } else {
                  v = __int_as_float(0x7fc00000);
                  if (a.status) atomicOr(a.status, HYTOPK_DEV_REPLAY_BAD_INDEX);
                }
              }
              a.out[(size_t)t * a.k_top + ja] = v;
            }
            if (jb >= 0) a.out[(size_t)tB * a.k_top + jb] = scB;
          } else if (REPLAY) {
            float v = sc;
            if (!valid) {
              if (s == -1) {
                v = -__int_as_float(0x7f800000);
              } else {
                v = __int_as_float(0x7fc00000);
                if (a.status) atomicOr(a.status, HYTOPK_DEV_REPLAY_BAD_INDEX);
              }
            }
            a.out[(size_t)t * a.k_top + j] = v;
          } else {
            a.rowbuf[(size_t)blockIdx.x * a.L + j] = sc;
          }
        }
      }
    }
    __syncthreads();
    if (*abort_flag) break;
    // ---- per-query completion (whole CTA) ----
    if (MODE == kRecover) {
      const int got = cta_row_topk(a.rowbuf + (size_t)blockIdx.x * a.L, ctx, a.k_top, sel, rsc);
      write_selection(sel, got, a.k_top, a.idx_out + (size_t)t * a.k_top,
                      a.scores_out ? a.scores_out + (size_t)t * a.k_top : nullptr);
      __syncthreads();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, C_::TMEM_COLS);
  }
}

// Shared memory of k_gather: q operand + max(stage ring, post-processing
// scratch) + barriers and weights.
template <int D, int DT, int H, int MODE>
inline int gather_smem_bytes(int k_top, int* u_bytes) {
  using C_ = Cfg<D, DT, H, MODE>;
  int post = 0;
  if (MODE == kRecover) post = (int)sizeof(RadixScratch) + sort_capacity(k_top) * 8;
  int u = C_::RING > post ? C_::RING : post;
  if (MODE == kReplayPair) u = C_::RING + 3 * k_top * 4;  // + xkey, rja, rjb
  u = (u + 15) / 16 * 16;
  *u_bytes = u;
  const int tail = 8 * C_::NBARS + 16 + 128 * 4;
  return 1024 + C_::U_OFF + u + tail;
}

// Host launch of one instantiation (dynamic shared memory set per call).
template <int D, int DT, int H, int MODE>
cudaError_t gather_go(const GArgs& a0, int grid, cudaStream_t st) {
  GArgs a = a0;
  int u = 0;
  const int smem = gather_smem_bytes<D, DT, H, MODE>(a.k_top, &u);
  a.u_bytes = u;
  auto fn = k_gather<D, DT, H, MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fn<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

// The sampled threshold runs on its own engine (threshold_engine.cuh).
inline thr::TArgs threshold_args(const GArgs& a) {
  thr::TArgs t{};
  t.k = a.k;
  t.k_scale = a.k_scale;
  t.L = a.L;
  t.k_top = a.k_top;
  t.perm = a.perm;
  t.qpos = a.qpos;
  t.qp = a.qp;
  t.wq = a.wq;
  t.thr = a.thr;
  t.override_thr = a.override_thr;
  t.n_pad = a.n_pad;
  t.status = a.status;
  return t;
}

template <int D, int DT, int H>
cudaError_t gather_modes(int mode, const GArgs& a, int grid, cudaStream_t st) {
  switch (mode) {
    case kThreshold: return thr::threshold_go<D, DT, H>(threshold_args(a), grid, st);
    case kReplay: return gather_go<D, DT, H, kReplay>(a, grid, st);
    case kRecover: return gather_go<D, DT, H, kRecover>(a, grid, st);
    case kReplayPair:
      if constexpr (H <= 64) return gather_go<D, DT, H, kReplayPair>(a, grid, st);
      break;
  }
  return cudaErrorInvalidValue;
}

// Every mode for the H values of the C ABI (powers of two up to 128).
template <int D, int DT>
cudaError_t gather_launch(int H, int mode, const GArgs& a, int grid, cudaStream_t st) {
  switch (H) {
    case 1: return gather_modes<D, DT, 1>(mode, a, grid, st);
    case 2: return gather_modes<D, DT, 2>(mode, a, grid, st);
    case 4: return gather_modes<D, DT, 4>(mode, a, grid, st);
    case 8: return gather_modes<D, DT, 8>(mode, a, grid, st);
    case 16: return gather_modes<D, DT, 16>(mode, a, grid, st);
    case 32: return gather_modes<D, DT, 32>(mode, a, grid, st);
    case 64: return gather_modes<D, DT, 64>(mode, a, grid, st);
    case 128: return gather_modes<D, DT, 128>(mode, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gather
}  // namespace hytopk

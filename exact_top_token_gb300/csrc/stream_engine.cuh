// stream_engine.cuh -- the tensor-core scoring engine over contiguous key
// tiles: the fused score + threshold filter of HyTopK (no score table) and
// the score-table writer of the two-pass path.
//
// HyScale explainer, HyTopK paragraph: the scoring kernel compares each score
// with the query's threshold on chip and writes only passing keys into a
// small per-query candidate buffer (atomic appends). Score-table paragraph:
// the conventional method writes every score to HBM instead (MODE 1 here).
//
// Work item = (key chunk of 64 or 256 tiles x 128 keys, query block of QB
// slots); the filter takes the longer chunks when there are work items enough
// for every SM without them (long contexts), since each item boundary costs a
// reload of the block's query operand and weights.
// One persistent CTA per SM walks items blockIdx.x, +gridDim.x, ... in
// chunk-major order, so the CTAs running at one time share a key chunk in L2.
//
//   warp 0  TMA producer: the block's q rows (256 (query, head) rows) once
//           per item, then the key tiles through a STAGES ring.
//   warp 1  TMEM allocator and MMA issuer: per key tile one 128 x 256 x d
//           product (keys x (query, head)) into one of two TMEM accumulators.
//   warps 2, 3 idle (they complete warpgroup 0, which hands registers to the
//           epilogue warpgroups with setmaxnreg).
//   warps 4..19 epilogue: TMEM lane = key, so each thread reduces its key's
//           H heads per query in registers: ReLU, times w*q_scale (packed
//           fp32 FMA), times k_scale; then the causal test and the threshold
//           test, and a warp-aggregated append to the candidate buffer.
//           A warp always reads the same 64 accumulator columns during an
//           item, so (for H <= 64) it keeps their weights in registers.
#pragma once

#include "tc.cuh"

namespace hytopk {
namespace stream {

constexpr int kChunkTiles = 64;       // tiles per key chunk (the score table, short contexts)
constexpr int kChunkTilesLong = 256;  // the filter at long contexts
constexpr int kChunkKeys = kChunkTiles * kTileKeys;
constexpr int kEpiWarps = 16;   // epilogue warps (4 per TMEM lane quadrant)
constexpr int kEpiWarp0 = 4;    // first epilogue warp: warpgroups 1..4 are the epilogue
constexpr int kThreads = kEpiWarp0 * 32 + kEpiWarps * 32;
// One CTA of kThreads per SM is launched with kRegsLaunch registers a thread
// (65536 / 640, rounded down to a multiple of 8). When the epilogue keeps its
// weights in registers, warpgroup 0 then shrinks to kRegsCtl and the epilogue
// warpgroups grow to kRegsEpi (setmaxnreg). setmaxnreg.inc waits until the
// CTA's pool (threads x launch registers) can serve it, so the split must fit
// in that pool.
constexpr int kRegsLaunch = 96;
constexpr int kRegsCtl = 32;
constexpr int kRegsEpi = 112;
static_assert(128 * kRegsCtl + (kThreads - 128) * kRegsEpi <= kThreads * kRegsLaunch,
              "register split exceeds the CTA's launch allocation");
constexpr int kMinSmem = 120 * 1024;  // keeps one CTA (and its 512 TMEM columns) per SM

// Candidate staging entries per query slot and work item of the filter: 1024
// per block of QB slots, and for 16 <= H <= 32 (whose warps stage into private
// regions of a quarter of this, flushed when full) at least 32 a region.
__host__ __device__ constexpr int stage_capacity(int H, int QB) {
  return (1024 / QB) > ((H >= 16 && H <= 32) ? 128 : 8) ? (1024 / QB)
                                                          : ((H >= 16 && H <= 32) ? 128 : 8);
}

template <int D, int DT, int H, int MODE_STAGING = 1>
struct Cfg {
  static constexpr int ES = DT == 0 ? 2 : 1;
  static constexpr int RB = D * ES;
  using Geo = tc::Geo<RB>;
  static constexpr int G = 256 / H;               // queries per MMA (N = 256 columns)
  static constexpr int NG = 1;                    // MMA groups per work item
  static constexpr int QB = G * NG;               // query slots per work item
  static constexpr int KT_BYTES = 128 * RB;
  static constexpr int QG_BYTES = 256 * RB;
  static constexpr int STAGES = RB == 256 ? 4 : (RB == 128 ? 6 : 8);
  // q operand buffers (a second buffer, loading the next item's q rows during
  // this item, measured slower at 1M keys: kept at one)
  static constexpr int QBUF = 1;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + QBUF * NG * QG_BYTES;
  static constexpr int BAR_OFF = K_OFF + STAGES * KT_BYTES;
  static constexpr int NBARS = 2 * STAGES + 4 + 4 + 8;   // + q full / empty [2], item ring [4]
  static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;      // tmem base, abort flag, item ring
  static constexpr int POS_OFF = MISC_OFF + 32;
  static constexpr int THR_OFF = POS_OFF + QB * 4;
  static constexpr int ROW_OFF = THR_OFF + QB * 4;
  // per-item candidate staging (filter): CAP entries per query slot of the block
  static constexpr int STAGE_CAP = stage_capacity(H, QB);
  static constexpr int SCNT_OFF = ROW_OFF + QB * 4;
  static constexpr int STAGE_OFF = ((SCNT_OFF + QB * 4) + 15) / 16 * 16;
  static constexpr int END = STAGE_OFF + (MODE_STAGING ? QB * STAGE_CAP * 8 : 0);
  static constexpr int SMEM = (END + 1024) > kMinSmem ? (END + 1024) : kMinSmem;
  // epilogue: each warp owns one TMEM lane quadrant (32 keys) and CW columns
  static constexpr int CW = H > (1024 / kEpiWarps) ? H : (1024 / kEpiWarps);
  static constexpr int ACTIVE_EPI = 4 * (256 / CW);  // warps that read accumulators
  // weights of the CW columns kept in registers for a whole item (H <= 64)
  static constexpr bool REG_W = CW == 64;
  static constexpr int KC = REG_W ? 16 : 32;  // TMEM columns per tcgen05.ld
  static_assert(H >= 1 && H <= 128 && (H & (H - 1)) == 0, "H must be a power of two <= 128");
  static_assert(RB == 64 || RB == 128 || RB == 256, "row bytes");
};

struct Args {
  // halved folded weights hw = w * q_scale / 2: [slots, H] (MODE 0) or
  // [rows padded to the block size, H] (MODE 1)
  const float* wq;
  // MODE 0 (filter): slots sorted by position; plan = chunk offsets
  const int32_t* qpos;
  const float* thr;
  int32_t* cnt;
  uint64_t* cand;
  const int32_t* plan;  // [nchunks + 1] item offsets per key chunk
  int chunk_tiles;      // tiles per key chunk (kChunkTiles or kChunkTilesLong)
  int C;
  int n_pad;
  int reverse;
  // MODE 1 (table): original queries row0..row0+rows-1
  const float* w;
  const float* q_scale;
  const int32_t* positions;
  float* table;
  int row0, rows, n;
  // shared
  const float* k_scale;
  int L;
  uint32_t* status;
  // MODE 0: global item counter (zeroed before the launch); null: items are
  // dealt round robin (MODE 1, whose items cost the same)
  uint32_t* work;
  // MODE 1 inside hytopk_select (the fallback past HYTOPK_MAX_RECOVERY_ROWS
  // failed queries): the failed-query counter; the launch does nothing unless
  // it exceeds that limit. Null: always run.
  const uint32_t* gate;
};

__device__ __forceinline__ int find_chunk(const int32_t* off, int nchunks, int item) {
  int lo = 0, hi = nchunks - 1;  // largest c with off[c] <= item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct Item {
  int block, tile0, ntiles;
};

template <int QB, int MODE>
__device__ __forceinline__ Item decode(const Args& a, int nchunks, int nblocks, int it) {
  Item r;
  int c;
  const int ct = a.chunk_tiles;
  if (MODE == 0) {
    c = find_chunk(a.plan, nchunks, it);
    r.block = it - __ldg(a.plan + c);
    const int maxpos = __ldg(a.qpos + r.block * QB);
    r.tile0 = c * ct;
    const int end = min(maxpos + 1, a.L);
    r.ntiles = min(ct, (end - r.tile0 * kTileKeys + kTileKeys - 1) / kTileKeys);
  } else {
    c = it / nblocks;
    r.block = it - c * nblocks;
    r.tile0 = c * ct;
    r.ntiles = min(ct, (a.L - r.tile0 * kTileKeys + kTileKeys - 1) / kTileKeys);
  }
  return r;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32)); }

// Canonical head reduction, shared by every scoring kernel of the library.
// The weights are stored halved (hw = w / 2) and ReLU(x) * w is evaluated as
// (x + |x|) * hw: 2x and w/2 are exact scalings, so the product is bit for
// bit ReLU(x) * w (for |w| >= 2^-125), while the add runs on the FMA pipe.
// Head pair p = (2p, 2p+1) accumulates into packed accumulator p % NA with
// one packed fp32 FMA (the first pair of each accumulator with a packed
// multiply, which gives the same value up to the sign of a zero); then the
// accumulators are combined with packed adds, t = (a0 + a1) + (a2 + a3), and
// total = lo(t) + hi(t). The sign of a zero total is made +0 by finish_score.
//
// With four accumulators, the last one takes its ReLU on the integer pipe
// instead: for finite x, the signed-integer maximum of x's bit pattern and 0
// is x when x >= +0 and +0 otherwise. That accumulator then sums ReLU(x) * hw,
// exactly half of what the (x + |x|) form gives at every step (halving is
// exact away from the subnormal range), and the combine doubles it exactly:
// t = (a0 + a1) + (a2 + (a3 + a3)). Splitting the ReLUs between the FMA and
// ALU pipes this way (one pair in four) shortens the epilogue of the score
// kernels.
template <int H>
struct HeadSum {
  static constexpr int NA = H >= 8 ? 4 : (H >= 2 ? H / 2 : 1);
  static constexpr bool kAluLast = NA == 4;
  uint64_t a[NA];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < NA; ++i) a[i] = 0ull;
  }
  // 2 ReLU(x) for accumulators 0 .. NA-2 (FMA pipe), ReLU(x) for the last
  // one when kAluLast (integer pipe)
  __device__ __forceinline__ static float relu_term(int s, float x) {
    if (kAluLast && s == NA - 1) return __int_as_float(max(__float_as_int(x), 0));
    return x + fabsf(x);
  }
  // heads h, h+1 (h even), halved weights hw0, hw1
  __device__ __forceinline__ void add_pair(int h, float x0, float x1, float hw0, float hw1) {
    const int s = (h >> 1) % NA;
    const float r0 = relu_term(s, x0), r1 = relu_term(s, x1);
    uint64_t r, w;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(r0), "f"(r1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(w) : "f"(hw0), "f"(hw1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a[s]) : "l"(r), "l"(w));
  }
  // the same with the two halved weights already packed as {hw0, hw1}; the
  // first pair of an accumulator (h < 2 NA) sets it, so no reset is needed
  __device__ __forceinline__ void add_pair_packed(int h, float x0, float x1, uint64_t w) {
    const int s = (h >> 1) % NA;
    const float r0 = relu_term(s, x0), r1 = relu_term(s, x1);
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(r0), "f"(r1));
    if (h < 2 * NA)
      asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(a[s]) : "l"(r), "l"(w));
    else
      asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a[s]) : "l"(r), "l"(w));
  }
  __device__ __forceinline__ float lane_sum(int i) const {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a[i]));
    return lo + hi;
  }
  __device__ __forceinline__ float total() const {
    if (NA == 1) return lane_sum(0);
    uint64_t t;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(a[0]), "l"(a[1]));
    if (NA == 4) {
      uint64_t a3x2, t23;
      asm("add.rn.f32x2 %0, %1, %1;" : "=l"(a3x2) : "l"(a[3]));
      asm("add.rn.f32x2 %0, %1, %2;" : "=l"(t23) : "l"(a[2]), "l"(a3x2));
      asm("add.rn.f32x2 %0, %0, %1;" : "+l"(t) : "l"(t23));
    }
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(t));
    return lo + hi;
  }
};

// H = 1: ReLU(x) * w with the halved weight, as above.
template <int H>
__device__ __forceinline__ float single_head_score(float x, float hw) {
  return (x + fabsf(x)) * hw;
}

// Append (score, key) to the query's candidate buffer; all 32 lanes call it.
// Candidates are staged per work item in shared memory (a shared atomic per
// warp reserves room); the item's flush reserves global room with one atomic
// per query. Entries beyond the staging capacity take the global path at once.
template <int CAP>
__device__ __forceinline__ void append_staged(bool pass, float score, int s, int jb, int slot,
                                              uint32_t* scnt, uint64_t* stage, int32_t* cnt,
                                              uint64_t* cand, int C) {
  const unsigned mask = __ballot_sync(0xffffffffu, pass);
  if (mask == 0u) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(scnt + jb, (uint32_t)__popc(mask));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (pass) {
    const uint32_t at = base + (uint32_t)__popc(mask & ((1u << lane) - 1u));
    const uint64_t key = cand_key(score, s);
    if (at < (uint32_t)CAP) {
      stage[jb * CAP + at] = key;
    } else {
      const int g = atomicAdd(cnt + slot, 1);
      if (g < C) cand[(size_t)slot * C + g] = key;
    }
  }
}

// Move one item's staged candidates to the global buffers: warp w flushes
// query slots w, w + kEpiWarps, ... and clears their staging counters.
template <int QB, int CAP>
__device__ __forceinline__ void flush_staged(int block, uint32_t* scnt, const uint64_t* stage,
                                             int32_t* cnt, uint64_t* cand, int C, int ewarp) {
  const int lane = threadIdx.x & 31;
  for (int jb = ewarp; jb < QB; jb += kEpiWarps) {
    const uint32_t n = min(scnt[jb], (uint32_t)CAP);
    if (n == 0) continue;
    const int slot = block * QB + jb;
    int base = 0;
    if (lane == 0) base = atomicAdd(cnt + slot, (int)n);
    base = __shfl_sync(0xffffffffu, base, 0);
    for (uint32_t i = lane; i < n; i += 32) {
      const int g = base + (int)i;
      if (g < C) cand[(size_t)slot * C + g] = stage[jb * CAP + i];
    }
  }
  __syncwarp();
  for (int jb = ewarp; jb < QB; jb += kEpiWarps)
    if (lane == 0) scnt[jb] = 0;
}

// Private staging, for warps that serve at most a few queries of the block:
// the (query, lane quadrant) pair owns a region of CAP4 entries and the warp
// keeps its fill level in a register, so an append needs no atomic.
//
// Move one private region to the query's global buffer (one atomic) and
// empty it; the whole warp calls it.
template <int CAP4>
__device__ __forceinline__ void flush_private(int region, int slot, uint32_t& fill,
                                              const uint64_t* stage, int32_t* cnt, uint64_t* cand,
                                              int C) {
  const uint32_t n = min(fill, (uint32_t)CAP4);
  fill = 0;
  if (n == 0) return;
  const int lane = threadIdx.x & 31;
  __syncwarp();
  int base = 0;
  if (lane == 0) base = atomicAdd(cnt + slot, (int)n);
  base = __shfl_sync(0xffffffffu, base, 0);
  for (uint32_t i = lane; i < n; i += 32) {
    const int g = base + (int)i;
    if (g < C) cand[(size_t)slot * C + g] = stage[region * CAP4 + i];
  }
  __syncwarp();
}

// Append (score, key) for the lanes where pass holds; the whole warp calls
// it. FLUSH_FULL (used with H <= 32, whose short-context queries can pass
// most keys): a region that cannot take this ballot's keys is flushed first,
// one atomic for the region (CAP4 >= 32). Otherwise (H = 64, a few dozen
// candidates per query and item) keys past the region go to the global buffer
// one atomic each; that branch-light form measured faster there.
template <int CAP4, bool FLUSH_FULL>
__device__ __forceinline__ void append_private(bool pass, float score, int s, int region, int slot,
                                               uint32_t& fill, uint64_t* stage, int32_t* cnt,
                                               uint64_t* cand, int C) {
  const unsigned mask = __ballot_sync(0xffffffffu, pass);
  if (mask == 0u) return;
  const int lane = threadIdx.x & 31;
  if constexpr (FLUSH_FULL) {
    static_assert(CAP4 >= 32, "a region must take one ballot's keys");
    const uint32_t np = (uint32_t)__popc(mask);
    if (fill + np > (uint32_t)CAP4) flush_private<CAP4>(region, slot, fill, stage, cnt, cand, C);
    if (pass) stage[region * CAP4 + fill + __popc(mask & ((1u << lane) - 1u))] = cand_key(score, s);
    fill += np;
  } else {
    if (pass) {
      const uint32_t at = fill + (uint32_t)__popc(mask & ((1u << lane) - 1u));
      const uint64_t key = cand_key(score, s);
      if (at < (uint32_t)CAP4) {
        stage[region * CAP4 + at] = key;
      } else {
        const int g = atomicAdd(cnt + slot, 1);
        if (g < C) cand[(size_t)slot * C + g] = key;
      }
    }
    fill += (uint32_t)__popc(mask);
  }
}

template <int D, int DT, int H, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    k_stream(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
             const Args a);

// Host side: a build whose launch register count is below kRegsLaunch would
// leave the epilogue's setmaxnreg.inc unserved, so it is refused before launch.
template <int D, int DT, int H, int MODE>
inline cudaError_t check_register_split() {
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, k_stream<D, DT, H, MODE>);
  if (e != cudaSuccess) return e;
  return fa.numRegs >= kRegsLaunch ? cudaSuccess : cudaErrorLaunchOutOfResources;
}

template <int D, int DT, int H, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    k_stream(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
             const Args a) {
  using C_ = Cfg<D, DT, H, MODE == 0 ? 1 : 0>;
  using Geo = typename C_::Geo;
  constexpr int G = C_::G, NG = C_::NG, QB = C_::QB, STAGES = C_::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  uint8_t* smem = tc::align1024(smem_dyn);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C_::BAR_OFF);
  uint64_t* k_full = bars;
  uint64_t* k_empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;       // [2]
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2]
  uint64_t* q_full = bars + 2 * STAGES + 4;       // [QBUF]
  uint64_t* q_empty = bars + 2 * STAGES + 6;      // [QBUF]
  uint64_t* item_full = bars + 2 * STAGES + 8;    // [4]
  uint64_t* item_empty = bars + 2 * STAGES + 12;  // [4]
  volatile int32_t* item_ring = reinterpret_cast<volatile int32_t*>(smem + C_::MISC_OFF + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C_::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C_::MISC_OFF + 4);
  int32_t* pos_s = reinterpret_cast<int32_t*>(smem + C_::POS_OFF);
  float* thr_s = reinterpret_cast<float*>(smem + C_::THR_OFF);
  int32_t* row_s = reinterpret_cast<int32_t*>(smem + C_::ROW_OFF);
  uint32_t* scnt_s = reinterpret_cast<uint32_t*>(smem + C_::SCNT_OFF);
  uint64_t* stage_s = reinterpret_cast<uint64_t*>(smem + C_::STAGE_OFF);
  constexpr int CAP = C_::STAGE_CAP;

  if (MODE == 1 && a.gate != nullptr &&
      *reinterpret_cast<const volatile uint32_t*>(a.gate) <= HYTOPK_MAX_RECOVERY_ROWS)
    return;  // uniform over the grid, before any barrier or TMEM is set up
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk_keys = a.chunk_tiles * kTileKeys;
  const int nchunks = (a.L + chunk_keys - 1) / chunk_keys;
  const int nblocks = MODE == 0 ? a.n_pad / QB : (a.rows + QB - 1) / QB;
  const int total = MODE == 0 ? __ldg(a.plan + nchunks) : nchunks * nblocks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      tc::mbar_init(k_full + i, 1);
      tc::mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(acc_full + i, 1);
      tc::mbar_init(acc_empty + i, C_::ACTIVE_EPI);
    }
    for (int i = 0; i < C_::QBUF; ++i) {
      tc::mbar_init(q_full + i, 1);
      tc::mbar_init(q_empty + i, 1);
    }
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(item_full + i, 1);
      tc::mbar_init(item_empty + i, 1 + kEpiWarps);
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  auto item_at = [&](int i) { return a.reverse ? total - 1 - i : i; };
  // The n-th item of this CTA. With a work counter (the filter, whose items
  // differ in cost: the causal edge, candidate appends) the TMA producer takes
  // the next item from the counter and publishes it through a 4-slot ring that
  // the MMA issuer and every epilogue warp read in the same order; without
  // one, items are dealt round robin. An index >= total ends the sequence.
  auto publish_item = [&](int n) -> int {  // TMA producer lane
    if (a.work == nullptr) return (int)blockIdx.x + n * (int)gridDim.x;
    const int slot = n & 3;
    if (!tc::mbar_wait(item_empty + slot, ((n >> 2) & 1) ^ 1u, abort_flag, a.status)) return -1;
    const int i = (int)atomicAdd(a.work, 1u);
    item_ring[slot] = i;
    tc::mbar_arrive(item_full + slot);
    return i;
  };
  auto take_item = [&](int n) -> int {  // MMA issuer lane, every epilogue lane
    if (a.work == nullptr) return (int)blockIdx.x + n * (int)gridDim.x;
    const int slot = n & 3;
    if (!tc::mbar_wait(item_full + slot, (n >> 2) & 1, abort_flag, a.status)) return -1;
    return item_ring[slot];
  };

  // Each role starts with its setmaxnreg, so that the register target of its
  // code is the one set there.
  if (warp < kEpiWarp0) {
    if constexpr (C_::REG_W) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == 0) {
      if (lane == 0) {
        // ---------------- TMA producer ----------------
        tc::tma_prefetch(&kmap);
        tc::tma_prefetch(&qmap);
        int stage = 0;
        uint32_t sphase = 0;
        uint32_t pending = 0, pend_phase = 0, q_loads = 0;  // issued loads, for a clean abort
        for (int n = 0;; ++n) {
          const int i = publish_item(n);
          if (i < 0 || i >= total) break;
          const Item itm = decode<QB, MODE>(a, nchunks, nblocks, item_at(i));
          // q buffer of the n-th item: n % QBUF, its (n / QBUF)-th use
          const int qb = n % C_::QBUF;
          const uint32_t qpar = (uint32_t)(n / C_::QBUF) & 1u;
          if (!tc::mbar_wait(q_empty + qb, qpar ^ 1u, abort_flag, a.status)) break;
          tc::mbar_expect_tx(q_full + qb, NG * C_::QG_BYTES);
          const int qrow0 = (MODE == 0 ? itm.block * QB : a.row0 + itm.block * QB) * H;
  #pragma unroll
          for (int g = 0; g < NG; ++g)
  #pragma unroll
            for (int at = 0; at < Geo::kAtoms; ++at)
              tc::tma_load_2d(smem + C_::Q_OFF + (qb * NG + g) * C_::QG_BYTES +
                                  at * 256 * Geo::kAtom,
                              &qmap, q_full + qb, at * Geo::kAtom / C_::ES, qrow0 + g * 256);
          ++q_loads;
          bool ok = true;
          for (int t = 0; t < itm.ntiles; ++t) {
            if (!tc::mbar_wait(k_empty + stage, sphase ^ 1u, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc::mbar_expect_tx(k_full + stage, C_::KT_BYTES);
  #pragma unroll
            for (int at = 0; at < Geo::kAtoms; ++at)
              tc::tma_load_2d(smem + C_::K_OFF + stage * C_::KT_BYTES + at * 128 * Geo::kAtom,
                              &kmap, k_full + stage, at * Geo::kAtom / C_::ES,
                              (itm.tile0 + t) * kTileKeys);
            pending |= 1u << stage;
            pend_phase = (pend_phase & ~(1u << stage)) | (sphase << stage);
            if (++stage == STAGES) {
              stage = 0;
              sphase ^= 1u;
            }
          }
          if (!ok) break;
        }
        if (*abort_flag) {
          // let the copies still in flight land before the CTA exits (bounded)
          const uint64_t t0 = tc::global_ns();
          for (int st = 0; st < STAGES; ++st)
            if (pending & (1u << st))
              while (!tc::mbar_try_wait(k_full + st, (pend_phase >> st) & 1u) &&
                     tc::global_ns() - t0 < 200000000ull) {
              }
          for (uint32_t j = q_loads > (uint32_t)C_::QBUF ? q_loads - C_::QBUF : 0u; j < q_loads; ++j)
            while (!tc::mbar_try_wait(q_full + j % C_::QBUF, (j / C_::QBUF) & 1u) &&
                   tc::global_ns() - t0 < 200000000ull) {
            }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t IDESC = tc::instr_desc(DT, 128, 256);
        // Descriptors of stage 0, K-step 0. The start address field (bits
        // 0-13, address / 16) is the only part that differs between stages
        // and K-steps, and shared-memory addresses stay below 256 KB, so a
        // descriptor is its template plus (byte offset / 16) in the low word.
        const uint64_t a_tmpl = tc::smem_desc(tc::smem_u32(smem + C_::K_OFF), Geo::kSbo, Geo::kSwizzle);
        const uint64_t b_tmpl = tc::smem_desc(tc::smem_u32(smem + C_::Q_OFF), Geo::kSbo, Geo::kSwizzle);
        const uint32_t a_lo = (uint32_t)a_tmpl, a_hi = (uint32_t)(a_tmpl >> 32);
        const uint32_t b_lo = (uint32_t)b_tmpl, b_hi = (uint32_t)(b_tmpl >> 32);
        uint32_t a_stage_lo = a_lo;  // a_lo + stage * KT_BYTES / 16
        int stage = 0, acc = 0;
        uint32_t sphase = 0, aphase = 0;
        for (int n = 0;; ++n) {
          const int i = take_item(n);
          if (a.work != nullptr && i >= 0) tc::mbar_arrive(item_empty + (n & 3));
          if (i < 0 || i >= total) break;
          const Item itm = decode<QB, MODE>(a, nchunks, nblocks, item_at(i));
          const int qb = n % C_::QBUF;
          if (!tc::mbar_wait(q_full + qb, (uint32_t)(n / C_::QBUF) & 1u, abort_flag, a.status))
            break;
          const uint32_t bq_lo = b_lo + (uint32_t)((qb * NG * C_::QG_BYTES) >> 4);
          tc::fence_after_sync();
          bool ok = true;
          for (int t = 0; t < itm.ntiles && ok; ++t) {
            if (!tc::mbar_wait(k_full + stage, sphase, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
  #pragma unroll
            for (int g = 0; g < NG; ++g) {
              if (!tc::mbar_wait(acc_empty + acc, aphase ^ 1u, abort_flag, a.status)) {
                ok = false;
                break;
              }
              tc::fence_after_sync();
              const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
  #pragma unroll
              for (int j = 0; j < Geo::kSteps; ++j) {
                const uint64_t adesc =
                    tc::desc_from_words(a_stage_lo + (Geo::step_offset(j, 128) >> 4), a_hi);
                const uint64_t bdesc = tc::desc_from_words(
                    bq_lo + ((g * C_::QG_BYTES + Geo::step_offset(j, 256)) >> 4), b_hi);
                tc::mma<DT>(d_tmem, adesc, bdesc, IDESC, j > 0 ? 1u : 0u);
              }
              tc::mma_commit(acc_full + acc);
              acc ^= 1;
              if (acc == 0) aphase ^= 1u;
            }
            tc::mma_commit(k_empty + stage);
            a_stage_lo += C_::KT_BYTES >> 4;
            if (++stage == STAGES) {
              stage = 0;
              a_stage_lo = a_lo;
              sphase ^= 1u;
            }
          }
          tc::mma_commit(q_empty + qb);
          if (!ok) break;
        }
      }
    }
  } else {
    if constexpr (C_::REG_W) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    // ---------------- epilogue ----------------
    constexpr int CW = C_::CW;
    constexpr int KC = C_::KC;
    constexpr bool REG_W = C_::REG_W;
    constexpr int NQS = CW / H;           // queries in a warp's column span
    constexpr bool REG_META = NQS <= 4;   // their position and threshold in registers
    const int e = warp - kEpiWarp0;
    const int quad = warp & 3;            // TMEM lane quadrant this warp may read
    const int sub = e >> 2;               // column span of this warp: [sub*CW, sub*CW+CW)
    const bool reads_tmem = sub * CW < 256;
    const int qlo = (sub * CW) / H;       // first query (within the block) of the span
    const int et = threadIdx.x - kEpiWarp0 * 32;
    int acc = 0;
    uint32_t aphase = 0;
    int prev_block = -1;
    // candidate staging: private regions (REG_META) or shared counters
    constexpr int CAP4 = CAP / 4;
    uint32_t fill[REG_META ? NQS : 1];
    if constexpr (REG_META) {
#pragma unroll
      for (int u = 0; u < NQS; ++u) fill[u] = 0;
    }
    if (MODE == 0 && !REG_META)
      for (int jb = et; jb < QB; jb += kEpiWarps * 32) scnt_s[jb] = 0;
    for (int n = 0;; ++n) {
      // every epilogue warp reads the same item sequence (lane 0's view,
      // after all lanes have read the slot), so the warps stay in step at
      // the named barriers below
      const int i = __shfl_sync(0xffffffffu, take_item(n), 0);
      if (a.work != nullptr && i >= 0) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(item_empty + (n & 3));
      }
      if (i < 0 || i >= total) break;
      const Item itm = decode<QB, MODE>(a, nchunks, nblocks, item_at(i));
      epi_sync();
      if (MODE == 0 && !REG_META && prev_block >= 0)
        flush_staged<QB, CAP>(prev_block, scnt_s, stage_s, a.cnt, a.cand, a.C, e);
      prev_block = itm.block;
      for (int jb = et; jb < QB; jb += kEpiWarps * 32) {
        if (MODE == 0) {
          const int slot = itm.block * QB + jb;
          pos_s[jb] = __ldg(a.qpos + slot);
          thr_s[jb] = __ldg(a.thr + slot);
          row_s[jb] = slot;
        } else {
          const int r = itm.block * QB + jb;
          int p = -1;
          if (r < a.rows) {
            p = __ldg(a.positions + a.row0 + r);
            if (p < 0 || p >= a.L) p = -1;
          }
          pos_s[jb] = p;
          row_s[jb] = r < a.rows ? r : -1;
        }
      }
      epi_sync();
      if (*abort_flag || !reads_tmem) continue;  // named-barrier count stays equal
      // halved weight of column c of the span is wrow[c] (workspace, warp-uniform)
      const float* wrow =
          a.wq + ((size_t)(MODE == 0 ? 0 : a.row0) + (size_t)itm.block * QB + qlo) * H;
      const int32_t* prow = pos_s + qlo;
      const float* trow = thr_s + qlo;
      const int32_t* rrow = row_s + qlo;
      // per item: the span's weights as packed pairs {hw[2c], hw[2c+1]}, and the
      // positions and thresholds of its queries
      uint64_t wp[REG_W ? CW / 2 : 1];
      if constexpr (REG_W) {
        if (MODE == 0) {  // slot rows: 256-byte aligned
#pragma unroll
          for (int u = 0; u < CW / 4; ++u) {
            const ulonglong2 w2 = __ldg(reinterpret_cast<const ulonglong2*>(wrow) + u);
            wp[2 * u] = w2.x;
            wp[2 * u + 1] = w2.y;
          }
        } else {  // rows from an arbitrary row0: 4-byte aligned only
#pragma unroll
          for (int u = 0; u < CW / 2; ++u)
            asm("mov.b64 %0, {%1, %2};"
                : "=l"(wp[u])
                : "f"(__ldg(wrow + 2 * u)), "f"(__ldg(wrow + 2 * u + 1)));
        }
      }
      int pv[REG_META ? NQS : 1];
      float tv[REG_META ? NQS : 1];
      if constexpr (REG_META) {
#pragma unroll
        for (int u = 0; u < NQS; ++u) {
          pv[u] = prow[u];
          tv[u] = trow[u];
        }
      }
      bool ok = true;
      const int s_first = itm.tile0 * kTileKeys + quad * 32 + lane;
      // key scales are read one tile ahead from an index clamped to L - 1: a
      // key at or past L (zero-filled by the tile load) fails the causal test
      // whatever its scale, and the clamped read stays inside k_scale
      const int s_last = a.L - 1;
      float ks_next = DT == 1 ? __ldg(a.k_scale + min(s_first, s_last)) : 1.0f;
      // TMEM address of this warp's lane quadrant and column span in
      // accumulator 0; accumulator 1 is 256 columns on
      const uint32_t tbase0 =
          tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(sub * CW);
      for (int t = 0; t < itm.ntiles && ok; ++t) {
        const int s = s_first + t * kTileKeys;
        const float ks = ks_next;
        if (DT == 1) ks_next = __ldg(a.k_scale + min(s + kTileKeys, s_last));
        if (!tc::mbar_wait(acc_full + acc, aphase, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t tbase = tbase0 + ((uint32_t)acc << 8);
        HeadSum<H> hs;
        if (!REG_W) hs.reset();
        float va[KC];
        auto reduce = [&](const float (&v)[KC], int ch) {
          constexpr int STEP = H == 1 ? 1 : (H == 2 ? 2 : 4);
#pragma unroll
          for (int j = 0; j < KC; j += STEP) {
            const int col = ch * KC + j;  // column within this warp's span
            const int qi = col / H;       // query within the span
            const int h = col % H;
            float sc = 0.0f;
            bool done = false;
            if (H == 1) {
              float hw;
              if constexpr (REG_W) {
                float lo, hi;
                asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(wp[col / 2]));
                hw = (col & 1) ? hi : lo;
              } else {
                hw = __ldg(wrow + col);
              }
              sc = single_head_score<H>(v[j], hw);
              done = true;
            } else if (REG_W) {
              hs.add_pair_packed(h, v[j], v[j + 1], wp[col / 2]);
              if (H >= 4) hs.add_pair_packed(h + 2, v[j + 2], v[j + 3], wp[col / 2 + 1]);
              done = (h + STEP == H);
            } else {
              const float4 w4 = __ldg(reinterpret_cast<const float4*>(wrow + col));
              hs.add_pair(h, v[j], v[j + 1], w4.x, w4.y);
              hs.add_pair(h + 2, v[j + 2], v[j + 3], w4.z, w4.w);
              done = (h + 4 == H);
            }
            if (done) {
              if (H >= 2) {
                sc = hs.total();
                if (!REG_W) hs.reset();
              }
              // the filter's keys carry the score through cand_key, which
              // takes -0 as +0, and -0 >= thr exactly when +0 >= thr, so the
              // filter skips finish_score's zero fixup (same bits kept)
              sc = MODE == 0 ? sc * ks : finish_score(sc, ks);
              int p;
              float thr;
              if constexpr (REG_META) {
                p = pv[qi];
                thr = tv[qi];
              } else {
                p = prow[qi];
                thr = trow[qi];
              }
              if (MODE == 0) {
                const bool pass = (s <= p) && (sc >= thr);
                if constexpr (REG_META)
                  append_private<CAP4, (H <= 32)>(pass, sc, s, (qlo + qi) * 4 + quad, rrow[qi],
                                                  fill[qi],
                                       stage_s, a.cnt, a.cand, a.C);
                else
                  append_staged<CAP>(pass, sc, s, qlo + qi, rrow[qi], scnt_s, stage_s, a.cnt,
                                     a.cand, a.C);
              } else {
                const int r = rrow[qi];
                if (r >= 0 && s < a.L)
                  a.table[(size_t)r * a.L + s] = (s <= p) ? sc : -__int_as_float(0x7f800000);
              }
            }
          }
        };
        if constexpr (REG_W) {
          // two buffers: the load of chunk ch + 1 is in flight while chunk ch
          // is reduced
          float vb[KC];
          constexpr int NCH = CW / KC;
          tc::tmem_ld_n(tbase, va);
          tc::tmem_wait_ld(va);
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            if (ch + 1 < NCH) tc::tmem_ld_n(tbase + (ch + 1) * KC, (ch & 1) ? va : vb);
            reduce((ch & 1) ? vb : va, ch);
            if (ch + 1 < NCH) tc::tmem_wait_ld((ch & 1) ? va : vb);
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < CW / KC; ++ch) {
            tc::tmem_ld_n(tbase + ch * KC, va);
            tc::tmem_wait_ld(va);
            reduce(va, ch);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(acc_empty + acc);
        acc ^= 1;
        if (acc == 0) aphase ^= 1u;
      }
      if constexpr (MODE == 0 && REG_META) {
#pragma unroll
        for (int u = 0; u < NQS; ++u)
          flush_private<CAP4>((qlo + u) * 4 + quad, rrow[u], fill[u], stage_s, a.cnt, a.cand,
                              a.C);
      }
    }
    if (MODE == 0 && !REG_META) {
      epi_sync();
      if (prev_block >= 0)
        flush_staged<QB, CAP>(prev_block, scnt_s, stage_s, a.cnt, a.cand, a.C, e);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace stream
}  // namespace hytopk

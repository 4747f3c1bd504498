// radix.cuh -- CTA-wide radix select and sort on ordered keys.
//
// The HyScale explainer (HyTopK paragraph) resolves ties at the k-th score
// with a radix select over positions and orders the kept entries with a radix
// sort, which makes the output independent of the order in which the
// unordered atomic appends filled the candidate buffer. Here a candidate is
// the 64-bit key desc32(score) << 32 | position: an MSB-first radix select
// over its upper 32 bits is the select on score, and over its lower 32 bits
// (reached only when scores tie at the boundary) the select over positions.
// The k selected keys are unique, so the final order (ascending key = score
// descending, position ascending) is a total order.
#pragma once

#include "common.cuh"

namespace hytopk {

// Block-wide: given hist[0..nbins), find the bin b where the running count
// crosses `target` (1-based): sum(hist[<b]) < target <= sum(hist[<=b]).
// Writes b and sum(hist[<b]) to out[0], out[1]. Needs blockDim.x % 32 == 0 and
// a `warp_sums` array of blockDim.x/32 entries. All threads must call it.
__device__ __forceinline__ void cta_find_crossing(const uint32_t* hist, int nbins, uint32_t target,
                                                  uint32_t* warp_sums, uint32_t* out) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int per = (nbins + nthr - 1) / nthr;
  if (tid == 0) {
    out[0] = 0;
    out[1] = 0;
  }
  const int b0 = tid * per;
  uint32_t local = 0;
  for (int b = b0; b < b0 + per && b < nbins; ++b) local += hist[b];
  // inclusive warp scan
  uint32_t incl = local;
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  uint32_t before_warp = 0;
  for (int w = 0; w < warp; ++w) before_warp += warp_sums[w];
  const uint32_t excl = before_warp + incl - local;
  if (excl < target && target <= excl + local) {
    uint32_t cum = excl;
    for (int b = b0; b < b0 + per && b < nbins; ++b) {
      if (cum + hist[b] >= target) {
        out[0] = (uint32_t)b;
        out[1] = cum;
        break;
      }
      cum += hist[b];
    }
  }
  __syncthreads();
}

// Warp-aggregated histogram increment. Scores of a query share their top bits,
// so most lanes of a warp hit the bin of its first active lane: those add
// their count with one shared atomic, the others one each. All 32 lanes must
// call it; `active` lanes contribute.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (act == 0u) return;
  const int first = __ffs(act) - 1;
  const uint32_t b0 = __shfl_sync(0xffffffffu, bin, first);
  const bool same = active && bin == b0;
  const unsigned m = __ballot_sync(0xffffffffu, same);
  if ((int)(threadIdx.x & 31) == first) atomicAdd(hist + b0, (uint32_t)__popc(m));
  else if (active && !same) atomicAdd(hist + bin, 1u);
}

// Shared-memory scratch of the selection helpers.
struct alignas(16) RadixScratch {
  uint32_t hist[4096];
  uint32_t warp_sums[32];
  uint32_t out[4];
  uint32_t counter;
};

// Selects the k_sel smallest of the unique keys list[0..cnt) into sel[0..k_sel)
// (shared memory, unordered). Returns the number written (min(cnt, k_sel)).
static __device__ int cta_select_smallest_u64(const uint64_t* list, int cnt, int k_sel, uint64_t* sel,
                                       RadixScratch& sc) {
  if (cnt <= k_sel) {
    for (int e = threadIdx.x; e < cnt; e += blockDim.x) sel[e] = list[e];
    __syncthreads();
    return cnt;
  }
  uint64_t prefix = 0;
  int pbits = 0;
  uint32_t krem = (uint32_t)k_sel;
  while (pbits < 64) {
    const int shift = 56 - pbits;
    for (int b = threadIdx.x; b < 256; b += blockDim.x) sc.hist[b] = 0;
    __syncthreads();
    for (int e0 = 0; e0 < cnt; e0 += blockDim.x) {
      const int e = e0 + threadIdx.x;
      const uint64_t key = e < cnt ? list[e] : 0ull;
      const bool in = e < cnt && (pbits == 0 || (key >> (64 - pbits)) == prefix);
      hist_add(sc.hist, (uint32_t)(key >> shift) & 255u, in);
    }
    __syncthreads();
    cta_find_crossing(sc.hist, 256, krem, sc.warp_sums, sc.out);
    const uint32_t bin = sc.out[0], before = sc.out[1];
    const bool whole_bin = (sc.hist[bin] == krem - before);
    krem -= before;
    prefix = (prefix << 8) | bin;
    pbits += 8;
    __syncthreads();
    if (whole_bin) break;
  }
  if (threadIdx.x == 0) sc.counter = 0;
  __syncthreads();
  const int drop = 64 - pbits;
  for (int e = threadIdx.x; e < cnt; e += blockDim.x) {
    const uint64_t key = list[e];
    if ((drop == 64 ? 0ull : (key >> drop)) <= prefix) {
      const uint32_t at = atomicAdd(&sc.counter, 1u);
      if (at < (uint32_t)k_sel) sel[at] = key;
    }
  }
  __syncthreads();
  return k_sel;
}

// Ascending bitonic sort of sel[0..n) in shared memory; entries n..P-1 (P =
// next power of two, within the buffer's capacity) are filled with ~0 and sort
// last.
static __device__ void cta_bitonic_u64(uint64_t* sel, int n) {
  int P = 1;
  while (P < n) P <<= 1;
  for (int e = n + threadIdx.x; e < P; e += blockDim.x) sel[e] = ~0ull;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < (P >> 1); i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t a = sel[lo], b = sel[hi];
        if ((a > b) == up) {
          sel[lo] = b;
          sel[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

// Ascending sort of sel[0..n) in shared memory (all threads call it; blockDim.x
// a multiple of 32). With at most 4 keys per thread it is a bucket sort: the
// upper 32 bits of the keys (the score part of a candidate key), less their
// minimum, are shifted right until their range fits 4096 ordered buckets, every
// key is counted, the counts are prefix-summed, each key is scattered into its
// bucket's range, and its final place in the bucket is the number of the
// bucket's keys below it (equal keys ordered by their scatter slot). A query's
// kept scores spread over their range, so a bucket holds a few keys. If a
// bucket holds more than kMaxBucket keys (many keys sharing a score) or there
// are more than 4 keys per thread, the bitonic network sorts instead; both
// give the same order. Uses sc.hist, sc.warp_sums and sc.out.
static __device__ void cta_sort_u64(uint64_t* sel, int n, RadixScratch& sc) {
  constexpr int NB = 4096, PER = 4;
  constexpr uint32_t kMaxBucket = 32;
  const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (n <= 1) {
    __syncthreads();
    return;
  }
  if (n > PER * T) {
    cta_bitonic_u64(sel, n);
    return;
  }
  if (tid == 0) {
    sc.out[0] = 0xffffffffu;
    sc.out[1] = 0u;
    sc.out[2] = 0u;
  }
  for (int b = tid; b < NB; b += T) sc.hist[b] = 0u;
  uint64_t key[PER];
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int i = tid + r * T;
    key[r] = i < n ? sel[i] : 0ull;
    if (i < n) {
      const uint32_t u = (uint32_t)(key[r] >> 32);
      lo = min(lo, u);
      hi = max(hi, u);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  __syncthreads();  // out[] and hist cleared, every key in registers
  if (lane == 0) {
    atomicMin(&sc.out[0], lo);
    atomicMax(&sc.out[1], hi);
  }
  __syncthreads();
  // bucket = (upper - min) >> sh, the smallest shift that maps the range
  // below NB (so at least NB / 2 buckets are in use when the range is wide)
  const uint32_t kmin = sc.out[0], range = sc.out[1] - kmin;
  const int width = range == 0u ? 0 : 32 - __clz(range);
  const int sh = width > 12 ? width - 12 : 0;
  int bin[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int i = tid + r * T;
    bin[r] = (int)(((uint32_t)(key[r] >> 32) - kmin) >> sh);
    if (i < n) atomicAdd(&sc.hist[bin[r]], 1u);
  }
  __syncthreads();
  // exclusive prefix sum of the counts; each thread owns a run of buckets
  const int per = (NB + T - 1) / T, b0 = tid * per, b1 = min(b0 + per, NB);
  uint32_t local = 0, big = 0;
  for (int b = b0; b < b1; ++b) {
    const uint32_t c = sc.hist[b];
    local += c;
    big = max(big, c);
  }
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
    big = max(big, __shfl_xor_sync(0xffffffffu, big, o));
  }
  if (lane == 31) sc.warp_sums[warp] = incl;
  if (lane == 0) atomicMax(&sc.out[2], big);
  __syncthreads();
  uint32_t run = incl - local;
  for (int w = 0; w < warp; ++w) run += sc.warp_sums[w];
  for (int b = b0; b < b1; ++b) {
    const uint32_t c = sc.hist[b];
    sc.hist[b] = run;
    run += c;
  }
  const bool crowded = sc.out[2] > kMaxBucket;
  __syncthreads();  // hist[b] = start of bucket b
  if (crowded) {  // sel is untouched so far
    cta_bitonic_u64(sel, n);
    return;
  }
  uint32_t slot[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int i = tid + r * T;
    slot[r] = 0u;
    if (i < n) {
      slot[r] = atomicAdd(&sc.hist[bin[r]], 1u);
      sel[slot[r]] = key[r];
    }
  }
  __syncthreads();  // hist[b] = end of bucket b = start of bucket b + 1
  uint32_t dst[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int i = tid + r * T;
    dst[r] = 0u;
    if (i < n) {
      const uint32_t start = bin[r] > 0 ? sc.hist[bin[r] - 1] : 0u, end = sc.hist[bin[r]];
      uint32_t below = 0;
      for (uint32_t j = start; j < end; ++j) {
        const uint64_t o = sel[j];
        below += (o < key[r] || (o == key[r] && j < slot[r])) ? 1u : 0u;
      }
      dst[r] = start + below;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < PER; ++r)
    if (tid + r * T < n) sel[dst[r]] = key[r];
  __syncthreads();
}

// Selection and order in one bucket pass, for lists of at most PER * NT
// unique keys (a query's candidates in the common case), NT = blockDim.x
// threads. Only the upper 32 bits of each key (the score part) are held in
// registers: hi[r] is that of list entry threadIdx.x + r * NT (loaded by the
// caller, who may read past cnt: entries at or past cnt are ignored). The
// upper halves less their minimum, shifted right until the range fits 4096
// ordered buckets, give each key a bucket; the buckets are counted and
// prefix-summed, which locates the bucket b* holding the k_sel-th smallest
// key. The keys of buckets up to b* are read again whole from the list and
// scattered by bucket into tmp; each one's final place is its bucket's start
// plus the number of the bucket's keys below it, and the places below k_sel
// are written to sel. The result is the k_sel smallest keys in ascending order
// in sel[0 .. k_sel) -- the radix select and sort of the list. Returns false,
// leaving sel untouched, when the list is longer than PER * NT or a bucket
// holds more than kMaxBucket keys (many equal scores); the caller then takes
// the general path. tmp needs room for k_sel + kMaxBucket keys.
//
// Thread t prefix-sums the buckets t * BPT .. t * BPT + BPT - 1 (BPT = 4096 /
// NT). Bucket b is kept at hist[(b % BPT) * NT + b / BPT], so that the BPT
// reads and writes of that sum are consecutive across each warp (no bank
// conflicts); counts, cursors and bucket bounds go through the same map.
constexpr uint32_t kMaxBucket = 32;

template <int PER, int NT>
static __device__ bool cta_select_sort_hi(const uint64_t* list, const uint32_t (&hi)[PER], int cnt,
                                          int k_sel, uint64_t* sel, uint64_t* tmp,
                                          RadixScratch& sc) {
  constexpr int NB = 4096, BPT = NB / NT;
  static_assert(NB % NT == 0 && NT % 32 == 0 && NT / 32 <= 32, "thread count");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (cnt > PER * NT) return false;
  if (k_sel <= 0) return true;
  if (tid == 0) {
    sc.out[0] = 0xffffffffu;
    sc.out[1] = 0u;
    sc.out[2] = 0u;
  }
  for (int b = tid; b < NB; b += NT) sc.hist[b] = 0u;
  uint32_t lo = 0xffffffffu, top = 0u;
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    if (tid + r * NT < cnt) {
      lo = min(lo, hi[r]);
      top = max(top, hi[r]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    top = max(top, __shfl_xor_sync(0xffffffffu, top, o));
  }
  __syncthreads();  // out[] and hist cleared
  if (lane == 0) {
    atomicMin(&sc.out[0], lo);
    atomicMax(&sc.out[1], top);
  }
  __syncthreads();
  const uint32_t kmin = sc.out[0], range = sc.out[1] - kmin;
  const int width = range == 0u ? 0 : 32 - __clz(range);
  const int sh = width > 12 ? width - 12 : 0;
  auto bucket = [&](uint32_t h) { return (h - kmin) >> sh; };
  auto slot = [](uint32_t b) { return (b % BPT) * NT + b / BPT; };
#pragma unroll
  for (int r = 0; r < PER; ++r)
    if (tid + r * NT < cnt) atomicAdd(&sc.hist[slot(bucket(hi[r]))], 1u);
  __syncthreads();
  // exclusive prefix sum; the bucket where the running count reaches k_sel;
  // the largest bucket
  uint32_t local = 0, big = 0;
#pragma unroll 1
  for (int j = 0; j < BPT; ++j) {
    const uint32_t c = sc.hist[j * NT + tid];
    local += c;
    big = max(big, c);
  }
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
    big = max(big, __shfl_xor_sync(0xffffffffu, big, o));
  }
  if (lane == 31) sc.warp_sums[warp] = incl;
  if (lane == 0) atomicMax(&sc.out[2], big);
  __syncthreads();
  uint32_t run = incl - local;
  for (int w = 0; w < warp; ++w) run += sc.warp_sums[w];
#pragma unroll 1
  for (int j = 0; j < BPT; ++j) {
    const uint32_t c = sc.hist[j * NT + tid];
    if (run < (uint32_t)k_sel && (uint32_t)k_sel <= run + c) sc.out[3] = (uint32_t)(tid * BPT + j);
    sc.hist[j * NT + tid] = run;
    run += c;
  }
  const bool crowded = sc.out[2] > kMaxBucket;
  __syncthreads();  // hist = start of each bucket; out[3] = b*
  if (crowded) return false;
  const uint32_t bstar = sc.out[3];
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int i = tid + r * NT;
    if (i < cnt) {
      const uint32_t b = bucket(hi[r]);
      if (b <= bstar) tmp[atomicAdd(&sc.hist[slot(b)], 1u)] = __ldg(list + i);
    }
  }
  __syncthreads();  // hist = end of each bucket up to b*
  const uint32_t scattered = sc.hist[slot(bstar)];
  for (uint32_t j = tid; j < scattered; j += NT) {
    const uint64_t key = tmp[j];
    const uint32_t b = bucket((uint32_t)(key >> 32));
    const uint32_t start = b > 0 ? sc.hist[slot(b - 1)] : 0u, end = sc.hist[slot(b)];
    uint32_t dst = start;
    for (uint32_t m = start; m < end; ++m) dst += tmp[m] < key ? 1u : 0u;
    if (dst < (uint32_t)k_sel) sel[dst] = key;
  }
  __syncthreads();
  return true;
}

// Write one query's sorted selection: k_eff keys then padding to k_top.
__device__ __forceinline__ void write_selection(const uint64_t* sel, int k_eff, int k_top,
                                                int32_t* idx_row, float* score_row) {
  for (int j = threadIdx.x; j < k_top; j += blockDim.x) {
    if (j < k_eff) {
      const uint64_t key = sel[j];
      idx_row[j] = (int32_t)(uint32_t)key;
      if (score_row) score_row[j] = desc32_score((uint32_t)(key >> 32));
    } else {
      idx_row[j] = -1;
      if (score_row) score_row[j] = -__int_as_float(0x7f800000);
    }
  }
}

// Four consecutive scores of a row starting at position s (s + 3 < ctx), read
// with one 16-byte load when the row is 16-byte aligned.
__device__ __forceinline__ float4 load4(const float* row, bool vec, int s) {
  if (vec) return *reinterpret_cast<const float4*>(row + s);
  return make_float4(row[s], row[s + 1], row[s + 2], row[s + 3]);
}

// Exact top-k of a full score row[0..ctx). A 12-bit histogram of desc32
// (one pass over the row) finds the bin holding the k-th best score. When the
// keys in and above that bin fit `list` (shared memory, `cap` keys; may be
// null), a second pass lists them there and they are radix selected and
// sorted in shared memory. Otherwise the radix select goes on over the row:
// further digits of 12 and 8 bits (one pass each, restricted to the keys under
// the prefix found so far; a pass that ends with a bin whose keys are all
// needed stops early) find the k-th best score, and a last pass keeps every
// score before it and, among the scores tied with it, the lowest positions
// (counted in position order across the CTA). Result: sel[0..min(k, ctx))
// sorted.
static __device__ int cta_row_topk(const float* row, int ctx, int k_top, uint64_t* sel,
                                   RadixScratch& sc, uint64_t* list = nullptr, int cap = 0) {
  const int k_eff = ctx < k_top ? ctx : k_top;
  if (k_eff <= 0) return 0;
  const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int n4 = ctx / 4;  // whole groups of four positions; the rest one by one
  // one pass over the row: f(score, position, in range) for every position,
  // four groups of four in flight per thread
  auto sweep = [&](auto&& f) {
    constexpr int U = 4;
    for (int i0 = 0; i0 < n4; i0 += U * T) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * T + tid;
        v[u] = i < n4 ? load4(row, vec, 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * T + tid;
        const bool in = i < n4;
        f(v[u].x, 4 * i, in);
        f(v[u].y, 4 * i + 1, in);
        f(v[u].z, 4 * i + 2, in);
        f(v[u].w, 4 * i + 3, in);
      }
    }
    for (int s0 = 4 * n4; s0 < ctx; s0 += T) {
      const int s = s0 + tid;
      f(s < ctx ? row[s] : 0.0f, s, s < ctx);
    }
  };
  // warp-aggregated append of the keys for which take holds
  auto append = [&](uint64_t* dst, float v, int s, bool take) {
    const unsigned mask = __ballot_sync(0xffffffffu, take);
    if (mask) {
      const int leader = __ffs(mask) - 1;
      uint32_t base = 0;
      if (lane == leader) base = atomicAdd(&sc.counter, (uint32_t)__popc(mask));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (take) dst[base + __popc(mask & ((1u << lane) - 1u))] = cand_key(v, s);
    }
  };
  uint32_t prefix = 0, need = (uint32_t)k_eff;
  int done = 0;
  bool whole = false;  // every key under the final prefix is kept
  for (int p = 0; p < 3 && !whole; ++p) {
    const int bits = p == 2 ? 8 : 12, shift = 32 - done - bits, nb = 1 << bits;
    for (int b = tid; b < nb; b += T) sc.hist[b] = 0;
    __syncthreads();
    sweep([&](float v, int, bool in) {
      const uint32_t d = desc32(v);
      in = in && (done == 0 || (d >> (32 - done)) == prefix);
      hist_add(sc.hist, (d >> shift) & (uint32_t)(nb - 1), in);
    });
    __syncthreads();
    cta_find_crossing(sc.hist, nb, need, sc.warp_sums, sc.out);
    const uint32_t bin = sc.out[0], before = sc.out[1];
    const uint32_t in_bin = sc.hist[bin];
    if (p == 0 && list != nullptr && (uint64_t)before + in_bin <= (uint64_t)cap) {
      // the keys in and above the bin fit the shared-memory list
      if (tid == 0) sc.counter = 0;
      __syncthreads();
      sweep([&](float v, int s, bool in) { append(list, v, s, in && (desc32(v) >> 20) <= bin); });
      __syncthreads();
      const int listed = (int)sc.counter;
      __syncthreads();
      const int got = cta_select_smallest_u64(list, listed, k_eff, sel, sc);
      cta_sort_u64(sel, got, sc);
      return got;
    }
    need -= before;
    prefix = (prefix << bits) | bin;
    done += bits;
    whole = in_bin == need;
    __syncthreads();
  }
  // Keep: desc32 >> (32 - done) below the prefix (all of them), and under the
  // prefix either all (whole) or, tied at the k-th score (done == 32), the
  // `need` lowest positions.
  const int drop = 32 - done;
  if (tid == 0) {
    sc.counter = 0;
    sc.out[2] = 0;  // tied keys seen so far
  }
  __syncthreads();
  if (whole) {
    sweep([&](float v, int s, bool in) {
      const uint32_t hi = desc32(v) >> drop;
      append(sel, v, s, in && hi <= prefix);
    });
    __syncthreads();
  } else {
    // positions in order, T*4 at a time, so that the tied keys are ranked by
    // position with one CTA scan per group
    const int groups = (ctx + 4 * T - 1) / (4 * T);
    for (int gi = 0; gi < groups; ++gi) {
      const int s = gi * 4 * T + 4 * tid;
      float v[4];
      bool in[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) in[j] = s + j < ctx;
      if (s + 3 < ctx) {
        const float4 f = load4(row, vec, s);
        v[0] = f.x;
        v[1] = f.y;
        v[2] = f.z;
        v[3] = f.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = in[j] ? row[s + j] : 0.0f;
      }
      // rank of this thread's first tied key: tied keys of earlier groups, of
      // earlier warps, of earlier lanes
      uint32_t ties = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) ties += (in[j] && desc32(v[j]) == prefix) ? 1u : 0u;
      uint32_t incl = ties;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (lane == 31) sc.warp_sums[warp] = incl;
      __syncthreads();
      uint32_t rank = sc.out[2] + incl - ties;
      for (int w = 0; w < warp; ++w) rank += sc.warp_sums[w];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t d = desc32(v[j]);
        const bool tie = in[j] && d == prefix;
        append(sel, v[j], s + j, in[j] && (d < prefix || (tie && rank < need)));
        rank += tie ? 1u : 0u;
      }
      __syncthreads();
      if (tid == T - 1) sc.out[2] = rank;  // the last thread's running rank
      const bool full = sc.counter >= (uint32_t)k_eff;
      __syncthreads();
      if (full) break;
    }
  }
  cta_sort_u64(sel, k_eff, sc);
  return k_eff;
}

}  // namespace hytopk

// prep.cu -- order the queries by position and pack them for the scoring
// kernels.
//
// Queries are placed in "slots" sorted by position, longest context first,
// so that a block of adjacent slots has nearly equal causal ranges (little
// masked work in a shared key tile) and the longest blocks are scheduled
// first. Packing copies each query's q rows to its slot, folds the fp8 query
// scale into the head weight and halves it (hw = w * q_scale / 2, valid
// because scales are positive; the halving is exact and is undone by the
// ReLU form (x + |x|) * hw of the epilogue), and records the position. Slots
// past n are padding with position -1 (no keys).
#include <climits>

#include "launch.h"

namespace hytopk {

namespace {

__device__ __forceinline__ int clean_position(const int32_t* positions, int t, int L) {
  const int p = positions[t];
  return (p >= 0 && p < L) ? p : -1;
}

// slot(t) = #{u : pos(u) > pos(t) or (pos(u) == pos(t) and u < t)}: a stable
// descending sort by rank counting. A block of 8 warps ranks 32 queries
// (4 per warp); the positions pass through shared memory 1024 at a time and
// the lanes of a warp split each tile, so the grid covers every SM.
constexpr int kRankWarps = 8, kRankPerWarp = 4, kRankTile = 1024;

__global__ void __launch_bounds__(kRankWarps * 32) k_rank_by_position(
    const int32_t* __restrict__ positions, int n, int L, int32_t* __restrict__ perm) {
  __shared__ int tile[kRankTile];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = (blockIdx.x * kRankWarps + warp) * kRankPerWarp;
  int mine[kRankPerWarp], rank[kRankPerWarp];
#pragma unroll
  for (int q = 0; q < kRankPerWarp; ++q) {
    mine[q] = t0 + q < n ? clean_position(positions, t0 + q, L) : INT_MIN;
    rank[q] = 0;
  }
  for (int base = 0; base < n; base += kRankTile) {
    for (int i = threadIdx.x; i < kRankTile; i += blockDim.x)
      tile[i] = base + i < n ? clean_position(positions, base + i, L) : INT_MIN;
    __syncthreads();
    const int lim = min(kRankTile, n - base);
    for (int j = lane; j < lim; j += 32) {
      const int pu = tile[j], u = base + j;
#pragma unroll
      for (int q = 0; q < kRankPerWarp; ++q)
        rank[q] += (pu > mine[q]) | ((pu == mine[q]) & (u < t0 + q));
    }
    __syncthreads();
  }
#pragma unroll
  for (int q = 0; q < kRankPerWarp; ++q) {
    const int r = __reduce_add_sync(0xffffffffu, rank[q]);
    if (lane == 0 && t0 + q < n) perm[r] = t0 + q;
  }
}

// Slot row of the packed query operand, in the key element type: a copy, or
// (e4m3 queries against bf16 keys) an exact conversion to bf16.
__global__ void __launch_bounds__(128) k_pack_queries(Problem p, SelectWs ws) {
  const int slot = blockIdx.x;
  const int t = slot < p.n ? ws.perm[slot] : -1;
  const int esize = p.dt == 0 ? 2 : 1;
  const size_t row_bytes = (size_t)p.H * p.d * esize;  // multiple of 16
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws.qp) + slot * row_bytes);
  const int nvec = (int)(row_bytes / 16);
  if (t < 0) {
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = make_uint4(0, 0, 0, 0);
    for (int h = threadIdx.x; h < p.H; h += blockDim.x) ws.wq[(size_t)slot * p.H + h] = 0.0f;
    if (threadIdx.x == 0) {
      ws.qpos[slot] = -1;
      ws.perm[slot] = -1;
    }
    return;
  }
  if (p.qdt == p.dt) {
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.q) +
                                                      (size_t)t * row_bytes);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = src[v];
  } else {  // e4m3 -> bf16: 8 codes in, 16 bytes out
    const uint2* src = reinterpret_cast<const uint2*>(reinterpret_cast<const uint8_t*>(p.q) +
                                                      (size_t)t * p.H * p.d);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) dst[v] = e4m3x8_to_bf16(src[v]);
  }
  for (int h = threadIdx.x; h < p.H; h += blockDim.x) {
    float wv = p.w[(size_t)t * p.H + h];
    if (p.qdt == 1) {
      const float qs = p.q_scale[(size_t)t * p.H + h];
      if (!(qs > 0.0f)) set_status(ws.counters, HYTOPK_DEV_BAD_SCALE);
      wv *= qs;
    }
    ws.wq[(size_t)slot * p.H + h] = 0.5f * wv;
  }
  if (threadIdx.x == 0) {
    const int pos = clean_position(p.positions, t, p.L);
    if (pos < 0) set_status(ws.counters, HYTOPK_DEV_BAD_POSITION);
    ws.qpos[slot] = pos;
  }
}

__global__ void k_check_key_scales(const float* __restrict__ k_scale, int L, uint32_t* counters) {
  bool bad = false;
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < L; s += gridDim.x * blockDim.x)
    bad |= !(k_scale[s] > 0.0f);
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(counters, HYTOPK_DEV_BAD_SCALE);
}

// Halved folded weights of the original queries (two-pass path): rows n..rows-1
// are zero padding.
__global__ void k_fold_weights(Problem p, int rows, float* __restrict__ hw) {
  const size_t total = (size_t)rows * p.H;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / p.H;
    float wv = 0.0f;
    if (t < (size_t)p.n) {
      wv = p.w[i];
      if (p.qdt == 1) wv *= p.q_scale[i];
    }
    hw[i] = 0.5f * wv;
  }
}

// q [n, H, d] e4m3 codes -> bf16 (exact), for paths that read q as given
__global__ void k_convert_queries(const uint2* __restrict__ q8, size_t n_chunks,
                                  uint4* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n_chunks;
       i += (size_t)gridDim.x * blockDim.x)
    out[i] = e4m3x8_to_bf16(q8[i]);
}

}  // namespace

cudaError_t launch_convert_queries(const Problem& p, void* out, cudaStream_t st) {
  const size_t n_chunks = (size_t)p.n * p.H * p.d / 8;
  if (n_chunks == 0) return cudaSuccess;
  k_convert_queries<<<512, 256, 0, st>>>(reinterpret_cast<const uint2*>(p.q), n_chunks,
                                         reinterpret_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_fold_weights(const Problem& p, int rows, float* hw, cudaStream_t st) {
  k_fold_weights<<<256, 256, 0, st>>>(p, rows, hw);
  return cudaGetLastError();
}

cudaError_t launch_prep(const Problem& p, const SelectWs& ws, cudaStream_t st) {
  constexpr int per_block = kRankWarps * kRankPerWarp;
  if (p.n > 0)
    k_rank_by_position<<<(p.n + per_block - 1) / per_block, kRankWarps * 32, 0, st>>>(
        p.positions, p.n, p.L, ws.perm);
  if (ws.n_pad > 0) k_pack_queries<<<ws.n_pad, 128, 0, st>>>(p, ws);
  if (p.dt == 1) {
    // four blocks per SM (about 16 scales a thread at 1M keys), fewer when L is small
    const int want = (p.L + 4 * 256 - 1) / (4 * 256), cap = 4 * num_sms();
    k_check_key_scales<<<want < cap ? want : cap, 256, 0, st>>>(p.k_scale, p.L, ws.counters);
  }
  return cudaGetLastError();
}

}  // namespace hytopk

// sharded.cu -- hytopk_select_sharded: exact selection with the keys split
// into ranges, one hytopk_select per range, then one merge per query.
//
// This is how a selection runs when each GPU of a context-parallel group holds
// one range of the keys (HyScale summary, "What the paper found", and the
// explainer's limits paragraph: context-parallel communication overlapped with
// selection). Here the ranges run one after another on one stream; the merge
// is the exchange step. Exactness: with one total order on (score, position)
// the k best of a union are among the k best of each part, so the merge of
// the per-range exact top-k lists is the exact top-k of the whole context.
#include "launch.h"
#include "radix.cuh"

namespace hytopk {
namespace {

constexpr int kMaxShards = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Keys per range: ceil(L / P) rounded up to whole key tiles.
int shard_keys(int L, int P) {
  const long long s = ((long long)L + P - 1) / P;
  return (int)((s + kTileKeys - 1) / kTileKeys * kTileKeys);
}

struct ShardLayout {
  size_t sel, pos, idx, sc, keys, stats, status, total;
};

ShardLayout shard_layout(int n, int L, int H, int d, int k_top, int capacity, hytopk_dtype dt,
                         int P) {
  ShardLayout s{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 1024);
    return at;
  };
  const size_t sel = hytopk_select_workspace_size(n, shard_keys(L, P), H, d, k_top, capacity, dt);
  if (sel == 0) return s;
  s.sel = take(sel);
  s.pos = take((size_t)n * 4);
  s.idx = take((size_t)n * k_top * 4);
  s.sc = take((size_t)n * k_top * 4);
  s.keys = take((size_t)n * P * k_top * 8);
  s.stats = take((size_t)P * sizeof(hytopk_stats));
  s.status = take(16);
  s.total = off;
  return s;
}

// Position of query t inside range [lo, hi): min(pos, hi - 1) - lo, or -1
// when the query sees no key of the range (its position is below lo). A
// position outside [0, L) is reported once, here, and gives -1 everywhere.
__global__ void k_shard_positions(const int32_t* __restrict__ positions, int n, int L, int lo,
                                  int hi, int32_t* __restrict__ out, uint32_t* status) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const int p = positions[t];
  const bool valid = p >= 0 && p < L;
  if (!valid && lo == 0) atomicOr(status, HYTOPK_DEV_BAD_POSITION);
  out[t] = (valid && p >= lo) ? min(p, hi - 1) - lo : -1;
}

// Range p's selection of each query as ordered keys, global positions:
// keys[t][p*k + j]; an empty entry (-1) becomes the largest key, which no
// real candidate equals (positions are below 2^31).
__global__ void k_collect_shard(const int32_t* __restrict__ idx, const float* __restrict__ sc,
                                int n, int k_top, int lo, int P, int p,
                                uint64_t* __restrict__ keys) {
  const size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (e >= (size_t)n * k_top) return;
  const size_t t = e / k_top;
  const int j = (int)(e - t * k_top);
  const int s = idx[e];
  keys[(t * P + p) * k_top + j] = s >= 0 ? cand_key(sc[e], s + lo) : ~0ull;
}

// One CTA per query: the exact k best of the union of the ranges' lists.
__global__ void __launch_bounds__(512) k_merge_shards(const int32_t* __restrict__ positions, int n,
                                                      int L, int k_top, int S, int used, int P,
                                                      const uint64_t* __restrict__ keys,
                                                      int32_t* __restrict__ idx_out,
                                                      float* __restrict__ scores_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RadixScratch& rsc = *reinterpret_cast<RadixScratch*>(smem_raw);
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw + sizeof(RadixScratch));
  const int t = blockIdx.x;
  const int pos = positions[t];
  int k_eff = 0;
  if (pos >= 0 && pos < L) {
    // entries the ranges hold for this query: sum of min(k, keys of the range <= pos)
    long long held = 0;
    for (int p = 0; p < used; ++p) {
      const long long lo = (long long)p * S;
      const long long hi = lo + S < L ? lo + S : L;
      const long long c = pos < lo ? 0 : (pos < hi ? pos - lo + 1 : hi - lo);
      held += c < k_top ? c : k_top;
    }
    k_eff = (int)(held < k_top ? held : k_top);
  }
  int got = 0;
  if (k_eff > 0) {
    got = cta_select_smallest_u64(keys + (size_t)t * P * k_top, used * k_top, k_eff, sel, rsc);
    cta_sort_u64(sel, got, rsc);
  }
  write_selection(sel, got, k_top, idx_out + (size_t)t * k_top,
                  scores_out ? scores_out + (size_t)t * k_top : nullptr);
}

// Sum of the ranges' statistics. The ranges see queries below their start as
// positions "outside the range"; that bit is dropped here and the call's own
// position check (k_shard_positions) supplies it instead.
__global__ void k_sum_stats(const hytopk_stats* __restrict__ per, int used, int n,
                            const uint32_t* status, hytopk_stats* out) {
  if (threadIdx.x != 0) return;
  hytopk_stats s{};
  for (int p = 0; p < used; ++p) {
    s.n_failed += per[p].n_failed;
    s.n_overflow += per[p].n_overflow;
    s.n_under_k += per[p].n_under_k;
    s.fallback_used |= per[p].fallback_used;
    s.total_candidates += per[p].total_candidates;
    s.device_status |= per[p].device_status & ~HYTOPK_DEV_BAD_POSITION;
  }
  s.device_status |= *status;
  s.n_queries = n;
  *out = s;
}

bool shard_args_ok(int L, int P) { return P >= 1 && P <= kMaxShards && L >= 1; }

}  // namespace
}  // namespace hytopk

using namespace hytopk;

extern "C" size_t hytopk_select_sharded_workspace_size(int n, int L, int H, int d, int k_top,
                                                       int capacity, hytopk_dtype dt,
                                                       int num_shards) {
  if (!shard_args_ok(L, num_shards) || n < 0) return 0;
  return shard_layout(n, L, H, d, k_top, capacity, dt, num_shards).total;
}

extern "C" hytopk_status hytopk_select_sharded(const void* q, const float* q_scale, const void* k,
                                               const float* k_scale, const float* w,
                                               const int32_t* positions, int n, int L, int H,
                                               int d, int k_top, hytopk_dtype dt, int num_shards,
                                               int32_t* idx_out, float* scores_out, int capacity,
                                               void* workspace, size_t workspace_bytes,
                                               hytopk_stats* stats_out, cudaStream_t stream) {
  if (!shard_args_ok(L, num_shards) || n < 0) return HYTOPK_INVALID_ARG;
  hytopk_status s = check_shape(n, L, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  if ((s = check_inputs(q, q_scale, k, k_scale, w, dt, n)) != HYTOPK_OK) return s;
  const int P = num_shards;
  const ShardLayout lay = shard_layout(n, L, H, d, k_top, capacity, dt, P);
  if (lay.total == 0)  // shape, dtype or capacity rejected: let hytopk_select say which
    return hytopk_select(q, q_scale, k, k_scale, w, positions, n, L, H, d, k_top, dt, idx_out,
                         scores_out, capacity, nullptr, 0, stats_out, stream);
  if (n == 0)
    return hytopk_select(q, q_scale, k, k_scale, w, positions, n, L, H, d, k_top, dt, idx_out,
                         scores_out, capacity, workspace, workspace_bytes, stats_out, stream);
  if (!positions || !idx_out || !workspace) return HYTOPK_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return HYTOPK_MISALIGNED;
  if (workspace_bytes < lay.total) return HYTOPK_WORKSPACE_TOO_SMALL;

  uint8_t* base = static_cast<uint8_t*>(workspace);
  void* sel_ws = base + lay.sel;
  const size_t sel_bytes = lay.pos - lay.sel;
  int32_t* pos_s = reinterpret_cast<int32_t*>(base + lay.pos);
  int32_t* idx_s = reinterpret_cast<int32_t*>(base + lay.idx);
  float* sc_s = reinterpret_cast<float*>(base + lay.sc);
  uint64_t* keys = reinterpret_cast<uint64_t*>(base + lay.keys);
  hytopk_stats* per = reinterpret_cast<hytopk_stats*>(base + lay.stats);
  uint32_t* status = reinterpret_cast<uint32_t*>(base + lay.status);

  const int S = shard_keys(L, P);
  const int used = (L + S - 1) / S;
  const int esize = dt == HYTOPK_E4M3 ? 1 : 2;  // key element bytes
  if (cudaMemsetAsync(status, 0, 4, stream) != cudaSuccess) return HYTOPK_CUDA_ERROR;
  const int pos_blocks = (n + 255) / 256;
  const size_t entries = (size_t)n * k_top;
  const unsigned collect_blocks = (unsigned)((entries + 255) / 256);
  for (int p = 0; p < used; ++p) {
    const int lo = p * S;
    const int hi = lo + S < L ? lo + S : L;
    k_shard_positions<<<pos_blocks, 256, 0, stream>>>(positions, n, L, lo, hi, pos_s, status);
    if (cudaGetLastError() != cudaSuccess) return HYTOPK_CUDA_ERROR;
    const void* k_range = static_cast<const uint8_t*>(k) + (size_t)lo * d * esize;
    const float* ks_range = k_scale ? k_scale + lo : nullptr;
    const hytopk_status st =
        hytopk_select(q, q_scale, k_range, ks_range, w, pos_s, n, hi - lo, H, d, k_top, dt, idx_s,
                      sc_s, capacity, sel_ws, sel_bytes, per + p, stream);
    if (st != HYTOPK_OK) return st;
    k_collect_shard<<<collect_blocks, 256, 0, stream>>>(idx_s, sc_s, n, k_top, lo, P, p, keys);
    if (cudaGetLastError() != cudaSuccess) return HYTOPK_CUDA_ERROR;
  }
  const size_t smem = select_smem_bytes(k_top);
  if (cudaFuncSetAttribute(k_merge_shards, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return HYTOPK_CUDA_ERROR;
  k_merge_shards<<<n, 512, smem, stream>>>(positions, n, L, k_top, S, used, P, keys, idx_out,
                                           scores_out);
  if (cudaGetLastError() != cudaSuccess) return HYTOPK_CUDA_ERROR;
  if (stats_out) {
    k_sum_stats<<<1, 32, 0, stream>>>(per, used, n, status, stats_out);
    if (cudaGetLastError() != cudaSuccess) return HYTOPK_CUDA_ERROR;
  }
  return HYTOPK_OK;
}

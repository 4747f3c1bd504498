// select.cu -- the check kernel, the exact selection over candidate buffers,
// the statistics, and the read-back half of the two-pass path.
//
// HyScale explainer, HyTopK paragraph: a check kernel flags any query whose
// candidates overflowed the buffer or number fewer than k; more than 64 such
// queries fall back to rescoring everything; the exact selection resolves
// ties at the k-th score by position and radix-sorts the k kept entries.
#include "launch.h"
#include "radix.cuh"

namespace hytopk {

namespace {

__global__ void k_check(Problem p, SelectWs ws) {
  const int slot = blockIdx.x * blockDim.x + threadIdx.x;
  if (slot >= ws.n_pad) return;
  const int t = ws.perm[slot];
  uint8_t failed = 0;
  if (t >= 0) {
    const int64_t ctx = (int64_t)ws.qpos[slot] + 1;
    const int c = ws.cnt[slot];
    const bool under = ctx > p.k_top && c < p.k_top;
    const bool over = ctx > p.k_top && c > ws.C;
    failed = under || over;
    if (under) atomicAdd(ws.counters + kCtrUnderK, 1u);
    if (over) atomicAdd(ws.counters + kCtrOverflow, 1u);
    if (failed) {
      const uint32_t at = atomicAdd(ws.counters + kCtrFailed, 1u);
      ws.failed_list[at] = slot;
    }
    atomicAdd(reinterpret_cast<unsigned long long*>(ws.counters + kCtrCandLo),
              (unsigned long long)c);
  }
  ws.failed[slot] = failed;
}

// One CTA per query slot: select and sort the k best candidates. A list of
// at most 16 keys per thread is selected and ordered by one bucket pass
// (cta_select_sort_hi) with only the keys' upper halves in registers, so that
// three CTAs share an SM; longer lists, or lists with crowded buckets (many
// equal scores), take the radix select over the list in global memory and
// the general sort.
constexpr int kSelectPer = 16;
constexpr int kSelectThreads = 512;

// Scatter room of the bucket pass: it runs on lists of at most
// kSelectPer * kSelectThreads keys and keeps k of them, and may scatter up to
// kMaxBucket - 1 keys past the k-th.
__host__ __device__ constexpr int select_tmp_keys(int k_top) {
  return (k_top < kSelectPer * kSelectThreads ? k_top : kSelectPer * kSelectThreads) +
         (int)kMaxBucket;
}

__global__ void __launch_bounds__(kSelectThreads, 3) k_select_candidates(Problem p, SelectWs ws,
                                                           int32_t* __restrict__ idx_out,
                                                           float* __restrict__ scores_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RadixScratch& sc = *reinterpret_cast<RadixScratch*>(smem_raw);
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw + sizeof(RadixScratch));
  uint64_t* tmp = sel + sort_capacity(p.k_top);  // select_tmp_keys(k_top) keys
  const int slot = blockIdx.x;
  // every read of the slot's state, the upper halves of its first candidates
  // included (the buffer has C entries whatever the count), is issued before
  // any is used
  const uint64_t* list = ws.cand + (size_t)slot * ws.C;
  const uint32_t* list_hi = reinterpret_cast<const uint32_t*>(list) + 1;
  uint32_t hi[kSelectPer];
#pragma unroll
  for (int r = 0; r < kSelectPer; ++r) {
    const int i = threadIdx.x + r * kSelectThreads;
    hi[r] = i < ws.C ? __ldg(list_hi + 2 * i) : 0xffffffffu;
  }
  const int t = ws.perm[slot];
  const uint32_t n_failed = ws.counters[kCtrFailed];
  const uint8_t failed = ws.failed[slot];
  const int cnt = min(ws.cnt[slot], ws.C);
  if (t < 0 || n_failed > HYTOPK_MAX_RECOVERY_ROWS || failed) return;
  const int k_eff = min(p.k_top, cnt);
  if (!cta_select_sort_hi<kSelectPer, kSelectThreads>(list, hi, cnt, k_eff, sel, tmp, sc)) {
    const int got = cta_select_smallest_u64(list, cnt, k_eff, sel, sc);
    cta_sort_u64(sel, got, sc);
  }
  write_selection(sel, k_eff, p.k_top, idx_out + (size_t)t * p.k_top,
                  scores_out ? scores_out + (size_t)t * p.k_top : nullptr);
}

__global__ void k_finalize(SelectWs ws, int n, hytopk_stats* stats) {
  if (threadIdx.x != 0) return;
  const uint32_t failed = ws.counters[kCtrFailed];
  stats->n_failed = (int32_t)failed;
  stats->n_overflow = (int32_t)ws.counters[kCtrOverflow];
  stats->n_under_k = (int32_t)ws.counters[kCtrUnderK];
  stats->fallback_used = failed > HYTOPK_MAX_RECOVERY_ROWS ? 1 : 0;
  stats->total_candidates = *reinterpret_cast<const int64_t*>(ws.counters + kCtrCandLo);
  stats->device_status = ws.counters[kCtrStatus];
  stats->n_queries = n;
}

// Read-back half of the two-pass path: exact top-k of each table row.
// Shared-memory list of the read-back (keys in and above the histogram bin of
// the k-th best score): what is left of about 110 KB per CTA (two CTAs per
// SM) after the selection scratch, if that holds k + 1024 keys; else none.
__host__ __device__ inline int table_list_keys(int k_top) {
  const size_t budget = 110 * 1024, fixed = sizeof(RadixScratch) + sort_capacity(k_top) * 8;
  const int keys = fixed < budget ? (int)((budget - fixed) / 8) : 0;
  return keys >= k_top + 1024 ? keys : 0;
}

// Rows are queries row0.. in the caller's order (two-pass path), or, with
// `perm` (the fallback of hytopk_select), slots row0.. whose query is perm[slot]
// and position qpos[slot]; with `gate`, the launch does nothing unless the
// failed-query counter exceeds HYTOPK_MAX_RECOVERY_ROWS.
__global__ void __launch_bounds__(512) k_table_topk(Problem p, int row0, int rows,
                                                    const float* __restrict__ table,
                                                    const int32_t* __restrict__ perm,
                                                    const int32_t* __restrict__ qpos,
                                                    const uint32_t* gate,
                                                    int32_t* __restrict__ idx_out,
                                                    float* __restrict__ scores_out) {
  if (gate != nullptr && *reinterpret_cast<const volatile uint32_t*>(gate) <=
                             HYTOPK_MAX_RECOVERY_ROWS)
    return;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RadixScratch& sc = *reinterpret_cast<RadixScratch*>(smem_raw);
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw + sizeof(RadixScratch));
  const int cap = table_list_keys(p.k_top);
  uint64_t* list = cap > 0 ? sel + sort_capacity(p.k_top) : nullptr;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    int t, pos;
    if (perm != nullptr) {
      t = perm[row0 + r];
      pos = qpos[row0 + r];
      if (t < 0) continue;
    } else {
      t = row0 + r;
      pos = p.positions[t];
    }
    const int ctx = (pos >= 0 && pos < p.L) ? pos + 1 : 0;
    const int got = cta_row_topk(table + (size_t)r * p.L, ctx, p.k_top, sel, sc, list, cap);
    write_selection(sel, got, p.k_top, idx_out + (size_t)t * p.k_top,
                    scores_out ? scores_out + (size_t)t * p.k_top : nullptr);
    __syncthreads();
  }
}

}  // namespace

size_t select_smem_bytes(int k_top) {
  return sizeof(RadixScratch) + (size_t)sort_capacity(k_top) * sizeof(uint64_t);
}

cudaError_t launch_check(const Problem& p, const SelectWs& ws, cudaStream_t st) {
  if (ws.n_pad == 0) return cudaSuccess;
  k_check<<<(ws.n_pad + 255) / 256, 256, 0, st>>>(p, ws);
  return cudaGetLastError();
}

cudaError_t launch_select(const Problem& p, const SelectWs& ws, int32_t* idx_out,
                          float* scores_out, cudaStream_t st) {
  if (ws.n_pad == 0) return cudaSuccess;
  const size_t smem = select_smem_bytes(p.k_top) + select_tmp_keys(p.k_top) * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(k_select_candidates,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_select_candidates<<<ws.n_pad, kSelectThreads, smem, st>>>(p, ws, idx_out, scores_out);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const SelectWs& ws, int n, hytopk_stats* stats, cudaStream_t st) {
  k_finalize<<<1, 32, 0, st>>>(ws, n, stats);
  return cudaGetLastError();
}

namespace {

cudaError_t table_topk(const Problem& p, int row0, int rows, const float* table,
                       const int32_t* perm, const int32_t* qpos, const uint32_t* gate,
                       int32_t* idx_out, float* scores_out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const size_t smem = select_smem_bytes(p.k_top) + (size_t)table_list_keys(p.k_top) * 8;
  cudaError_t e =
      cudaFuncSetAttribute(k_table_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // the same shared-memory carveout as the table writer that runs before it,
  // so that the SMs need not be reconfigured between the two
  e = cudaFuncSetAttribute(k_table_topk, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const int grid = rows < kTableCtas ? rows : kTableCtas;
  k_table_topk<<<grid, 512, smem, st>>>(p, row0, rows, table, perm, qpos, gate, idx_out,
                                        scores_out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_table_topk(const Problem& p, int row0, int rows, const float* table,
                              int32_t* idx_out, float* scores_out, cudaStream_t st) {
  return table_topk(p, row0, rows, table, nullptr, nullptr, nullptr, idx_out, scores_out, st);
}

cudaError_t launch_fallback_topk(const Problem& p, const SelectWs& ws, int slot0, int rows,
                                 const float* table, int32_t* idx_out, float* scores_out,
                                 cudaStream_t st) {
  return table_topk(p, slot0, rows, table, ws.perm, ws.qpos, ws.counters + kCtrFailed, idx_out,
                    scores_out, st);
}

}  // namespace hytopk

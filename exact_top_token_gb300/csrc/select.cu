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

// One CTA per query slot: select and sort the k best candidates. Capped at 32
// registers so that four CTAs (64 warps) share an SM: the kernel waits on L2
// reads of the candidate lists and on CTA barriers, and the extra warps hide
// that (0.65 -> 0.58 ms at 1M keys, against 40 registers and three CTAs).
__global__ void __launch_bounds__(512, 4) k_select_candidates(Problem p, SelectWs ws,
                                                           int32_t* __restrict__ idx_out,
                                                           float* __restrict__ scores_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RadixScratch& sc = *reinterpret_cast<RadixScratch*>(smem_raw);
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw + sizeof(RadixScratch));
  const int slot = blockIdx.x;
  const int t = ws.perm[slot];
  if (t < 0) return;
  if (ws.counters[kCtrFailed] > HYTOPK_MAX_RECOVERY_ROWS || ws.failed[slot]) return;
  const int cnt = min(ws.cnt[slot], ws.C);
  const int k_eff = min(p.k_top, cnt);
  const int got = cta_select_smallest_u64(ws.cand + (size_t)slot * ws.C, cnt, k_eff, sel, sc);
  cta_sort_u64(sel, got, sc);
  write_selection(sel, got, p.k_top, idx_out + (size_t)t * p.k_top,
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
__global__ void __launch_bounds__(512) k_table_topk(Problem p, int row0, int rows,
                                                    const float* __restrict__ table,
                                                    uint64_t* __restrict__ lists,
                                                    int32_t* __restrict__ idx_out,
                                                    float* __restrict__ scores_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RadixScratch& sc = *reinterpret_cast<RadixScratch*>(smem_raw);
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw + sizeof(RadixScratch));
  uint64_t* list = lists + (size_t)blockIdx.x * p.L;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int t = row0 + r;
    const int pos = p.positions[t];
    const int ctx = (pos >= 0 && pos < p.L) ? pos + 1 : 0;
    const int got = cta_row_topk(table + (size_t)r * p.L, ctx, p.k_top, list, sel, sc);
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
  const size_t smem = select_smem_bytes(p.k_top);
  cudaError_t e = cudaFuncSetAttribute(k_select_candidates,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_select_candidates<<<ws.n_pad, 512, smem, st>>>(p, ws, idx_out, scores_out);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const SelectWs& ws, int n, hytopk_stats* stats, cudaStream_t st) {
  k_finalize<<<1, 32, 0, st>>>(ws, n, stats);
  return cudaGetLastError();
}

cudaError_t launch_table_topk(const Problem& p, int row0, int rows, const float* table,
                              uint64_t* lists, int n_lists, int32_t* idx_out, float* scores_out,
                              cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const size_t smem = select_smem_bytes(p.k_top);
  cudaError_t e =
      cudaFuncSetAttribute(k_table_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = rows < n_lists ? rows : n_lists;
  k_table_topk<<<grid, 512, smem, st>>>(p, row0, rows, table, lists, idx_out, scores_out);
  return cudaGetLastError();
}

}  // namespace hytopk

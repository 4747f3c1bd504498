// varlen.cu -- packed variable-length batches: B sequences concatenated along
// the query and key axes, each selected, replayed or differentiated on its
// own rows.
//
// Long-context training packs several sequences into one step; every query
// selects among the keys of its own sequence only (HyScale summary: learned
// sparse attention selects, per query, among the previous tokens of its
// sequence). The sequences run one after another on the caller's stream with
// the whole HyTopK selection each, reusing one workspace.
#include "launch.h"

namespace hytopk {
namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int key_bytes(hytopk_dtype dt) { return dt == HYTOPK_E4M3 ? 1 : 2; }
int query_bytes(hytopk_dtype dt) { return dt == HYTOPK_BF16 ? 2 : 1; }

// Host check of the two offset arrays: B >= 1, start at 0, non-decreasing,
// every sequence with queries has keys.
bool valid_offsets(const int32_t* cu_q, const int32_t* cu_k, int B) {
  if (B < 1 || !cu_q || !cu_k || cu_q[0] != 0 || cu_k[0] != 0) return false;
  for (int b = 0; b < B; ++b) {
    if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return false;
    if (cu_q[b + 1] > cu_q[b] && cu_k[b + 1] == cu_k[b]) return false;
  }
  return true;
}

// The largest per-sequence selection workspace (0 if a sequence is rejected).
size_t select_need(const int32_t* cu_q, const int32_t* cu_k, int B, int H, int d, int k_top,
                   int capacity, hytopk_dtype dt) {
  size_t need = 0;
  for (int b = 0; b < B; ++b) {
    const int nb = cu_q[b + 1] - cu_q[b], Lb = cu_k[b + 1] - cu_k[b];
    if (nb == 0) continue;
    const size_t s = hytopk_select_workspace_size(nb, Lb, H, d, k_top, capacity, dt);
    if (s == 0) return 0;
    need = s > need ? s : need;
  }
  return need;
}

size_t stats_bytes(int B) { return align_up((size_t)B * sizeof(hytopk_stats), 1024); }

__global__ void k_sum_stats(const hytopk_stats* __restrict__ per, int B, int n,
                            hytopk_stats* out) {
  if (threadIdx.x != 0) return;
  hytopk_stats s{};
  for (int b = 0; b < B; ++b) {
    s.n_failed += per[b].n_failed;
    s.n_overflow += per[b].n_overflow;
    s.n_under_k += per[b].n_under_k;
    s.fallback_used |= per[b].fallback_used;
    s.total_candidates += per[b].total_candidates;
    s.device_status |= per[b].device_status;
  }
  s.n_queries = n;
  *out = s;
}

}  // namespace
}  // namespace hytopk

using namespace hytopk;

extern "C" size_t hytopk_select_varlen_workspace_size(const int32_t* cu_q, const int32_t* cu_k,
                                                      int B, int H, int d, int k_top,
                                                      int capacity, hytopk_dtype dt) {
  if (!valid_offsets(cu_q, cu_k, B)) return 0;
  const size_t need = select_need(cu_q, cu_k, B, H, d, k_top, capacity, dt);
  if (need == 0 && cu_q[B] > 0) return 0;
  return align_up(need, 1024) + stats_bytes(B);
}

extern "C" hytopk_status hytopk_select_varlen(const void* q, const float* q_scale, const void* k,
                                              const float* k_scale, const float* w,
                                              const int32_t* positions, const int32_t* cu_q,
                                              const int32_t* cu_k, int B, int H, int d, int k_top,
                                              hytopk_dtype dt, int32_t* idx_out,
                                              float* scores_out, int capacity, void* workspace,
                                              size_t workspace_bytes, hytopk_stats* stats_out,
                                              cudaStream_t stream) {
  if (!valid_offsets(cu_q, cu_k, B)) return HYTOPK_INVALID_ARG;
  const int n = cu_q[B], L = cu_k[B];
  hytopk_status s = check_shape(n, L > 0 ? L : 1, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  if ((s = check_inputs(q, q_scale, k, k_scale, w, dt, n)) != HYTOPK_OK) return s;
  if (n == 0) {
    if (stats_out && cudaMemsetAsync(stats_out, 0, sizeof(hytopk_stats), stream) != cudaSuccess)
      return HYTOPK_CUDA_ERROR;
    return HYTOPK_OK;
  }
  if (!positions || !idx_out || !workspace) return HYTOPK_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return HYTOPK_MISALIGNED;
  const size_t need = select_need(cu_q, cu_k, B, H, d, k_top, capacity, dt);
  if (need == 0) return HYTOPK_INVALID_ARG;  // capacity below k_top
  const size_t sel_bytes = align_up(need, 1024);
  if (workspace_bytes < sel_bytes + stats_bytes(B)) return HYTOPK_WORKSPACE_TOO_SMALL;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  hytopk_stats* per = reinterpret_cast<hytopk_stats*>(base + sel_bytes);
  if (stats_out && cudaMemsetAsync(per, 0, (size_t)B * sizeof(hytopk_stats), stream) != cudaSuccess)
    return HYTOPK_CUDA_ERROR;
  const size_t qrow = (size_t)H * d * query_bytes(dt), krow = (size_t)d * key_bytes(dt);
  for (int b = 0; b < B; ++b) {
    const int q0 = cu_q[b], nb = cu_q[b + 1] - q0, k0 = cu_k[b], Lb = cu_k[b + 1] - k0;
    if (nb == 0) continue;
    s = hytopk_select(static_cast<const uint8_t*>(q) + (size_t)q0 * qrow,
                      q_scale ? q_scale + (size_t)q0 * H : nullptr,
                      static_cast<const uint8_t*>(k) + (size_t)k0 * krow,
                      k_scale ? k_scale + k0 : nullptr, w + (size_t)q0 * H, positions + q0, nb,
                      Lb, H, d, k_top, dt, idx_out + (size_t)q0 * k_top,
                      scores_out ? scores_out + (size_t)q0 * k_top : nullptr, capacity, base,
                      sel_bytes, stats_out ? per + b : nullptr, stream);
    if (s != HYTOPK_OK) return s;
  }
  if (stats_out) {
    k_sum_stats<<<1, 32, 0, stream>>>(per, B, n, stats_out);
    if (cudaGetLastError() != cudaSuccess) return HYTOPK_CUDA_ERROR;
  }
  return HYTOPK_OK;
}

extern "C" hytopk_status hytopk_replay_varlen(const void* q, const float* q_scale, const void* k,
                                              const float* k_scale, const float* w,
                                              const int32_t* idx, const int32_t* cu_q,
                                              const int32_t* cu_k, int B, int H, int d, int k_top,
                                              hytopk_dtype dt, float* scores_out,
                                              uint32_t* dev_status, cudaStream_t stream) {
  if (!valid_offsets(cu_q, cu_k, B)) return HYTOPK_INVALID_ARG;
  const int n = cu_q[B], L = cu_k[B];
  hytopk_status s = check_shape(n, L > 0 ? L : 1, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  if ((s = check_inputs(q, q_scale, k, k_scale, w, dt, n)) != HYTOPK_OK) return s;
  if (n == 0) return HYTOPK_OK;
  if (!idx || !scores_out) return HYTOPK_INVALID_ARG;
  const size_t qrow = (size_t)H * d * query_bytes(dt), krow = (size_t)d * key_bytes(dt);
  for (int b = 0; b < B; ++b) {
    const int q0 = cu_q[b], nb = cu_q[b + 1] - q0, k0 = cu_k[b], Lb = cu_k[b + 1] - k0;
    if (nb == 0) continue;
    s = hytopk_replay(static_cast<const uint8_t*>(q) + (size_t)q0 * qrow,
                      q_scale ? q_scale + (size_t)q0 * H : nullptr,
                      static_cast<const uint8_t*>(k) + (size_t)k0 * krow,
                      k_scale ? k_scale + k0 : nullptr, w + (size_t)q0 * H,
                      idx + (size_t)q0 * k_top, nb, Lb, H, d, k_top, dt,
                      scores_out + (size_t)q0 * k_top, dev_status, stream);
    if (s != HYTOPK_OK) return s;
  }
  return HYTOPK_OK;
}

extern "C" hytopk_status hytopk_replay_backward_varlen(
    const void* q, const float* q_scale, const void* k, const float* k_scale, const float* w,
    const int32_t* idx, const float* grad, const int32_t* cu_q, const int32_t* cu_k, int B, int H,
    int d, int k_top, hytopk_dtype dt, float* dq, float* dk, float* dw, uint32_t* dev_status,
    cudaStream_t stream) {
  if (!valid_offsets(cu_q, cu_k, B)) return HYTOPK_INVALID_ARG;
  const int n = cu_q[B], L = cu_k[B];
  hytopk_status s = check_shape(n, L > 0 ? L : 1, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  if ((s = check_inputs(q, q_scale, k, k_scale, w, dt, n)) != HYTOPK_OK) return s;
  if (n == 0) return HYTOPK_OK;
  if (!idx || !grad || !dq || !dk || !dw) return HYTOPK_INVALID_ARG;
  const size_t qrow = (size_t)H * d * query_bytes(dt), krow = (size_t)d * key_bytes(dt);
  for (int b = 0; b < B; ++b) {
    const int q0 = cu_q[b], nb = cu_q[b + 1] - q0, k0 = cu_k[b], Lb = cu_k[b + 1] - k0;
    if (nb == 0) continue;
    const size_t e0 = (size_t)q0 * k_top;
    s = hytopk_replay_backward(static_cast<const uint8_t*>(q) + (size_t)q0 * qrow,
                               q_scale ? q_scale + (size_t)q0 * H : nullptr,
                               static_cast<const uint8_t*>(k) + (size_t)k0 * krow,
                               k_scale ? k_scale + k0 : nullptr, w + (size_t)q0 * H, idx + e0,
                               grad + e0, nb, Lb, H, d, k_top, dt, dq + (size_t)q0 * H * d,
                               dk + (size_t)k0 * d, dw + (size_t)q0 * H, dev_status, stream);
    if (s != HYTOPK_OK) return s;
  }
  return HYTOPK_OK;
}

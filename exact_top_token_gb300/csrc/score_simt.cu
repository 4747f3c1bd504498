// score_simt.cu -- scoring phases on the CUDA cores: sampled threshold,
// recovery rescoring and replay.
//
// Every kernel evaluates the same per-(query, key) arithmetic
// (score_key_simt in common.cuh): raw-element dots in fp32 with fused
// multiply-adds over i = 0..d-1, ReLU, fused weighted sum over h = 0..H-1,
// then the key scale. The filter, recovery, replay and table kernels
// therefore return identical bits for the same (query, key).
#include "launch.h"
#include "radix.cuh"

namespace hytopk {

namespace {

// Decode the packed query rows of one slot (raw, [H][D]) and its folded
// weights into shared memory.
template <int D, int DT>
__device__ __forceinline__ void load_query(const void* qbase, size_t row0, int H, const float* wq,
                                           float* qf, float* wsm) {
  for (int i = threadIdx.x; i < H * D; i += blockDim.x) qf[i] = load_elem<DT>(qbase, row0 * D + i);
  for (int h = threadIdx.x; h < H; h += blockDim.x) wsm[h] = wq[h];
}

__device__ __forceinline__ float key_scale(const Problem& p, int s) {
  return p.dt == 1 ? p.k_scale[s] : 1.0f;
}

// ---- sampled threshold ---------------------------------------------------------
// One CTA per slot: score the M evenly spaced samples p_j = floor(j*ctx/M)
// and take the r-th best (HyScale explainer: HyTopK paragraph, worked example).
template <int D, int DT>
__global__ void __launch_bounds__(256) k_threshold_simt(Problem p, SelectWs ws,
                                                        const float* override_thr) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RadixScratch& sc = *reinterpret_cast<RadixScratch*>(smem_raw);
  float* qf = reinterpret_cast<float*>(smem_raw + sizeof(RadixScratch));
  float* wsm = qf + p.H * D;
  uint32_t* keys = reinterpret_cast<uint32_t*>(wsm + p.H);
  const int slot = blockIdx.x;
  const int t = ws.perm[slot];
  const int64_t ctx = (int64_t)ws.qpos[slot] + 1;
  if (t < 0 || ctx <= p.k_top) {
    if (threadIdx.x == 0) ws.thr[slot] = -__int_as_float(0x7f800000);
    return;
  }
  if (override_thr) {
    if (threadIdx.x == 0) ws.thr[slot] = override_thr[t];
    return;
  }
  const int M = sample_count(ctx);
  const int r = threshold_rank(ctx, p.k_top, M);
  load_query<D, DT>(ws.qp, (size_t)slot * p.H, p.H, ws.wq + (size_t)slot * p.H, qf, wsm);
  __syncthreads();
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    const int s = sample_position(ctx, M, j);
    float kr[D];
    load_key_row<D, DT>(p.k, (size_t)s, kr);
    keys[j] = desc32(score_key_simt<D>(qf, wsm, p.H, kr, key_scale(p, s)));
  }
  __syncthreads();
  const uint32_t v = cta_kth_smallest_u32(keys, M, (uint32_t)r, sc);
  if (threadIdx.x == 0) ws.thr[slot] = desc32_score(v);
}

// ---- recovery -------------------------------------------------------------------------
// Persistent CTAs rescore failed queries (or, past the 64-query limit, every
// query) over their whole context into a private row, then select exactly.
template <int D, int DT>
__global__ void __launch_bounds__(256) k_recover_simt(Problem p, SelectWs ws,
                                                      int32_t* __restrict__ idx_out,
                                                      float* __restrict__ scores_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RadixScratch& sc = *reinterpret_cast<RadixScratch*>(smem_raw);
  __shared__ int item_sh;
  const uint32_t n_failed = ws.counters[kCtrFailed];
  const bool fallback = n_failed > HYTOPK_MAX_RECOVERY_ROWS;
  const int total = fallback ? ws.n_pad : (int)n_failed;
  if (total == 0) return;
  const size_t P = (size_t)sort_capacity(p.k_top);
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem_raw + sizeof(RadixScratch));
  float* qf = reinterpret_cast<float*>(sel + P);
  float* wsm = qf + p.H * D;
  float* row = ws.rowbuf + (size_t)blockIdx.x * p.L;
  uint64_t* list = ws.rowlist + (size_t)blockIdx.x * p.L;
  for (;;) {
    if (threadIdx.x == 0) item_sh = (int)atomicAdd(ws.counters + kCtrRecoverWork, 1u);
    __syncthreads();
    const int item = item_sh;
    __syncthreads();
    if (item >= total) break;
    const int slot = fallback ? item : ws.failed_list[item];
    const int t = ws.perm[slot];
    if (t < 0) continue;
    const int ctx = ws.qpos[slot] + 1;
    load_query<D, DT>(ws.qp, (size_t)slot * p.H, p.H, ws.wq + (size_t)slot * p.H, qf, wsm);
    __syncthreads();
    for (int s = threadIdx.x; s < ctx; s += blockDim.x) {
      float kr[D];
      load_key_row<D, DT>(p.k, (size_t)s, kr);
      row[s] = score_key_simt<D>(qf, wsm, p.H, kr, key_scale(p, s));
    }
    __syncthreads();
    const int got = cta_row_topk(row, ctx, p.k_top, list, sel, sc);
    write_selection(sel, got, p.k_top, idx_out + (size_t)t * p.k_top,
                    scores_out ? scores_out + (size_t)t * p.k_top : nullptr);
    __syncthreads();
  }
}

// ---- replay ---------------------------------------------------------------------------
// One CTA per query: rescore only the stored indices (HyScale explainer,
// selection-replay paragraph).
template <int D, int DT>
__global__ void __launch_bounds__(128) k_replay_simt(Problem p, const int32_t* __restrict__ idx,
                                                     float* __restrict__ out, uint32_t* status) {
  extern __shared__ __align__(16) float rsm[];
  float* qf = rsm;
  float* wsm = qf + p.H * D;
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < p.H * D; i += blockDim.x)
    qf[i] = load_elem<DT>(p.q, (size_t)t * p.H * D + i);
  for (int h = threadIdx.x; h < p.H; h += blockDim.x) {
    float wv = p.w[(size_t)t * p.H + h];
    if (p.dt == 1) wv *= p.q_scale[(size_t)t * p.H + h];
    wsm[h] = wv;
  }
  __syncthreads();
  bool bad = false;
  for (int j = threadIdx.x; j < p.k_top; j += blockDim.x) {
    const int s = idx[(size_t)t * p.k_top + j];
    float v;
    if (s == -1) {
      v = -__int_as_float(0x7f800000);
    } else if (s < 0 || s >= p.L) {
      v = __int_as_float(0x7fc00000);
      bad = true;
    } else {
      float kr[D];
      load_key_row<D, DT>(p.k, (size_t)s, kr);
      v = score_key_simt<D>(qf, wsm, p.H, kr, key_scale(p, s));
    }
    out[(size_t)t * p.k_top + j] = v;
  }
  if (bad && status) atomicOr(status, HYTOPK_DEV_REPLAY_BAD_INDEX);
}

#define HYTOPK_DISPATCH(D_, DT_, CALL)                 \
  do {                                                 \
    if ((D_) == 64 && (DT_) == 0) { CALL(64, 0); }     \
    else if ((D_) == 64 && (DT_) == 1) { CALL(64, 1); } \
    else if ((D_) == 128 && (DT_) == 0) { CALL(128, 0); } \
    else { CALL(128, 1); }                             \
  } while (0)

template <typename F>
cudaError_t set_smem(F* fn, size_t bytes) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_threshold(const Problem& p, const SelectWs& ws, const float* override_thr,
                             cudaStream_t st) {
  if (ws.n_pad == 0) return cudaSuccess;
  const size_t smem = sizeof(RadixScratch) + ((size_t)p.H * p.d + p.H + kMaxSamples) * 4;
  cudaError_t e = cudaSuccess;
#define CALL(D, DT)                                                             \
  e = set_smem(k_threshold_simt<D, DT>, smem);                                  \
  if (e == cudaSuccess) k_threshold_simt<D, DT><<<ws.n_pad, 256, smem, st>>>(p, ws, override_thr);
  HYTOPK_DISPATCH(p.d, p.dt, CALL);
#undef CALL
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_recover(const Problem& p, const SelectWs& ws, int32_t* idx_out,
                           float* scores_out, cudaStream_t st) {
  if (ws.n_pad == 0) return cudaSuccess;
  const size_t P = (size_t)sort_capacity(p.k_top);
  const size_t smem = sizeof(RadixScratch) + P * 8 + ((size_t)p.H * p.d + p.H) * 4;
  cudaError_t e = cudaSuccess;
#define CALL(D, DT)                                        \
  e = set_smem(k_recover_simt<D, DT>, smem);               \
  if (e == cudaSuccess)                                    \
    k_recover_simt<D, DT><<<kRecoveryCtas, 256, smem, st>>>(p, ws, idx_out, scores_out);
  HYTOPK_DISPATCH(p.d, p.dt, CALL);
#undef CALL
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_replay(const Problem& p, const int32_t* idx, float* out, uint32_t* status,
                          cudaStream_t st) {
  if (p.n == 0) return cudaSuccess;
  const size_t smem = ((size_t)p.H * p.d + p.H) * 4;
  cudaError_t e = cudaSuccess;
#define CALL(D, DT)                                    \
  e = set_smem(k_replay_simt<D, DT>, smem);            \
  if (e == cudaSuccess) k_replay_simt<D, DT><<<p.n, 128, smem, st>>>(p, idx, out, status);
  HYTOPK_DISPATCH(p.d, p.dt, CALL);
#undef CALL
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hytopk

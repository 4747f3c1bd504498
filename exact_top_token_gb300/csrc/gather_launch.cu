// gather_launch.cu -- host launchers of the gather engine: the sampled
// threshold and recovery phases of hytopk_select, hytopk_replay and the paired
// replay of hytopk_replay_grouped.
#include "gather_engine.cuh"
#include "launch.h"

namespace hytopk {

cudaError_t launch_gather_d64_bf16(int H, int mode, const gather::GArgs& a, int grid,
                                   cudaStream_t st);
cudaError_t launch_gather_d64_e4m3(int H, int mode, const gather::GArgs& a, int grid,
                                   cudaStream_t st);
cudaError_t launch_gather_d128_bf16(int H, int mode, const gather::GArgs& a, int grid,
                                    cudaStream_t st);
cudaError_t launch_gather_d128_e4m3(int H, int mode, const gather::GArgs& a, int grid,
                                    cudaStream_t st);
cudaError_t launch_gather_d32_bf16(int H, int mode, const gather::GArgs& a, int grid,
                                   cudaStream_t st);
cudaError_t launch_gather_d256_e4m3(int H, int mode, const gather::GArgs& a, int grid,
                                    cudaStream_t st);

namespace {

cudaError_t dispatch(const Problem& p, int mode, const gather::GArgs& a, int grid,
                     cudaStream_t st) {
  if (grid <= 0) return cudaSuccess;
  if (p.dt == 0) {
    if (p.d == 32) return launch_gather_d32_bf16(p.H, mode, a, grid, st);
    if (p.d == 64) return launch_gather_d64_bf16(p.H, mode, a, grid, st);
    return launch_gather_d128_bf16(p.H, mode, a, grid, st);
  }
  if (p.d == 64) return launch_gather_d64_e4m3(p.H, mode, a, grid, st);
  if (p.d == 128) return launch_gather_d128_e4m3(p.H, mode, a, grid, st);
  return launch_gather_d256_e4m3(p.H, mode, a, grid, st);
}

gather::GArgs base_args(const Problem& p) {
  gather::GArgs a{};
  a.k = p.k;
  a.k_scale = p.k_scale;
  a.L = p.L;
  a.k_top = p.k_top;
  a.n = p.n;
  return a;
}

void slot_args(gather::GArgs& a, const SelectWs& ws) {
  a.perm = ws.perm;
  a.qpos = ws.qpos;
  a.qp = ws.qp;
  a.wq = ws.wq;
  a.thr = ws.thr;
  a.n_pad = ws.n_pad;
  a.counters = ws.counters;
  a.failed_list = ws.failed_list;
  a.rowbuf = ws.rowbuf;
  a.status = ws.counters + kCtrStatus;
}

int capped_grid(int items) {
  const int g = 2 * num_sms();
  return items < g ? items : g;
}

}  // namespace

cudaError_t launch_threshold(const Problem& p, const SelectWs& ws, const float* override_thr,
                             cudaStream_t st) {
  gather::GArgs a = base_args(p);
  slot_args(a, ws);
  a.override_thr = override_thr;
  return dispatch(p, gather::kThreshold, a, capped_grid(ws.n_pad), st);
}

cudaError_t launch_recover(const Problem& p, const SelectWs& ws, int32_t* idx_out,
                           float* scores_out, cudaStream_t st) {
  gather::GArgs a = base_args(p);
  slot_args(a, ws);
  a.idx_out = idx_out;
  a.scores_out = scores_out;
  return dispatch(p, gather::kRecover, a, ws.n_pad > 0 ? kRecoveryCtas : 0, st);
}

cudaError_t launch_replay(const Problem& p, const int32_t* idx, float* out, uint32_t* status,
                          cudaStream_t st) {
  gather::GArgs a = base_args(p);
  a.q = p.q;
  a.q_scale = p.q_scale;
  a.q_e4m3 = p.qdt == 1 && p.dt == 0;
  a.w = p.w;
  a.idx = idx;
  a.out = out;
  a.status = status;
  return dispatch(p, gather::kReplay, a, capped_grid(p.n), st);
}

bool replay_pair_supported(const Problem& p) {
  return p.H <= 64 && p.k_top <= gather::kMaxPairTopK;
}

cudaError_t launch_replay_pair(const Problem& p, const int32_t* idx, float* out, uint32_t* status,
                               cudaStream_t st) {
  gather::GArgs a = base_args(p);
  a.q = p.q;
  a.q_scale = p.q_scale;
  a.q_e4m3 = p.qdt == 1 && p.dt == 0;
  a.w = p.w;
  a.idx = idx;
  a.out = out;
  a.status = status;
  return dispatch(p, gather::kReplayPair, a, capped_grid((p.n + 1) / 2), st);
}

}  // namespace hytopk

// gather_launch.cu -- host launchers of the gather engine: the sampled
// threshold and recovery phases of hytopk_select, and hytopk_replay.
#include "gather_engine.cuh"
#include "launch.h"

namespace hytopk {

cudaError_t launch_gather_d64_bf16(int H, int mode, const CUtensorMap& km,
                                    const gather::GArgs& a, int items,
                                   cudaStream_t st);
cudaError_t launch_gather_d64_e4m3(int H, int mode, const CUtensorMap& km,
                                    const gather::GArgs& a, int items,
                                   cudaStream_t st);
cudaError_t launch_gather_d128_bf16(int H, int mode, const CUtensorMap& km,
                                    const gather::GArgs& a, int items,
                                    cudaStream_t st);
cudaError_t launch_gather_d128_e4m3(int H, int mode, const CUtensorMap& km,
                                    const gather::GArgs& a, int items,
                                    cudaStream_t st);

namespace {

// Tensor map of the keys for TMA gathers: boxes one row high, one swizzle atom
// (128 or 64 bytes) wide.
cudaError_t dispatch(const Problem& p, int mode, const gather::GArgs& a, int items,
                     cudaStream_t st) {
  if (items <= 0) return cudaSuccess;
  const int rb = p.d * (p.dt == 0 ? 2 : 1);
  const int atom = rb >= 128 ? 128 : 64;
  CUtensorMap km;
  if (!make_tmap_2d(&km, p.k, p.dt, (uint64_t)p.d, (uint64_t)p.L, atom / (p.dt == 0 ? 2 : 1), 1,
                    atom))
    return cudaErrorInvalidValue;
  if (p.d == 64)
    return p.dt == 0 ? launch_gather_d64_bf16(p.H, mode, km, a, items, st)
                     : launch_gather_d64_e4m3(p.H, mode, km, a, items, st);
  return p.dt == 0 ? launch_gather_d128_bf16(p.H, mode, km, a, items, st)
                   : launch_gather_d128_e4m3(p.H, mode, km, a, items, st);
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
  a.rowlist = ws.rowlist;
  a.status = ws.counters + kCtrStatus;
}

}  // namespace

cudaError_t launch_threshold(const Problem& p, const SelectWs& ws, const float* override_thr,
                             cudaStream_t st) {
  gather::GArgs a = base_args(p);
  slot_args(a, ws);
  a.override_thr = override_thr;
  return dispatch(p, gather::kThreshold, a, ws.n_pad, st);
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
  a.w = p.w;
  a.idx = idx;
  a.out = out;
  a.status = status;
  return dispatch(p, gather::kReplay, a, p.n, st);
}

}  // namespace hytopk

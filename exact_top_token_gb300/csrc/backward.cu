// backward.cu -- hytopk_replay_backward: gradients of the indexer score at the
// selected entries (the engine is backward_engine.cuh).
#include "backward_engine.cuh"
#include "launch.h"

namespace hytopk {

cudaError_t launch_backward_bf16(int d, int H, const bwd::BArgs& a, int grid, cudaStream_t st);
cudaError_t launch_backward_e4m3(int d, int H, const bwd::BArgs& a, int grid, cudaStream_t st);
cudaError_t launch_backward_bf16_small(int d, int H, const bwd::BArgs& a, int grid,
                                       cudaStream_t st);
cudaError_t launch_backward_e4m3_small(int d, int H, const bwd::BArgs& a, int grid,
                                       cudaStream_t st);

}  // namespace hytopk

using namespace hytopk;

extern "C" hytopk_status hytopk_replay_backward(const void* q, const float* q_scale, const void* k,
                                                const float* k_scale, const float* w,
                                                const int32_t* idx, const float* grad, int n,
                                                int L, int H, int d, int k_top, hytopk_dtype dt,
                                                float* dq, float* dk, float* dw,
                                                uint32_t* dev_status, cudaStream_t stream) {
  hytopk_status s = check_shape(n, L, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  if ((s = check_inputs(q, q_scale, k, k_scale, w, dt, n)) != HYTOPK_OK) return s;
  if (H > 64 || (d != 64 && d != 128)) return HYTOPK_UNSUPPORTED;
  if (n == 0) return HYTOPK_OK;
  if (!idx || !grad || !dq || !dk || !dw) return HYTOPK_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dq) & 15u) || (reinterpret_cast<uintptr_t>(dk) & 15u))
    return HYTOPK_MISALIGNED;
  bwd::BArgs a{};
  a.q = q;
  a.q_scale = q_scale;
  a.k = k;
  a.k_scale = k_scale;
  a.w = w;
  a.idx = idx;
  a.grad = grad;
  a.dq = dq;
  a.dk = dk;
  a.dw = dw;
  a.n = n;
  a.L = L;
  a.k_top = k_top;
  a.q_e4m3 = dt != HYTOPK_BF16;
  a.status = dev_status;
  const int grid = n < num_sms() ? n : num_sms();
  const bool e4 = dt == HYTOPK_E4M3;
  const cudaError_t e = H < 16 ? (e4 ? launch_backward_e4m3_small(d, H, a, grid, stream)
                                     : launch_backward_bf16_small(d, H, a, grid, stream))
                               : (e4 ? launch_backward_e4m3(d, H, a, grid, stream)
                                     : launch_backward_bf16(d, H, a, grid, stream));
  return e == cudaSuccess ? HYTOPK_OK : HYTOPK_CUDA_ERROR;
}

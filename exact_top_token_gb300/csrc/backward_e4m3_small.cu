// backward_e4m3_small.cu -- instantiations of the backward engine for e4m3 inputs
// with fewer than 16 heads (padded to 16 inside the engine); a translation
// unit of its own so that the library compiles in parallel.
#include "backward_engine.cuh"
#include "launch.h"

namespace hytopk {

namespace {

template <int D, int H>
cudaError_t go(const bwd::BArgs& a, int grid, cudaStream_t st) {
  constexpr int smem = bwd::Cfg<D, 1, H>::SMEM;
  auto fn = bwd::k_backward<D, 1, H>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fn<<<grid, bwd::kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_e4m3_small(int d, int H, const bwd::BArgs& a, int grid,
                                       cudaStream_t st) {
  if (d == 64) {
    if (H == 1) return go<64, 1>(a, grid, st);
    if (H == 2) return go<64, 2>(a, grid, st);
    if (H == 4) return go<64, 4>(a, grid, st);
    if (H == 8) return go<64, 8>(a, grid, st);
  } else if (d == 128) {
    if (H == 1) return go<128, 1>(a, grid, st);
    if (H == 2) return go<128, 2>(a, grid, st);
    if (H == 4) return go<128, 4>(a, grid, st);
    if (H == 8) return go<128, 8>(a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hytopk

// backward_e4m3.cu -- instantiations of the backward engine for e4m3 inputs
// (one translation unit per dtype so that the library compiles in parallel).
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

cudaError_t launch_backward_e4m3(int d, int H, const bwd::BArgs& a, int grid, cudaStream_t st) {
  if (d == 64) {
    if (H == 16) return go<64, 16>(a, grid, st);
    if (H == 32) return go<64, 32>(a, grid, st);
    if (H == 64) return go<64, 64>(a, grid, st);
  } else if (d == 128) {
    if (H == 16) return go<128, 16>(a, grid, st);
    if (H == 32) return go<128, 32>(a, grid, st);
    if (H == 64) return go<128, 64>(a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hytopk

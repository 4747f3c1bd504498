// gather_d32_bf16.cu -- instantiations of the tensor-core gather engine
// (threshold sampling, replay, recovery) for d = 32, bf16 inputs.
#include "gather_engine.cuh"
#include "launch.h"

namespace hytopk {

namespace {

template <int H, int MODE>
cudaError_t go(const gather::GArgs& a0, int grid, cudaStream_t st) {
  gather::GArgs a = a0;
  int u = 0;
  const int smem = gather::gather_smem_bytes<32, 0, H, MODE>(a.k_top, &u);
  a.u_bytes = u;
  auto fn = gather::k_gather<32, 0, H, MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fn<<<grid, gather::kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_d32_bf16(int H, int mode, const gather::GArgs& a, int grid,
                                     cudaStream_t st) {
  switch (H) {
    case 1: return mode == 0 ? go<1, 0>(a, grid, st) : mode == 1 ? go<1, 1>(a, grid, st) : go<1, 2>(a, grid, st);
    case 2: return mode == 0 ? go<2, 0>(a, grid, st) : mode == 1 ? go<2, 1>(a, grid, st) : go<2, 2>(a, grid, st);
    case 4: return mode == 0 ? go<4, 0>(a, grid, st) : mode == 1 ? go<4, 1>(a, grid, st) : go<4, 2>(a, grid, st);
    case 8: return mode == 0 ? go<8, 0>(a, grid, st) : mode == 1 ? go<8, 1>(a, grid, st) : go<8, 2>(a, grid, st);
    case 16: return mode == 0 ? go<16, 0>(a, grid, st) : mode == 1 ? go<16, 1>(a, grid, st) : go<16, 2>(a, grid, st);
    case 32: return mode == 0 ? go<32, 0>(a, grid, st) : mode == 1 ? go<32, 1>(a, grid, st) : go<32, 2>(a, grid, st);
    case 64: return mode == 0 ? go<64, 0>(a, grid, st) : mode == 1 ? go<64, 1>(a, grid, st) : go<64, 2>(a, grid, st);
    case 128: return mode == 0 ? go<128, 0>(a, grid, st) : mode == 1 ? go<128, 1>(a, grid, st) : go<128, 2>(a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hytopk

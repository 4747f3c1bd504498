// stream_d32_bf16.cu -- instantiations of the tensor-core streaming engine
// for d = 32, bf16 inputs (one translation unit per (d, dtype) so that the
// library compiles in parallel).
#include "launch.h"
#include "stream_engine.cuh"

namespace hytopk {

namespace {

template <int H, int MODE>
cudaError_t go(const CUtensorMap& km, const CUtensorMap& qm, const stream::Args& a, int grid,
               cudaStream_t st) {
  constexpr int smem = stream::Cfg<32, 0, H>::SMEM;
  auto fn = stream::k_stream<32, 0, H, MODE>;
  cudaError_t e = stream::check_register_split<32, 0, H, MODE>();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (MODE == 1) {  // the table writer alternates with the read-back: one carveout for both
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  fn<<<grid, stream::kThreads, smem, st>>>(km, qm, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stream_d32_bf16(int H, int mode, const CUtensorMap& km, const CUtensorMap& qm,
                                     const stream::Args& a, int grid, cudaStream_t st) {
  switch (H) {
    case 1: return mode ? go<1, 1>(km, qm, a, grid, st) : go<1, 0>(km, qm, a, grid, st);
    case 2: return mode ? go<2, 1>(km, qm, a, grid, st) : go<2, 0>(km, qm, a, grid, st);
    case 4: return mode ? go<4, 1>(km, qm, a, grid, st) : go<4, 0>(km, qm, a, grid, st);
    case 8: return mode ? go<8, 1>(km, qm, a, grid, st) : go<8, 0>(km, qm, a, grid, st);
    case 16: return mode ? go<16, 1>(km, qm, a, grid, st) : go<16, 0>(km, qm, a, grid, st);
    case 32: return mode ? go<32, 1>(km, qm, a, grid, st) : go<32, 0>(km, qm, a, grid, st);
    case 64: return mode ? go<64, 1>(km, qm, a, grid, st) : go<64, 0>(km, qm, a, grid, st);
    case 128: return mode ? go<128, 1>(km, qm, a, grid, st) : go<128, 0>(km, qm, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hytopk

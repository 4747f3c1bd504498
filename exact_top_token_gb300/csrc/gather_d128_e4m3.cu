// gather_d128_e4m3.cu -- instantiations of the tensor-core gather engine
// (threshold sampling, replay, recovery) for d = 128, e4m3 inputs.
#include "gather_engine.cuh"
#include "launch.h"

namespace hytopk {

namespace {

// items: queries to process. The grid is the number of CTAs resident at once
// (persistent CTAs), except for recovery, which has one scratch row per CTA.
template <int H, int MODE>
cudaError_t go(const CUtensorMap& km, const gather::GArgs& a0, int items, cudaStream_t st) {
  gather::GArgs a = a0;
  int u = 0;
  const int smem = gather::gather_smem_bytes<128, 1, H, MODE>(a.k_top, &u);
  a.u_bytes = u;
  auto fn = gather::k_gather<128, 1, H, MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = items;
  if (MODE != gather::kRecover) {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, gather::kThreads, smem);
    if (e != cudaSuccess) return e;
    const int resident = (per_sm > 0 ? per_sm : 1) * num_sms();
    grid = items < resident ? items : resident;
  }
  if (grid <= 0) return cudaSuccess;
  fn<<<grid, gather::kThreads, smem, st>>>(km, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_d128_e4m3(int H, int mode, const CUtensorMap& km,
                                     const gather::GArgs& a, int items, cudaStream_t st) {
  switch (H) {
    case 1: return mode == 0 ? go<1, 0>(km, a, items, st) : mode == 1 ? go<1, 1>(km, a, items, st) : go<1, 2>(km, a, items, st);
    case 2: return mode == 0 ? go<2, 0>(km, a, items, st) : mode == 1 ? go<2, 1>(km, a, items, st) : go<2, 2>(km, a, items, st);
    case 4: return mode == 0 ? go<4, 0>(km, a, items, st) : mode == 1 ? go<4, 1>(km, a, items, st) : go<4, 2>(km, a, items, st);
    case 8: return mode == 0 ? go<8, 0>(km, a, items, st) : mode == 1 ? go<8, 1>(km, a, items, st) : go<8, 2>(km, a, items, st);
    case 16: return mode == 0 ? go<16, 0>(km, a, items, st) : mode == 1 ? go<16, 1>(km, a, items, st) : go<16, 2>(km, a, items, st);
    case 32: return mode == 0 ? go<32, 0>(km, a, items, st) : mode == 1 ? go<32, 1>(km, a, items, st) : go<32, 2>(km, a, items, st);
    case 64: return mode == 0 ? go<64, 0>(km, a, items, st) : mode == 1 ? go<64, 1>(km, a, items, st) : go<64, 2>(km, a, items, st);
    case 128: return mode == 0 ? go<128, 0>(km, a, items, st) : mode == 1 ? go<128, 1>(km, a, items, st) : go<128, 2>(km, a, items, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hytopk

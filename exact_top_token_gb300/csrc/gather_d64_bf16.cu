// gather_d64_bf16.cu -- instantiations of the tensor-core gather engine
// (threshold sampling, replay, paired replay, recovery) for d = 64, bf16 keys.
#include "gather_engine.cuh"
#include "launch.h"

namespace hytopk {

cudaError_t launch_gather_d64_bf16(int H, int mode, const gather::GArgs& a, int grid,
                                   cudaStream_t st) {
  return gather::gather_launch<64, 0>(H, mode, a, grid, st);
}

}  // namespace hytopk

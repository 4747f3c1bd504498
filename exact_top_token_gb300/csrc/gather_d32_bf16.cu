// gather_d32_bf16.cu -- instantiations of the tensor-core gather engine
// (threshold sampling, replay, paired replay, recovery) for d = 32, bf16 keys.
#include "gather_engine.cuh"
#include "launch.h"

namespace hytopk {

cudaError_t launch_gather_d32_bf16(int H, int mode, const gather::GArgs& a, int grid,
                                   cudaStream_t st) {
  return gather::gather_launch<32, 0>(H, mode, a, grid, st);
}

}  // namespace hytopk

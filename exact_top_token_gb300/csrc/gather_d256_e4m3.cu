// gather_d256_e4m3.cu -- instantiations of the tensor-core gather engine
// (threshold sampling, replay, paired replay, recovery) for d = 256, e4m3 keys.
#include "gather_engine.cuh"
#include "launch.h"

namespace hytopk {

cudaError_t launch_gather_d256_e4m3(int H, int mode, const gather::GArgs& a, int grid,
                                    cudaStream_t st) {
  return gather::gather_launch<256, 1>(H, mode, a, grid, st);
}

}  // namespace hytopk

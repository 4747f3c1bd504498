// launch.h -- host-side launchers of the HyTopK kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace hytopk {

// prep.cu
cudaError_t launch_prep(const Problem& p, const SelectWs& ws, cudaStream_t st);

// score_*.cu: the scoring phases
cudaError_t launch_threshold(const Problem& p, const SelectWs& ws, const float* override_thr,
                             cudaStream_t st);
cudaError_t launch_filter(const Problem& p, const SelectWs& ws, int reverse, cudaStream_t st);
cudaError_t launch_recover(const Problem& p, const SelectWs& ws, int32_t* idx_out,
                           float* scores_out, cudaStream_t st);
cudaError_t launch_replay(const Problem& p, const int32_t* idx, float* out, uint32_t* status,
                          cudaStream_t st);
cudaError_t launch_table(const Problem& p, int row0, int rows, float* table, uint32_t* status,
                         cudaStream_t st);

// select.cu
cudaError_t launch_check(const Problem& p, const SelectWs& ws, cudaStream_t st);
cudaError_t launch_select(const Problem& p, const SelectWs& ws, int32_t* idx_out,
                          float* scores_out, cudaStream_t st);
cudaError_t launch_finalize(const SelectWs& ws, int n, hytopk_stats* stats, cudaStream_t st);
cudaError_t launch_table_topk(const Problem& p, int row0, int rows, const float* table,
                              uint64_t* lists, int n_lists, int32_t* idx_out, float* scores_out,
                              cudaStream_t st);

// Shared-memory bytes of the candidate selection for k_top.
size_t select_smem_bytes(int k_top);

}  // namespace hytopk

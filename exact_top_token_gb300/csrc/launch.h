// launch.h -- host-side launchers of the HyTopK kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"

namespace hytopk {

// prep.cu
cudaError_t launch_prep(const Problem& p, const SelectWs& ws, cudaStream_t st);
cudaError_t launch_fold_weights(const Problem& p, int rows, float* hw, cudaStream_t st);
// e4m3 q -> bf16 copy [n, H, d] (the mixed dtype's paths that read q as given)
cudaError_t launch_convert_queries(const Problem& p, void* out, cudaStream_t st);

// score_*.cu: the scoring phases
cudaError_t launch_threshold(const Problem& p, const SelectWs& ws, const float* override_thr,
                             cudaStream_t st);
cudaError_t launch_filter(const Problem& p, const SelectWs& ws, int reverse, cudaStream_t st);
cudaError_t launch_recover(const Problem& p, const SelectWs& ws, int32_t* idx_out,
                           float* scores_out, cudaStream_t st);
cudaError_t launch_replay(const Problem& p, const int32_t* idx, float* out, uint32_t* status,
                          cudaStream_t st);
// adjacent queries 2i, 2i+1 replayed together over the union of their indices
bool replay_pair_supported(const Problem& p);
cudaError_t launch_replay_pair(const Problem& p, const int32_t* idx, float* out, uint32_t* status,
                               cudaStream_t st);
cudaError_t launch_table(const Problem& p, int row0, int rows, float* table, const float* hw,
                         uint32_t* status, cudaStream_t st);

// select.cu
cudaError_t launch_check(const Problem& p, const SelectWs& ws, cudaStream_t st);
cudaError_t launch_select(const Problem& p, const SelectWs& ws, int32_t* idx_out,
                          float* scores_out, cudaStream_t st);
cudaError_t launch_finalize(const SelectWs& ws, int n, hytopk_stats* stats, cudaStream_t st);
cudaError_t launch_table_topk(const Problem& p, int row0, int rows, const float* table,
                              int32_t* idx_out, float* scores_out, cudaStream_t st);
// The fallback of hytopk_select past HYTOPK_MAX_RECOVERY_ROWS failed queries:
// slots slot0 .. slot0 + rows - 1 scored into a table (slot order, one row of
// L scores each) and their exact top-k read back. Both launches do nothing
// unless the failed-query counter exceeds the limit.
struct FallbackMaps {
  CUtensorMap km, qm;  // keys; slot-packed queries
};
cudaError_t prepare_fallback_table(const Problem& p, const SelectWs& ws, FallbackMaps* m);
cudaError_t launch_fallback_table(const Problem& p, const SelectWs& ws, const FallbackMaps& m,
                                  int slot0, int rows, float* table, cudaStream_t st);
cudaError_t launch_fallback_topk(const Problem& p, const SelectWs& ws, int slot0, int rows,
                                 const float* table, int32_t* idx_out, float* scores_out,
                                 cudaStream_t st);

// tmap.cu
bool make_tmap_2d(CUtensorMap* map, const void* base, int dt, uint64_t inner_elems, uint64_t rows,
                  uint32_t box_inner_elems, uint32_t box_rows, int swizzle_bytes);
int num_sms();
int stream_chunks(int L);
cudaError_t launch_plan(const SelectWs& ws, int L, int qb, int chunk_tiles, cudaStream_t st);

// Shared-memory bytes of the candidate selection for k_top.
size_t select_smem_bytes(int k_top);

// Host-side argument checks shared by the entry points (api.cu).
hytopk_status check_shape(int n, int L, int H, int d, int k_top, hytopk_dtype dt);
hytopk_status check_inputs(const void* q, const float* q_scale, const void* k,
                           const float* k_scale, const float* w, hytopk_dtype dt, int n);

}  // namespace hytopk

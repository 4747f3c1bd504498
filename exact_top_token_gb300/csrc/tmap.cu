// tmap.cu -- TMA tensor maps (host side) and the work plan of the filter.
#include <cudaTypedefs.h>

#include "launch.h"
#include "stream_engine.cuh"

namespace hytopk {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Exclusive prefix sum over a block of 1024 threads; returns the block total.
__device__ int block_exclusive_scan(int v, int* excl, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) before += warp_tot[w];
    total += warp_tot[w];
  }
  *excl = before + incl - v;
  __syncthreads();
  return total;
}

// plan[c] = number of filter work items before key chunk c: chunk c holds one
// item per query block whose largest position reaches the chunk (blocks are
// sorted by position, descending, so they are a prefix). plan[nchunks] = total.
__global__ void __launch_bounds__(1024) k_plan(const int32_t* __restrict__ qpos, int nblocks,
                                               int qb, int nchunks, int chunk_keys,
                                               int32_t* __restrict__ plan) {
  __shared__ int warp_tot[32];
  int carry = 0;
  for (int base = 0; base < nchunks; base += 1024) {
    const int c = base + threadIdx.x;
    int nb = 0;
    if (c < nchunks) {
      const int key0 = c * chunk_keys;
      int lo = 0, hi = nblocks;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (qpos[mid * qb] >= key0) lo = mid + 1;
        else hi = mid;
      }
      nb = lo;
    }
    int excl;
    const int tot = block_exclusive_scan(nb, &excl, warp_tot);
    if (c < nchunks) plan[c] = carry + excl;
    carry += tot;
  }
  if (threadIdx.x == 0) plan[nchunks] = carry;
}

}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* base, int dt, uint64_t inner_elems, uint64_t rows,
                  uint32_t box_inner_elems, uint32_t box_rows, int swizzle_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int es = dt == 0 ? 2 : 1;
  const cuuint64_t dims[2] = {inner_elems, rows};
  const cuuint64_t strides[1] = {inner_elems * es};
  const cuuint32_t box[2] = {box_inner_elems, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = fn(map, dt == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                        2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

// Key chunks at the shortest chunk length: an upper bound on the filter's
// chunk count (the size of the plan).
int stream_chunks(int L) { return (L + stream::kChunkKeys - 1) / stream::kChunkKeys; }

cudaError_t launch_plan(const SelectWs& ws, int L, int qb, int chunk_tiles, cudaStream_t st) {
  const int chunk_keys = chunk_tiles * kTileKeys;
  k_plan<<<1, 1024, 0, st>>>(ws.qpos, ws.n_pad / qb, qb, (L + chunk_keys - 1) / chunk_keys,
                             chunk_keys, ws.plan);
  return cudaGetLastError();
}

}  // namespace hytopk

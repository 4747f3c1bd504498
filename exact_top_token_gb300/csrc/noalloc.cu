// noalloc.cu -- hytopk_select_noalloc: the exact top-k selection for callers
// that cannot allocate device memory themselves.
//
// Some callers can neither call cudaMalloc nor hand the library a workspace
// of the size hytopk_select asks for: code that runs inside a host framework
// which owns the whole device-memory budget through its own pool and forbids
// any allocation outside it, and latency-critical paths where an allocation
// (and the device synchronisation cudaMalloc/cudaFree can imply) is not
// acceptable. For them the library keeps one fixed scratch array in device
// memory, below, and runs the normal hytopk_select on it.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds HYTOPK_NOALLOC_SCRATCH_BYTES for it until the
// process exits. In host code its name is only a host-side stand-in, so its
// device address is looked up with cudaGetSymbolAddress, once per device and
// with that device current, the first time the entry point runs on that
// device. Nothing here allocates: no cudaMalloc, cudaFree or allocating
// library routine is called.
#include <mutex>

#include "launch.h"

namespace {

constexpr size_t kScratchBytes = HYTOPK_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 128;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call per device). Returns nullptr on a CUDA error.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" hytopk_status hytopk_select_noalloc(const void* q, const float* q_scale, const void* k,
                                               const float* k_scale, const float* w,
                                               const int32_t* positions, int n, int L, int H,
                                               int d, int k_top, hytopk_dtype dt,
                                               int32_t* idx_out, float* scores_out, int capacity,
                                               hytopk_stats* stats_out, cudaStream_t stream) {
  // the argument checks of hytopk_select, in its order, before the size check
  hytopk_status s = hytopk::check_shape(n, L, H, d, k_top, dt);
  if (s != HYTOPK_OK) return s;
  s = hytopk::check_inputs(q, q_scale, k, k_scale, w, dt, n);
  if (s != HYTOPK_OK) return s;
  if (capacity < 0 || (capacity > 0 && capacity < k_top)) return HYTOPK_INVALID_ARG;
  if (n > 0 && (!positions || !idx_out)) return HYTOPK_INVALID_ARG;
  const size_t need = hytopk_select_workspace_size(n, L, H, d, k_top, capacity, dt);
  if (need == 0) return HYTOPK_INVALID_ARG;
  if (need > kScratchBytes) return HYTOPK_WORKSPACE_TOO_SMALL;
  void* scratch = scratch_on_current_device();
  if (!scratch) return HYTOPK_CUDA_ERROR;
  // hytopk_select clears every counter and count it relies on at the start of
  // each call, so what a previous call left in the array does not matter.
  return hytopk_select(q, q_scale, k, k_scale, w, positions, n, L, H, d, k_top, dt, idx_out,
                       scores_out, capacity, scratch, kScratchBytes, stats_out, stream);
}

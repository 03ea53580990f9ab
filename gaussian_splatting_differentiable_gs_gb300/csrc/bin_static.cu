// bin_static.cu -- gs_bin_and_sort_static: binning without a caller workspace.
//
// gs_bin_and_sort needs a scratch workspace that the caller allocates.  Some
// callers cannot allocate device memory at the point where they bin: a host
// application whose own allocator owns every byte of the GPU and hands out
// no extra buffers, a render or training loop that must not stall on an
// allocation in the middle of a frame, or a plug-in that only ever receives
// the input and output buffers it is given.  For them this variant keeps its
// scratch in one file-scope device array sized for a bounded problem, so the
// call itself allocates nothing.
//
// Costs and limits:
//  - the array (kStaticWsBytes) is part of the library image: every GPU that
//    loads the library holds it until the process exits;
//  - at most kStaticMaxRows projected rows (n_views * n) and at most
//    kStaticMaxIsect intersections; larger problems are rejected;
//  - all calls share the one array, so two calls whose work overlaps on the
//    GPU (different streams, or different host threads) race and corrupt each
//    other's results: serialise them;
//  - the array keeps what the previous call left in it; the call clears the
//    parts that must start at zero itself (the status words are carried over
//    on purpose so that a device-side wait that ran out in one call is
//    reported by the next, as with gs_bin_and_sort).
#include <mutex>

#include "gs_internal.cuh"

namespace {

constexpr int64_t kStaticMaxRows = GS_BIN_STATIC_MAX_ROWS;
constexpr int64_t kStaticMaxIsect = GS_BIN_STATIC_MAX_ISECT;
constexpr size_t kStaticWsBytes = size_t(14) << 20;

// The scratch itself.  Host code may not pass this name to a kernel (on the
// host it is only a stand-in for the device symbol); its device address is
// looked up once per device below.
static __device__ __align__(256) unsigned char g_bin_scratch[kStaticWsBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: device address of the array,
// and a zeroed status header.
gs_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return GS_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    if (gs_bin_workspace_bytes(kStaticMaxRows, kStaticMaxIsect) > kStaticWsBytes)
      return GS_ERR_DEVICE_CHECK;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bin_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return GS_ERR_CUDA;
    }
    if (cudaMemset(p, 0, 256) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      (void)cudaGetLastError();
      return GS_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GS_OK;
}

}  // namespace

extern "C" gs_status gs_bin_and_sort_static(int64_t n, int32_t n_views, const gs_splat* splats,
                                            const int32_t* tile_counts, int32_t width, int32_t height, int64_t capacity,
                                            uint64_t* keys, uint32_t* vals, int64_t* ranges,
                                            int64_t* n_isect, void* stream) {
  if (n < 0 || n_views < 1 || n_views > GS_MAX_VIEWS || capacity < 0) return GS_ERR_INVALID_ARG;
  // n > max / n_views rather than n * n_views > max: the product could overflow
  if (n > kStaticMaxRows / n_views || capacity > kStaticMaxIsect) return GS_ERR_INVALID_ARG;
  void* ws = nullptr;
  const gs_status st = scratch_for_current_device(&ws);
  if (st != GS_OK) return st;
  return gs_bin_and_sort(n, n_views, splats, tile_counts, width, height, ws, kStaticWsBytes,
                         capacity, keys, vals, ranges, n_isect, stream);
}

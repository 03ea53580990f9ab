// prune.cu -- gs_prune_mask and gs_compact_index: pruning of Gaussians
// bounded by the per-tile working set the compositing kernels keep on chip.
//
// "ByteSplat: Efficient Distributed 3D Gaussian Splatting Training ...",
// abstract: pruning that considers both rendering quality and per-tile
// shared-memory constraints, so that fused forward + backward rasterization
// keeps its working set on chip.  Rule (the pages give only the intent):
//   working set of a tile = its list positions [0, L), L = the largest
//     n_contrib over the tile's pixels (nothing behind it is composited);
//   a tile is over capacity when L > K;
//   theta_t = the K-th largest importance among the tile's working set;
//   a Gaussian is pruned when, in some over-capacity tile of some view, it
//     lies in the working set with importance < theta_t and importance < tau
//     (the quality floor: Gaussians that weigh >= tau in some pixel stay).
// Importance is a per-row input (gs_rasterize_fwd_importance gives each
// row's largest blending weight alpha T); a Gaussian's importance in a view
// is its row's.
#include <stdint.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kPT = 256;  // threads per tile CTA
constexpr int kBins = 256;

// One CTA per (view, tile).
__global__ void __launch_bounds__(kPT) prune_tile_kernel(
    int64_t n, int32_t tiles_x, int64_t T, int32_t W, int32_t H, const uint32_t* __restrict__ vals,
    const int64_t* __restrict__ ranges, const int32_t* __restrict__ n_contrib,
    const float* __restrict__ importance, int64_t K, float tau, uint8_t* __restrict__ mask) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t s_max;
  __shared__ uint32_t s_sel[2];  // chosen digit, count strictly above it
  const int tid = threadIdx.x;
  const int64_t flat = blockIdx.x;
  const int64_t view = flat / T;
  const int32_t tile = (int32_t)(flat - view * T);
  const int tile_x = tile % tiles_x, tile_y = tile / tiles_x;
  const int64_t start = ranges[2 * flat], end = ranges[2 * flat + 1];
  // working set: the largest n_contrib over the tile's pixels
  if (tid == 0) s_max = 0;
  __syncthreads();
  {
    const int px = tile_x * GS_TILE + (tid & 15), py = tile_y * GS_TILE + (tid >> 4);
    uint32_t c = 0;
    if (px < W && py < H) c = (uint32_t)max(0, n_contrib[view * (int64_t)W * H + (int64_t)py * W + px]);
    c = __reduce_max_sync(0xffffffffu, c);
    if ((tid & 31) == 0) atomicMax(&s_max, c);
  }
  __syncthreads();
  const int64_t L = min((int64_t)s_max, end - start);
  if (L <= K) return;
  const float* vimp = importance + view * n;
  auto imp_bits = [&](int64_t i) {
    const uint32_t id = min(__ldg(vals + start + i), (uint32_t)(n - 1));
    return __float_as_uint(fmaxf(__ldg(vimp + id), 0.f));  // >= 0: bits order as values
  };
  // K-th largest importance: most-significant-digit radix select, 4 x 8 bits
  uint32_t prefix = 0, want = (uint32_t)K;  // rank among entries matching prefix
  for (int pass = 3; pass >= 0; --pass) {
    const int shift = 8 * pass;
    const uint32_t hi_mask = pass == 3 ? 0u : (0xFFFFFFFFu << (shift + 8));
    hist[tid] = 0;
    __syncthreads();
    for (int64_t i = tid; i < L; i += kPT) {
      const uint32_t b = imp_bits(i);
      if ((b & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(b >> shift) & 0xFF], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t above = 0;
      int d = kBins - 1;
      for (; d > 0; --d) {
        if (above + hist[d] >= want) break;
        above += hist[d];
      }
      s_sel[0] = (uint32_t)d;
      s_sel[1] = above;
    }
    __syncthreads();
    prefix |= s_sel[0] << shift;
    want -= s_sel[1];
    __syncthreads();
  }
  const float theta = __uint_as_float(prefix);
  for (int64_t i = tid; i < L; i += kPT) {
    const uint32_t id = min(__ldg(vals + start + i), (uint32_t)(n - 1));
    const float v = fmaxf(__ldg(vimp + id), 0.f);
    if (v < theta && v < tau) mask[id] = 1;
  }
}

constexpr int kCT = 256;        // compaction threads
constexpr int kCItems = 16;     // flags per thread
constexpr int kCPart = kCT * kCItems;

// per-partition count of kept (mask == 0) entries
__global__ void __launch_bounds__(kCT) count_keep_kernel(int64_t n, const uint8_t* __restrict__ mask,
                                                         int64_t* __restrict__ part_count) {
  __shared__ int s_w[kCT / 32];
  const int64_t base = (int64_t)blockIdx.x * kCPart;
  int c = 0;
  for (int k = 0; k < kCItems; ++k) {
    const int64_t i = base + (int64_t)k * kCT + threadIdx.x;
    c += (i < n && mask[i] == 0) ? 1 : 0;
  }
  c = __reduce_add_sync(0xffffffffu, c);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < kCT / 32; ++w) t += s_w[w];
    part_count[blockIdx.x] = t;
  }
}

// exclusive scan of the partition counts in one CTA (sequential over chunks
// of kCT); total into *n_keep
__global__ void __launch_bounds__(kCT) scan_counts_kernel(int64_t parts, int64_t* __restrict__ part_count,
                                                          int64_t* __restrict__ n_keep) {
  __shared__ int64_t s[kCT];
  __shared__ int64_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t c0 = 0; c0 < parts; c0 += kCT) {
    const int64_t i = c0 + threadIdx.x;
    const int64_t v = i < parts ? part_count[i] : 0;
    s[threadIdx.x] = v;
    __syncthreads();
    for (int o = 1; o < kCT; o <<= 1) {
      const int64_t y = threadIdx.x >= o ? s[threadIdx.x - o] : 0;
      __syncthreads();
      s[threadIdx.x] += y;
      __syncthreads();
    }
    if (i < parts) part_count[i] = carry + s[threadIdx.x] - v;
    __syncthreads();
    if (threadIdx.x == kCT - 1) carry += s[kCT - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_keep = carry;
}

// idx[k] = index of the k-th kept entry (order preserved)
__global__ void __launch_bounds__(kCT) write_keep_kernel(int64_t n, const uint8_t* __restrict__ mask,
                                                         const int64_t* __restrict__ part_start,
                                                         uint32_t* __restrict__ idx) {
  __shared__ int s_w[kCT / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t base = (int64_t)blockIdx.x * kCPart;
  int64_t off = part_start[blockIdx.x];
  for (int k = 0; k < kCItems; ++k) {
    const int64_t i = base + (int64_t)k * kCT + threadIdx.x;
    const bool keep = i < n && mask[i] == 0;
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_w[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kCT / 32; ++w) {
      before += w < warp ? s_w[w] : 0;
      total += s_w[w];
    }
    if (keep) idx[off + before + __popc(bal & ((1u << lane) - 1u))] = (uint32_t)i;
    off += total;
    __syncthreads();
  }
}

}  // namespace
}  // namespace gs

using namespace gs;

extern "C" gs_status gs_prune_mask(int64_t n, int32_t n_views, int32_t width, int32_t height,
                                   const uint32_t* vals, const int64_t* ranges,
                                   const int32_t* n_contrib, const float* importance,
                                   int64_t capacity, float tau, uint8_t* mask, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || capacity < 1 || !ranges || !n_contrib || (n > 0 && (!importance || !mask)))
    return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  cudaStream_t st = (cudaStream_t)stream;
  GS_CUDA(cudaMemsetAsync(mask, 0, (size_t)n, st));
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE;
  prune_tile_kernel<<<(unsigned)(n_views * T), kPT, 0, st>>>(n, tiles_x, T, width, height, vals,
                                                              ranges, n_contrib, importance,
                                                              capacity, tau, mask);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" size_t gs_compact_workspace_bytes(int64_t n) {
  return sizeof(int64_t) * (size_t)(div_up(n > 0 ? n : 1, kCPart) + 1);
}

extern "C" gs_status gs_compact_index(int64_t n, const uint8_t* mask, void* workspace,
                                      size_t ws_bytes, uint32_t* idx, int64_t* n_keep,
                                      void* stream) {
  if (n < 0 || n > (int64_t)0xFFFFFFFFll || !n_keep || !workspace ||
      ws_bytes < gs_compact_workspace_bytes(n) || (n > 0 && (!mask || !idx)))
    return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (n == 0) {
    GS_CUDA(cudaMemsetAsync(n_keep, 0, sizeof(int64_t), st));
    return GS_OK;
  }
  const int64_t parts = div_up(n, kCPart);
  int64_t* part = reinterpret_cast<int64_t*>(workspace);
  count_keep_kernel<<<(unsigned)parts, kCT, 0, st>>>(n, mask, part);
  GS_CHECK_LAUNCH();
  scan_counts_kernel<<<1, kCT, 0, st>>>(parts, part, n_keep);
  GS_CHECK_LAUNCH();
  write_keep_kernel<<<(unsigned)parts, kCT, 0, st>>>(n, mask, part, idx);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

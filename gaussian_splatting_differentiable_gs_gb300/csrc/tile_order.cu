// tile_order.cu -- gs_tile_order: the order in which the compositing CTAs
// start.
#include <stdint.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

// Launch order of the compositing CTAs: a tile's cost grows with its list
// length, which spans four orders of magnitude in clustered scenes, and CTAs
// start roughly in grid order, so a long list that starts late leaves the
// other SMs idle at the end of the kernel.  Longest lists first (the
// longest-processing-time-first rule of list scheduling) starts them while
// the short ones fill the gaps: order = tiles by descending
// floor(log2(list length)), empty tiles last, ties in tile order.  One CTA.
constexpr int kOrdThreads = 1024;
constexpr int kOrdWarps = kOrdThreads / 32;
constexpr int kOrdBuckets = 34;  // 0: empty; 1 + floor(log2 len) <= 33 (len < 2^33)

__device__ __forceinline__ uint32_t bucket_of_len(int64_t len) {
  return len > 0 ? (uint32_t)min(64 - __clzll((unsigned long long)len), kOrdBuckets - 1) : 0u;
}

__device__ __forceinline__ uint32_t order_bucket(const int64_t* ranges, int64_t f) {
  const longlong2 r = __ldg(reinterpret_cast<const longlong2*>(ranges) + f);
  return bucket_of_len(r.y - r.x);
}

constexpr int kOrdCache = 40960;  // tiles whose buckets are kept in shared memory

__global__ void __launch_bounds__(kOrdThreads) tile_order_kernel(int64_t n_flat,
                                                                 const int64_t* __restrict__ ranges,
                                                                 uint32_t* __restrict__ order) {
  __shared__ uint32_t s_start[kOrdBuckets];
  __shared__ uint32_t s_wcount[kOrdWarps][kOrdBuckets];
  __shared__ uint8_t s_bucket[kOrdCache];  // the first pass's buckets, read again by the second
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool cached = n_flat <= kOrdCache;
  if (tid < kOrdBuckets) s_start[tid] = 0;
  __syncthreads();
  constexpr int kBatch = 8;  // tiles per thread whose loads are in flight together
  for (int64_t base = 0; base < n_flat; base += kBatch * kOrdThreads) {
    uint32_t bk[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t f = base + (int64_t)u * kOrdThreads + tid;
      bk[u] = f < n_flat ? order_bucket(ranges, f) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t f = base + (int64_t)u * kOrdThreads + tid;
      if (f < n_flat) {
        if (cached) s_bucket[f] = (uint8_t)bk[u];
        atomicAdd(&s_start[bk[u]], 1u);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {  // exclusive starts, longest bucket first, empty tiles last
    uint32_t run = 0;
    for (int b = kOrdBuckets - 1; b >= 0; --b) {
      const uint32_t c = s_start[b];
      s_start[b] = run;
      run += c;
    }
  }
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t base = 0; base < n_flat; base += kOrdThreads) {
    const int64_t f = base + tid;
    const bool valid = f < n_flat;
    const uint32_t b = !valid ? (uint32_t)kOrdBuckets : cached ? (uint32_t)s_bucket[f]
                                                                : order_bucket(ranges, f);
    const uint32_t peers = __match_any_sync(0xffffffffu, b);
    for (int k = lane; k < kOrdBuckets; k += 32) s_wcount[warp][k] = 0;  // all 34 buckets
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) s_wcount[warp][b] = __popc(peers);
    __syncthreads();
    if (valid) {
      uint32_t pos = s_start[b] + __popc(peers & lt);
      for (int w = 0; w < warp; ++w) pos += s_wcount[w][b];
      order[pos] = (uint32_t)f;
    }
    __syncthreads();
    if (tid < kOrdBuckets) {
      uint32_t c = 0;
      for (int w = 0; w < kOrdWarps; ++w) c += s_wcount[w][tid];
      s_start[tid] += c;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace gs

using namespace gs;

extern "C" gs_status gs_tile_order(int64_t n_flat, const int64_t* ranges, uint32_t* order,
                                   void* stream) {
  if (n_flat < 0 || n_flat > (int64_t)0xFFFFFFFFll || (n_flat > 0 && (!ranges || !order)) ||
      !aligned16(ranges))
    return GS_ERR_INVALID_ARG;
  if (n_flat == 0) return GS_OK;
  tile_order_kernel<<<1, kOrdThreads, 0, (cudaStream_t)stream>>>(n_flat, ranges, order);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

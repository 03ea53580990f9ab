// binning.cu -- gs_bin_and_sort: per-tile depth-sorted intersection lists.
//
// "per-tile sorted lists of Gaussian-to-pixel intersections" ("AMD ROCm team
// open-sources distributed 3D Gaussian Splatting training", per-tile
// intersection bullet).  Stages, all in-house kernels:
//   1. single-pass exclusive scan of the per-row tile counts with decoupled
//      look-back (Merrill & Garland, cited in "A Scalable PyTorch Abstraction
//      for Multi-GPU Gaussian Splatting", references);
//   2-3. key emission, one thread per projected row, counting the digits of
//      every radix pass on the way (no separate histogram read of the keys);
//   4. stable LSD radix sort, 8-bit digits, one kernel per pass that ranks its
//      partition, resolves the partition's global digit offsets by decoupled
//      look-back and scatters ("onesweep"; radix sorting per Merrill &
//      Grimshaw, same reference list);
//   5. tile range extraction.
//
// Device waits: the look-backs are the only waits.  Each partition takes its
// index from an atomic ticket, so it only ever waits for partitions that are
// already running.  Every wait is bounded; when a bound is hit the partition
// publishes an error flag (successors propagate it), writes nothing, sets
// the workspace status word and returns.
#include <stddef.h>
#include <stdint.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;
constexpr int kScanPart = kScanThreads * kScanItems;   // rows per scan partition

constexpr int kSortThreads = 512;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortKpt = 8;                             // keys per thread
constexpr int kSortPart = kSortThreads * kSortKpt;      // keys per sort partition
constexpr int kRadix = 256;
constexpr int kMaxPasses = 8;

constexpr uint32_t kSpinLimit = 1u << 22;               // x ~100 ns sleep: >0.4 s

constexpr uint64_t kFlagAgg = 1, kFlagInc = 2, kFlagErr = 3;
constexpr unsigned int kErrCapacity = kWsErrCapacity;  // intersections exceed capacity

// Workspace header, at offset 0 of the caller's workspace.
struct WsHeader {
  unsigned long long total;        // intersections I (written by the scan)
  unsigned int error;              // sticky device status (0 = ok)
  unsigned int scan_ticket;
  unsigned int pass_ticket[kMaxPasses];
  unsigned int pad[52];
};
static_assert(sizeof(WsHeader) == 256, "header size");
static_assert(offsetof(WsHeader, error) == kWsStatusOffset, "status word offset");

struct WsLayout {
  size_t hist, digit_start, offsets, scan_status, sort_status, keys_alt, vals_alt, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t n_rows, int64_t capacity) {
  WsLayout L;
  size_t off = sizeof(WsHeader);
  L.hist = off;        off += align256(sizeof(uint32_t) * kMaxPasses * kRadix);
  L.digit_start = off; off += align256(sizeof(uint32_t) * kMaxPasses * kRadix);
  L.offsets = off;     off += align256(sizeof(int64_t) * (size_t)(n_rows > 0 ? n_rows : 1));
  L.scan_status = off; off += align256(sizeof(uint64_t) * (size_t)div_up(n_rows > 0 ? n_rows : 1, kScanPart));
  L.sort_status = off;
  off += align256(sizeof(uint64_t) * kRadix * (size_t)div_up(capacity > 0 ? capacity : 1, kSortPart));
  L.keys_alt = off;    off += align256(sizeof(uint64_t) * (size_t)(capacity > 0 ? capacity : 1));
  L.vals_alt = off;    off += align256(sizeof(uint32_t) * (size_t)(capacity > 0 ? capacity : 1));
  L.total = off;
  return L;
}

__device__ __forceinline__ uint64_t ld_volatile(const uint64_t* p) {
  return *reinterpret_cast<const volatile uint64_t*>(p);
}
__device__ __forceinline__ void st_volatile(uint64_t* p, uint64_t v) {
  *reinterpret_cast<volatile uint64_t*>(p) = v;
}

// ---------------------------------------------------------------------------
// 1. scan of tile counts -> inclusive int64 offsets, total I.
// Scan status word: value << 2 | flag.
__global__ void __launch_bounds__(kScanThreads) scan_tiles_kernel(
    int64_t n_rows, const int4* __restrict__ splat_tail, int64_t* __restrict__ offsets,
    uint64_t* __restrict__ status, WsHeader* __restrict__ hdr) {
  __shared__ int s_part;
  __shared__ long long s_warp[kScanThreads / 32];
  __shared__ long long s_prefix;
  __shared__ int s_err;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_part = (int)atomicAdd(&hdr->scan_ticket, 1u);
    s_err = 0;
  }
  __syncthreads();
  const int64_t part = s_part;
  const int64_t base = part * kScanPart + (int64_t)tid * kScanItems;
  int64_t v[kScanItems];
  long long sum = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t r = base + i;
    // the tile count is the 4th word of the record's last 16 bytes
    v[i] = r < n_rows ? (int64_t)splat_tail[3 * r + 2].w : 0;
    sum += v[i];
  }
  // block-wide inclusive scan of the per-thread sums
  long long incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < kScanThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kScanThreads / 32) s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const long long block_total = s_warp[kScanThreads / 32 - 1];
  const long long thread_excl = incl - sum + (warp > 0 ? s_warp[warp - 1] : 0);
  // decoupled look-back (thread 0)
  if (tid == 0) {
    long long prefix = 0;
    if (part == 0) {
      st_volatile(&status[0], ((uint64_t)block_total << 2) | kFlagInc);
    } else {
      st_volatile(&status[part], ((uint64_t)block_total << 2) | kFlagAgg);
      int64_t j = part - 1;
      bool err = false;
      while (j >= 0) {
        uint64_t s;
        uint32_t spins = 0;
        while (((s = ld_volatile(&status[j])) & 3u) == 0) {
          if (++spins > kSpinLimit) break;
          __nanosleep(100);
        }
        const uint64_t f = s & 3u;
        if (f == 0 || f == kFlagErr) { err = true; break; }
        prefix += (long long)(s >> 2);
        if (f == kFlagInc) break;
        --j;
      }
      if (err) {
        st_volatile(&status[part], kFlagErr);
        atomicOr(&hdr->error, 1u);
        s_err = 1;
      } else {
        __threadfence();
        st_volatile(&status[part], ((uint64_t)(prefix + block_total) << 2) | kFlagInc);
      }
    }
    s_prefix = prefix;
    if (!s_err && (part + 1) * kScanPart >= n_rows) hdr->total = (unsigned long long)(prefix + block_total);
  }
  __syncthreads();
  if (s_err) return;
  long long run = s_prefix + thread_excl;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    run += v[i];
    if (base + i < n_rows) offsets[base + i] = run;
  }
}

// ---------------------------------------------------------------------------
// 2. emission of (key, id) pairs, one thread per row, and the digit
//    histograms of every radix pass.  The low 32 key bits (depth) are the same
//    for all keys of a row, so their digits are counted once per row with the
//    row's tile count as weight; the tile digits are counted per key.
//    A row whose rectangle disagrees with its stored tile count (records not
//    produced by gs_project) writes nothing and raises the device-check bit, so
//    emission never leaves the row's scanned slot range.
__global__ void __launch_bounds__(256) emit_kernel(int64_t n, int64_t n_rows, int32_t tiles_x,
                                                   int32_t tiles_y, int64_t T, int32_t passes,
                                                   const float4* __restrict__ splats,
                                                   const int64_t* __restrict__ offsets,
                                                   uint64_t* __restrict__ keys,
                                                   uint32_t* __restrict__ vals,
                                                   uint32_t* __restrict__ hist,
                                                   WsHeader* __restrict__ hdr) {
  __shared__ uint32_t sh[kMaxPasses * kRadix];
  __shared__ unsigned int s_err;
  // the asynchronous path leaves the lists unbuilt when they exceed capacity
  // or when the scan's look-back gave up (its offsets are then incomplete);
  // the status word comes from earlier kernels: one load per CTA
  if (threadIdx.x == 0) s_err = hdr->error;
  for (int i = threadIdx.x; i < passes * kRadix; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  if (s_err & (1u | kErrCapacity)) return;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n_rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const float4 tail = splats[3 * r + 2];
    const int32_t tiles = __float_as_int(tail.w);
    if (tiles <= 0) continue;
    const float4 head = splats[3 * r];
    const int32_t radius = __float_as_int(tail.z);
    int32_t x0, x1, y0, y1;
    tile_rect(head.x, head.y, radius, tiles_x, tiles_y, x0, x1, y0, y1);
    if ((int64_t)(x1 - x0) * (y1 - y0) != tiles) {
      atomicOr(&hdr->error, 2u);
      continue;
    }
    const int64_t view = r / n;
    const uint32_t g = (uint32_t)(r - view * n);
    const uint32_t dbits = __float_as_uint(tail.y);
#pragma unroll
    for (int p = 0; p < 4; ++p) atomicAdd(&sh[p * kRadix + ((dbits >> (8 * p)) & 0xFF)], (uint32_t)tiles);
    int64_t o = offsets[r] - tiles;
    for (int32_t ty = y0; ty < y1; ++ty)
      for (int32_t tx = x0; tx < x1; ++tx) {
        const uint64_t flat = (uint64_t)(view * T + (int64_t)ty * tiles_x + tx);
        keys[o] = (flat << 32) | (uint64_t)dbits;
        vals[o] = g;
        ++o;
        for (int p = 4; p < passes; ++p)
          atomicAdd(&sh[p * kRadix + ((flat >> (8 * (p - 4))) & 0xFF)], 1u);
      }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < passes * kRadix; i += blockDim.x)
    if (sh[i]) atomicAdd(&hist[i], sh[i]);
}

// exclusive scan of each pass's 256 digit counts; one block per pass
__global__ void __launch_bounds__(kRadix) hist_scan_kernel(const uint32_t* __restrict__ hist,
                                                           uint32_t* __restrict__ digit_start) {
  __shared__ uint32_t s_w[kRadix / 32];
  const int p = blockIdx.x, d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const uint32_t c = hist[p * kRadix + d];
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  uint32_t add = 0;
  for (int w = 0; w < warp; ++w) add += s_w[w];
  digit_start[p * kRadix + d] = add + incl - c;
}

// ---------------------------------------------------------------------------
// 4. one stable radix pass (onesweep).  Sort status word:
//    value << 8 | tag << 2 | flag, tag = pass + 1 (stale entries of an earlier
//    pass read as not ready).
struct SortSmem {
  uint32_t warp_hist[kSortWarps][kRadix];
  uint32_t local_start[kRadix];
  unsigned long long global_base[kRadix];
  uint32_t scan_w[kSortWarps];
  int part;
  int err;
  int64_t count;
  uint64_t keys[kSortPart];
  uint32_t vals[kSortPart];
};

__global__ void __launch_bounds__(kSortThreads, 3) onesweep_kernel(
    int64_t count, int32_t pass, const uint64_t* __restrict__ keys_in,
    const uint32_t* __restrict__ vals_in, uint64_t* __restrict__ keys_out,
    uint32_t* __restrict__ vals_out, const uint32_t* __restrict__ digit_start,
    uint64_t* __restrict__ status, WsHeader* __restrict__ hdr) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmem& S = *reinterpret_cast<SortSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int shift = 8 * pass;
  const uint64_t tag = (uint64_t)(pass + 1) << 2;
  for (int i = tid; i < kSortWarps * kRadix; i += kSortThreads) (&S.warp_hist[0][0])[i] = 0;
  if (tid == 0) {
    S.part = (int)atomicAdd(&hdr->pass_ticket[pass], 1u);
    S.err = 0;
    // count < 0: the intersection count is the scan's total (asynchronous
    // path, grid sized by capacity; surplus partitions hold the highest
    // tickets, so no real partition looks back at them); -1 on overflow
    if (count < 0) S.count = (hdr->error & kErrCapacity) ? -1 : (int64_t)hdr->total;
  }
  __syncthreads();
  if (count < 0) {
    count = S.count;
    if (count < 0) return;
  }
  const int64_t part = S.part;
  const int64_t pbase = part * kSortPart;
  if (pbase >= count) return;
  const int64_t wbase = pbase + (int64_t)warp * 32 * kSortKpt;
  // load (warp-striped: item i of lane l is element wbase + 32 i + l) and rank
  uint64_t key[kSortKpt];
  uint32_t val[kSortKpt];
  uint32_t rank[kSortKpt];
#pragma unroll
  for (int i = 0; i < kSortKpt; ++i) {
    const int64_t idx = wbase + 32 * i + lane;
    const bool valid = idx < count;
    key[i] = valid ? keys_in[idx] : 0ull;
    val[i] = valid ? vals_in[idx] : 0u;
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < kSortKpt; ++i) {
    const int64_t idx = wbase + 32 * i + lane;
    const uint32_t d = idx < count ? (uint32_t)((key[i] >> shift) & 0xFF) : 256u;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    uint32_t basec = 0;
    if (d < 256u) basec = S.warp_hist[warp][d];
    __syncwarp();
    if (d < 256u && lane == __ffs(peers) - 1) S.warp_hist[warp][d] = basec + __popc(peers);
    __syncwarp();
    rank[i] = basec + __popc(peers & lt_mask);
  }
  __syncthreads();
  // per digit (threads 0..255, i.e. warps 0..7): exclusive prefix over warps,
  // partition count, aggregate published first so successors can proceed
  const bool dthread = tid < kRadix;
  const int d = tid;
  uint32_t my_count = 0, incl = 0;
  if (dthread) {
    uint32_t run = 0;
#pragma unroll
    for (int w = 0; w < kSortWarps; ++w) {
      const uint32_t c = S.warp_hist[w][d];
      S.warp_hist[w][d] = run;
      run += c;
    }
    my_count = run;
    if (part == 0)
      st_volatile(&status[d], ((uint64_t)my_count << 8) | tag | kFlagInc);
    else
      st_volatile(&status[part * kRadix + d], ((uint64_t)my_count << 8) | tag | kFlagAgg);
    incl = my_count;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) S.scan_w[warp] = incl;
  }
  __syncthreads();
  if (dthread) {
    // exclusive scan of the counts over digits -> local start of each digit
    uint32_t add = 0;
    for (int w = 0; w < warp; ++w) add += S.scan_w[w];
    S.local_start[d] = add + incl - my_count;
    // look back for this digit
    unsigned long long excl = 0;
    if (part > 0) {
      int64_t j = part - 1;
      bool err = false;
      while (j >= 0) {
        uint64_t s;
        uint32_t spins = 0;
        for (;;) {
          s = ld_volatile(&status[j * kRadix + d]);
          const uint64_t f = s & 3u;
          if (f == kFlagErr) break;
          if (f != 0 && (s & 0xFCu) == tag) break;
          if (++spins > kSpinLimit) { s = kFlagErr; break; }
          __nanosleep(100);
        }
        const uint64_t f = s & 3u;
        if (f == kFlagErr) { err = true; break; }
        excl += (unsigned long long)(s >> 8);
        if (f == kFlagInc) break;
        --j;
      }
      if (err) {
        st_volatile(&status[part * kRadix + d], tag | kFlagErr);
        atomicOr(&hdr->error, 1u);
        S.err = 1;
      } else {
        st_volatile(&status[part * kRadix + d], ((uint64_t)(excl + my_count) << 8) | tag | kFlagInc);
      }
    }
    S.global_base[d] = (unsigned long long)digit_start[pass * kRadix + d] + excl;
  }
  __syncthreads();
  if (S.err) return;
  // place the partition in smem in sorted (digit-major, stable) order
#pragma unroll
  for (int i = 0; i < kSortKpt; ++i) {
    const int64_t idx = wbase + 32 * i + lane;
    if (idx < count) {
      const uint32_t dd = (uint32_t)((key[i] >> shift) & 0xFF);
      const uint32_t pos = S.local_start[dd] + S.warp_hist[warp][dd] + rank[i];
      S.keys[pos] = key[i];
      S.vals[pos] = val[i];
    }
  }
  __syncthreads();
  const int64_t n_here = count - pbase < kSortPart ? count - pbase : kSortPart;
  for (int j = tid; j < n_here; j += kSortThreads) {
    const uint64_t k = S.keys[j];
    const uint32_t dd = (uint32_t)((k >> shift) & 0xFF);
    const unsigned long long gpos = S.global_base[dd] + (unsigned long long)(j - S.local_start[dd]);
    if (gpos < (unsigned long long)count) {
      keys_out[gpos] = k;
      vals_out[gpos] = S.vals[j];
    }
  }
}

// ---------------------------------------------------------------------------
// 5. [first, last + 1) of each (view, tile) in the sorted keys.
__global__ void __launch_bounds__(256) ranges_kernel(int64_t count, uint64_t n_flat,
                                                     const uint64_t* __restrict__ keys,
                                                     int64_t* __restrict__ ranges,
                                                     const WsHeader* __restrict__ hdr) {
  if (count < 0) {  // asynchronous path: the scan's total, nothing on overflow
    __shared__ int64_t s_count;
    if (threadIdx.x == 0) s_count = (hdr->error & kErrCapacity) ? -1 : (int64_t)hdr->total;
    __syncthreads();
    count = s_count;
    if (count < 0) return;
  }
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const uint64_t f = keys[i] >> 32;
  if (f >= n_flat) return;
  if (i == 0 || (keys[i - 1] >> 32) != f) ranges[2 * f] = i;
  if (i == count - 1 || (keys[i + 1] >> 32) != f) ranges[2 * f + 1] = i + 1;
}

// ---------------------------------------------------------------------------
// Morton order of the Gaussians ("A Scalable PyTorch Abstraction for
// Multi-GPU Gaussian Splatting", references: Morton order).  Each mean is
// quantised to 21 bits per axis inside the means' bounding box,
//   q = clamp(floor((x - lo) * (2^21 / (hi - lo))), 0, 2^21 - 1)   (fp32),
// and the bits are interleaved, bit i of q_x at code bit 3i, of q_y at 3i+1,
// of q_z at 3i+2.  A stable radix sort of (code, index) gives the order.
constexpr int kMortonPasses = 8;  // 63 code bits

// float -> uint32 with the same order (atomic min / max of floats)
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// box[0..2] = ordered bits of the minimum mean x, y, z, box[3..5] of the
// maximum (initialised to all ones / zero)
__global__ void __launch_bounds__(256) bbox_kernel(int64_t n, const float* __restrict__ params,
                                                   uint32_t* __restrict__ box) {
  uint32_t lo[3] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu}, hi[3] = {0u, 0u, 0u};
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const uint32_t o = ordered_bits(params[a * n + i]);
      lo[a] = min(lo[a], o);
      hi[a] = max(hi[a], o);
    }
  }
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    lo[a] = __reduce_min_sync(0xffffffffu, lo[a]);
    hi[a] = __reduce_max_sync(0xffffffffu, hi[a]);
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      atomicMin(&box[a], lo[a]);
      atomicMax(&box[3 + a], hi[a]);
    }
  }
}

// The low 21 bits of v moved to bits 0, 3, 6, ..., 60 (bit spreading by
// shifts and masks).
__device__ __forceinline__ uint64_t spread3(uint32_t v) {
  uint64_t x = v & 0x1FFFFFu;
  x = (x | x << 32) & 0x001F00000000FFFFull;
  x = (x | x << 16) & 0x001F0000FF0000FFull;
  x = (x | x << 8) & 0x100F00F00F00F00Full;
  x = (x | x << 4) & 0x10C30C30C30C30C3ull;
  x = (x | x << 2) & 0x1249249249249249ull;
  return x;
}

__device__ __forceinline__ uint32_t quantize21(float v, float lo, float s) {
  const float t = floorf(__fmul_rn(__fsub_rn(v, lo), s));
  return (uint32_t)fminf(fmaxf(t, 0.f), 2097151.f);  // NaN -> 0
}

// keys[i] = Morton code of Gaussian i, vals[i] = i, and the digit histograms
// of the eight radix passes
__global__ void __launch_bounds__(256) morton_kernel(int64_t n, const float* __restrict__ params,
                                                     const uint32_t* __restrict__ box,
                                                     uint64_t* __restrict__ keys,
                                                     uint32_t* __restrict__ vals,
                                                     uint32_t* __restrict__ hist) {
  __shared__ uint32_t sh[kMortonPasses * kRadix];
  for (int i = threadIdx.x; i < kMortonPasses * kRadix; i += blockDim.x) sh[i] = 0;
  float lo[3], sc[3];
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    lo[a] = from_ordered(box[a]);
    const float ext = __fsub_rn(from_ordered(box[3 + a]), lo[a]);
    sc[a] = ext > 0.f ? __fdiv_rn(2097152.f, ext) : 0.f;
  }
  __syncthreads();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t code = spread3(quantize21(params[i], lo[0], sc[0])) |
                          spread3(quantize21(params[n + i], lo[1], sc[1])) << 1 |
                          spread3(quantize21(params[2 * n + i], lo[2], sc[2])) << 2;
    keys[i] = code;
    vals[i] = (uint32_t)i;
#pragma unroll
    for (int p = 0; p < kMortonPasses; ++p) atomicAdd(&sh[p * kRadix + ((code >> (8 * p)) & 0xFF)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kMortonPasses * kRadix; i += blockDim.x)
    if (sh[i]) atomicAdd(&hist[i], sh[i]);
}

// dst[r][i] = src[r][idx[i]] for r < rows, i < n_dst (idx clamped into range)
__global__ void __launch_bounds__(256) gather_columns_kernel(int64_t rows, int64_t n_src,
                                                             int64_t n_dst,
                                                             const float* __restrict__ src,
                                                             const uint32_t* __restrict__ idx,
                                                             float* __restrict__ dst) {
  const int64_t total = rows * n_dst;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / n_dst, i = t - r * n_dst;
    const uint32_t j = min(__ldg(idx + i), (uint32_t)(n_src - 1));
    dst[t] = __ldg(src + r * n_src + j);
  }
}

// Publishes the intersection count and sets the capacity bit of the status
// word when it exceeds capacity, clears it otherwise (the bit describes the
// latest call; the timeout and device-check bits stay until read).
__global__ void check_capacity_kernel(WsHeader* __restrict__ hdr, int64_t capacity,
                                      int64_t* __restrict__ n_isect) {
  const unsigned long long total = *reinterpret_cast<volatile unsigned long long*>(&hdr->total);
  if (n_isect) *n_isect = (int64_t)total;
  if ((int64_t)total > capacity) atomicOr(&hdr->error, kErrCapacity);
  else atomicAnd(&hdr->error, ~kErrCapacity);
}

// The onesweep kernel's shared-memory attribute, set once per device (the
// asynchronous path is captured into graphs after an eager call).
cudaError_t ensure_sort_attr() {
  static bool done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(onesweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sizeof(SortSmem));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

int bit_length(uint64_t v) {
  int b = 0;
  while (v) { ++b; v >>= 1; }
  return b;
}

}  // namespace
}  // namespace gs

using namespace gs;

extern "C" size_t gs_bin_workspace_bytes(int64_t n_rows, int64_t capacity) {
  if (n_rows < 0 || capacity < 0) return 0;
  return ws_layout(n_rows, capacity).total;
}

extern "C" int32_t gs_key_bits(int32_t n_views, int32_t width, int32_t height) {
  if (n_views < 1 || width < 1 || height < 1) return 0;
  const int64_t flat = (int64_t)n_views * tiles_per_view(width, height);
  const int b = bit_length((uint64_t)(flat - 1));
  return 32 + (b > 0 ? b : 1);
}

extern "C" gs_status gs_selftest_lookback_timeout(void* workspace, size_t ws_bytes, void* stream) {
  // One scan partition is launched with ticket 1, so it looks back at
  // partition 0, which never runs: its bounded wait must run out, flag the
  // error and return.  Reads and writes no row data (zero rows).
  const WsLayout L = ws_layout(1, 1);
  if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  uint64_t* scan_status = reinterpret_cast<uint64_t*>(ws + L.scan_status);
  GS_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st));
  GS_CUDA(cudaMemsetAsync(scan_status, 0, sizeof(uint64_t) * 2, st));
  const unsigned one = 1;
  GS_CUDA(cudaMemcpyAsync(&hdr->scan_ticket, &one, sizeof(one), cudaMemcpyHostToDevice, st));
  scan_tiles_kernel<<<1, kScanThreads, 0, st>>>(0, nullptr, reinterpret_cast<int64_t*>(ws + L.offsets),
                                               scan_status, hdr);
  GS_CHECK_LAUNCH();
  return gs_workspace_status(workspace, stream);
}

extern "C" gs_status gs_workspace_status(void* workspace, void* stream) {
  if (!workspace) return GS_ERR_INVALID_ARG;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(workspace);
  unsigned int err = 0;
  GS_CUDA(cudaMemcpyAsync(&err, &hdr->error, sizeof(err), cudaMemcpyDeviceToHost,
                          (cudaStream_t)stream));
  GS_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  if (err) {
    GS_CUDA(cudaMemsetAsync(&hdr->error, 0, sizeof(unsigned int), (cudaStream_t)stream));
    if (err & 1u) return GS_ERR_TIMEOUT;
    return (err & kErrCapacity) ? GS_ERR_CAPACITY : GS_ERR_DEVICE_CHECK;
  }
  return GS_OK;
}

extern "C" gs_status gs_bin_and_sort(int64_t n, int32_t n_views, const gs_splat* splats,
                                     int32_t width, int32_t height, void* workspace,
                                     size_t ws_bytes, int64_t capacity, uint64_t* keys,
                                     uint32_t* vals, int64_t* ranges, int64_t* n_isect,
                                     void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || capacity < 0 || capacity > (int64_t)0xFFFFFFFFll || !n_isect || !workspace)
    return GS_ERR_INVALID_ARG;
  const int64_t n_rows = n * n_views;
  const WsLayout L = ws_layout(n_rows, capacity);
  if (ws_bytes < L.total || !aligned16(workspace)) return GS_ERR_INVALID_ARG;
  if (!ranges || (n_rows > 0 && (!splats || !aligned16(splats))) ||
      (capacity > 0 && (!keys || !vals)))
    return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint32_t* digit_start = reinterpret_cast<uint32_t*>(ws + L.digit_start);
  int64_t* offsets = reinterpret_cast<int64_t*>(ws + L.offsets);
  uint64_t* scan_status = reinterpret_cast<uint64_t*>(ws + L.scan_status);
  uint64_t* sort_status = reinterpret_cast<uint64_t*>(ws + L.sort_status);
  uint64_t* keys_alt = reinterpret_cast<uint64_t*>(ws + L.keys_alt);
  uint32_t* vals_alt = reinterpret_cast<uint32_t*>(ws + L.vals_alt);
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE, tiles_y = (height + GS_TILE - 1) / GS_TILE;
  if (n_views * T > (int64_t)0xFFFFFFFFll) return GS_ERR_INVALID_ARG;  // flat index in 32 key bits

  // 1. scan (tickets, total and histograms reset; the status word is kept)
  GS_CUDA(cudaMemsetAsync(&hdr->scan_ticket, 0, sizeof(WsHeader) - offsetof(WsHeader, scan_ticket), st));
  GS_CUDA(cudaMemsetAsync(&hdr->total, 0, sizeof(hdr->total), st));
  GS_CUDA(cudaMemsetAsync(hist, 0, sizeof(uint32_t) * kMaxPasses * kRadix, st));
  const int64_t scan_parts = div_up(n_rows, kScanPart);
  if (n_rows > 0) {
    GS_CUDA(cudaMemsetAsync(scan_status, 0, sizeof(uint64_t) * (size_t)scan_parts, st));
    scan_tiles_kernel<<<(unsigned)scan_parts, kScanThreads, 0, st>>>(
        n_rows, reinterpret_cast<const int4*>(splats), offsets, scan_status, hdr);
    GS_CHECK_LAUNCH();
  }
  struct { unsigned long long total; unsigned int error; unsigned int pad; } h{};
  GS_CUDA(cudaMemcpyAsync(&h, hdr, 16, cudaMemcpyDeviceToHost, st));
  GS_CUDA(cudaStreamSynchronize(st));
  if (h.error & ~kErrCapacity) {  // a capacity bit can only be left by an asynchronous call
    GS_CUDA(cudaMemsetAsync(&hdr->error, 0, sizeof(unsigned int), st));
    return (h.error & 1u) ? GS_ERR_TIMEOUT : GS_ERR_DEVICE_CHECK;
  }
  const int64_t I = (int64_t)h.total;
  *n_isect = I;
  if (I > capacity) return GS_ERR_CAPACITY;
  check_capacity_kernel<<<1, 1, 0, st>>>(hdr, capacity, nullptr);  // clears the bit
  GS_CHECK_LAUNCH();
  GS_CUDA(cudaMemsetAsync(ranges, 0, sizeof(int64_t) * 2 * (size_t)(n_views * T), st));
  if (I == 0) return GS_OK;

  const int passes = (gs_key_bits(n_views, width, height) + 7) / 8;
  uint64_t* k_a = (passes % 2 == 0) ? keys : keys_alt;
  uint32_t* v_a = (passes % 2 == 0) ? vals : vals_alt;
  uint64_t* k_b = (passes % 2 == 0) ? keys_alt : keys;
  uint32_t* v_b = (passes % 2 == 0) ? vals_alt : vals;
  // 2-3. emission into the buffer that ends up holding the sorted result, with
  //      the digit histograms of every pass
  int dev = 0, sms = 0;
  GS_CUDA(cudaGetDevice(&dev));
  GS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t emit_blocks = div_up(n_rows, 256) < 8 * sms ? div_up(n_rows, 256) : 8 * sms;
  emit_kernel<<<(unsigned)emit_blocks, 256, 0, st>>>(n, n_rows, tiles_x, tiles_y, T, passes,
                                                              reinterpret_cast<const float4*>(splats),
                                                              offsets, k_a, v_a, hist, hdr);
  GS_CHECK_LAUNCH();
  hist_scan_kernel<<<passes, kRadix, 0, st>>>(hist, digit_start);
  GS_CHECK_LAUNCH();
  // 4. radix passes
  const int64_t sort_parts = div_up(I, kSortPart);
  GS_CUDA(cudaMemsetAsync(sort_status, 0, sizeof(uint64_t) * kRadix * (size_t)sort_parts, st));
  const size_t smem = sizeof(SortSmem);
  GS_CUDA(ensure_sort_attr());
  for (int p = 0; p < passes; ++p) {
    onesweep_kernel<<<(unsigned)sort_parts, kSortThreads, smem, st>>>(
        I, p, k_a, v_a, k_b, v_b, digit_start, sort_status, hdr);
    GS_CHECK_LAUNCH();
    uint64_t* tk = k_a; k_a = k_b; k_b = tk;
    uint32_t* tv = v_a; v_a = v_b; v_b = tv;
  }
  // 5. ranges
  ranges_kernel<<<(unsigned)div_up(I, 256), 256, 0, st>>>(I, (uint64_t)(n_views * T), keys, ranges,
                                                          hdr);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

// ---------------------------------------------------------------------------
// Morton order entry points

static size_t morton_ws_bytes(int64_t n) {
  return ws_layout(0, n).total + align256(sizeof(uint64_t) * (size_t)(n > 0 ? n : 1));
}

extern "C" size_t gs_morton_workspace_bytes(int64_t n) { return morton_ws_bytes(n); }

extern "C" gs_status gs_morton_order(int64_t n, const float* params, void* workspace,
                                     size_t ws_bytes, uint32_t* perm, void* stream) {
  if (n < 0 || n > (int64_t)0xFFFFFFFFll || !workspace || !aligned16(workspace) ||
      ws_bytes < morton_ws_bytes(n) || (n > 0 && (!params || !perm)))
    return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(0, n);
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint32_t* digit_start = reinterpret_cast<uint32_t*>(ws + L.digit_start);
  uint64_t* sort_status = reinterpret_cast<uint64_t*>(ws + L.sort_status);
  uint64_t* keys_b = reinterpret_cast<uint64_t*>(ws + L.keys_alt);
  uint32_t* vals_b = reinterpret_cast<uint32_t*>(ws + L.vals_alt);
  uint64_t* keys_a = reinterpret_cast<uint64_t*>(ws + L.total);
  uint32_t* box = hdr->pad;  // six words of the header's spare space
  GS_CUDA(cudaMemsetAsync(&hdr->scan_ticket, 0, sizeof(WsHeader) - offsetof(WsHeader, scan_ticket), st));
  GS_CUDA(cudaMemsetAsync(box, 0xFF, 3 * sizeof(uint32_t), st));
  GS_CUDA(cudaMemsetAsync(hist, 0, sizeof(uint32_t) * kMaxPasses * kRadix, st));
  int dev = 0, sms = 0;
  GS_CUDA(cudaGetDevice(&dev));
  GS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t blocks = div_up(n, 256) < 8 * sms ? div_up(n, 256) : 8 * sms;
  bbox_kernel<<<(unsigned)blocks, 256, 0, st>>>(n, params, box);
  GS_CHECK_LAUNCH();
  // eight passes (even): emission into (keys_a, perm) leaves the result there
  morton_kernel<<<(unsigned)blocks, 256, 0, st>>>(n, params, box, keys_a, perm, hist);
  GS_CHECK_LAUNCH();
  hist_scan_kernel<<<kMortonPasses, kRadix, 0, st>>>(hist, digit_start);
  GS_CHECK_LAUNCH();
  const int64_t sort_parts = div_up(n, kSortPart);
  GS_CUDA(cudaMemsetAsync(sort_status, 0, sizeof(uint64_t) * kRadix * (size_t)sort_parts, st));
  const size_t smem = sizeof(SortSmem);
  GS_CUDA(ensure_sort_attr());
  uint64_t* k_in = keys_a;
  uint32_t* v_in = perm;
  uint64_t* k_out = keys_b;
  uint32_t* v_out = vals_b;
  for (int p = 0; p < kMortonPasses; ++p) {
    onesweep_kernel<<<(unsigned)sort_parts, kSortThreads, smem, st>>>(
        n, p, k_in, v_in, k_out, v_out, digit_start, sort_status, hdr);
    GS_CHECK_LAUNCH();
    uint64_t* tk = k_in; k_in = k_out; k_out = tk;
    uint32_t* tv = v_in; v_in = v_out; v_out = tv;
  }
  return GS_OK;
}

extern "C" gs_status gs_gather_columns(int64_t rows, int64_t n_src, int64_t n_dst,
                                       const float* src, const uint32_t* idx, float* dst,
                                       void* stream) {
  if (rows < 0 || n_src < 0 || n_dst < 0 || n_src > (int64_t)0xFFFFFFFFll ||
      (n_dst > 0 && n_src == 0) ||
      (rows > 0 && n_dst > 0 && (!src || !idx || !dst || src == dst)))
    return GS_ERR_INVALID_ARG;
  if (rows == 0 || n_dst == 0) return GS_OK;
  int dev = 0, sms = 0;
  GS_CUDA(cudaGetDevice(&dev));
  GS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t blocks = div_up(rows * n_dst, 256) < 16 * sms ? div_up(rows * n_dst, 256) : 16 * sms;
  gather_columns_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(rows, n_src, n_dst, src,
                                                                            idx, dst);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

// ---------------------------------------------------------------------------
// gs_bin_and_sort without a host synchronisation (graph-capturable): launch
// shapes follow `capacity`, the kernels read the intersection count from the
// workspace, and an overflow is reported through the workspace status word.
extern "C" gs_status gs_bin_and_sort_async(int64_t n, int32_t n_views, const gs_splat* splats,
                                           int32_t width, int32_t height, void* workspace,
                                           size_t ws_bytes, int64_t capacity, uint64_t* keys,
                                           uint32_t* vals, int64_t* ranges, int64_t* n_isect,
                                           void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || capacity < 1 || capacity > (int64_t)0xFFFFFFFFll || !workspace || !n_isect)
    return GS_ERR_INVALID_ARG;
  const int64_t n_rows = n * n_views;
  const WsLayout L = ws_layout(n_rows, capacity);
  if (ws_bytes < L.total || !aligned16(workspace) || !ranges || !keys || !vals ||
      (n_rows > 0 && (!splats || !aligned16(splats))))
    return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint32_t* digit_start = reinterpret_cast<uint32_t*>(ws + L.digit_start);
  int64_t* offsets = reinterpret_cast<int64_t*>(ws + L.offsets);
  uint64_t* scan_status = reinterpret_cast<uint64_t*>(ws + L.scan_status);
  uint64_t* sort_status = reinterpret_cast<uint64_t*>(ws + L.sort_status);
  uint64_t* keys_alt = reinterpret_cast<uint64_t*>(ws + L.keys_alt);
  uint32_t* vals_alt = reinterpret_cast<uint32_t*>(ws + L.vals_alt);
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE, tiles_y = (height + GS_TILE - 1) / GS_TILE;
  if (n_views * T > (int64_t)0xFFFFFFFFll) return GS_ERR_INVALID_ARG;
  const int64_t n_flat = n_views * T;

  GS_CUDA(cudaMemsetAsync(&hdr->scan_ticket, 0, sizeof(WsHeader) - offsetof(WsHeader, scan_ticket), st));
  GS_CUDA(cudaMemsetAsync(&hdr->total, 0, sizeof(hdr->total), st));
  GS_CUDA(cudaMemsetAsync(hist, 0, sizeof(uint32_t) * kMaxPasses * kRadix, st));
  GS_CUDA(cudaMemsetAsync(ranges, 0, sizeof(int64_t) * 2 * (size_t)n_flat, st));
  if (n_rows > 0) {
    const int64_t scan_parts = div_up(n_rows, kScanPart);
    GS_CUDA(cudaMemsetAsync(scan_status, 0, sizeof(uint64_t) * (size_t)scan_parts, st));
    scan_tiles_kernel<<<(unsigned)scan_parts, kScanThreads, 0, st>>>(
        n_rows, reinterpret_cast<const int4*>(splats), offsets, scan_status, hdr);
    GS_CHECK_LAUNCH();
  }
  check_capacity_kernel<<<1, 1, 0, st>>>(hdr, capacity, n_isect);
  GS_CHECK_LAUNCH();
  if (n_rows == 0) return GS_OK;
  const int passes = (gs_key_bits(n_views, width, height) + 7) / 8;
  uint64_t* k_a = (passes % 2 == 0) ? keys : keys_alt;
  uint32_t* v_a = (passes % 2 == 0) ? vals : vals_alt;
  uint64_t* k_b = (passes % 2 == 0) ? keys_alt : keys;
  uint32_t* v_b = (passes % 2 == 0) ? vals_alt : vals;
  int dev = 0, sms = 0;
  GS_CUDA(cudaGetDevice(&dev));
  GS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t emit_blocks = div_up(n_rows, 256) < 8 * sms ? div_up(n_rows, 256) : 8 * sms;
  emit_kernel<<<(unsigned)emit_blocks, 256, 0, st>>>(n, n_rows, tiles_x, tiles_y, T, passes,
                                                     reinterpret_cast<const float4*>(splats),
                                                     offsets, k_a, v_a, hist, hdr);
  GS_CHECK_LAUNCH();
  hist_scan_kernel<<<passes, kRadix, 0, st>>>(hist, digit_start);
  GS_CHECK_LAUNCH();
  const int64_t sort_parts = div_up(capacity, kSortPart);
  GS_CUDA(cudaMemsetAsync(sort_status, 0, sizeof(uint64_t) * kRadix * (size_t)sort_parts, st));
  const size_t smem = sizeof(SortSmem);
  GS_CUDA(ensure_sort_attr());
  for (int p = 0; p < passes; ++p) {
    onesweep_kernel<<<(unsigned)sort_parts, kSortThreads, smem, st>>>(
        -1, p, k_a, v_a, k_b, v_b, digit_start, sort_status, hdr);
    GS_CHECK_LAUNCH();
    uint64_t* tk = k_a; k_a = k_b; k_b = tk;
    uint32_t* tv = v_a; v_a = v_b; v_b = tv;
  }
  ranges_kernel<<<(unsigned)div_up(capacity, 256), 256, 0, st>>>(-1, (uint64_t)n_flat, keys, ranges,
                                                                hdr);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

// binning.cu -- gs_bin_and_sort: per-tile depth-sorted intersection lists.
//
// "per-tile sorted lists of Gaussian-to-pixel intersections" ("AMD ROCm team
// open-sources distributed 3D Gaussian Splatting training", per-tile
// intersection bullet), ordered by (view, tile, depth) with equal depths in
// Gaussian order.  The depth order is a property of a projected row, not of
// its intersections, so the rows are sorted by depth once and their
// intersections emitted in that order; a stable sort on the tile index alone
// then finishes the lists.  Stages, all in-house kernels:
//   1. compaction of the visible rows (rows in order: a decoupled look-back
//      over their counts, Merrill & Garland, cited in "A Scalable PyTorch
//      Abstraction for Multi-GPU Gaussian Splatting", references), with the
//      intersection total and the digit histograms of the depth passes;
//   2. stable LSD radix sort of the rows on their 32 depth bits, 8-bit
//      digits, one kernel per pass that ranks its partition, resolves the
//      partition's global digit offsets by decoupled look-back and scatters
//      ("onesweep"; radix sorting per Merrill & Grimshaw, same reference
//      list); an element is one 64-bit word, sort digits in the high half,
//      the row index (view * n + g) in the low half;
//   3. emission of each row's tiles in depth order (a second look-back scan
//      gives the offsets; a partition's outputs are spread evenly over its
//      threads), with the digit histograms of the tile passes; an
//      intersection carries its row's position in depth order, whose
//      (depth, Gaussian id) word the emission also writes, in depth order;
//   4. the same radix passes on the tile index (ceil(tile bits / 8) passes);
//      the last one writes the final (tile << 32 | depth) keys and ids;
//   5. tile ranges, marked by the last tile pass.
// The result is the stable sort of (tile << 32 | depth) keys emitted in row
// order, bit for bit.
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

constexpr int kCompThreads = 256;
constexpr int kCompWarps = kCompThreads / 32;
constexpr int kCompItems = 8;                           // rows per thread and chunk (warp-striped)
constexpr int kCompChunk = kCompThreads * kCompItems;   // rows per chunk
// chunks per compaction partition: 1 below 2^21 rows (enough partitions to
// fill the GPU), 4 up to 2^27, 8 beyond (fewer partitions shorten the
// look-back chain, which sets the pace of a call over hundreds of millions of
// mostly culled rows)
inline int comp_chunks(int64_t n_rows) {
  return n_rows < ((int64_t)1 << 21) ? 1 : (n_rows < ((int64_t)1 << 27) ? 4 : 8);
}

constexpr int kEmitThreads = 512;
constexpr int kEmitItems = 4;
constexpr int kEmitPart = kEmitThreads * kEmitItems;    // sorted rows per emission partition
// emission in balanced chunks of kEmitChunk intersections per CTA, chosen
// when rows average at least kEmitChunkMinTiles tiles (else one CTA per
// partition of kEmitPart rows: cheaper when rows are small, e.g. 2.5 tiles a
// row on the 1080p ring scene, 0.21 against 0.35 ms; slower when they are
// large, 168 tiles a row on the 4K cluster scene, 16.8 against 11.5 ms)
constexpr int kEmitChunk = 2048;
constexpr int64_t kEmitChunkMinTiles = 8;

constexpr int kSortThreads = 512;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortKpt = 8;                             // keys per thread
constexpr int kSortPart = kSortThreads * kSortKpt;      // keys per sort partition
// the binning's radix passes: the same partition, over fewer, fuller threads
// (one thread per digit in the digit phases)
constexpr int kPassThreads = 512;
constexpr int kPassWarps = kPassThreads / 32;
constexpr int kPassKpt = kSortPart / kPassThreads;       // keys per thread
constexpr int kPassMinBlocks = 3;
static_assert(kPassThreads * kPassKpt == kSortPart && kPassThreads >= 256, "pass shape");
constexpr int kRadix = 256;
constexpr int kMaxPasses = 8;
constexpr int kDepthPasses = 4;                         // 32 depth bits

constexpr uint32_t kSpinLimit = 1u << 22;               // x ~100 ns sleep: >0.4 s

constexpr uint64_t kFlagAgg = 1, kFlagInc = 2, kFlagErr = 3;
constexpr unsigned int kErrCapacity = kWsErrCapacity;  // intersections exceed capacity
constexpr unsigned int kErrStop = 1u | kErrCapacity;    // later stages do nothing

// Workspace header, at offset 0 of the caller's workspace.
struct WsHeader {
  unsigned long long total;        // intersections I
  unsigned int error;              // sticky device status (0 = ok)
  unsigned int scan_ticket;        // compaction partitions
  unsigned long long rows;         // visible rows R
  unsigned int emit_ticket;        // emission partitions
  unsigned int pass_ticket[kMaxPasses];
  unsigned int pad[49];
};
static_assert(sizeof(WsHeader) == 256, "header size");
static_assert(offsetof(WsHeader, error) == kWsStatusOffset, "status word offset");
static_assert(offsetof(WsHeader, rows) == 16, "counts in the first 24 bytes");

// Workspace layout.  row_rect[r] (r = view * n + g, written for the visible
// rows only) = first flat tile | width << 32 | height << 48 of the row's tile
// rectangle; row_d[s] (s < R: the row's position in depth order) = depth bits
// << 32 | Gaussian id, written at emission and gathered by the last tile pass
// (an intersection carries s, so the gathers of a partition, which is in
// depth order within each tile digit, fall in a narrow window of row_d).
// tmp: one capacity-sized key buffer; the row sort ping-pongs between it and
// the caller's key buffer (R <= I <= capacity), as do the tile passes.
struct WsLayout {
  size_t hist, digit_start, scan_status, emit_status, sort_status, row_d, row_rect, erow, chunk_row,
      tmp, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int64_t n_rows, int64_t capacity) {
  const int64_t r = n_rows > 0 ? n_rows : 1, c = capacity > 0 ? capacity : 1;
  const int64_t sort_parts = div_up(r, kSortPart) > div_up(c, kSortPart) ? div_up(r, kSortPart)
                                                                         : div_up(c, kSortPart);
  WsLayout L;
  size_t off = sizeof(WsHeader);
  L.hist = off;        off += align256(sizeof(uint32_t) * kMaxPasses * kRadix);
  L.digit_start = off; off += align256(sizeof(uint32_t) * kMaxPasses * kRadix);
  L.scan_status = off; off += align256(sizeof(uint64_t) * (size_t)div_up(r, kCompChunk));
  L.emit_status = off; off += align256(sizeof(uint64_t) * (size_t)div_up(r, kEmitPart));
  L.sort_status = off; off += align256(sizeof(uint64_t) * kRadix * (size_t)sort_parts);
  L.row_d = off;       off += align256(sizeof(uint64_t) * (size_t)r);
  L.row_rect = off;    off += align256(sizeof(uint64_t) * (size_t)r);
  L.erow = off;        off += align256(sizeof(uint4) * (size_t)r);
  L.chunk_row = off;   off += align256(sizeof(uint32_t) * (size_t)(div_up(c, kEmitChunk) + 1));
  L.tmp = off;         off += align256(sizeof(uint64_t) * (size_t)c);
  L.total = off;
  return L;
}

__device__ __forceinline__ uint64_t ld_volatile(const uint64_t* p) {
  return *reinterpret_cast<const volatile uint64_t*>(p);
}
__device__ __forceinline__ void st_volatile(uint64_t* p, uint64_t v) {
  *reinterpret_cast<volatile uint64_t*>(p) = v;
}

// Lanes whose valid 8-bit digit equals this lane's (bit-sliced ballots).
// Whole-warp call; the result is meaningful for valid lanes only.
__device__ __forceinline__ uint32_t peers_of_digit(uint32_t d, bool valid) {
  uint32_t peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const uint32_t m = __ballot_sync(0xffffffffu, (d >> b) & 1u);
    peers &= ((d >> b) & 1u) ? m : ~m;
  }
  return peers;
}

// Decoupled look-back of partition `part` by one warp (all 32 lanes call;
// status word: value << 2 | flag): lane 0 publishes the aggregate, the warp
// reads 32 predecessors at a time and stops at the nearest inclusive prefix;
// returns the exclusive prefix (all lanes), -1 when a wait ran out.
__device__ long long lookback_prefix_warp(uint64_t* status, int64_t part, long long agg,
                                          WsHeader* hdr) {
  const int lane = threadIdx.x & 31;
  if (part == 0) {
    if (lane == 0) st_volatile(&status[0], ((uint64_t)agg << 2) | kFlagInc);
    return 0;
  }
  if (lane == 0) st_volatile(&status[part], ((uint64_t)agg << 2) | kFlagAgg);
  long long prefix = 0;
  int64_t hi = part - 1;
  for (;;) {
    const int64_t j = hi - lane;
    uint64_t s = kFlagInc;  // before partition 0: an inclusive zero
    if (j >= 0) {
      uint32_t spins = 0;
      while (((s = ld_volatile(&status[j])) & 3u) == 0) {
        if (++spins > kSpinLimit) break;
        __nanosleep(100);
      }
    }
    const uint64_t f = s & 3u;
    if (__any_sync(0xffffffffu, f == 0 || f == kFlagErr)) {
      if (lane == 0) {
        st_volatile(&status[part], kFlagErr);
        atomicOr(&hdr->error, 1u);
      }
      return -1;
    }
    const uint32_t inc = __ballot_sync(0xffffffffu, f == kFlagInc);
    const int stop = inc ? __ffs(inc) - 1 : 31;
    long long v = lane <= stop ? (long long)(s >> 2) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    prefix += v;
    if (inc) break;
    hi -= 32;
  }
  if (lane == 0) {
    __threadfence();
    st_volatile(&status[part], ((uint64_t)(prefix + agg) << 2) | kFlagInc);
  }
  return prefix;
}

// ---------------------------------------------------------------------------
// 1. Compaction of the visible rows (tile count > 0), in row order.  Per
//    visible row r at compact index c: the depth-sort element (depth bits <<
//    32 | r) into sort_in[c] (when c < capacity) and row_rect[r]; the
//    intersection total I into the header (block sums added atomically) and
//    R by the last partition; the depth-digit histograms.  Positive depths
//    order as their bit patterns.  The visible rows are found from the tile
//    counts alone (the array, else the records' tile words), so that a
//    partition publishes its aggregate for the look-back after one round of
//    loads; their records are read after the look-back.  A row whose
//    rectangle disagrees with its count (records not produced by
//    gs_project) raises the device-check bit and keeps its position with an
//    empty rectangle: it emits nothing and adds nothing to I.
// A row's tile count: the array's, else the record's tile word (0 past the end).
__device__ __forceinline__ int32_t row_count(int64_t r, int64_t n_rows,
                                             const float4* __restrict__ splats,
                                             const int32_t* __restrict__ counts) {
  if (r >= n_rows) return 0;
  return counts ? __ldg(counts + r) : __float_as_int(splats[3 * r + 2].w);
}

template <int kCompChunks>
__global__ void __launch_bounds__(kCompThreads, 4) compact_rows_kernel(
    int64_t n_rows, int64_t n, int32_t tiles_x, int32_t tiles_y, int64_t T, int64_t capacity,
    const float4* __restrict__ splats, const int32_t* __restrict__ counts,
    uint64_t* __restrict__ sort_in,
    uint64_t* __restrict__ row_rect, uint32_t* __restrict__ hist,
    uint64_t* __restrict__ status, WsHeader* __restrict__ hdr) {
  __shared__ uint32_t sh[kDepthPasses * kRadix];
  __shared__ uint32_t s_warp[kCompChunks][kCompWarps];
  __shared__ unsigned long long s_tiles[kCompWarps];
  __shared__ uint8_t s_lidx[kCompWarps][16 * kCompItems];  // a sparse warp chunk's visible
  __shared__ int32_t s_lcnt[kCompWarps][16 * kCompItems];  // rows (offsets), their counts
  __shared__ long long s_prefix;
  __shared__ int s_part;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_part = (int)atomicAdd(&hdr->scan_ticket, 1u);
  for (int i = tid; i < kDepthPasses * kRadix; i += kCompThreads) sh[i] = 0;
  __syncthreads();
  const int64_t part = s_part;
  // item i of lane l of warp w in chunk k: row
  // part * kRows + k * kCompChunk + w * 32 * kCompItems + 32 i + l
  constexpr int kRows = kCompChunk * kCompChunks;
  const int64_t wbase = part * kRows + (int64_t)warp * 32 * kCompItems + lane;
  // 1. the rows with a positive tile count, per chunk and warp: the
  //    partition's aggregate for the look-back is published after one round
  //    of 4-byte loads (the tile-count array), however few rows are visible
#pragma unroll
  for (int k = 0; k < kCompChunks; ++k) {
    int32_t cnt[kCompItems];
#pragma unroll
    for (int i = 0; i < kCompItems; ++i)
      cnt[i] = row_count(wbase + (int64_t)k * kCompChunk + 32 * i, n_rows, splats, counts);
    uint32_t wc = 0;
#pragma unroll
    for (int i = 0; i < kCompItems; ++i) wc += __popc(__ballot_sync(0xffffffffu, cnt[i] > 0));
    if (lane == 0) s_warp[k][warp] = wc;
  }
  __syncthreads();
  uint32_t block_count = 0;
#pragma unroll
  for (int k = 0; k < kCompChunks; ++k)
#pragma unroll
    for (int w = 0; w < kCompWarps; ++w) block_count += s_warp[k][w];
  if (warp == 0) {
    const long long prefix = lookback_prefix_warp(status, part, (long long)block_count, hdr);
    if (lane == 0) {
      s_prefix = prefix;
      if (prefix >= 0 && (part + 1) * kRows >= n_rows)
        hdr->rows = (unsigned long long)(prefix + block_count);
    }
  }
  __syncthreads();
  // 2. the same counts again (cached), and the visible rows' records,
  //    checked against the counts and written at their compact positions.  A
  //    row whose rectangle disagrees with its count raises the device-check
  //    bit and keeps its position with an empty rectangle (it emits no
  //    intersection and adds nothing to the total)
  unsigned long long tiles_sum = 0;
  if (s_prefix >= 0) {
    const uint32_t lt = (1u << lane) - 1u;
    int64_t base = s_prefix;
#pragma unroll 1
    for (int k = 0; k < kCompChunks; ++k) {
      uint32_t before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < kCompWarps; ++w) {
        before += w < warp ? s_warp[k][w] : 0u;
        total += s_warp[k][w];
      }
      const int64_t c = base + before;
      const int64_t cbase = part * kRows + (int64_t)k * kCompChunk + warp * 32 * kCompItems;
      int32_t cnt[kCompItems];
      int nvis = 0;
#pragma unroll
      for (int i = 0; i < kCompItems; ++i) {
        cnt[i] = row_count(cbase + 32 * i + lane, n_rows, splats, counts);
        nvis += __popc(__ballot_sync(0xffffffffu, cnt[i] > 0));
      }
      // one visible row: its rectangle checked against its count, its sort
      // element written at compact index ci and its rectangle at r, its depth
      // digits counted
      auto emit_row = [&](uint32_t r, int32_t cq, float2 mean, float dep, int32_t rad,
                          int64_t ci) {
        const uint32_t view = r / (uint32_t)n;  // rows < 2^32
        int32_t x0, x1, y0, y1;
        tile_rect(mean.x, mean.y, rad, tiles_x, tiles_y, x0, x1, y0, y1);
        uint64_t rect = 0;
        if ((int64_t)(x1 - x0) * (y1 - y0) == cq) {
          const uint32_t first = (uint32_t)((int64_t)view * T + (int64_t)y0 * tiles_x + x0);
          rect = (uint64_t)first | ((uint64_t)(x1 - x0) << 32) | ((uint64_t)(y1 - y0) << 48);
          tiles_sum += (unsigned long long)cq;
        } else {
          atomicOr(&hdr->error, 2u);
        }
        const uint32_t dbits = __float_as_uint(dep);
        if (ci < capacity) sort_in[ci] = ((uint64_t)dbits << 32) | (uint64_t)r;
        row_rect[r] = rect;
#pragma unroll
        for (int p = 0; p < kDepthPasses; ++p)
          atomicAdd(&sh[p * kRadix + ((dbits >> (8 * p)) & 0xFF)], 1u);
      };
      // every visible row's record fields are requested before the first is
      // used, so a chunk waits for one round of loads
      float2 mean[kCompItems];
      float dep[kCompItems];
      int32_t rad[kCompItems];
      if (nvis > 16 * kCompItems) {
        // mostly visible: item by item, in place
#pragma unroll
        for (int i = 0; i < kCompItems; ++i) {
          mean[i] = make_float2(0.f, 0.f);
          dep[i] = 0.f;
          rad[i] = 0;
          if (cnt[i] > 0) {
            const float* rec = reinterpret_cast<const float*>(splats + 3 * (cbase + 32 * i + lane));
            mean[i] = __ldg(reinterpret_cast<const float2*>(rec));
            dep[i] = __ldg(rec + 9);
            rad[i] = __float_as_int(__ldg(rec + 10));
          }
        }
        int64_t cc = c;
#pragma unroll
        for (int i = 0; i < kCompItems; ++i) {
          const uint32_t m = __ballot_sync(0xffffffffu, cnt[i] > 0);
          if (cnt[i] > 0)
            emit_row((uint32_t)(cbase + 32 * i + lane), cnt[i], mean[i], dep[i], rad[i],
                     cc + __popc(m & lt));
          cc += __popc(m);
        }
      } else {
        // sparse: the visible rows listed in row order, then one per lane
        uint8_t* lidx = s_lidx[warp];
        int32_t* lcnt = s_lcnt[warp];
        int at = 0;
#pragma unroll
        for (int i = 0; i < kCompItems; ++i) {
          const uint32_t m = __ballot_sync(0xffffffffu, cnt[i] > 0);
          if (cnt[i] > 0) {
            lidx[at + __popc(m & lt)] = (uint8_t)(32 * i + lane);
            lcnt[at + __popc(m & lt)] = cnt[i];
          }
          at += __popc(m);
        }
        __syncwarp();
#pragma unroll
        for (int q = 0; q < kCompItems / 2; ++q) {
          const int j = 32 * q + lane;
          mean[q] = make_float2(0.f, 0.f);
          dep[q] = 0.f;
          rad[q] = 0;
          if (j < nvis) {
            const float* rec = reinterpret_cast<const float*>(splats + 3 * (cbase + lidx[j]));
            mean[q] = __ldg(reinterpret_cast<const float2*>(rec));
            dep[q] = __ldg(rec + 9);
            rad[q] = __float_as_int(__ldg(rec + 10));
          }
        }
#pragma unroll
        for (int q = 0; q < kCompItems / 2; ++q) {
          const int j = 32 * q + lane;
          if (j < nvis)
            emit_row((uint32_t)cbase + lidx[j], lcnt[j], mean[q], dep[q], rad[q], c + j);
        }
        __syncwarp();  // the list is rewritten by the next chunk
      }
      base += total;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tiles_sum += __shfl_xor_sync(0xffffffffu, tiles_sum, o);
  if (lane == 0) s_tiles[warp] = tiles_sum;
  __syncthreads();
  if (tid == 0) {
    unsigned long long bt = 0;
#pragma unroll
    for (int w = 0; w < kCompWarps; ++w) bt += s_tiles[w];
    if (bt) atomicAdd(&hdr->total, bt);
  }
  for (int i = tid; i < kDepthPasses * kRadix; i += kCompThreads)
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

// Look-back of one digit of radix partition `part` (status word: value << 8 |
// tag << 2 | flag): the exclusive prefix of the digit over the partitions
// before `part`, summing aggregates back to the nearest inclusive prefix.
// The predecessors are read kLookWindow at a time (independent loads in
// flight together) rather than one by one: a partition that arrives while
// its k nearest predecessors are still looking back walks k steps, and with
// one dependent L2 round trip per step that walk, not the data movement, set
// the pace of a pass.  Each wait is bounded; false when one ran out (or a
// predecessor failed).
constexpr int kLookWindow = 8;

__device__ __forceinline__ bool digit_lookback(const uint64_t* status, int64_t part, int d,
                                               uint64_t tag, unsigned long long& excl) {
  excl = 0;
  int64_t j = part - 1;  // partition 0 is inclusive: every walk ends there at the latest
  while (j >= 0) {
    uint64_t s[kLookWindow];
#pragma unroll
    for (int i = 0; i < kLookWindow; ++i)
      s[i] = j - i >= 0 ? ld_volatile(&status[(j - i) * kRadix + d]) : (tag | kFlagInc);
#pragma unroll
    for (int i = 0; i < kLookWindow; ++i) {
      uint64_t v = s[i];
      uint32_t spins = 0;
      while ((v & 3u) != kFlagErr && ((v & 3u) == 0 || (v & 0xFCu) != tag)) {
        if (++spins > kSpinLimit) return false;
        __nanosleep(100);
        v = ld_volatile(&status[(j - i) * kRadix + d]);
      }
      if ((v & 3u) == kFlagErr) return false;
      excl += (unsigned long long)(v >> 8);
      if ((v & 3u) == kFlagInc) return true;
    }
    j -= kLookWindow;
  }
  return true;
}

// ---------------------------------------------------------------------------
// 2, 4. One stable radix pass over 64-bit keys on the 8 bits at `shift`
//    (onesweep).  Sort status word: value << 8 | tag << 2 | flag, tag =
//    pass + 1 (stale entries of an earlier pass read as not ready).  kFinal:
//    the last tile pass, which writes key (tile << 32 | depth bits) and the
//    Gaussian id of the element's row, read from row_d at the row's depth
//    position s (the element's low 32 bits), instead, and marks
//    the tile ranges: a partition's keys, placed in shared memory, are in
//    full tile order (its input is ordered by the lower tile digits), so each
//    run of one tile in it is contiguous in the output; its ends go into
//    ranges by atomic maxima (the start as count - position), decoded by
//    ranges_fix_kernel.
//    kMode: 0 a pass, 1 the last tile pass (above), 2 the first tile pass of
//    the balanced emission, which makes its partition's elements instead of
//    loading them: element t (in depth order) lies in the last row whose
//    first output position (erow) is <= t, found by binary search among the
//    rows of t's emission chunk (chunk_row), so the emitted list never passes
//    through memory.  Same elements as emit_chunks_kernel.
struct SortSmem64 {
  uint32_t warp_hist[kPassWarps][kRadix];
  uint32_t local_start[kRadix];
  unsigned long long global_base[kRadix];
  uint32_t scan_w[kPassWarps];
  int part;
  int err;
  long long count;
  long long rows;
  uint64_t keys[kSortPart];
};

template <int kMode>
__global__ void __launch_bounds__(kPassThreads, kPassMinBlocks) onesweep64_kernel(
    int64_t count, int32_t pass, int32_t shift, const uint64_t* __restrict__ keys_in,
    uint64_t* __restrict__ keys_out, const uint32_t* __restrict__ digit_start,
    uint64_t* __restrict__ status, WsHeader* __restrict__ hdr, const uint64_t* __restrict__ row_d,
    uint32_t* __restrict__ vals_out, uint32_t n, unsigned long long* __restrict__ ranges,
    const uint4* __restrict__ erow, const uint32_t* __restrict__ chunk_row, int32_t tiles_x) {
  constexpr bool kFinal = kMode == 1;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmem64& S = *reinterpret_cast<SortSmem64*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t tag = (uint64_t)(pass + 1) << 2;
  const int hs = shift - 32;  // the digit lies in the high word
  for (int i = tid; i < kPassWarps * kRadix; i += kPassThreads) (&S.warp_hist[0][0])[i] = 0;
  if (tid == 0) {
    S.part = (int)atomicAdd(&hdr->pass_ticket[pass], 1u);
    S.err = 0;
    // count < 0 (asynchronous path, grid sized by an upper bound; surplus
    // partitions hold the highest tickets, so no real partition looks back
    // at them): -1 the intersections, -2 the visible rows, read from the
    // header; nothing to do after an overflow or a wait that ran out
    if (count < 0)
      S.count = (hdr->error & kErrStop) ? -1
                                        : (long long)(count == -1 ? hdr->total : hdr->rows);
    if (kMode == 2) S.rows = (long long)hdr->rows;
  }
  __syncthreads();
  if (count < 0) {
    count = S.count;
    if (count < 0) return;
  }
  const int64_t part = S.part;
  const int64_t pbase = part * kSortPart;
  if (pbase >= count) return;
  const int n_here = count - pbase < kSortPart ? (int)(count - pbase) : kSortPart;
  const int wbase = warp * 32 * kPassKpt;
  // load or make (warp-striped: item i of lane l is element wbase + 32 i + l) and rank
  uint64_t key[kPassKpt];
  if constexpr (kMode == 2) {
    // a warp's 256 elements lie in one emission chunk (kEmitChunk is a
    // multiple of 256 and of no partition boundary's offset); the rows of
    // chunk q are chunk_row[q] .. chunk_row[q + 1] (the last one: R - 1)
    static_assert(kEmitChunk % (32 * kPassKpt) == 0 && kSortPart % kEmitChunk == 0, "chunks");
    const int64_t q = (pbase + wbase) / kEmitChunk;
    const bool any = pbase + wbase < count;  // else no element of the warp is real
    int a0 = any ? (int)chunk_row[q] : 0;
    const int b0 = !any ? 0 : ((q + 1) * kEmitChunk < count ? (int)chunk_row[q + 1]
                                                            : (int)(S.rows - 1));
#pragma unroll
    for (int i = 0; i < kPassKpt; ++i) {
      const int li = wbase + 32 * i + lane;
      key[i] = 0ull;
      if (li < n_here) {
        const uint32_t t = (uint32_t)(pbase + li);  // I < 2^32
        int a = a0, b = b0;  // the last row whose first position is <= t
        while (a < b) {
          const int mid = (a + b + 1) >> 1;
          if (__ldg(&erow[mid].x) <= t) a = mid; else b = mid - 1;
        }
        a0 = a;  // a lane's elements ascend
        const uint4 r = __ldg(erow + a);
        const uint32_t i2 = t - r.x, w = r.z & 0xFFFFu;
        uint32_t ty;
        if (i2 < (1u << 24)) {  // exact in fp32: the reciprocal's quotient is off by at most one
          ty = __float2uint_rz(__fmul_rn((float)i2, __frcp_rn((float)w)));
          if (ty * w > i2) --ty;
          else if ((ty + 1) * w <= i2) ++ty;
        } else {
          ty = i2 / w;
        }
        const uint32_t flat = r.y + ty * (uint32_t)tiles_x + (i2 - ty * w);
        key[i] = ((uint64_t)flat << 32) | (uint64_t)r.w;
      }
    }
  } else {
    const uint64_t* src = keys_in + pbase;
#pragma unroll
    for (int i = 0; i < kPassKpt; ++i) {
      const int li = wbase + 32 * i + lane;
      key[i] = li < n_here ? src[li] : 0ull;
    }
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  // rank of each key among the warp's keys of its digit (< 32 kPassKpt <=
  // 65536: two to a register)
  uint32_t rank2[(kPassKpt + 1) / 2] = {};
#pragma unroll
  for (int i = 0; i < kPassKpt; ++i) {
    const bool valid = wbase + 32 * i + lane < n_here;
    const uint32_t d = ((uint32_t)(key[i] >> 32) >> hs) & 0xFFu;
    const uint32_t peers = peers_of_digit(d, valid);
    uint32_t basec = 0;
    if (valid) basec = S.warp_hist[warp][d];
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) S.warp_hist[warp][d] = basec + __popc(peers);
    __syncwarp();
    rank2[i / 2] |= ((basec + __popc(peers & lt_mask)) & 0xFFFFu) << (16 * (i % 2));
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
    for (int w = 0; w < kPassWarps; ++w) {
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
  }
  __syncthreads();
  // place the partition in smem in sorted (digit-major, stable) order; the
  // keys leave the registers before the look-back
#pragma unroll
  for (int i = 0; i < kPassKpt; ++i) {
    if (wbase + 32 * i + lane < n_here) {
      const uint32_t dd = ((uint32_t)(key[i] >> 32) >> hs) & 0xFFu;
      S.keys[S.local_start[dd] + S.warp_hist[warp][dd] + ((rank2[i / 2] >> (16 * (i % 2))) & 0xFFFFu)] =
          key[i];
    }
  }
  if (dthread) {
    unsigned long long excl = 0;
    if (part > 0) {
      if (digit_lookback(status, part, d, tag, excl)) {
        st_volatile(&status[part * kRadix + d], ((uint64_t)(excl + my_count) << 8) | tag | kFlagInc);
      } else {
        st_volatile(&status[part * kRadix + d], tag | kFlagErr);
        atomicOr(&hdr->error, 1u);
        S.err = 1;
      }
    }
    // global position of the digit's first key, less its local start
    S.global_base[d] = (unsigned long long)digit_start[pass * kRadix + d] + excl -
                       (unsigned long long)S.local_start[d];
  }
  __syncthreads();
  if (S.err) return;
  for (int j = tid; j < n_here; j += kPassThreads) {
    const uint64_t k = S.keys[j];
    const uint32_t dd = ((uint32_t)(k >> 32) >> hs) & 0xFFu;
    const unsigned long long gpos = S.global_base[dd] + (unsigned long long)j;
    if (gpos < (unsigned long long)count) {
      if constexpr (kFinal) {
        const uint64_t u = __ldg(row_d + (uint32_t)k);  // depth bits, Gaussian id
        keys_out[gpos] = (k & 0xFFFFFFFF00000000ull) | (u >> 32);
        vals_out[gpos] = (uint32_t)u;
        const uint32_t f = (uint32_t)(k >> 32);
        if (j == 0 || (uint32_t)(S.keys[j - 1] >> 32) != f)
          atomicMax(&ranges[2 * (uint64_t)f], (unsigned long long)count - gpos);
        if (j == n_here - 1 || (uint32_t)(S.keys[j + 1] >> 32) != f)
          atomicMax(&ranges[2 * (uint64_t)f + 1], gpos + 1ull);
      } else {
        keys_out[gpos] = k;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 3. Emission in depth order.  The sorted rows are cut into partitions of
//    kEmitPart; a partition scans its rows' tile counts (the look-back across
//    partitions gives its output offset), then its threads write the
//    partition's intersections at consecutive positions, each finding its
//    row by binary search over the partition's inclusive counts: element
//    (flat tile << 32 | s), s the row's position in depth order, tiles of a
//    row in raster order; and row_d[s].  Also the digit histograms of the
//    tile passes.  count < 0: R from the header.
__global__ void __launch_bounds__(kEmitThreads) emit_sorted_kernel(
    int64_t count, int32_t tiles_x, int32_t tile_passes, uint32_t n,
    const uint64_t* __restrict__ sorted, const uint64_t* __restrict__ row_rect,
    uint64_t* __restrict__ row_d, uint64_t* __restrict__ out, uint32_t* __restrict__ hist,
    uint64_t* __restrict__ status, WsHeader* __restrict__ hdr) {
  __shared__ uint32_t s_incl[kEmitPart];   // inclusive tile counts, partition-local
  __shared__ uint32_t s_first[kEmitPart];  // first flat tile of the row's rectangle
  __shared__ uint32_t s_w[kEmitPart];      // rectangle width
  __shared__ uint32_t s_c[kEmitPart];      // the row's position in depth order
  __shared__ uint32_t sh[4 * kRadix];
  __shared__ uint32_t s_warp[kEmitThreads / 32];
  __shared__ long long s_count, s_prefix;
  __shared__ int s_part;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    // the status word and R come from earlier kernels: one load per CTA
    s_count = (hdr->error & kErrStop) ? -1 : (count < 0 ? (long long)hdr->rows : count);
    s_part = (int)atomicAdd(&hdr->emit_ticket, 1u);
  }
  for (int i = tid; i < tile_passes * kRadix; i += kEmitThreads) sh[i] = 0;
  __syncthreads();
  const long long R = s_count;
  const int64_t part = s_part, pbase = part * kEmitPart;
  if (R < 0 || pbase >= R) return;
  const int n_here = R - pbase < kEmitPart ? (int)(R - pbase) : kEmitPart;
  for (int e = tid; e < kEmitPart; e += kEmitThreads) {
    uint32_t t = 0;
    if (e < n_here) {
      const uint64_t u = sorted[pbase + e];  // depth bits << 32 | row
      const uint32_t r = (uint32_t)u;
      const uint64_t rc = __ldg(row_rect + r);
      const uint32_t w = (uint32_t)(rc >> 32) & 0xFFFFu, h = (uint32_t)(rc >> 48);
      t = w * h;
      s_first[e] = (uint32_t)rc;
      s_w[e] = w;
      s_c[e] = (uint32_t)(pbase + e);  // R < 2^32
      row_d[pbase + e] = (u & 0xFFFFFFFF00000000ull) | (uint64_t)(r % n);
    }
    s_incl[e] = t;
  }
  __syncthreads();
  // block scan: thread tid owns elements [tid * kEmitItems, + kEmitItems)
  uint32_t v[kEmitItems];
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < kEmitItems; ++k) {
    v[k] = s_incl[tid * kEmitItems + k];
    sum += v[k];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  uint32_t run = incl - sum, block_total = 0;
#pragma unroll
  for (int w = 0; w < kEmitThreads / 32; ++w) {
    run += w < warp ? s_warp[w] : 0u;
    block_total += s_warp[w];
  }
#pragma unroll
  for (int k = 0; k < kEmitItems; ++k) {
    run += v[k];
    s_incl[tid * kEmitItems + k] = run;
  }
  if (warp == 0) {
    const long long prefix = lookback_prefix_warp(status, part, (long long)block_total, hdr);
    if (lane == 0) s_prefix = prefix;
  }
  __syncthreads();
  if (s_prefix < 0) return;
  uint64_t* dst = out + s_prefix;
  for (uint32_t t = tid; t < block_total; t += kEmitThreads) {
    int lo = 0, hi = n_here - 1;  // first e with s_incl[e] > t
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_incl[mid] > t) hi = mid; else lo = mid + 1;
    }
    const uint32_t i = t - (lo > 0 ? s_incl[lo - 1] : 0u);
    const uint32_t w = s_w[lo];
    const uint32_t ty = i / w, tx = i - ty * w;
    const uint32_t flat = s_first[lo] + ty * (uint32_t)tiles_x + tx;
    dst[t] = ((uint64_t)flat << 32) | (uint64_t)s_c[lo];
    for (int p = 0; p < tile_passes; ++p) atomicAdd(&sh[p * kRadix + ((flat >> (8 * p)) & 0xFF)], 1u);
  }
  __syncthreads();
  for (int i = tid; i < tile_passes * kRadix; i += kEmitThreads)
    if (sh[i]) atomicAdd(&hist[kDepthPasses * kRadix + i], sh[i]);
}

// 3 (balanced form).  Two kernels.  row_scan_kernel scans the sorted rows'
//    tile counts (partitions of kEmitPart rows, decoupled look-back as
//    above) into each row's first output position and writes per sorted row
//    s erow = (position, first flat tile, width | height << 16, s) and row_d[s]
//    and, for every chunk of kEmitChunk outputs that starts inside the row,
//    chunk_row[chunk] = the row.  emit_chunks_kernel then gives every CTA
//    one chunk of outputs -- the same number whatever the rows' sizes, where
//    partitions of rows differ by orders of magnitude in output -- loads the
//    chunk's rows into shared memory and finds each output's row by binary
//    search among them; a row's tile (ty, tx) comes from a float reciprocal
//    of its width, corrected to the exact quotient.  Same outputs, bit for
//    bit, as emit_sorted_kernel.
__global__ void __launch_bounds__(kEmitThreads) row_scan_kernel(
    int64_t count, int32_t tiles_x, int32_t tile_passes, uint32_t n,
    const uint64_t* __restrict__ sorted, const uint64_t* __restrict__ row_rect,
    uint64_t* __restrict__ row_d, uint4* __restrict__ erow,
    uint32_t* __restrict__ chunk_row, uint32_t* __restrict__ hist, uint64_t* __restrict__ status,
    WsHeader* __restrict__ hdr) {
  __shared__ uint32_t s_warp[kEmitThreads / 32];
  // the tile passes' digit counts of the partition's intersections, from the
  // rows' rectangles: a tile row of a rectangle is a run of consecutive flat
  // indices, so the lowest digit of its tiles covers a cyclic range of bins
  // (added as a difference array: diff[lo]++, diff[hi]--) and each higher
  // digit is constant over whole sub-runs
  __shared__ int32_t s_diff[kRadix + 1];
  __shared__ uint32_t s_hi[3 * kRadix];
  __shared__ uint32_t s_wrap;  // whole turns of the lowest digit (added to every bin)
  __shared__ long long s_count, s_prefix;
  __shared__ int s_part;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_count = (hdr->error & kErrStop) ? -1 : (count < 0 ? (long long)hdr->rows : count);
    s_part = (int)atomicAdd(&hdr->emit_ticket, 1u);
    s_wrap = 0;
  }
  for (int i = tid; i <= kRadix; i += kEmitThreads) s_diff[i] = 0;
  for (int i = tid; i < 3 * kRadix; i += kEmitThreads) s_hi[i] = 0;
  __syncthreads();
  const long long R = s_count;
  const int64_t part = s_part, pbase = part * kEmitPart;
  if (R < 0 || pbase >= R) return;
  // thread tid owns rows pbase + tid * kEmitItems + [0, kEmitItems)
  uint32_t c[kEmitItems], first[kEmitItems], wh[kEmitItems], t[kEmitItems];
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < kEmitItems; ++k) {
    const int64_t e = pbase + tid * kEmitItems + k;
    t[k] = 0;
    if (e < R) {
      const uint64_t u = sorted[e];  // depth bits << 32 | row
      const uint32_t r = (uint32_t)u;
      c[k] = (uint32_t)e;  // R < 2^32
      row_d[e] = (u & 0xFFFFFFFF00000000ull) | (uint64_t)(r % n);
      const uint64_t rc = __ldg(row_rect + r);
      const uint32_t w = (uint32_t)(rc >> 32) & 0xFFFFu, h = (uint32_t)(rc >> 48);
      first[k] = (uint32_t)rc;
      wh[k] = w | (h << 16);
      t[k] = w * h;
    }
    sum += t[k];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  uint32_t run = incl - sum, block_total = 0;
#pragma unroll
  for (int w = 0; w < kEmitThreads / 32; ++w) {
    run += w < warp ? s_warp[w] : 0u;
    block_total += s_warp[w];
  }
  if (warp == 0) {
    const long long prefix = lookback_prefix_warp(status, part, (long long)block_total, hdr);
    if (lane == 0) s_prefix = prefix;
  }
  __syncthreads();
  if (s_prefix < 0) return;
  unsigned long long pos = (unsigned long long)s_prefix + run;
#pragma unroll
  for (int k = 0; k < kEmitItems; ++k) {
    const int64_t e = pbase + tid * kEmitItems + k;
    if (e < R) {
      erow[e] = make_uint4((uint32_t)pos, first[k], wh[k], c[k]);
      // the chunks whose first output lies in [pos, pos + t)
      for (unsigned long long q = div_up((int64_t)pos, kEmitChunk);
           q * kEmitChunk < pos + t[k]; ++q)
        chunk_row[q] = (uint32_t)e;
    }
    pos += t[k];
  }
  // digit counts of the tile passes
#pragma unroll
  for (int k = 0; k < kEmitItems; ++k) {
    if (pbase + tid * kEmitItems + k >= R) continue;
    const uint32_t w = wh[k] & 0xFFFFu, h = wh[k] >> 16;
    for (uint32_t y = 0; y < h; ++y) {
      const uint32_t f = first[k] + y * (uint32_t)tiles_x;  // tiles f .. f + w - 1
      const uint32_t lo = f & 0xFFu, rem = w & 0xFFu;
      if (w >> 8) atomicAdd(&s_wrap, w >> 8);
      if (rem) {
        atomicAdd(&s_diff[lo], 1);
        if (lo + rem <= (uint32_t)kRadix) {
          atomicAdd(&s_diff[lo + rem], -1);
        } else {
          atomicAdd(&s_diff[kRadix], -1);
          atomicAdd(&s_diff[0], 1);
          atomicAdd(&s_diff[lo + rem - kRadix], -1);
        }
      }
      for (int p = 1; p < tile_passes; ++p) {
        const uint32_t shift = 8u * (uint32_t)p;
        for (uint32_t a = f, end = f + w; a < end;) {
          const uint32_t next = ((a >> shift) + 1u) << shift;  // next change of digit p
          const uint32_t b = next > a && next < end ? next : end;
          atomicAdd(&s_hi[(p - 1) * kRadix + ((a >> shift) & 0xFFu)], b - a);
          a = b;
        }
      }
    }
  }
  __syncthreads();
  if (tid < kRadix) {  // bin d of the lowest digit: the prefix sum of diff up to d, plus the turns
    int32_t run = 0;
    for (int i = 0; i <= tid; ++i) run += s_diff[i];
    const uint32_t c0 = (uint32_t)run + s_wrap;
    if (c0) atomicAdd(&hist[kDepthPasses * kRadix + tid], c0);
    for (int p = 1; p < tile_passes; ++p)
      if (s_hi[(p - 1) * kRadix + tid])
        atomicAdd(&hist[(kDepthPasses + p) * kRadix + tid], s_hi[(p - 1) * kRadix + tid]);
  }
}

__global__ void __launch_bounds__(kEmitThreads) emit_chunks_kernel(
    int32_t tiles_x, const uint4* __restrict__ erow, const uint32_t* __restrict__ chunk_row,
    uint64_t* __restrict__ out, const WsHeader* __restrict__ hdr) {
  __shared__ uint4 s_row[kEmitChunk + 1];
  __shared__ long long s_total, s_rows;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_total = (hdr->error & kErrStop) ? -1 : (long long)hdr->total;
    s_rows = (long long)hdr->rows;
  }
  __syncthreads();
  const long long I = s_total, R = s_rows;
  const long long t0 = (long long)blockIdx.x * kEmitChunk;
  if (I < 0 || t0 >= I) return;
  const int n_here = I - t0 < kEmitChunk ? (int)(I - t0) : kEmitChunk;
  const long long nchunks = div_up(I, kEmitChunk);
  // the rows holding outputs t0 .. t0 + n_here - 1 (at most kEmitChunk, each
  // row holding at least one; the next chunk's first row may be one more)
  const uint32_t ra = chunk_row[blockIdx.x];
  const uint32_t rb = blockIdx.x + 1 < nchunks ? chunk_row[blockIdx.x + 1] : (uint32_t)(R - 1);
  const int m = (int)(rb - ra) + 1;
  for (int i = tid; i < m; i += kEmitThreads) s_row[i] = erow[ra + i];
  __syncthreads();
  for (int j = tid; j < n_here; j += kEmitThreads) {
    const uint32_t t = (uint32_t)(t0 + j);
    int lo = 0, hi = m - 1;  // the last row whose first position is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_row[mid].x <= t) lo = mid; else hi = mid - 1;
    }
    const uint4 r = s_row[lo];
    const uint32_t i = t - r.x, w = r.z & 0xFFFFu;
    uint32_t ty;
    if (i < (1u << 24)) {  // exact in fp32: the reciprocal's quotient is off by at most one
      ty = __float2uint_rz(__fmul_rn((float)i, __frcp_rn((float)w)));
      if (ty * w > i) --ty;
      else if ((ty + 1) * w <= i) ++ty;
    } else {
      ty = i / w;
    }
    const uint32_t tx = i - ty * w;
    const uint32_t flat = r.y + ty * (uint32_t)tiles_x + tx;
    out[t] = ((uint64_t)flat << 32) | (uint64_t)r.w;
  }
}

// ---------------------------------------------------------------------------
// 5. Tile ranges [first, last + 1): the last tile pass leaves count - first
//    (0 for an empty tile) in ranges[2 f]; decoded here.  count < 0: the
//    intersection total from the header (nothing after an overflow).
__global__ void __launch_bounds__(256) ranges_fix_kernel(int64_t count, int64_t n_flat,
                                                         int64_t* __restrict__ ranges,
                                                         const WsHeader* __restrict__ hdr) {
  if (count < 0) {
    __shared__ int64_t s_count;
    if (threadIdx.x == 0) s_count = (hdr->error & kErrStop) ? -1 : (int64_t)hdr->total;
    __syncthreads();
    count = s_count;
    if (count < 0) return;
  }
  for (int64_t f = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; f < n_flat;
       f += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = ranges[2 * f];
    if (e > 0) ranges[2 * f] = count - e;
  }
}

// ---------------------------------------------------------------------------
// One stable radix pass over (key, value) pairs, for the Morton order ("onesweep",
// as the key-only passes below).  Sort status word: value << 8 | tag << 2 |
// flag, tag = pass + 1 (stale entries of an earlier pass read as not ready).
struct SortSmemKV {
  uint32_t warp_hist[kSortWarps][kRadix];
  uint32_t local_start[kRadix];
  unsigned long long global_base[kRadix];
  uint32_t scan_w[kSortWarps];
  int part;
  int err;
  uint64_t keys[kSortPart];
  uint32_t vals[kSortPart];
};

__global__ void __launch_bounds__(kSortThreads, 3) onesweep_kv_kernel(
    int64_t count, int32_t pass, const uint64_t* __restrict__ keys_in,
    const uint32_t* __restrict__ vals_in, uint64_t* __restrict__ keys_out,
    uint32_t* __restrict__ vals_out, const uint32_t* __restrict__ digit_start,
    uint64_t* __restrict__ status, WsHeader* __restrict__ hdr) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmemKV& S = *reinterpret_cast<SortSmemKV*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int shift = 8 * pass;
  const uint64_t tag = (uint64_t)(pass + 1) << 2;
  for (int i = tid; i < kSortWarps * kRadix; i += kSortThreads) (&S.warp_hist[0][0])[i] = 0;
  if (tid == 0) {
    S.part = (int)atomicAdd(&hdr->pass_ticket[pass], 1u);
    S.err = 0;
  }
  __syncthreads();
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
    const uint32_t peers = peers_of_digit(d, d < 256u);
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
  }
  __syncthreads();
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
  if (dthread) {
    unsigned long long excl = 0;
    if (part > 0) {
      if (digit_lookback(status, part, d, tag, excl)) {
        st_volatile(&status[part * kRadix + d], ((uint64_t)(excl + my_count) << 8) | tag | kFlagInc);
      } else {
        st_volatile(&status[part * kRadix + d], tag | kFlagErr);
        atomicOr(&hdr->error, 1u);
        S.err = 1;
      }
    }
    S.global_base[d] = (unsigned long long)digit_start[pass * kRadix + d] + excl;
  }
  __syncthreads();
  if (S.err) return;
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

// The sort kernels' shared-memory attribute, set once per device (the
// asynchronous path is captured into graphs after an eager call).
cudaError_t ensure_sort_attr() {
  static bool done[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(onesweep_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sizeof(SortSmemKV));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(onesweep64_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SortSmem64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(onesweep64_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SortSmem64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(onesweep64_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SortSmem64));

  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

int bit_length(uint64_t v) {
  int b = 0;
  while (v) { ++b; v >>= 1; }
  return b;
}

// Pointers into a binning workspace.
struct BinBufs {
  WsHeader* hdr;
  uint32_t *hist, *digit_start;
  uint64_t *scan_status, *emit_status, *sort_status, *row_d, *row_rect, *tmp;
  uint4* erow;
  uint32_t* chunk_row;
};

BinBufs bin_bufs(void* workspace, const WsLayout& L) {
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  BinBufs b;
  b.hdr = reinterpret_cast<WsHeader*>(ws);
  b.hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  b.digit_start = reinterpret_cast<uint32_t*>(ws + L.digit_start);
  b.scan_status = reinterpret_cast<uint64_t*>(ws + L.scan_status);
  b.emit_status = reinterpret_cast<uint64_t*>(ws + L.emit_status);
  b.erow = reinterpret_cast<uint4*>(ws + L.erow);
  b.chunk_row = reinterpret_cast<uint32_t*>(ws + L.chunk_row);
  b.sort_status = reinterpret_cast<uint64_t*>(ws + L.sort_status);
  b.row_d = reinterpret_cast<uint64_t*>(ws + L.row_d);
  b.row_rect = reinterpret_cast<uint64_t*>(ws + L.row_rect);
  b.tmp = reinterpret_cast<uint64_t*>(ws + L.tmp);
  return b;
}

// Problem shape shared by the binning entry points.
struct BinShape {
  int64_t n, n_rows, T, n_flat;
  int32_t tiles_x, tiles_y;
  int tile_passes;
};

bool bin_shape(int64_t n, int32_t n_views, int32_t width, int32_t height, BinShape& s) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1)
    return false;
  s.n = n;
  s.n_rows = n * n_views;
  s.tiles_x = (width + GS_TILE - 1) / GS_TILE;
  s.tiles_y = (height + GS_TILE - 1) / GS_TILE;
  s.T = tiles_per_view(width, height);
  s.n_flat = n_views * s.T;
  // row index and flat tile index in 32 bits, rectangle sides in 16
  if (s.n_rows > (int64_t)0xFFFFFFFFll || s.n_flat > (int64_t)0xFFFFFFFFll || s.tiles_x > 0xFFFF ||
      s.tiles_y > 0xFFFF)
    return false;
  const int b = bit_length((uint64_t)(s.n_flat - 1));
  s.tile_passes = ((b > 0 ? b : 1) + 7) / 8;
  return true;
}

// Where the compaction writes the depth-sort elements: the buffer the four
// depth passes end in, chosen so that the tile passes end their chain in
// the caller's keys with the last pass reading the other buffer.
uint64_t* rows_buffer(const BinShape& s, const BinBufs& b, uint64_t* keys) {
  return s.tile_passes % 2 == 0 ? b.tmp : keys;
}

gs_status launch_compaction(const BinShape& s, const BinBufs& b, const gs_splat* splats,
                            const int32_t* counts, int64_t capacity, uint64_t* keys,
                            cudaStream_t st) {
  const int chunks = comp_chunks(s.n_rows);
  const int64_t parts = div_up(s.n_rows, (int64_t)chunks * kCompChunk);
  GS_CUDA(cudaMemsetAsync(b.scan_status, 0, sizeof(uint64_t) * (size_t)parts, st));
  auto kernel = chunks == 1 ? compact_rows_kernel<1>
                            : (chunks == 4 ? compact_rows_kernel<4> : compact_rows_kernel<8>);
  kernel<<<(unsigned)parts, kCompThreads, 0, st>>>(
      s.n_rows, s.n, s.tiles_x, s.tiles_y, s.T, capacity, reinterpret_cast<const float4*>(splats),
      counts, rows_buffer(s, b, keys), b.row_rect, b.hist, b.scan_status, b.hdr);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

// Stages 2-5.  rows / isect: the counts, or -2 / -1 to have the kernels read
// them from the header (grids then sized by rows_max / isect_max).
gs_status launch_sort_stages(const BinShape& s, const BinBufs& b, int64_t rows, int64_t isect,
                             int64_t rows_max, int64_t isect_max, uint64_t* keys, uint32_t* vals,
                             int64_t* ranges, cudaStream_t st) {
  uint64_t* ra = rows_buffer(s, b, keys);
  uint64_t* rb = ra == keys ? b.tmp : keys;
  const int64_t parts_r = div_up(rows_max, kSortPart), parts_i = div_up(isect_max, kSortPart);
  GS_CUDA(cudaMemsetAsync(b.sort_status, 0,
                          sizeof(uint64_t) * kRadix * (size_t)(parts_r > parts_i ? parts_r : parts_i),
                          st));
  hist_scan_kernel<<<kDepthPasses, kRadix, 0, st>>>(b.hist, b.digit_start);
  GS_CHECK_LAUNCH();
  GS_CUDA(ensure_sort_attr());
  const size_t smem = sizeof(SortSmem64);
  uint64_t* in = ra;
  uint64_t* out = rb;
  for (int p = 0; p < kDepthPasses; ++p) {
    onesweep64_kernel<0><<<(unsigned)parts_r, kPassThreads, smem, st>>>(
        rows, p, 32 + 8 * p, in, out, b.digit_start, b.sort_status, b.hdr, nullptr, nullptr, 0u,
        nullptr, nullptr, nullptr, 0);
    GS_CHECK_LAUNCH();
    uint64_t* t = in; in = out; out = t;
  }
  // the sorted rows are back in ra
  const int64_t eparts = div_up(rows_max, kEmitPart);
  GS_CUDA(cudaMemsetAsync(b.emit_status, 0, sizeof(uint64_t) * (size_t)eparts, st));
  // the balanced emission; with two tile passes or more its list is made
  // by the first tile pass itself (onesweep64_kernel<2>) instead
  const bool chunked = isect_max >= kEmitChunkMinTiles * rows_max;
  const bool generate = chunked && s.tile_passes > 1;
  if (chunked) {
    row_scan_kernel<<<(unsigned)eparts, kEmitThreads, 0, st>>>(
        rows, s.tiles_x, s.tile_passes, (uint32_t)s.n, ra, b.row_rect, b.row_d, b.erow,
        b.chunk_row, b.hist,
        b.emit_status, b.hdr);
    GS_CHECK_LAUNCH();
    if (!generate)
      emit_chunks_kernel<<<(unsigned)div_up(isect_max, kEmitChunk), kEmitThreads, 0, st>>>(
          s.tiles_x, b.erow, b.chunk_row, rb, b.hdr);
  } else {
    emit_sorted_kernel<<<(unsigned)eparts, kEmitThreads, 0, st>>>(
        rows, s.tiles_x, s.tile_passes, (uint32_t)s.n, ra, b.row_rect, b.row_d, rb, b.hist,
        b.emit_status, b.hdr);
  }
  GS_CHECK_LAUNCH();
  hist_scan_kernel<<<s.tile_passes, kRadix, 0, st>>>(b.hist + kDepthPasses * kRadix,
                                                     b.digit_start + kDepthPasses * kRadix);
  GS_CHECK_LAUNCH();
  in = rb;
  for (int q = 0; q < s.tile_passes; ++q) {
    const int p = kDepthPasses + q;
    if (q == s.tile_passes - 1) {
      onesweep64_kernel<1><<<(unsigned)parts_i, kPassThreads, smem, st>>>(
          isect, p, 32 + 8 * q, in, keys, b.digit_start, b.sort_status, b.hdr, b.row_d, vals,
          (uint32_t)s.n, reinterpret_cast<unsigned long long*>(ranges), nullptr, nullptr, 0);
    } else if (q == 0 && generate) {
      out = in == keys ? b.tmp : keys;
      onesweep64_kernel<2><<<(unsigned)parts_i, kPassThreads, smem, st>>>(
          isect, p, 32, nullptr, out, b.digit_start, b.sort_status, b.hdr, nullptr, nullptr, 0u,
          nullptr, b.erow, b.chunk_row, s.tiles_x);
      in = out;
    } else {
      out = in == keys ? b.tmp : keys;
      onesweep64_kernel<0><<<(unsigned)parts_i, kPassThreads, smem, st>>>(
          isect, p, 32 + 8 * q, in, out, b.digit_start, b.sort_status, b.hdr, nullptr, nullptr, 0u,
          nullptr, nullptr, nullptr, 0);
      in = out;
    }
    GS_CHECK_LAUNCH();
  }
  const int64_t fix_blocks = div_up(s.n_flat, 256) < 1024 ? div_up(s.n_flat, 256) : 1024;
  ranges_fix_kernel<<<(unsigned)fix_blocks, 256, 0, st>>>(isect, s.n_flat, ranges, b.hdr);
  GS_CHECK_LAUNCH();
  return GS_OK;
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
  // One compaction partition is launched with ticket 1, so it looks back at
  // partition 0, which never runs: its bounded wait must run out, flag the
  // error and return.  Reads and writes no row data (zero rows).
  const WsLayout L = ws_layout(1, 1);
  if (!workspace || ws_bytes < L.total || !aligned16(workspace)) return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const BinBufs b = bin_bufs(workspace, L);
  GS_CUDA(cudaMemsetAsync(b.hdr, 0, sizeof(WsHeader), st));
  GS_CUDA(cudaMemsetAsync(b.scan_status, 0, sizeof(uint64_t) * 2, st));
  const unsigned one = 1;
  GS_CUDA(cudaMemcpyAsync(&b.hdr->scan_ticket, &one, sizeof(one), cudaMemcpyHostToDevice, st));
  compact_rows_kernel<4><<<1, kCompThreads, 0, st>>>(0, 1, 1, 1, 1, 1, nullptr, nullptr, b.tmp,
                                                     b.row_rect, b.hist, b.scan_status,
                                                     b.hdr);
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
                                     const int32_t* tile_counts, int32_t width, int32_t height, void* workspace,
                                     size_t ws_bytes, int64_t capacity, uint64_t* keys,
                                     uint32_t* vals, int64_t* ranges, int64_t* n_isect,
                                     void* stream) {
  BinShape s;
  if (!bin_shape(n, n_views, width, height, s) || capacity < 0 ||
      capacity > (int64_t)0xFFFFFFFFll || !n_isect || !workspace)
    return GS_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(s.n_rows, capacity);
  if (ws_bytes < L.total || !aligned16(workspace)) return GS_ERR_INVALID_ARG;
  if (!ranges || (s.n_rows > 0 && (!splats || !aligned16(splats))) || !aligned4(tile_counts) ||
      (capacity > 0 && (!keys || !vals)))
    return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const BinBufs b = bin_bufs(workspace, L);

  // 1. compaction (tickets, counts and histograms reset; the status word is kept)
  GS_CUDA(cudaMemsetAsync(&b.hdr->scan_ticket, 0,
                          sizeof(WsHeader) - offsetof(WsHeader, scan_ticket), st));
  GS_CUDA(cudaMemsetAsync(&b.hdr->total, 0, sizeof(b.hdr->total), st));
  GS_CUDA(cudaMemsetAsync(b.hist, 0, sizeof(uint32_t) * kMaxPasses * kRadix, st));
  if (s.n_rows > 0) {
    const gs_status e = launch_compaction(s, b, splats, tile_counts, capacity, keys, st);
    if (e != GS_OK) return e;
  }
  struct { unsigned long long total; unsigned int error, ticket; unsigned long long rows; } h{};
  static_assert(sizeof(h) == 24, "header prefix");
  GS_CUDA(cudaMemcpyAsync(&h, b.hdr, sizeof(h), cudaMemcpyDeviceToHost, st));
  GS_CUDA(cudaStreamSynchronize(st));
  if (h.error & ~kErrCapacity) {  // a capacity bit can only be left by an asynchronous call
    GS_CUDA(cudaMemsetAsync(&b.hdr->error, 0, sizeof(unsigned int), st));
    return (h.error & 1u) ? GS_ERR_TIMEOUT : GS_ERR_DEVICE_CHECK;
  }
  const int64_t I = (int64_t)h.total, R = (int64_t)h.rows;
  *n_isect = I;
  if (I > capacity) return GS_ERR_CAPACITY;
  check_capacity_kernel<<<1, 1, 0, st>>>(b.hdr, capacity, nullptr);  // clears the bit
  GS_CHECK_LAUNCH();
  GS_CUDA(cudaMemsetAsync(ranges, 0, sizeof(int64_t) * 2 * (size_t)s.n_flat, st));
  if (I == 0) return GS_OK;
  return launch_sort_stages(s, b, R, I, R, I, keys, vals, ranges, st);
}

// ---------------------------------------------------------------------------
// Morton order entry points

struct MortonLayout {
  size_t hist, digit_start, sort_status, keys_a, keys_b, vals_b, total;
};

inline MortonLayout morton_layout(int64_t n) {
  const size_t m = (size_t)(n > 0 ? n : 1);
  MortonLayout L;
  size_t off = sizeof(WsHeader);
  L.hist = off;        off += align256(sizeof(uint32_t) * kMaxPasses * kRadix);
  L.digit_start = off; off += align256(sizeof(uint32_t) * kMaxPasses * kRadix);
  L.sort_status = off; off += align256(sizeof(uint64_t) * kRadix * (size_t)div_up((int64_t)m, kSortPart));
  L.keys_a = off;      off += align256(sizeof(uint64_t) * m);
  L.keys_b = off;      off += align256(sizeof(uint64_t) * m);
  L.vals_b = off;      off += align256(sizeof(uint32_t) * m);
  L.total = off;
  return L;
}

static size_t morton_ws_bytes(int64_t n) { return morton_layout(n).total; }

extern "C" size_t gs_morton_workspace_bytes(int64_t n) { return morton_ws_bytes(n); }

extern "C" gs_status gs_morton_order(int64_t n, const float* params, void* workspace,
                                     size_t ws_bytes, uint32_t* perm, void* stream) {
  if (n < 0 || n > (int64_t)0xFFFFFFFFll || !workspace || !aligned16(workspace) ||
      ws_bytes < morton_ws_bytes(n) || (n > 0 && (!params || !perm)))
    return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const MortonLayout L = morton_layout(n);
  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + L.hist);
  uint32_t* digit_start = reinterpret_cast<uint32_t*>(ws + L.digit_start);
  uint64_t* sort_status = reinterpret_cast<uint64_t*>(ws + L.sort_status);
  uint64_t* keys_b = reinterpret_cast<uint64_t*>(ws + L.keys_b);
  uint32_t* vals_b = reinterpret_cast<uint32_t*>(ws + L.vals_b);
  uint64_t* keys_a = reinterpret_cast<uint64_t*>(ws + L.keys_a);
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
  const size_t smem = sizeof(SortSmemKV);
  GS_CUDA(ensure_sort_attr());
  uint64_t* k_in = keys_a;
  uint32_t* v_in = perm;
  uint64_t* k_out = keys_b;
  uint32_t* v_out = vals_b;
  for (int p = 0; p < kMortonPasses; ++p) {
    onesweep_kv_kernel<<<(unsigned)sort_parts, kSortThreads, smem, st>>>(
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
// shapes follow the row count and `capacity`, the kernels read the counts
// from the workspace, and an overflow is reported through the workspace
// status word.
extern "C" gs_status gs_bin_and_sort_async(int64_t n, int32_t n_views, const gs_splat* splats,
                                           const int32_t* tile_counts, int32_t width,
                                           int32_t height, void* workspace, size_t ws_bytes,
                                           int64_t capacity, uint64_t* keys, uint32_t* vals,
                                           int64_t* ranges, int64_t* n_isect, void* stream) {
  BinShape s;
  if (!bin_shape(n, n_views, width, height, s) || capacity < 1 ||
      capacity > (int64_t)0xFFFFFFFFll || !workspace || !n_isect)
    return GS_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(s.n_rows, capacity);
  if (ws_bytes < L.total || !aligned16(workspace) || !ranges || !keys || !vals ||
      (s.n_rows > 0 && (!splats || !aligned16(splats))) || !aligned4(tile_counts))
    return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const BinBufs b = bin_bufs(workspace, L);
  GS_CUDA(cudaMemsetAsync(&b.hdr->scan_ticket, 0,
                          sizeof(WsHeader) - offsetof(WsHeader, scan_ticket), st));
  GS_CUDA(cudaMemsetAsync(&b.hdr->total, 0, sizeof(b.hdr->total), st));
  GS_CUDA(cudaMemsetAsync(b.hist, 0, sizeof(uint32_t) * kMaxPasses * kRadix, st));
  GS_CUDA(cudaMemsetAsync(ranges, 0, sizeof(int64_t) * 2 * (size_t)s.n_flat, st));
  if (s.n_rows > 0) {
    const gs_status e = launch_compaction(s, b, splats, tile_counts, capacity, keys, st);
    if (e != GS_OK) return e;
  }
  check_capacity_kernel<<<1, 1, 0, st>>>(b.hdr, capacity, n_isect);
  GS_CHECK_LAUNCH();
  if (s.n_rows == 0) return GS_OK;
  return launch_sort_stages(s, b, -2, -1, s.n_rows, capacity, keys, vals, ranges, st);
}

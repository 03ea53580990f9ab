// raster.cu -- gs_rasterize_fwd, gs_rasterize_bwd, gs_rasterize_fused (and
// gs_rasterize_fused_acc) and gs_zero_grads.
//
// Front-to-back alpha compositing over per-tile sorted lists and its
// analytic backward ("ByteSplat": forward and backward rasterization;
// "On Scaling Up 3D Gaussian Splatting Training": 16x16 pixel blocks and the
// opacity saturation depth at which a pixel stops).
//
// One CTA per (view, 16x16 tile).  The tile's Gaussians are gathered by id
// into shared memory in batches of kBatch with cp.async, double buffered: the
// next batch is in flight while the current one is composited.
//
// Clustered scenes make most pairs skips (alpha < 1/255) and leave a few
// pixels of a tile unsaturated long after the rest have stopped.  Measures
// that cut the work without changing any decision or the order of
// accumulation:
//  - staging: for every entry of a batch, its exponent expanded about the
//    tile pixel where it peaks (exact per-pixel offsets, see below) and the
//    bounding box of the ellipse where alpha may reach 1/255; pairs outside
//    it are skipped, the exact alpha test decides everything inside;
//  - forward: each warp walks only the entries whose box touches its pixels
//    (a ballot-compacted sub-list that keeps list order); pixel state lives
//    in shared memory and, at every batch, the still-open pixels are packed
//    onto the first threads of the CTA, so the per-pair loop runs on full
//    warps and finished warps stop issuing;
//  - backward: each quarter-warp (eight lanes, a 4x2 pixel block) walks its
//    own entry list, the four quarters of a warp in lockstep; a pair's
//    gradient is reduced over the quarter (nine values in ten shuffles)
//    and added to shared memory by one atomic per value;
//  - fused call with a workspace: the forward records, per batch and per
//    quarter, which entries it composited; the backward walks exactly those
//    and hands the quarters to warps by descending count of recorded
//    entries, so that quarters of similar length share a warp;
//  - zeroing of the gradient records the backward adds to: only the pairs
//    of rows of which one is visible, as a call of its own so that it can
//    run beside the binning on another stream;
//  - launch order: CTA b composites tile tile_order[b] when given
//    (gs_tile_order in tile_order.cu: longest lists first), which shortens
//    the kernel's tail.
#include <stdint.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kRT = 256;      // threads per CTA = pixels per tile
constexpr int kWarps = kRT / 32;
// List entries per batch: 192 keeps a CTA of the fused kernel under 37 KB of
// shared memory, so that six CTAs share an SM (the kernels are bound by how
// many warps an SM can switch between: at three CTAs per SM the fused kernel
// took 44 % longer than at five).
constexpr int kBatch = 192;
constexpr int kWords = kBatch / 32;  // 32-bit words of a per-batch entry mask

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Pair exponent.  The pages define, for pixel centre p and a projected
// Gaussian (mean m, conic Q = [[a, b], [b, c]], opacity o),
//   power = -(d^T Q d)/2,  d = p - m,   raw alpha = o e^power.
// Evaluated literally in fp32 this loses accuracy when m lies far from the
// tile (street-level views put the means of elongated ground footprints
// thousands of pixels off screen): p - m then rounds, and Q, near-singular,
// turns a 1e-3 px rounding of d into an error of order one in the exponent.
// So each entry is expanded, once per tile at staging, about a pixel centre
// z of the tile (the one where its exponent is largest):
//   ln o + power(p) = P + G.l - (l^T Q l)/2,   l = p - z,
//   P = ln o - (e^T Q e)/2,  G = -Q e,  e = z - m,
// with P and G computed by error-free transformations to about twice fp32
// precision.  l is a small integer vector, exact, and the terms are of the
// size of the exponent near the footprint, so the per-pair evaluation is as
// accurate as for a Gaussian centred on the tile.  Folding ln o into P turns
// the 1/255 test into a test on the exponent alone.

// Knuth's two-sum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// a1 b1 + a2 b2 as s + e (FMA two-products, then a two-sum of the leading
// parts): the dot product to about twice fp32 precision.
__device__ __forceinline__ void dot2(float a1, float b1, float a2, float b2, float& s, float& e) {
  const float p1 = __fmul_rn(a1, b1), e1 = __fmaf_rn(a1, b1, -p1);
  const float p2 = __fmul_rn(a2, b2), e2 = __fmaf_rn(a2, b2, -p2);
  float t;
  two_sum(p1, p2, s, t);
  e = __fadd_rn(t, __fadd_rn(e1, e2));
}

struct Expansion {
  float P, gx, gy;  // ln o - (e^T Q e)/2 and -Q e, rounded once
  float ex, ey;     // e = z - m, rounded
};

__device__ __forceinline__ Expansion expand_at(float zx, float zy, float mx, float my, float a,
                                               float b, float c, float lno) {
  float ex, exl, ey, eyl;
  two_sum(zx, -mx, ex, exl);
  two_sum(zy, -my, ey, eyl);
  float qx, qxl, qy, qyl;  // Q e
  dot2(a, ex, b, ey, qx, qxl);
  qxl = __fmaf_rn(a, exl, __fmaf_rn(b, eyl, qxl));
  dot2(b, ex, c, ey, qy, qyl);
  qyl = __fmaf_rn(b, exl, __fmaf_rn(c, eyl, qyl));
  float s, sl;  // e^T Q e
  dot2(ex, qx, ey, qy, s, sl);
  sl = __fmaf_rn(ex, qxl, __fmaf_rn(ey, qyl, __fmaf_rn(exl, qx, __fmaf_rn(eyl, qy, sl))));
  Expansion r;
  r.P = __fmaf_rn(-0.5f, s, __fmaf_rn(-0.5f, sl, lno));
  r.gx = -__fadd_rn(qx, qxl);
  r.gy = -__fadd_rn(qy, qyl);
  r.ex = ex;
  r.ey = ey;
  return r;
}

// A box bound in grid indices, clamped to [-1, 16] (NaN -> -1).
__device__ __forceinline__ signed char clamp_index(float v) {
  return (signed char)fminf(fmaxf(v, -1.f), 16.f);
}

// Pixel-centre grid index (0..15) of the tile nearest to coordinate v.
__device__ __forceinline__ float snap(float v, float origin) {
  return fminf(fmaxf(rintf(__fsub_rn(__fsub_rn(v, origin), 0.5f)), 0.f), 15.f);
}

struct Batch {
  float4 a[kBatch];  // as loaded: mean_x, mean_y, conic_a, conic_b
                     // staged:    G_x, G_y, P, -a/2
  float4 b[kBatch];  // as loaded: conic_c, opacity, color_r, color_g
                     // staged:    -b, -c/2, z_x, z_y (grid index in the tile)
  float4 c[kBatch];  // as loaded: color_b, depth, radius, tiles
                     // staged:    color_r, color_g, color_b, opacity
  char4 box[kBatch];  // grid-index box (x0, x1, y0, y1) outside of which
                     // alpha < 1/255 for sure; clamped to [-1, 16]
};

// ln 255, and the exponent below which a pair is skipped without computing
// alpha: alpha = e^exponent < 1/255 there with a margin of 1e-3 (>> the
// rounding error of the exponent).
constexpr float kLn255 = 5.5412635451584f;
constexpr float kPrefilterMargin = 1e-3f;
constexpr float kExpSkip = -kLn255 - kPrefilterMargin;

// Staging of entry j of a landed batch for the tile with origin (ox, oy):
// expansion point, expansion, and the bounding box of the ellipse
// d^T Q d <= 2 (ln(255 o) + margin), half-widths sqrt(q (Q^-1)_xx) and
// sqrt(q (Q^-1)_yy), det Q by Kahan's compensated 2x2 determinant (the plain
// a c - b^2 cancels for elongated footprints).  e_out (backward only)
// receives e = z - m.
__device__ __forceinline__ void stage_entry(Batch& B, int j, float ox, float oy, float2* e_out) {
  const float4 A = B.a[j];
  const float4 Bv = B.b[j];
  const float4 Cv = B.c[j];
  const float mx = A.x, my = A.y, ca = A.z, cb = A.w, cc = Bv.x, o = Bv.y;
  const float lno = __logf(o);
  // Expansion point: the maximum of the exponent over the tile's pixel-centre
  // box, snapped to the grid.  Inside the box that is the mean; outside, the
  // better of the maxima along the (at most two) edges that face the mean,
  // compared by a plain fp32 quadratic (a wrong pick can only happen between
  // near-equal candidates, either of which serves).  Only the choice of z
  // depends on these approximate values; selects keep the warp converged.
  const float x0 = ox + 0.5f, x1 = ox + 15.5f, y0 = oy + 0.5f, y1 = oy + 15.5f;
  const bool inx = mx >= x0 && mx <= x1, iny = my >= y0 && my <= y1;
  const float X = mx < x0 ? x0 : x1, Y = my < y0 ? y0 : y1;
  const float ys = my - __fdividef(cb, cc) * (X - mx);  // edge x = X
  const float xs = mx - __fdividef(cb, ca) * (Y - my);  // edge y = Y
  const float c1x = !inx ? X : (!iny ? xs : mx), c1y = !inx ? ys : (!iny ? Y : my);
  const float c2x = (!inx && !iny) ? xs : c1x, c2y = (!inx && !iny) ? Y : c1y;
  const float k1x = snap(c1x, ox), k1y = snap(c1y, oy);
  const float k2x = snap(c2x, ox), k2y = snap(c2y, oy);
  const float d1x = ox + k1x + 0.5f - mx, d1y = oy + k1y + 0.5f - my;
  const float d2x = ox + k2x + 0.5f - mx, d2y = oy + k2y + 0.5f - my;
  const float s1 = ca * d1x * d1x + 2.f * cb * d1x * d1y + cc * d1y * d1y;
  const float s2 = ca * d2x * d2x + 2.f * cb * d2x * d2y + cc * d2y * d2y;
  const bool second = s2 < s1;
  const float kx = second ? k2x : k1x, ky = second ? k2y : k1y;
  const Expansion E = expand_at(ox + kx + 0.5f, oy + ky + 0.5f, mx, my, ca, cb, cc, lno);
  B.a[j] = make_float4(E.gx, E.gy, E.P, -0.5f * ca);
  B.b[j] = make_float4(-cb, -0.5f * cc, kx, ky);
  B.c[j] = make_float4(Bv.z, Bv.w, Cv.x, o);
  if (e_out) e_out[j] = make_float2(E.ex, E.ey);
  // bounding box in grid indices of the tile: pixel k's centre is at index
  // coordinate k and the ellipse centre at k - e; the padding (1e-3 px +
  // 1e-4 hw) exceeds the rounding of k - e (|e| <= hw + 16 when the ellipse
  // reaches the tile)
  char4 box = make_char4(16, -1, 16, -1);  // empty
  const float q = 2.f * (kLn255 + lno + kPrefilterMargin);
  if (q > 0.f) {
    const float w = __fmul_rn(cb, cb);
    const float det = __fadd_rn(__fmaf_rn(ca, cc, -w), __fmaf_rn(-cb, cb, w));
    // approximate division and square root: the 1e-4 relative padding covers
    // their few-ulp errors; det 0 gives inf or NaN, an indefinite Q NaN
    const float qx = __fdividef(q * cc, det), qy = __fdividef(q * ca, det);
    const float hw = qx * rsqrtf(qx) * 1.0001f + 1e-3f;
    const float hh = qy * rsqrtf(qy) * 1.0001f + 1e-3f;
    if (hw >= 0.f && hh >= 0.f && hw < 1e30f && hh < 1e30f) {  // else keep all
      const float cxk = kx - E.ex, cyk = ky - E.ey;
      box = make_char4(clamp_index(ceilf(cxk - hw)), clamp_index(floorf(cxk + hw)),
                       clamp_index(ceilf(cyk - hh)), clamp_index(floorf(cyk + hh)));
    } else {
      box = make_char4(-1, 16, -1, 16);
    }
  }
  B.box[j] = box;
}

// ln o + power of a staged entry at the pixel with grid index (ix, iy), with
// a fixed rounding sequence shared by the forward and the backward so both
// take identical decisions; (lx, ly) = l, the exact offsets from z.
__device__ __forceinline__ float pair_exponent(const float4& A, const float4& Bv, float ix,
                                               float iy, float& lx, float& ly) {
  lx = __fsub_rn(ix, Bv.z);
  ly = __fsub_rn(iy, Bv.w);
  const float t1 = __fmaf_rn(A.w, lx, __fmaf_rn(Bv.x, ly, A.x));  // G_x - a l_x/2 - b l_y
  const float t2 = __fmaf_rn(Bv.y, ly, A.y);                      // G_y - c l_y/2
  return __fmaf_rn(lx, t1, __fmaf_rn(ly, t2, A.z));
}

__device__ __forceinline__ bool box_hits(char4 b, int x0, int x1, int y0, int y1) {
  return !(b.y < x0 || b.x > x1 || b.w < y0 || b.z > y1);
}

// Pixel p of the tile (0..255): warp w = p >> 5 covers an 8x4 block and each
// quarter of the warp (lanes 8q..8q+7) a 4x2 block of it -- quarters 0, 1 on
// top (left, right), 2, 3 below -- so that the eight lanes of a quarter form
// one phase of a 128-bit shared-memory access.
__device__ __forceinline__ void pixel_of(int p, int tile_x, int tile_y, int& px, int& py) {
  const int warp = p >> 5, q = (p >> 3) & 3, r = p & 7;
  px = tile_x * GS_TILE + (warp & 1) * 8 + (q & 1) * 4 + (r & 3);
  py = tile_y * GS_TILE + (warp >> 1) * 4 + (q >> 1) * 2 + (r >> 2);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums over the eight lanes of a quarter.  quarter_sum8 reduces 8 values by
// recursive halving (at each of three exchange rounds a lane keeps half of its
// values and sends the other half to its partner: 7 shuffles); lane r of the
// quarter (r = lane & 7) returns the quarter's sum of value r.
__device__ __forceinline__ float quarter_sum8(const float v[8], int lane) {
  const bool h1 = lane & 4, h2 = lane & 2, h3 = lane & 1;
  float k1[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = h1 ? v[4 + i] : v[i];
    const float send = h1 ? v[i] : v[4 + i];
    k1[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  float k2[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = h2 ? k1[2 + i] : k1[i];
    const float send = h2 ? k1[i] : k1[2 + i];
    k2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  return (h3 ? k2[1] : k2[0]) + __shfl_xor_sync(0xffffffffu, h3 ? k2[0] : k2[1], 1);
}

__device__ __forceinline__ float quarter_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v + __shfl_xor_sync(0xffffffffu, v, 1);
}

// Pixel state of a tile during the forward pass, by pixel index.
struct PixState {
  float T[kRT], Tl[kRT], C0[kRT], C1[kRT], C2[kRT];  // T = T + Tl (double-float)
  int32_t last[kRT];
  uint8_t done[kRT];
  uint8_t list[kRT];  // open pixels, packed
};

__device__ __forceinline__ void pix_init(PixState& P, int tid, int tile_x, int tile_y, int W,
                                         int H) {
  int px, py;
  pixel_of(tid, tile_x, tile_y, px, py);
  P.T[tid] = 1.f;
  P.Tl[tid] = 0.f;
  P.C0[tid] = P.C1[tid] = P.C2[tid] = 0.f;
  P.last[tid] = 0;
  P.done[tid] = (px < W && py < H) ? 0 : 1;
}

// Writes into wl[0..] the entries j < cnt (ascending) whose box meets the
// grid-index rectangle [x0, x1] x [y0, y1]; returns their number.  Whole-warp
// call.
__device__ __forceinline__ int warp_sublist(const Batch& B, int cnt, int x0, int x1, int y0,
                                            int y1, uint8_t* wl, int lane) {
  int n = 0;
  for (int c0 = 0; c0 < cnt; c0 += 32) {
    const int j = c0 + lane;
    const bool hit = j < cnt && box_hits(B.box[j], x0, x1, y0, y1);
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (hit) wl[n + __popc(bal & ((1u << lane) - 1u))] = (uint8_t)j;
    n += __popc(bal);
  }
  __syncwarp();
  return n;
}

// Forward compositing of staged batch k over the m open pixels packed in
// P.list[0..m): each worker thread takes one open pixel; each warp walks the
// entries whose box meets its pixels.  With `rec`, every composited pair also
// sets bit j of the record of its pixel's 4x2 quarter (p >> 3).
template <bool kCount, bool kImp, int kUnroll>
__device__ __forceinline__ void fwd_batch(PixState& P, const Batch& B, uint8_t* wl, int cnt, int k,
                                          int m, int tile_x, int tile_y, int tid, int warp,
                                          int lane, unsigned long long& n_tested,
                                          unsigned long long& n_included, const uint32_t* ids,
                                          float* imp, int32_t* pix_counts, int64_t plane,
                                          int32_t W, uint32_t (*rec)[kWords]) {
  if (warp * 32 >= m) return;
  const bool worker = tid < m;
  const int p = worker ? P.list[tid] : 0;
  int px, py;
  pixel_of(p, tile_x, tile_y, px, py);
  const int kx = px - tile_x * GS_TILE, ky = py - tile_y * GS_TILE;  // grid index
  const float ix = (float)kx, iy = (float)ky;
  const int x0 = __reduce_min_sync(0xffffffffu, worker ? kx : 1 << 30);
  const int x1 = __reduce_max_sync(0xffffffffu, worker ? kx : -(1 << 30));
  const int y0 = __reduce_min_sync(0xffffffffu, worker ? ky : 1 << 30);
  const int y1 = __reduce_max_sync(0xffffffffu, worker ? ky : -(1 << 30));
  const int nw = warp_sublist(B, cnt, x0, x1, y0, y1, wl, lane);
  if (!worker) return;
  // T is carried as an unevaluated sum Tr + Tl, so its rounding error does
  // not grow with the number of contributors (city-scale lists reach 10^4
  // entries); the colour of this batch is summed apart and added once at the
  // end of the batch.
  float Tr = P.T[p], Tl = P.Tl[p];
  float C0 = 0.f, C1 = 0.f, C2 = 0.f;
  int32_t last = P.last[p];
  int done = 0;
  int stop_j = cnt;
  int32_t n_inc = 0;
  const int32_t base1 = k * kBatch + 1;  // 1-based list position of entry 0
#pragma unroll kUnroll
  for (int i = 0; i < nw; ++i) {
    const int j = wl[i];
    const float4 A = B.a[j];
    const float4 Bv = B.b[j];
    float lx, ly;
    const float ex = pair_exponent(A, Bv, ix, iy, lx, ly);
    if (ex < kExpSkip) continue;
    const float alpha = fminf(kAlphaMax, __expf(ex));
    if (alpha < kAlphaMin) continue;
    const float om = __fsub_rn(1.f, alpha);
    const float oml = __fsub_rn(__fsub_rn(1.f, om), alpha);  // 1 - alpha = om + oml
    const float ph = __fmul_rn(Tr, om);
    const float lo = __fmaf_rn(Tr, oml, __fmaf_rn(Tl, om, __fmaf_rn(Tr, om, -ph)));
    const float Tn = __fadd_rn(ph, lo);
    if (Tn < kTMin) { done = 1; stop_j = j + 1; break; }
    const float w = __fmul_rn(alpha, Tr);
    const float4 Cv = B.c[j];
    C0 = __fmaf_rn(w, Cv.x, C0);
    C1 = __fmaf_rn(w, Cv.y, C1);
    C2 = __fmaf_rn(w, Cv.z, C2);
    Tl = __fsub_rn(lo, __fsub_rn(Tn, ph));
    Tr = Tn;
    last = base1 + j;
    if (kCount) ++n_inc;
    if (rec) atomicOr(&rec[p >> 3][j >> 5], 1u << (j & 31));
    // largest blending weight of the Gaussian (w >= 0: the bits order as the values)
    if (kImp) atomicMax(reinterpret_cast<unsigned int*>(imp + ids[j]), __float_as_uint(w));
  }
  if (kCount) {
    n_tested += stop_j;
    n_included += n_inc;
    if (pix_counts) {  // this batch's share of the pixel's tested / composited pairs
      const int64_t q = (int64_t)py * W + px;
      atomicAdd(pix_counts + q, stop_j);
      atomicAdd(pix_counts + plane + q, n_inc);
    }
  }
  P.T[p] = Tr;
  P.Tl[p] = Tl;
  P.C0[p] = __fadd_rn(P.C0[p], C0);
  P.C1[p] = __fadd_rn(P.C1[p], C1);
  P.C2[p] = __fadd_rn(P.C2[p], C2);
  P.last[p] = last;
  P.done[p] = done;
}

// The forward over a tile's list [start, end): batches of kBatch gathered by
// cp.async into the two slots of `b` (batch k in slot k & 1), one batch
// ahead.  The open pixels are counted at the end of each batch, before the
// next one is prefetched, so when every pixel has stopped the last batch
// composited is still staged in its slot; on return `staged` holds the
// batch index staged in each slot (-1: none).  With `ids`/`E` the staging
// also records each entry's id and e = z - m (for a backward that reuses the
// slots).  slot(s, i) names the batch index staged in slot i.  kImp: also
// record each Gaussian's largest blending weight into imp (ids required).
__device__ __forceinline__ int& slot(int2& s, int i) { return i ? s.y : s.x; }

template <bool kCount, bool kImp = false, int kUnroll = 1>
__device__ __forceinline__ void fwd_tile(PixState& P, Batch* b, uint32_t (*ids)[kBatch],
                                         float2 (*E)[kBatch], uint8_t (*wl)[kBatch], int32_t* wcount,
                                         const float4* vsplat, const uint32_t* __restrict__ vals,
                                         int64_t n, int64_t start, int64_t end, int tile_x,
                                         int tile_y, float ox, float oy, int tid, int warp,
                                         int lane, int2& staged,
                                         unsigned long long& n_tested,
                                         unsigned long long& n_included, float* imp = nullptr,
                                         int32_t* pix_counts = nullptr, int64_t plane = 0,
                                         int32_t W = 0, uint32_t (*rec)[kWords] = nullptr,
                                         uint32_t* __restrict__ rec_out = nullptr) {
  const int64_t len = end - start;
  const int nb = (int)((len + kBatch - 1) / kBatch);
  staged = make_int2(-1, -1);
  auto issue = [&](int k) {
    const int64_t e = start + (int64_t)k * kBatch + tid;
    if (tid < kBatch && e < end) {
      // ids come from gs_bin_and_sort; clamping keeps a corrupt list in bounds
      const uint32_t id = min(__ldg(vals + e), (uint32_t)(n - 1));
      const float4* src = vsplat + 3 * (int64_t)id;
      Batch& B = b[k & 1];
      if (ids) ids[k & 1][tid] = id;
      cp_async16(&B.a[tid], src);
      cp_async16(&B.b[tid], src + 1);
      cp_async16(&B.c[tid], src + 2);
    }
    cp_async_commit();
  };
  if (nb > 0) issue(0);
  unsigned bal = __ballot_sync(0xffffffffu, !P.done[tid]);
  if (lane == 0) wcount[warp] = __popc(bal);
  for (int k = 0; k < nb; ++k) {
    cp_async_wait<0>();
    __syncthreads();  // batch k landed; the open-pixel counts are visible
    int off = 0, m = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcount[w];
      off += w < warp ? c : 0;
      m += c;
    }
    if (m == 0) break;
    if (k + 1 < nb) {
      issue(k + 1);
      slot(staged, (k + 1) & 1) = -1;
    }
    Batch& B = b[k & 1];
    const int cnt = (int)min((int64_t)kBatch, len - (int64_t)k * kBatch);
    if (tid < cnt) stage_entry(B, tid, ox, oy, E ? E[k & 1] : nullptr);
    slot(staged, k & 1) = k;
    if ((bal >> lane) & 1u) P.list[off + __popc(bal & ((1u << lane) - 1u))] = tid;
    __syncthreads();
    fwd_batch<kCount, kImp, kUnroll>(P, B, wl[warp], cnt, k, m, tile_x, tile_y, tid, warp, lane,
                                     n_tested, n_included, ids ? ids[k & 1] : nullptr, imp,
                                     pix_counts, plane, W, rec_out ? rec : nullptr);
    __syncthreads();  // pixel state written; slot k & 1 free for batch k + 2
    if (rec_out && tid < kRT / 8 * kWords) {  // this batch's record of the composited entries
      __stcg(rec_out + (int64_t)k * (kRT / 8 * kWords) + tid, (&rec[0][0])[tid]);
      (&rec[0][0])[tid] = 0u;
    }
    bal = __ballot_sync(0xffffffffu, !P.done[tid]);
    if (lane == 0) wcount[warp] = __popc(bal);
  }
  cp_async_wait<0>();
  __syncthreads();
}

// Backward pairs of one staged batch for this thread's pixel (list positions
// lo + j), back to front; per-entry sums into acc.  The lane's quarter walks
// the entries set in its mask qw[0..nw) (bit j of word j >> 5), highest
// first; the four quarters of the warp advance together, one entry each per
// step, so a step costs the longest of four short lists, and a pair's
// gradient is reduced over the quarter's eight lanes (10 shuffles).  A
// quarter that has no entry left, or no contributing lane, adds nothing.
__device__ __forceinline__ void bwd_walk(const Batch& B, float (*acc)[9], const uint32_t* qw,
                                         int nw, int lo, float ix, float iy, int last, float& Tr,
                                         float& S0, float& S1, float& S2, float g0, float g1,
                                         float g2, int lane) {
  const int r = lane & 7;
  int wi = nw - 1;
  uint32_t bits = wi >= 0 ? qw[wi] : 0u;
  while (true) {
    while (bits == 0u && wi > 0) bits = qw[--wi];
    const bool act = bits != 0u;
    if (!__any_sync(0xffffffffu, act)) break;
    int j = 0;
    if (act) {
      const int b = 31 - __clz(bits);
      bits ^= 1u << b;
      j = (wi << 5) | b;
    }
    const int pos = lo + j;
    float v[9];
#pragma unroll
    for (int c = 0; c < 9; ++c) v[c] = 0.f;
    bool contrib = false;
    if (act && pos < last) {
      const float4 A = B.a[j];
      const float4 Bv = B.b[j];
      float lx, ly;
      const float ex = pair_exponent(A, Bv, ix, iy, lx, ly);
      if (ex >= kExpSkip) {
        const float raw = __expf(ex);
        const float alpha = fminf(kAlphaMax, raw);
        if (alpha >= kAlphaMin) {
          contrib = true;
          const float4 Cv = B.c[j];
          const float oma = 1.f - alpha;
          const float rinv = __fdividef(1.f, oma);  // ~2 ulp; decides nothing
          const float Ti = Tr * rinv;
          const float w = alpha * Ti;
          v[6] = w * g0;
          v[7] = w * g1;
          v[8] = w * g2;
          const float dalpha = (g0 * Cv.x + g1 * Cv.y + g2 * Cv.z) * Ti -
                               (g0 * S0 + g1 * S1 + g2 * S2) * rinv;
          S0 += w * Cv.x;
          S1 += w * Cv.y;
          S2 += w * Cv.z;
          Tr = Ti;
          if (raw < kAlphaMax) {
            // moments of dL/dpower over the entry's pixels in the offsets
            // l = p - z; the flush turns them into the mean, conic and
            // opacity gradients with d = l + e
            const float dpow = dalpha * raw;
            const float p1 = dpow * lx, p2 = dpow * ly;
            v[0] = p1;
            v[1] = p2;
            v[2] = p1 * lx;
            v[3] = p1 * ly;
            v[4] = p2 * ly;
            v[5] = dpow;
          }
        }
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, contrib);
    if (bal) {
      // value r of the quarter ends on lane r (one shared atomic each), value
      // 8 on every lane; only quarters with a contributing lane add
      const float s8 = quarter_sum8(v, lane);
      const float s9 = quarter_sum(v[8]);
      if ((bal >> (lane & 24)) & 0xffu) {
        atomicAdd(&acc[j][r], s8);
        if (r == 0) atomicAdd(&acc[j][8], s9);
      }
    }
  }
  __syncwarp();
}

// The masks of the warp's quarters for one staged batch (cnt entries): the
// entries whose box meets the quarter's 4x2 block (origin wx0, wy0 of the
// warp's 8x4 block) and that lie below the quarter's last contributor
// (qlast[q]); into qm[q][0..nw), *nw = the words to walk.  Whole-warp call.
__device__ __forceinline__ int box_masks(const Batch& B, uint32_t (*qm)[kWords],
                                         const int32_t* qlast, int cnt, int lo, int wx0, int wy0,
                                         int lane) {
  const int4 ql = *reinterpret_cast<const int4*>(qlast);
  const int t0 = max(0, min(cnt, ql.x - lo)), t1 = max(0, min(cnt, ql.y - lo));
  const int t2 = max(0, min(cnt, ql.z - lo)), t3 = max(0, min(cnt, ql.w - lo));
  const int nchunk = (max(max(t0, t1), max(t2, t3)) + 31) >> 5;
  for (int c = 0; c < nchunk; ++c) {
    const int j = (c << 5) + lane;
    const char4 bx = B.box[j];  // j < kBatch; entries >= cnt are excluded by the tops
    const bool xl = !(bx.y < wx0 || bx.x > wx0 + 3), xr = !(bx.y < wx0 + 4 || bx.x > wx0 + 7);
    const bool yt = !(bx.w < wy0 || bx.z > wy0 + 1), yb = !(bx.w < wy0 + 2 || bx.z > wy0 + 3);
    const unsigned b0 = __ballot_sync(0xffffffffu, xl && yt && j < t0);
    const unsigned b1 = __ballot_sync(0xffffffffu, xr && yt && j < t1);
    const unsigned b2 = __ballot_sync(0xffffffffu, xl && yb && j < t2);
    const unsigned b3 = __ballot_sync(0xffffffffu, xr && yb && j < t3);
    if (lane == 0) {
      qm[0][c] = b0;
      qm[1][c] = b1;
      qm[2][c] = b2;
      qm[3][c] = b3;
    }
  }
  __syncwarp();
  return nchunk;
}

// Descending order of the 32 quarters of a tile by a per-quarter count (ties
// by quarter index): lane L of the calling warp returns the index of the
// L-th largest.  Bitonic network over the warp's lanes; whatever the counts,
// the result is a permutation of 0..31.
__device__ __forceinline__ int quarter_rank_order(int count, int lane) {
  int key = count, val = lane;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int ok = __shfl_xor_sync(0xffffffffu, key, j);
      const int ov = __shfl_xor_sync(0xffffffffu, val, j);
      const bool other_first = ok > key || (ok == key && ov < val);  // other precedes mine
      const bool keep_first = ((lane & k) == 0) == ((lane & j) == 0);
      if (keep_first == other_first) {
        key = ok;
        val = ov;
      }
    }
  }
  return val;
}

// The last contributor of each quarter of the warp (the largest `last` over
// its eight pixels) into qlast[0..3]; whole-warp call.
__device__ __forceinline__ void quarter_last(int last, int32_t* qlast, int lane) {
  int m = max(last, __shfl_xor_sync(0xffffffffu, last, 4));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
  if ((lane & 7) == 0) qlast[lane >> 3] = m;
  __syncwarp();
}

// Flush of a batch's per-entry sums (entries tid < cnt) into the row
// gradients of the view, then the sums are cleared.
__device__ __forceinline__ void bwd_flush(const Batch& B, const float2* E, const uint32_t* id,
                                          float (*acc)[9], int cnt, float4* __restrict__ vgrads,
                                          int tid) {
  if (tid >= cnt) return;
  float* a = acc[tid];
  bool nz = false;
#pragma unroll
  for (int c = 0; c < 9; ++c) nz |= a[c] != 0.f;
  if (nz) {
    float4* dst = vgrads + 3 * (int64_t)id[tid];
    // with s = sum dL/dpower, sx = sum dL/dpower l_x, ... and d = l + e:
    //   dL/dm = Q sum dL/dpower d = Q (sx, sy) - s G   (G = -Q e, staged to
    //   full precision: Q e itself cancels for far, elongated footprints),
    //   dL/d(a, b, c) = -(1/2, 1, 1/2) sum dL/dpower (d_x^2, d_x d_y, d_y^2),
    //   dL/do = s / o
    const float s0 = a[5], sx = a[0], sy = a[1];
    const float2 e = E[tid];
    const float4 A = B.a[tid], Bv = B.b[tid];
    const float ca = -2.f * A.w, cb = -Bv.x, cc = -2.f * Bv.y;
    const float gmx = ca * sx + cb * sy - s0 * A.x;
    const float gmy = cb * sx + cc * sy - s0 * A.y;
    const float dy = sy + e.y * s0;  // sum dL/dpower d_y
    const float gca = -0.5f * (a[2] + e.x * (2.f * sx + e.x * s0));
    const float gcb = -(a[3] + e.x * dy + e.y * sx);
    const float gcc = -0.5f * (a[4] + e.y * (2.f * sy + e.y * s0));
    const float dop = s0 / B.c[tid].w;  // staged opacity
    atomicAdd(dst, make_float4(gmx, gmy, gca, gcb));
    atomicAdd(dst + 1, make_float4(gcc, dop, a[6], a[7]));
    atomicAdd(reinterpret_cast<float*>(dst + 2), a[8]);
  }
#pragma unroll
  for (int c = 0; c < 9; ++c) a[c] = 0.f;
}

template <bool kImp>
struct FwdSmem {
  Batch b[2];
  uint32_t id[2][kImp ? kBatch : 1];  // ids of the staged entries (importance variant)
  PixState px;
  int32_t wcount[kWarps];
  uint8_t wl[kWarps][kBatch];  // per-warp entry sub-lists
};

// kCount: also accumulate the pairs tested / included into counts[0..1]
// (instrumentation for work accounting: "tested" counts every list entry a
// pixel passes before it stops, whether or not its box was visited).
// kImp: also record every row's largest blending weight alpha T into imp.
template <bool kCount, bool kImp>
__global__ void __launch_bounds__(kRT, 6) raster_fwd_kernel(
    int64_t n, int32_t tiles_x, int64_t T, int32_t W, int32_t H, const float4* __restrict__ splats,
    const uint32_t* __restrict__ vals, const int64_t* __restrict__ ranges,
    const uint32_t* __restrict__ tile_order, float bg0, float bg1, float bg2, float* __restrict__ image, float* __restrict__ T_final,
    int32_t* __restrict__ n_contrib, unsigned long long* __restrict__ counts,
    int32_t* __restrict__ pix_counts, float* __restrict__ imp) {
  __shared__ FwdSmem<kImp> S;
  unsigned long long n_tested = 0, n_included = 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t flat = tile_order ? (int64_t)tile_order[blockIdx.x] : (int64_t)blockIdx.x;
  const int64_t view = flat / T;
  const int32_t tile = (int32_t)(flat - view * T);
  const int tile_x = tile % tiles_x, tile_y = tile / tiles_x;
  const float ox = (float)(tile_x * GS_TILE), oy = (float)(tile_y * GS_TILE);
  pix_init(S.px, tid, tile_x, tile_y, W, H);
  int2 staged;
  fwd_tile<kCount, kImp>(S.px, S.b, kImp ? reinterpret_cast<uint32_t(*)[kBatch]>(&S.id[0][0]) : nullptr,
                         nullptr, S.wl, S.wcount,
                         splats + 3 * view * n, vals, n, ranges[2 * flat], ranges[2 * flat + 1],
                         tile_x, tile_y, ox, oy, tid, warp, lane, staged, n_tested, n_included,
                         kImp ? imp + view * n : nullptr,
                         pix_counts ? pix_counts + view * (int64_t)W * H : nullptr,
                         (int64_t)gridDim.x / T * W * H, W);
  {
    int px, py;
    pixel_of(tid, tile_x, tile_y, px, py);
    if (px < W && py < H) {
      const int64_t HW = (int64_t)W * H;
      const int64_t pix = (int64_t)py * W + px;
      const float Tr = S.px.T[tid];
      image[(view * 3 + 0) * HW + pix] = S.px.C0[tid] + Tr * bg0;
      image[(view * 3 + 1) * HW + pix] = S.px.C1[tid] + Tr * bg1;
      image[(view * 3 + 2) * HW + pix] = S.px.C2[tid] + Tr * bg2;
      T_final[view * HW + pix] = Tr;
      n_contrib[view * HW + pix] = S.px.last[tid];
    }
  }
  if (kCount) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_tested += __shfl_xor_sync(0xffffffffu, n_tested, o);
      n_included += __shfl_xor_sync(0xffffffffu, n_included, o);
    }
    if (lane == 0) {
      atomicAdd(&counts[0], n_tested);
      atomicAdd(&counts[1], n_included);
    }
  }
}

struct BwdSmem {
  Batch b[2];
  float2 e[2][kBatch];  // e = z - m of the staged entries
  uint32_t id[2][kBatch];
  float acc[kBatch][9];
  uint32_t qm[kWarps][4][kWords];  // per-quarter entry masks of the batch
  alignas(16) int32_t qlast[kWarps][4];  // per-quarter last contributor
  int max_last;
};

__global__ void __launch_bounds__(kRT, 6) raster_bwd_kernel(
    int64_t n, int32_t tiles_x, int64_t T, int32_t W, int32_t H, const float4* __restrict__ splats,
    const uint32_t* __restrict__ vals, const int64_t* __restrict__ ranges,
    const uint32_t* __restrict__ tile_order, float bg0, float bg1, float bg2, const float* __restrict__ T_final, const int32_t* __restrict__ n_contrib,
    const float* __restrict__ dL_dimage, float4* __restrict__ grads) {
  __shared__ BwdSmem S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t flat = tile_order ? (int64_t)tile_order[blockIdx.x] : (int64_t)blockIdx.x;
  const int64_t view = flat / T;
  const int32_t tile = (int32_t)(flat - view * T);
  const int tile_x = tile % tiles_x, tile_y = tile / tiles_x;
  const float ox = (float)(tile_x * GS_TILE), oy = (float)(tile_y * GS_TILE);
  int px, py;
  pixel_of(tid, tile_x, tile_y, px, py);
  const bool inside = px < W && py < H;
  const float ix = (float)(px - tile_x * GS_TILE), iy = (float)(py - tile_y * GS_TILE);
  // grid-index origin of this warp's 8x4 block
  const int wx0 = (warp & 1) * 8, wy0 = (warp >> 1) * 4;
  const int64_t start = ranges[2 * flat];
  const int64_t HW = (int64_t)W * H;
  const int64_t pix = (int64_t)py * W + px;
  float Tr = 0.f, g0 = 0.f, g1 = 0.f, g2 = 0.f;
  int32_t last = 0;
  if (inside) {
    Tr = T_final[view * HW + pix];
    last = n_contrib[view * HW + pix];
    g0 = dL_dimage[(view * 3 + 0) * HW + pix];
    g1 = dL_dimage[(view * 3 + 1) * HW + pix];
    g2 = dL_dimage[(view * 3 + 2) * HW + pix];
  }
  float S0 = Tr * bg0, S1 = Tr * bg1, S2 = Tr * bg2;
  if (tid == 0) S.max_last = 0;
  for (int i = tid; i < kBatch * 9; i += kRT) (&S.acc[0][0])[i] = 0.f;
  __syncthreads();
  const int warp_last = __reduce_max_sync(0xffffffffu, last);
  if (lane == 0) atomicMax(&S.max_last, warp_last);
  quarter_last(last, S.qlast[warp], lane);
  __syncthreads();
  const int max_last = S.max_last;
  const int nb = (max_last + kBatch - 1) / kBatch;
  const float4* vsplat = splats + 3 * view * n;

  // batch k covers list positions [hi - cnt, hi), hi = max_last - k * kBatch,
  // stored at smem slots 0..cnt-1 in position order
  auto issue = [&](int k) {
    const int hi = max_last - k * kBatch;
    const int cnt = min(kBatch, hi);
    if (tid < cnt) {
      const int64_t e = start + (hi - cnt) + tid;
      const uint32_t id = min(__ldg(vals + e), (uint32_t)(n - 1));
      const float4* src = vsplat + 3 * (int64_t)id;
      Batch& B = S.b[k & 1];
      S.id[k & 1][tid] = id;
      cp_async16(&B.a[tid], src);
      cp_async16(&B.b[tid], src + 1);
      cp_async16(&B.c[tid], src + 2);
    }
    cp_async_commit();
  };

  if (nb > 0) issue(0);
  for (int k = 0; k < nb; ++k) {
    if (k + 1 < nb) issue(k + 1); else cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    Batch& B = S.b[k & 1];
    const int hi = max_last - k * kBatch;
    const int cnt = min(kBatch, hi);
    const int lo = hi - cnt;
    float2* E = S.e[k & 1];
    if (tid < cnt) stage_entry(B, tid, ox, oy, E);
    __syncthreads();
    const int nw = box_masks(B, S.qm[warp], S.qlast[warp], cnt, lo, wx0, wy0, lane);
    bwd_walk(B, S.acc, S.qm[warp][(lane >> 3) & 3], nw, lo, ix, iy, last, Tr, S0, S1, S2, g0, g1,
             g2, lane);
    __syncthreads();
    bwd_flush(B, E, S.id[k & 1], S.acc, cnt, grads + 3 * view * n, tid);
    __syncthreads();
  }
  cp_async_wait<0>();
}

// Forward, L1 loss and backward of one tile in one CTA ("ByteSplat": forward
// and backward rasterization fused into a single kernel that keeps the
// intermediates on chip).  The per-pixel results of the forward (T, the last
// contributor, the colour and its L1 gradient) stay in registers and shared
// memory instead of a round trip through T_final, n_contrib and dL/dimage,
// and the batches still staged in shared memory when the forward ends (the
// last one composited, or the last two when the list runs out) are reused
// by the backward without a new gather or staging.  The backward walks the
// forward's batches (0-aligned) from the one holding the tile's last
// contributor down to the first.
struct FusedSmem {
  Batch b[2];
  float2 e[2][kBatch];
  uint32_t id[2][kBatch];
  union {
    struct {
      PixState px;
      uint32_t rec[kRT / 8][kWords];  // the batch's composited entries per quarter
      uint8_t wl[kWarps][kBatch];     // per-warp entry sub-lists
    } fw;  // forward
    struct {
      float acc[kBatch][9];
      alignas(16) uint32_t qm[kWarps][4][kWords];  // masks of quarter warp * 4 + q
      alignas(16) int32_t qlast[kWarps][4];
      // per-pixel state between batches, for a warp that takes other quarters
      float pT[kRT], pS0[kRT], pS1[kRT], pS2[kRT];
      int32_t plast[kRT];
      uint8_t pg[kRT];     // signs of the L1 gradient, 2 bits per channel
    } bw;  // backward
  } u;
  int32_t wcount[kWarps];
  float lsum[kWarps];
  int max_last;
};

__global__ void __launch_bounds__(kRT, 6) raster_fused_kernel(
    int64_t n, int32_t tiles_x, int64_t T, int32_t W, int32_t H, const float4* __restrict__ splats,
    const uint32_t* __restrict__ vals, const int64_t* __restrict__ ranges,
    const uint32_t* __restrict__ tile_order, float bg0, float bg1, float bg2, const float* __restrict__ target, float inv_count, float* __restrict__ image,
    float* __restrict__ T_final, int32_t* __restrict__ n_contrib, float* __restrict__ loss,
    float4* __restrict__ grads, uint32_t* __restrict__ recs, int64_t rec_slots) {
  __shared__ FusedSmem S;
  unsigned long long n_tested = 0, n_included = 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t flat = tile_order ? (int64_t)tile_order[blockIdx.x] : (int64_t)blockIdx.x;
  const int64_t view = flat / T;
  const int32_t tile = (int32_t)(flat - view * T);
  const int tile_x = tile % tiles_x, tile_y = tile / tiles_x;
  const float ox = (float)(tile_x * GS_TILE), oy = (float)(tile_y * GS_TILE);
  const int64_t start = ranges[2 * flat], end = ranges[2 * flat + 1];
  const float4* vsplat = splats + 3 * view * n;
  pix_init(S.u.fw.px, tid, tile_x, tile_y, W, H);
  // the workspace keeps, per batch of the tile, which entries the forward
  // composited into each 4x2 quarter (kRec words, slot g = start / kBatch + k
  // + flat: distinct for every (tile, batch) since the lists are contiguous
  // in tile order); without it (or beyond its end) the backward walks the
  // boxes
  constexpr int kRec = kRT / 8 * kWords;
  const int64_t nbt = (end - start + kBatch - 1) / kBatch;
  const int64_t slot0 = start / kBatch + flat;
  uint32_t* rec_out = (recs && nbt > 0 && slot0 + nbt <= rec_slots) ? recs + slot0 * kRec : nullptr;
  if (tid < kRec) (&S.u.fw.rec[0][0])[tid] = 0u;
  int2 staged;
  // the walk unrolled by 8: the pairs of a sub-list are mostly skips, and the
  // loop overhead and load latency of one entry at a time dominate them
  // (this kernel only: the separate forward, at a different occupancy, is
  // slower unrolled)
  fwd_tile<false, false, 8>(S.u.fw.px, S.b, S.id, S.e, S.u.fw.wl, S.wcount, vsplat, vals, n,
                            start, end, tile_x, tile_y, ox, oy, tid, warp, lane, staged, n_tested,
                            n_included, nullptr, nullptr, 0, 0, S.u.fw.rec, rec_out);

  // forward results, L1 loss and its gradient, in registers; thread tid owns
  // pixel tid from here on
  int px, py;
  pixel_of(tid, tile_x, tile_y, px, py);
  const bool inside = px < W && py < H;
  float Tr = S.u.fw.px.T[tid];
  const int32_t last = inside ? S.u.fw.px.last[tid] : 0;
  float g0 = 0.f, g1 = 0.f, g2 = 0.f, l1 = 0.f;
  if (inside) {
    const int64_t HW = (int64_t)W * H;
    const int64_t pix = (int64_t)py * W + px;
    const float c0 = S.u.fw.px.C0[tid] + Tr * bg0;
    const float c1 = S.u.fw.px.C1[tid] + Tr * bg1;
    const float c2 = S.u.fw.px.C2[tid] + Tr * bg2;
    image[(view * 3 + 0) * HW + pix] = c0;
    image[(view * 3 + 1) * HW + pix] = c1;
    image[(view * 3 + 2) * HW + pix] = c2;
    T_final[view * HW + pix] = Tr;
    n_contrib[view * HW + pix] = last;
    auto sgn = [&](float d) { return d > 0.f ? inv_count : (d < 0.f ? -inv_count : 0.f); };
    const float d0 = c0 - __ldcs(target + (view * 3 + 0) * HW + pix);
    const float d1 = c1 - __ldcs(target + (view * 3 + 1) * HW + pix);
    const float d2 = c2 - __ldcs(target + (view * 3 + 2) * HW + pix);
    l1 = fabsf(d0) + fabsf(d1) + fabsf(d2);
    g0 = sgn(d0);
    g1 = sgn(d1);
    g2 = sgn(d2);
  } else {
    Tr = 0.f;
  }
  l1 = warp_sum(l1);
  if (lane == 0) S.lsum[warp] = l1;
  if (tid == 0) S.max_last = 0;
  __syncthreads();  // the forward's pixel state is read; its space becomes acc
  for (int i = tid; i < kBatch * 9; i += kRT) (&S.u.bw.acc[0][0])[i] = 0.f;
  const int warp_last = __reduce_max_sync(0xffffffffu, last);
  if (lane == 0) atomicMax(&S.max_last, warp_last);
  quarter_last(last, S.u.bw.qlast[warp], lane);
  if (tid == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += S.lsum[w];
    atomicAdd(loss, t * inv_count);
  }
  __syncthreads();
  const int max_last = S.max_last;
  const float ix = (float)(px - tile_x * GS_TILE), iy = (float)(py - tile_y * GS_TILE);
  const int wx0 = (warp & 1) * 8, wy0 = (warp >> 1) * 4;
  float S0 = Tr * bg0, S1 = Tr * bg1, S2 = Tr * bg2;
  // With the forward's record, each batch's 32 quarters are handed to the
  // warps in descending order of their recorded entries (warp w takes the
  // quarters ranked 4w..4w+3): a warp's step costs the longest of its four
  // lists, and grouping lists of like length wastes fewer lanes.  A pixel's
  // state then lives in shared memory between batches.
  const bool regroup = rec_out != nullptr;
  if (regroup) {
    S.u.bw.pT[tid] = Tr;
    S.u.bw.pS0[tid] = S0;
    S.u.bw.pS1[tid] = S1;
    S.u.bw.pS2[tid] = S2;
    S.u.bw.plast[tid] = last;
    const auto code = [](float g) { return g > 0.f ? 1u : (g < 0.f ? 2u : 0u); };
    S.u.bw.pg[tid] = (uint8_t)(code(g0) | code(g1) << 2 | code(g2) << 4);
  }
  // backward: batch k covers list positions [k kBatch, min((k+1) kBatch, max_last))
  // in slot k & 1, gathered and staged unless the forward left it there
  auto issue = [&](int k) {
    const int lo = k * kBatch;
    const int cnt = min(kBatch, max_last - lo);
    if (tid < cnt) {
      const uint32_t id = min(__ldg(vals + start + lo + tid), (uint32_t)(n - 1));
      const float4* src = vsplat + 3 * (int64_t)id;
      Batch& B = S.b[k & 1];
      S.id[k & 1][tid] = id;
      cp_async16(&B.a[tid], src);
      cp_async16(&B.b[tid], src + 1);
      cp_async16(&B.c[tid], src + 2);
    }
    cp_async_commit();
  };
  // the record of batch k (kRec words, 16-byte pieces) into the mask space
  auto issue_rec = [&](int k) {
    if (tid < kRec / 4)
      cp_async16(&S.u.bw.qm[0][0][0] + 4 * tid, rec_out + (int64_t)k * kRec + 4 * tid);
    cp_async_commit();
  };
  const int kt = max_last > 0 ? (max_last - 1) / kBatch : -1;
  if (kt >= 0 && slot(staged, kt & 1) != kt) {
    issue(kt);
    slot(staged, kt & 1) = -1;
  }
  if (kt >= 0 && regroup) issue_rec(kt);
  // One barrier a batch besides the walk's: batch k - 1 is gathered, and
  // batch k - 1's record fetched, only after the barrier that follows the
  // walk (record) or the flush (slot) of the batch that used the space last.
  for (int k = kt; k >= 0; --k) {
    cp_async_wait<0>();
    __syncthreads();  // batch k and its record landed; batch k + 1 flushed, its slot free
    if (k >= 1 && slot(staged, (k - 1) & 1) != k - 1) {
      issue(k - 1);
      slot(staged, (k - 1) & 1) = -1;
    }
    Batch& B = S.b[k & 1];
    const int lo = k * kBatch;
    const int cnt = min(kBatch, max_last - lo);
    if (slot(staged, k & 1) != k) {
      if (tid < cnt) stage_entry(B, tid, ox, oy, S.e[k & 1]);
      slot(staged, k & 1) = k;
      __syncthreads();
    }
    if (regroup) {
      // the batch's record (quarter Q's words at Q * kWords); every warp
      // ranks the quarters itself and takes those ranked 4w..4w+3
      const uint32_t* qall = &S.u.bw.qm[0][0][0];
      int c = 0;
#pragma unroll
      for (int w = 0; w < kWords; ++w) c += __popc(qall[lane * kWords + w]);
      const int ranked = quarter_rank_order(c, lane);
      const int Q = __shfl_sync(0xffffffffu, ranked, warp * 4 + ((lane >> 3) & 3));
      const int p = Q * 8 + (lane & 7);
      int qx, qy;
      pixel_of(p, tile_x, tile_y, qx, qy);
      float T = S.u.bw.pT[p], s0 = S.u.bw.pS0[p], s1 = S.u.bw.pS1[p], s2 = S.u.bw.pS2[p];
      const uint32_t gc = S.u.bw.pg[p];
      const auto sg = [&](uint32_t c2) { return c2 == 1u ? inv_count : (c2 == 2u ? -inv_count : 0.f); };
      bwd_walk(B, S.u.bw.acc, qall + Q * kWords, kWords, lo, (float)(qx - tile_x * GS_TILE),
               (float)(qy - tile_y * GS_TILE), S.u.bw.plast[p], T, s0, s1, s2, sg(gc & 3u),
               sg((gc >> 2) & 3u), sg((gc >> 4) & 3u), lane);
      S.u.bw.pT[p] = T;
      S.u.bw.pS0[p] = s0;
      S.u.bw.pS1[p] = s1;
      S.u.bw.pS2[p] = s2;
    } else {
      const int nw = box_masks(B, S.u.bw.qm[warp], S.u.bw.qlast[warp], cnt, lo, wx0, wy0, lane);
      bwd_walk(B, S.u.bw.acc, S.u.bw.qm[warp][(lane >> 3) & 3], nw, lo, ix, iy, last, Tr, S0, S1,
               S2, g0, g1, g2, lane);
    }
    __syncthreads();  // the walk is done: sums complete, record and masks free
    if (regroup && k >= 1) issue_rec(k - 1);
    bwd_flush(B, S.e[k & 1], S.id[k & 1], S.u.bw.acc, cnt, grads + 3 * view * n, tid);
  }
  cp_async_wait<0>();
}

// Zeroes the gradient records of the rows with a positive tile count (the
// only rows whose gradients the compositing writes and the projection
// backward reads): 4 bytes read a row, 48 written a visible row.  Rows go in
// pairs, 96 bytes = three whole 32-byte sectors, both zeroed when either is
// visible: a lone 48-byte record half-fills a sector, and the partial writes
// cost the memory a read.  One thread per pair of rows (one 8-byte load of
// the two counts, six 16-byte stores): where few rows are visible most
// threads only read.
__global__ void __launch_bounds__(256) zero_visible_grads_kernel(int64_t rows,
                                                                 const int32_t* __restrict__ counts,
                                                                 float4* __restrict__ grads) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // rows 2q, 2q + 1
  const int64_t r = 2 * q;
  if (r >= rows) return;
  bool any;
  if (r + 1 < rows && ((reinterpret_cast<uintptr_t>(counts) & 7u) == 0)) {
    const int2 c = __ldg(reinterpret_cast<const int2*>(counts) + q);
    any = c.x > 0 || c.y > 0;
  } else {
    any = __ldg(counts + r) > 0 || (r + 1 < rows && __ldg(counts + r + 1) > 0);
  }
  if (!any) return;
  const int nv = r + 1 < rows ? 6 : 3;
  float4* g = grads + 3 * r;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int v = 0; v < 6; ++v)
    if (v < nv) g[v] = z;
}

// The same zeroing by a grid smaller than the pairs, striding over them four
// pairs a round with their counts loaded together: a launch meant to run
// beside other kernels takes a few CTAs per SM instead of filling the GPU
// ahead of them, and still keeps loads in flight.
__global__ void __launch_bounds__(256) zero_visible_grads_strided_kernel(
    int64_t rows, const int32_t* __restrict__ counts, float4* __restrict__ grads) {
  const bool even = (reinterpret_cast<uintptr_t>(counts) & 7u) == 0;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t pairs = (rows + 1) / 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t q0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q0 < pairs; q0 += 4 * stride) {
    bool any[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t q = q0 + u * stride, r = 2 * q;
      any[u] = false;
      if (q < pairs) {
        if (r + 1 < rows && even) {
          const int2 c = __ldg(reinterpret_cast<const int2*>(counts) + q);
          any[u] = c.x > 0 || c.y > 0;
        } else {
          any[u] = __ldg(counts + r) > 0 || (r + 1 < rows && __ldg(counts + r + 1) > 0);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!any[u]) continue;
      const int64_t r = 2 * (q0 + u * stride);
      const int nv = r + 1 < rows ? 6 : 3;
      float4* g = grads + 3 * r;
#pragma unroll
      for (int v = 0; v < 6; ++v)
        if (v < nv) g[v] = z;
    }
  }
}

// The gradient records' zeroing before a backward: every row, or with tile
// counts only the visible ones.
constexpr int kZeroSideCtas = 2;

// max_blocks > 0: the striding kernel on a grid of at most max_blocks (a
// zeroing meant to run beside other kernels); else one thread per pair.
gs_status zero_grads(int64_t rows, const int32_t* counts, gs_splat_grad* grads, cudaStream_t st,
                     int64_t max_blocks = 0) {
  if (rows <= 0) return GS_OK;
  if (!counts) {
    GS_CUDA(cudaMemsetAsync(grads, 0, sizeof(gs_splat_grad) * (size_t)rows, st));
    return GS_OK;
  }
  const int64_t blocks = div_up(div_up(rows, 2), 256);
  if (max_blocks > 0 && blocks > max_blocks)
    zero_visible_grads_strided_kernel<<<(unsigned)max_blocks, 256, 0, st>>>(
        rows, counts, reinterpret_cast<float4*>(grads));
  else
    zero_visible_grads_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        rows, counts, reinterpret_cast<float4*>(grads));
  GS_CHECK_LAUNCH();
  return GS_OK;
}

}  // namespace
}  // namespace gs

using namespace gs;


static gs_status rasterize_fwd_impl(int64_t n, int32_t n_views, const gs_splat* splats,
                                    int32_t width, int32_t height, const uint32_t* vals,
                                    const int64_t* ranges, const uint32_t* tile_order,
                                    const float* bg, float* image,
                                    float* T_final, int32_t* n_contrib, uint64_t* counts,
                                    int32_t* pix_counts, float* importance, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || !bg || !ranges || !image || !T_final || !n_contrib)
    return GS_ERR_INVALID_ARG;
  if (n > 0 && (!splats || !aligned16(splats))) return GS_ERR_INVALID_ARG;
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE;
  const unsigned grid = (unsigned)(n_views * T);
  unsigned long long* c = reinterpret_cast<unsigned long long*>(counts);
  const float4* sp = reinterpret_cast<const float4*>(splats);
  cudaStream_t st = (cudaStream_t)stream;
  if (importance) {
    if (n > 0) GS_CUDA(cudaMemsetAsync(importance, 0, sizeof(float) * (size_t)(n * n_views), st));
    raster_fwd_kernel<false, true><<<grid, kRT, 0, st>>>(n, tiles_x, T, width, height, sp, vals,
                                                         ranges, tile_order, bg[0], bg[1], bg[2], image,
                                                         T_final, n_contrib, c, nullptr, importance);
  } else if (counts) {
    if (pix_counts)
      GS_CUDA(cudaMemsetAsync(pix_counts, 0,
                              sizeof(int32_t) * 2 * (size_t)n_views * width * height, st));
    raster_fwd_kernel<true, false><<<grid, kRT, 0, st>>>(n, tiles_x, T, width, height, sp, vals,
                                                         ranges, tile_order, bg[0], bg[1], bg[2], image,
                                                         T_final, n_contrib, c, pix_counts, nullptr);
  } else {
    raster_fwd_kernel<false, false><<<grid, kRT, 0, st>>>(n, tiles_x, T, width, height, sp, vals,
                                                          ranges, tile_order, bg[0], bg[1], bg[2], image,
                                                          T_final, n_contrib, c, nullptr, nullptr);
  }
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" gs_status gs_rasterize_fwd(int64_t n, int32_t n_views, const gs_splat* splats,
                                      int32_t width, int32_t height, const uint32_t* vals,
                                      const int64_t* ranges, const uint32_t* tile_order,
                                      const float* bg, float* image, float* T_final,
                                      int32_t* n_contrib, void* stream) {
  return rasterize_fwd_impl(n, n_views, splats, width, height, vals, ranges, tile_order, bg, image,
                            T_final, n_contrib, nullptr, nullptr, nullptr, stream);
}

extern "C" gs_status gs_rasterize_fwd_counted(int64_t n, int32_t n_views, const gs_splat* splats,
                                              int32_t width, int32_t height, const uint32_t* vals,
                                              const int64_t* ranges, const uint32_t* tile_order,
                                              const float* bg, float* image, float* T_final,
                                              int32_t* n_contrib, uint64_t* counts,
                                              int32_t* pixel_counts, void* stream) {
  if (!counts) return GS_ERR_INVALID_ARG;
  return rasterize_fwd_impl(n, n_views, splats, width, height, vals, ranges, tile_order, bg, image,
                            T_final, n_contrib, counts, pixel_counts, nullptr, stream);
}

extern "C" gs_status gs_rasterize_fwd_importance(int64_t n, int32_t n_views, const gs_splat* splats,
                                                 int32_t width, int32_t height,
                                                 const uint32_t* vals, const int64_t* ranges,
                                                 const uint32_t* tile_order, const float* bg,
                                                 float* image, float* T_final, int32_t* n_contrib,
                                                 float* importance, void* stream) {
  if (!importance && n > 0) return GS_ERR_INVALID_ARG;
  return rasterize_fwd_impl(n, n_views, splats, width, height, vals, ranges, tile_order, bg, image,
                            T_final, n_contrib, nullptr, nullptr, importance, stream);
}

extern "C" size_t gs_rasterize_workspace_bytes(int32_t n_views, int32_t width, int32_t height,
                                               int64_t capacity) {
  if (n_views < 1 || width < 1 || height < 1 || capacity < 0) return 0;
  const int64_t slots = div_up(capacity, kBatch) + (int64_t)n_views * tiles_per_view(width, height) + 1;
  return (size_t)slots * (kRT / 8 * kWords) * sizeof(uint32_t);
}

// gs_rasterize_fused and gs_rasterize_fused_acc: the same launch, with or
// without the zeroing of the gradient records in front of it.
static gs_status rasterize_fused_impl(int64_t n, int32_t n_views, const gs_splat* splats,
                                      const int32_t* tile_counts, int32_t width, int32_t height,
                                      const uint32_t* vals, const int64_t* ranges,
                                      const uint32_t* tile_order, const float* bg,
                                      const float* target, float* image, float* T_final,
                                      int32_t* n_contrib, float* loss, gs_splat_grad* grads,
                                      void* workspace, size_t ws_bytes, bool zero, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || !bg || !ranges || !target || !image || !T_final || !n_contrib || !loss)
    return GS_ERR_INVALID_ARG;
  if (n > 0 && (!splats || !grads || !aligned16(splats) || !aligned16(grads)))
    return GS_ERR_INVALID_ARG;
  if (workspace && !aligned16(workspace)) return GS_ERR_INVALID_ARG;
  if (!aligned4(tile_counts)) return GS_ERR_INVALID_ARG;
  const int64_t rec_slots = workspace ? (int64_t)(ws_bytes / (kRT / 8 * kWords * sizeof(uint32_t))) : 0;
  cudaStream_t st = (cudaStream_t)stream;
  GS_CUDA(cudaMemsetAsync(loss, 0, sizeof(float), st));
  if (zero) {
    const gs_status zs = zero_grads(n * n_views, tile_counts, grads, st);
    if (zs != GS_OK) return zs;
  }
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE;
  const double count = 3.0 * (double)n_views * (double)width * (double)height;
  raster_fused_kernel<<<(unsigned)(n_views * T), kRT, 0, st>>>(
      n, tiles_x, T, width, height, reinterpret_cast<const float4*>(splats), vals, ranges,
      tile_order, bg[0], bg[1], bg[2], target, (float)(1.0 / count), image, T_final, n_contrib, loss,
      reinterpret_cast<float4*>(grads), rec_slots > 0 ? static_cast<uint32_t*>(workspace) : nullptr,
      rec_slots);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" gs_status gs_rasterize_fused(int64_t n, int32_t n_views, const gs_splat* splats,
                                        const int32_t* tile_counts, int32_t width, int32_t height,
                                        const uint32_t* vals, const int64_t* ranges,
                                        const uint32_t* tile_order, const float* bg,
                                        const float* target, float* image, float* T_final,
                                        int32_t* n_contrib, float* loss, gs_splat_grad* grads,
                                        void* workspace, size_t ws_bytes, void* stream) {
  return rasterize_fused_impl(n, n_views, splats, tile_counts, width, height, vals, ranges,
                              tile_order, bg, target, image, T_final, n_contrib, loss, grads,
                              workspace, ws_bytes, true, stream);
}

extern "C" gs_status gs_rasterize_fused_acc(int64_t n, int32_t n_views, const gs_splat* splats,
                                            const int32_t* tile_counts, int32_t width,
                                            int32_t height, const uint32_t* vals,
                                            const int64_t* ranges, const uint32_t* tile_order,
                                            const float* bg, const float* target, float* image,
                                            float* T_final, int32_t* n_contrib, float* loss,
                                            gs_splat_grad* grads, void* workspace,
                                            size_t ws_bytes, void* stream) {
  return rasterize_fused_impl(n, n_views, splats, tile_counts, width, height, vals, ranges,
                              tile_order, bg, target, image, T_final, n_contrib, loss, grads,
                              workspace, ws_bytes, false, stream);
}

extern "C" gs_status gs_zero_grads(int64_t n, int32_t n_views, const int32_t* tile_counts,
                                   gs_splat_grad* grads, int32_t beside, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS)
    return GS_ERR_INVALID_ARG;
  if (n > 0 && (!grads || !aligned16(grads))) return GS_ERR_INVALID_ARG;
  if (!aligned4(tile_counts)) return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  if (!beside) return zero_grads(n * n_views, tile_counts, grads, (cudaStream_t)stream);
  // beside other work: a small grid (kZeroSideCtas CTAs per SM, striding), as
  // a grid of one thread per pair of rows would hold the other stream's
  // kernels back until it drained
  int dev = 0, sms = 0;
  GS_CUDA(cudaGetDevice(&dev));
  GS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  return zero_grads(n * n_views, tile_counts, grads, (cudaStream_t)stream,
                    (int64_t)kZeroSideCtas * (sms > 0 ? sms : 1));
}

extern "C" gs_status gs_rasterize_bwd(int64_t n, int32_t n_views, const gs_splat* splats,
                                      const int32_t* tile_counts, int32_t width, int32_t height, const uint32_t* vals,
                                      const int64_t* ranges, const uint32_t* tile_order,
                                      const float* bg, const float* T_final,
                                      const int32_t* n_contrib, const float* dL_dimage,
                                      gs_splat_grad* grads, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || !bg || !ranges || !T_final || !n_contrib || !dL_dimage)
    return GS_ERR_INVALID_ARG;
  if (n > 0 && (!splats || !grads || !aligned16(splats) || !aligned16(grads)))
    return GS_ERR_INVALID_ARG;
  if (!aligned4(tile_counts)) return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const gs_status zs = zero_grads(n * n_views, tile_counts, grads, st);
  if (zs != GS_OK) return zs;
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE;
  raster_bwd_kernel<<<(unsigned)(n_views * T), kRT, 0, st>>>(
      n, tiles_x, T, width, height, reinterpret_cast<const float4*>(splats), vals, ranges,
      tile_order, bg[0], bg[1], bg[2], T_final, n_contrib, dL_dimage, reinterpret_cast<float4*>(grads));
  GS_CHECK_LAUNCH();
  return GS_OK;
}

// raster.cu -- gs_rasterize_fwd and gs_rasterize_bwd.
//
// Front-to-back alpha compositing over per-tile sorted lists and its
// analytic backward ("ByteSplat": forward and backward rasterization;
// "On Scaling Up 3D Gaussian Splatting Training": 16x16 pixel blocks and the
// opacity saturation depth at which a pixel stops).
//
// One CTA per (view, 16x16 tile), one pixel per thread.  Warps cover 8x4
// pixel blocks, so the per-pair skip/stop decisions of a warp are spatially
// coherent.  The tile's Gaussians are gathered by id into shared memory in
// batches of 256 with cp.async, double buffered: the next batch is in flight
// while the current one is composited.  The block stops as soon as every
// pixel has saturated (barrier count), and the backward starts each warp at
// its own last contributor.
#include <stdint.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

constexpr int kRT = 256;  // threads per CTA = pixels per tile

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// The pair terms with a fixed rounding sequence, shared by the forward and
// the backward so both take identical skip decisions:
//   power = -(a dx^2 + c dy^2)/2 - b dx dy,   raw alpha = opacity e^power.
__device__ __forceinline__ float pair_power(float dx, float dy, float ca, float cb, float cc) {
  const float s = __fmaf_rn(__fmul_rn(ca, dx), dx, __fmul_rn(__fmul_rn(cc, dy), dy));
  const float t = __fmul_rn(__fmul_rn(cb, dx), dy);
  return __fmaf_rn(-0.5f, s, -t);
}

struct Batch {
  float4 a[kRT];   // mean_x, mean_y, conic_a, conic_b
  float4 b[kRT];   // conic_c, opacity, color_r, color_g
  float c[kRT];    // color_b
};

__device__ __forceinline__ void pixel_of(int tid, int tile_x, int tile_y, int& px, int& py) {
  const int warp = tid >> 5, lane = tid & 31;
  px = tile_x * GS_TILE + (warp & 1) * 8 + (lane & 7);
  py = tile_y * GS_TILE + (warp >> 1) * 4 + (lane >> 3);
}

// kCount: also accumulate the pairs tested / included into counts[0..1]
// (instrumentation for work accounting; the compositing is identical).
template <bool kCount>
__global__ void __launch_bounds__(kRT) raster_fwd_kernel(
    int64_t n, int32_t tiles_x, int64_t T, int32_t W, int32_t H, const float4* __restrict__ splats,
    const uint32_t* __restrict__ vals, const int64_t* __restrict__ ranges, float bg0, float bg1,
    float bg2, float* __restrict__ image, float* __restrict__ T_final,
    int32_t* __restrict__ n_contrib, unsigned long long* __restrict__ counts) {
  __shared__ Batch sb[2];
  unsigned long long n_tested = 0, n_included = 0;
  const int tid = threadIdx.x;
  const int64_t flat = blockIdx.x;
  const int64_t view = flat / T;
  const int32_t tile = (int32_t)(flat - view * T);
  const int tile_x = tile % tiles_x, tile_y = tile / tiles_x;
  int px, py;
  pixel_of(tid, tile_x, tile_y, px, py);
  const bool inside = px < W && py < H;
  const float pxc = (float)px + 0.5f, pyc = (float)py + 0.5f;
  const int64_t start = ranges[2 * flat], end = ranges[2 * flat + 1];
  const int64_t len = end - start;
  const int nb = (int)((len + kRT - 1) / kRT);
  const float4* vsplat = splats + 3 * view * n;

  float Tr = 1.f, C0 = 0.f, C1 = 0.f, C2 = 0.f;
  int32_t last = 0;
  int done = inside ? 0 : 1;

  auto issue = [&](int k) {
    const int64_t e = start + (int64_t)k * kRT + tid;
    if (e < end) {
      // ids come from gs_bin_and_sort; clamping keeps a corrupt list in bounds
      const uint32_t id = min(__ldg(vals + e), (uint32_t)(n - 1));
      const float4* src = vsplat + 3 * (int64_t)id;
      Batch& B = sb[k & 1];
      cp_async16(&B.a[tid], src);
      cp_async16(&B.b[tid], src + 1);
      cp_async4(&B.c[tid], src + 2);
    }
    cp_async_commit();
  };

  if (nb > 0) issue(0);
  for (int k = 0; k < nb; ++k) {
    if (k + 1 < nb) issue(k + 1); else cp_async_commit();
    cp_async_wait<1>();
    if (__syncthreads_count(done) == kRT) break;
    const Batch& B = sb[k & 1];
    const int cnt = (int)min((int64_t)kRT, len - (int64_t)k * kRT);
    if (!done) {
      for (int j = 0; j < cnt; ++j) {
        const float4 A = B.a[j];
        const float4 Bv = B.b[j];
        if (kCount) ++n_tested;
        const float dx = __fsub_rn(pxc, A.x), dy = __fsub_rn(pyc, A.y);
        const float power = pair_power(dx, dy, A.z, A.w, Bv.x);
        const float alpha = fminf(kAlphaMax, __fmul_rn(Bv.y, __expf(power)));
        if (alpha < kAlphaMin) continue;
        const float Tn = __fmul_rn(Tr, __fsub_rn(1.f, alpha));
        if (Tn < kTMin) { done = 1; break; }
        if (kCount) ++n_included;
        const float w = alpha * Tr;
        C0 += w * Bv.z;
        C1 += w * Bv.w;
        C2 += w * B.c[j];
        Tr = Tn;
        last = k * kRT + j + 1;
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  if (inside) {
    const int64_t HW = (int64_t)W * H;
    const int64_t pix = (int64_t)py * W + px;
    image[(view * 3 + 0) * HW + pix] = C0 + Tr * bg0;
    image[(view * 3 + 1) * HW + pix] = C1 + Tr * bg1;
    image[(view * 3 + 2) * HW + pix] = C2 + Tr * bg2;
    T_final[view * HW + pix] = Tr;
    n_contrib[view * HW + pix] = last;
  }
  if (kCount) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      n_tested += __shfl_xor_sync(0xffffffffu, n_tested, o);
      n_included += __shfl_xor_sync(0xffffffffu, n_included, o);
    }
    if ((tid & 31) == 0) {
      atomicAdd(&counts[0], n_tested);
      atomicAdd(&counts[1], n_included);
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct BwdSmem {
  Batch b[2];
  uint32_t id[2][kRT];
  float acc[kRT][9];
  int max_last;
};

__global__ void __launch_bounds__(kRT) raster_bwd_kernel(
    int64_t n, int32_t tiles_x, int64_t T, int32_t W, int32_t H, const float4* __restrict__ splats,
    const uint32_t* __restrict__ vals, const int64_t* __restrict__ ranges, float bg0, float bg1,
    float bg2, const float* __restrict__ T_final, const int32_t* __restrict__ n_contrib,
    const float* __restrict__ dL_dimage, float4* __restrict__ grads) {
  __shared__ BwdSmem S;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t flat = blockIdx.x;
  const int64_t view = flat / T;
  const int32_t tile = (int32_t)(flat - view * T);
  const int tile_x = tile % tiles_x, tile_y = tile / tiles_x;
  int px, py;
  pixel_of(tid, tile_x, tile_y, px, py);
  const bool inside = px < W && py < H;
  const float pxc = (float)px + 0.5f, pyc = (float)py + 0.5f;
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
  for (int i = tid; i < kRT * 9; i += kRT) (&S.acc[0][0])[i] = 0.f;
  __syncthreads();
  const int warp_last = __reduce_max_sync(0xffffffffu, last);
  if (lane == 0) atomicMax(&S.max_last, warp_last);
  __syncthreads();
  const int max_last = S.max_last;
  const int nb = (max_last + kRT - 1) / kRT;
  const float4* vsplat = splats + 3 * view * n;

  // batch k covers list positions [hi - cnt, hi), hi = max_last - k*256,
  // stored at smem slots 0..cnt-1 in position order
  auto issue = [&](int k) {
    const int hi = max_last - k * kRT;
    const int cnt = min(kRT, hi);
    if (tid < cnt) {
      const int64_t e = start + (hi - cnt) + tid;
      const uint32_t id = min(__ldg(vals + e), (uint32_t)(n - 1));
      const float4* src = vsplat + 3 * (int64_t)id;
      Batch& B = S.b[k & 1];
      S.id[k & 1][tid] = id;
      cp_async16(&B.a[tid], src);
      cp_async16(&B.b[tid], src + 1);
      cp_async4(&B.c[tid], src + 2);
    }
    cp_async_commit();
  };

  if (nb > 0) issue(0);
  for (int k = 0; k < nb; ++k) {
    if (k + 1 < nb) issue(k + 1); else cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const Batch& B = S.b[k & 1];
    const int hi = max_last - k * kRT;
    const int cnt = min(kRT, hi);
    const int lo = hi - cnt;
    // positions at or above the warp's last contributor cannot contribute
    const int jtop = min(cnt, warp_last - lo);
    for (int j = jtop - 1; j >= 0; --j) {
      const int pos = lo + j;
      float v[9];
#pragma unroll
      for (int c = 0; c < 9; ++c) v[c] = 0.f;
      bool contrib = false;
      if (pos < last) {
        const float4 A = B.a[j];
        const float4 Bv = B.b[j];
        const float dx = __fsub_rn(pxc, A.x), dy = __fsub_rn(pyc, A.y);
        const float power = pair_power(dx, dy, A.z, A.w, Bv.x);
        const float e = __expf(power);
        const float raw = __fmul_rn(Bv.y, e);
        const float alpha = fminf(kAlphaMax, raw);
        if (alpha >= kAlphaMin) {
          contrib = true;
          const float cb = B.c[j];
          const float oma = 1.f - alpha;
          const float rinv = 1.f / oma;
          const float Ti = Tr * rinv;
          const float w = alpha * Ti;
          v[6] = w * g0;
          v[7] = w * g1;
          v[8] = w * g2;
          const float dalpha = (g0 * Bv.z + g1 * Bv.w + g2 * cb) * Ti -
                               (g0 * S0 + g1 * S1 + g2 * S2) * rinv;
          S0 += w * Bv.z;
          S1 += w * Bv.w;
          S2 += w * cb;
          Tr = Ti;
          if (raw < kAlphaMax) {
            const float dpow = dalpha * raw;
            v[5] = dalpha * e;
            v[0] = dpow * (A.z * dx + A.w * dy);
            v[1] = dpow * (A.w * dx + Bv.x * dy);
            v[2] = -0.5f * dpow * dx * dx;
            v[3] = -dpow * dx * dy;
            v[4] = -0.5f * dpow * dy * dy;
          }
        }
      }
      if (__any_sync(0xffffffffu, contrib)) {
#pragma unroll
        for (int c = 0; c < 9; ++c) v[c] = warp_sum(v[c]);
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < 9; ++c)
            if (v[c] != 0.f) atomicAdd(&S.acc[j][c], v[c]);
        }
      }
    }
    __syncthreads();
    if (tid < cnt) {
      float* a = S.acc[tid];
      bool nz = false;
#pragma unroll
      for (int c = 0; c < 9; ++c) nz |= a[c] != 0.f;
      if (nz) {
        float4* dst = grads + 3 * (view * n + (int64_t)S.id[k & 1][tid]);
        atomicAdd(dst, make_float4(a[0], a[1], a[2], a[3]));
        atomicAdd(dst + 1, make_float4(a[4], a[5], a[6], a[7]));
        atomicAdd(reinterpret_cast<float*>(dst + 2), a[8]);
      }
#pragma unroll
      for (int c = 0; c < 9; ++c) a[c] = 0.f;
    }
    __syncthreads();
  }
  cp_async_wait<0>();
}

}  // namespace
}  // namespace gs

using namespace gs;

static gs_status rasterize_fwd_impl(int64_t n, int32_t n_views, const gs_splat* splats,
                                    int32_t width, int32_t height, const uint32_t* vals,
                                    const int64_t* ranges, const float* bg, float* image,
                                    float* T_final, int32_t* n_contrib, uint64_t* counts,
                                    void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || !bg || !ranges || !image || !T_final || !n_contrib)
    return GS_ERR_INVALID_ARG;
  if (n > 0 && (!splats || !aligned16(splats))) return GS_ERR_INVALID_ARG;
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE;
  const unsigned grid = (unsigned)(n_views * T);
  unsigned long long* c = reinterpret_cast<unsigned long long*>(counts);
  if (counts)
    raster_fwd_kernel<true><<<grid, kRT, 0, (cudaStream_t)stream>>>(
        n, tiles_x, T, width, height, reinterpret_cast<const float4*>(splats), vals, ranges, bg[0],
        bg[1], bg[2], image, T_final, n_contrib, c);
  else
    raster_fwd_kernel<false><<<grid, kRT, 0, (cudaStream_t)stream>>>(
        n, tiles_x, T, width, height, reinterpret_cast<const float4*>(splats), vals, ranges, bg[0],
        bg[1], bg[2], image, T_final, n_contrib, c);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" gs_status gs_rasterize_fwd(int64_t n, int32_t n_views, const gs_splat* splats,
                                      int32_t width, int32_t height, const uint32_t* vals,
                                      const int64_t* ranges, const float* bg, float* image,
                                      float* T_final, int32_t* n_contrib, void* stream) {
  return rasterize_fwd_impl(n, n_views, splats, width, height, vals, ranges, bg, image, T_final,
                            n_contrib, nullptr, stream);
}

extern "C" gs_status gs_rasterize_fwd_counted(int64_t n, int32_t n_views, const gs_splat* splats,
                                              int32_t width, int32_t height, const uint32_t* vals,
                                              const int64_t* ranges, const float* bg, float* image,
                                              float* T_final, int32_t* n_contrib, uint64_t* counts,
                                              void* stream) {
  if (!counts) return GS_ERR_INVALID_ARG;
  return rasterize_fwd_impl(n, n_views, splats, width, height, vals, ranges, bg, image, T_final,
                            n_contrib, counts, stream);
}

extern "C" gs_status gs_rasterize_bwd(int64_t n, int32_t n_views, const gs_splat* splats,
                                      int32_t width, int32_t height, const uint32_t* vals,
                                      const int64_t* ranges, const float* bg, const float* T_final,
                                      const int32_t* n_contrib, const float* dL_dimage,
                                      gs_splat_grad* grads, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 ||
      height < 1 || !bg || !ranges || !T_final || !n_contrib || !dL_dimage)
    return GS_ERR_INVALID_ARG;
  if (n > 0 && (!splats || !grads || !aligned16(splats) || !aligned16(grads)))
    return GS_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (n > 0) GS_CUDA(cudaMemsetAsync(grads, 0, sizeof(gs_splat_grad) * (size_t)(n * n_views), st));
  const int64_t T = tiles_per_view(width, height);
  const int32_t tiles_x = (width + GS_TILE - 1) / GS_TILE;
  raster_bwd_kernel<<<(unsigned)(n_views * T), kRT, 0, st>>>(
      n, tiles_x, T, width, height, reinterpret_cast<const float4*>(splats), vals, ranges, bg[0],
      bg[1], bg[2], T_final, n_contrib, dL_dimage, reinterpret_cast<float4*>(grads));
  GS_CHECK_LAUNCH();
  return GS_OK;
}

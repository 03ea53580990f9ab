// gs_internal.cuh -- device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gs.h"

namespace gs {

constexpr float kDilation = 0.3f;          // added to the 2D covariance diagonal
constexpr float kClampFov = 1.3f;          // J uses x/z, y/z clamped to 1.3 half-FOV
constexpr float kAlphaMax = 0.99f;         // alpha cap
constexpr float kAlphaMin = 1.0f / 255.0f; // pairs below are skipped
constexpr float kTMin = 1e-4f;             // stop before T drops below
constexpr float kRadiusSigma = 3.0f;       // footprint radius in std deviations
constexpr float kRadiusCap = 1073741824.0f;  // 2^30, keeps radius an int32

// Per-camera constants, passed to kernels by value.
struct CamK {
  float R[9];
  float t[3];
  float fx, fy, cx, cy;
  float near_z, far_z;
  float lim_x, lim_y;   // clamp limits of x/z, y/z for J
  float campos[3];      // camera centre in world space, -R^T t
};

struct CamSet {
  CamK c[GS_MAX_VIEWS];
  int32_t n_views;
  int32_t width, height;
  int32_t tiles_x, tiles_y;
};

inline bool cams_valid(const gs_camera* cams, int32_t n_views) {
  if (!cams || n_views < 1 || n_views > GS_MAX_VIEWS) return false;
  for (int v = 0; v < n_views; ++v) {
    const gs_camera& c = cams[v];
    if (c.width <= 0 || c.height <= 0 || c.width != cams[0].width || c.height != cams[0].height)
      return false;
    if (!(c.fx > 0.f) || !(c.fy > 0.f) || !(c.near_z > 0.f) || !(c.far_z > c.near_z)) return false;
  }
  return true;
}

inline CamSet make_camset(const gs_camera* cams, int32_t n_views) {
  CamSet s{};
  s.n_views = n_views;
  s.width = cams[0].width;
  s.height = cams[0].height;
  s.tiles_x = (s.width + GS_TILE - 1) / GS_TILE;
  s.tiles_y = (s.height + GS_TILE - 1) / GS_TILE;
  for (int v = 0; v < n_views; ++v) {
    const gs_camera& c = cams[v];
    CamK& k = s.c[v];
    for (int i = 0; i < 9; ++i) k.R[i] = c.R[i];
    for (int i = 0; i < 3; ++i) k.t[i] = c.t[i];
    k.fx = c.fx; k.fy = c.fy; k.cx = c.cx; k.cy = c.cy;
    k.near_z = c.near_z; k.far_z = c.far_z;
    k.lim_x = (float)(1.3 * (0.5 * (double)c.width) / (double)c.fx);
    k.lim_y = (float)(1.3 * (0.5 * (double)c.height) / (double)c.fy);
    for (int i = 0; i < 3; ++i)
      k.campos[i] = (float)(-((double)c.R[i] * c.t[0] + (double)c.R[3 + i] * c.t[1] +
                              (double)c.R[6 + i] * c.t[2]));
  }
  return s;
}

inline int64_t tiles_per_view(int32_t width, int32_t height) {
  return (int64_t)((width + GS_TILE - 1) / GS_TILE) * ((height + GS_TILE - 1) / GS_TILE);
}

// Footprint rectangle in tile units, fp32 with one IEEE rounding per step
// (no contraction), so that every implementation of the definition agrees
// bit for bit:  x0 = clamp(floor((mx - r)/16), 0, TX), x1 = clamp(ceil((mx + r)/16), 0, TX).
__device__ __forceinline__ void tile_rect(float mx, float my, int32_t radius, int32_t tiles_x,
                                          int32_t tiles_y, int32_t& x0, int32_t& x1, int32_t& y0,
                                          int32_t& y1) {
  const float fr = (float)radius;
  const float ft = (float)GS_TILE;
  float fx0 = floorf(__fdiv_rn(__fsub_rn(mx, fr), ft));
  float fx1 = ceilf(__fdiv_rn(__fadd_rn(mx, fr), ft));
  float fy0 = floorf(__fdiv_rn(__fsub_rn(my, fr), ft));
  float fy1 = ceilf(__fdiv_rn(__fadd_rn(my, fr), ft));
  fx0 = fminf(fmaxf(fx0, 0.0f), (float)tiles_x);
  fx1 = fminf(fmaxf(fx1, 0.0f), (float)tiles_x);
  fy0 = fminf(fmaxf(fy0, 0.0f), (float)tiles_y);
  fy1 = fminf(fmaxf(fy1, 0.0f), (float)tiles_y);
  x0 = (int32_t)fx0;
  x1 = (int32_t)fx1;
  y0 = (int32_t)fy0;
  y1 = (int32_t)fy1;
}

__host__ __device__ inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Binning workspace: byte offset of the device status word, and its bit for
// "intersections exceed capacity" (set by the asynchronous binning).
constexpr size_t kWsStatusOffset = 8;
constexpr unsigned int kWsErrCapacity = 4u;

}  // namespace gs

#define GS_CHECK_LAUNCH()                                  \
  do {                                                     \
    if (cudaPeekAtLastError() != cudaSuccess) {            \
      (void)cudaGetLastError();                            \
      return GS_ERR_CUDA;                                  \
    }                                                      \
  } while (0)

#define GS_CUDA(call)                                      \
  do {                                                     \
    if ((call) != cudaSuccess) {                           \
      (void)cudaGetLastError();                            \
      return GS_ERR_CUDA;                                  \
    }                                                      \
  } while (0)

// project.cu -- gs_project and gs_project_bwd.
//
// EWA projection of 3D Gaussians with SH degree-3 colour (the 3D Gaussian
// Splatting model of Kerbl et al., cited in "A Scalable PyTorch Abstraction
// for Multi-GPU Gaussian Splatting", references; the "3D-to-2D Gaussian
// transformations" of "On Scaling Up 3D Gaussian Splatting Training",
// rendering-speed answer) and its exact backward.
//
// One thread per Gaussian reads its 59 parameters once (coalesced rows of
// the [59][n] SoA array) and loops over the views, so the parameter traffic
// is paid once per step however many cameras are batched.  HBM-bound.
// With a tile-count array, a culled row costs 4 written bytes (its count)
// instead of a record, and the backward reads the counts to find the rows
// it needs, so that scenes where a few per cent of the rows are visible
// move only what is visible.
#include <math.h>

#include "gs_internal.cuh"

namespace gs {
namespace {

// Real SH basis constants, degree <= 3 (l = 0..3, m = -l..l; sqrt(2) Re/Im of
// the complex harmonics with Condon-Shortley phase), from their closed forms.
struct ShK {
  float k0, k1, k2, k3, k4, k5, k6, k7, k8, k9;
};
__device__ __forceinline__ ShK sh_k() {
  ShK s;
  s.k0 = (float)(0.5 * 0.5641895835477563);       // 1/(2 sqrt(pi))
  s.k1 = (float)(0.4886025119029199);             // sqrt(3/(4 pi))
  s.k2 = (float)(1.0925484305920792);             // sqrt(15/(4 pi))
  s.k3 = (float)(0.31539156525252005);            // sqrt(5/(16 pi))
  s.k4 = (float)(0.5462742152960396);             // sqrt(15/(16 pi))
  s.k5 = (float)(0.5900435899266435);             // sqrt(35/(32 pi))
  s.k6 = (float)(2.890611442640554);              // sqrt(105/(4 pi))
  s.k7 = (float)(0.4570457994644658);             // sqrt(21/(32 pi))
  s.k8 = (float)(0.3731763325901154);             // sqrt(7/(16 pi))
  s.k9 = (float)(1.445305721320277);              // sqrt(105/(16 pi))
  return s;
}

__device__ __forceinline__ void sh_eval(float x, float y, float z, float Y[16]) {
  const ShK k = sh_k();
  const float xx = x * x, yy = y * y, zz = z * z;
  Y[0] = k.k0;
  Y[1] = -k.k1 * y;
  Y[2] = k.k1 * z;
  Y[3] = -k.k1 * x;
  Y[4] = k.k2 * x * y;
  Y[5] = -k.k2 * y * z;
  Y[6] = k.k3 * (2.f * zz - xx - yy);
  Y[7] = -k.k2 * x * z;
  Y[8] = k.k4 * (xx - yy);
  Y[9] = -k.k5 * y * (3.f * xx - yy);
  Y[10] = k.k6 * x * y * z;
  Y[11] = -k.k7 * y * (4.f * zz - xx - yy);
  Y[12] = k.k8 * z * (2.f * zz - 3.f * xx - 3.f * yy);
  Y[13] = -k.k7 * x * (4.f * zz - xx - yy);
  Y[14] = k.k9 * z * (xx - yy);
  Y[15] = -k.k5 * x * (xx - 3.f * yy);
}

// sum_k e[k] * grad Y_k at (x, y, z) (gradient of the polynomials)
__device__ __forceinline__ void sh_grad_dot(float x, float y, float z, const float e[16],
                                            float g[3]) {
  const ShK k = sh_k();
  const float xx = x * x, yy = y * y, zz = z * z;
  float gx = 0.f, gy = 0.f, gz = 0.f;
  gy += e[1] * (-k.k1);
  gz += e[2] * k.k1;
  gx += e[3] * (-k.k1);
  gx += e[4] * k.k2 * y;           gy += e[4] * k.k2 * x;
  gy += e[5] * (-k.k2 * z);        gz += e[5] * (-k.k2 * y);
  gx += e[6] * (-2.f * k.k3 * x);  gy += e[6] * (-2.f * k.k3 * y);  gz += e[6] * (4.f * k.k3 * z);
  gx += e[7] * (-k.k2 * z);        gz += e[7] * (-k.k2 * x);
  gx += e[8] * (2.f * k.k4 * x);   gy += e[8] * (-2.f * k.k4 * y);
  gx += e[9] * (-6.f * k.k5 * x * y);
  gy += e[9] * (-3.f * k.k5 * (xx - yy));
  gx += e[10] * k.k6 * y * z;      gy += e[10] * k.k6 * x * z;      gz += e[10] * k.k6 * x * y;
  gx += e[11] * (2.f * k.k7 * x * y);
  gy += e[11] * (-k.k7 * (4.f * zz - xx - 3.f * yy));
  gz += e[11] * (-8.f * k.k7 * y * z);
  gx += e[12] * (-6.f * k.k8 * x * z);
  gy += e[12] * (-6.f * k.k8 * y * z);
  gz += e[12] * (k.k8 * (6.f * zz - 3.f * xx - 3.f * yy));
  gx += e[13] * (-k.k7 * (4.f * zz - 3.f * xx - yy));
  gy += e[13] * (2.f * k.k7 * x * y);
  gz += e[13] * (-8.f * k.k7 * x * z);
  gx += e[14] * (2.f * k.k9 * x * z);
  gy += e[14] * (-2.f * k.k9 * y * z);
  gz += e[14] * (k.k9 * (xx - yy));
  gx += e[15] * (-3.f * k.k5 * (xx - yy));
  gy += e[15] * (6.f * k.k5 * x * y);
  g[0] = gx;
  g[1] = gy;
  g[2] = gz;
}

// View-independent part of one Gaussian.
struct Gauss {
  float mu[3];
  float scale[3];
  float qn[4];
  float qinv;   // 1/|q|
  float Rq[9];
  float M[9];   // Rq diag(scale)
  float S[6];   // Sigma: xx, xy, xz, yy, yz, zz
  float opacity;
};

__device__ __forceinline__ void load_gauss(const float* __restrict__ P, int64_t n, Gauss& G) {
  for (int i = 0; i < 3; ++i) G.mu[i] = __ldg(P + i * n);
  for (int i = 0; i < 3; ++i) G.scale[i] = expf(__ldg(P + (3 + i) * n));
  float q[4];
  for (int i = 0; i < 4; ++i) q[i] = __ldg(P + (6 + i) * n);
  const float qq = q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3];
  G.qinv = 1.0f / sqrtf(qq);
  for (int i = 0; i < 4; ++i) G.qn[i] = q[i] * G.qinv;
  const float w = G.qn[0], x = G.qn[1], y = G.qn[2], z = G.qn[3];
  G.Rq[0] = 1.f - 2.f * (y * y + z * z);
  G.Rq[1] = 2.f * (x * y - w * z);
  G.Rq[2] = 2.f * (x * z + w * y);
  G.Rq[3] = 2.f * (x * y + w * z);
  G.Rq[4] = 1.f - 2.f * (x * x + z * z);
  G.Rq[5] = 2.f * (y * z - w * x);
  G.Rq[6] = 2.f * (x * z - w * y);
  G.Rq[7] = 2.f * (y * z + w * x);
  G.Rq[8] = 1.f - 2.f * (x * x + y * y);
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j) G.M[3 * i + j] = G.Rq[3 * i + j] * G.scale[j];
  const float* M = G.M;
  G.S[0] = M[0] * M[0] + M[1] * M[1] + M[2] * M[2];
  G.S[1] = M[0] * M[3] + M[1] * M[4] + M[2] * M[5];
  G.S[2] = M[0] * M[6] + M[1] * M[7] + M[2] * M[8];
  G.S[3] = M[3] * M[3] + M[4] * M[4] + M[5] * M[5];
  G.S[4] = M[3] * M[6] + M[4] * M[7] + M[5] * M[8];
  G.S[5] = M[6] * M[6] + M[7] * M[7] + M[8] * M[8];
  G.opacity = 1.0f / (1.0f + expf(-__ldg(P + 10 * n)));
}

// View-dependent geometry of one Gaussian in one camera.
struct ViewGeom {
  float p[3];          // camera-space mean
  float tpos[2];       // clamped x, y used by J
  bool clamped[2];
  float J00, J02, J11, J12;
  float T[6];          // J W, 2x3
  float a, b, c;       // dilated 2D covariance
  float det;
  bool ok;             // inside near/far and det > 0
};

__device__ __forceinline__ void view_geom(const Gauss& G, const CamK& C, ViewGeom& V) {
  const float* W = C.R;
  for (int i = 0; i < 3; ++i)
    V.p[i] = W[3 * i] * G.mu[0] + W[3 * i + 1] * G.mu[1] + W[3 * i + 2] * G.mu[2] + C.t[i];
  const float x = V.p[0], y = V.p[1], z = V.p[2];
  V.ok = false;
  if (!(z >= C.near_z) || z > C.far_z) return;
  const float rz = 1.0f / z;
  float ux = x * rz, uy = y * rz;
  V.clamped[0] = ux < -C.lim_x || ux > C.lim_x;
  V.clamped[1] = uy < -C.lim_y || uy > C.lim_y;
  ux = fminf(fmaxf(ux, -C.lim_x), C.lim_x);
  uy = fminf(fmaxf(uy, -C.lim_y), C.lim_y);
  V.tpos[0] = ux * z;
  V.tpos[1] = uy * z;
  V.J00 = C.fx * rz;
  V.J11 = C.fy * rz;
  V.J02 = -C.fx * V.tpos[0] * rz * rz;
  V.J12 = -C.fy * V.tpos[1] * rz * rz;
  for (int j = 0; j < 3; ++j) {
    V.T[j] = V.J00 * W[j] + V.J02 * W[6 + j];
    V.T[3 + j] = V.J11 * W[3 + j] + V.J12 * W[6 + j];
  }
  const float* S = G.S;
  const float* T = V.T;
  float TS0[3], TS1[3];
  TS0[0] = T[0] * S[0] + T[1] * S[1] + T[2] * S[2];
  TS0[1] = T[0] * S[1] + T[1] * S[3] + T[2] * S[4];
  TS0[2] = T[0] * S[2] + T[1] * S[4] + T[2] * S[5];
  TS1[0] = T[3] * S[0] + T[4] * S[1] + T[5] * S[2];
  TS1[1] = T[3] * S[1] + T[4] * S[3] + T[5] * S[4];
  TS1[2] = T[3] * S[2] + T[4] * S[4] + T[5] * S[5];
  V.a = TS0[0] * T[0] + TS0[1] * T[1] + TS0[2] * T[2] + kDilation;
  V.b = TS0[0] * T[3] + TS0[1] * T[4] + TS0[2] * T[5];
  V.c = TS1[0] * T[3] + TS1[1] * T[4] + TS1[2] * T[5] + kDilation;
  V.det = V.a * V.c - V.b * V.b;
  V.ok = V.det > 0.0f;
}

// Footprint of one Gaussian in one view: its view geometry, projected mean,
// radius and tile count (0 = culled).
__device__ __forceinline__ int32_t view_footprint(const Gauss& G, const CamK& C, const CamSet& cs,
                                                  ViewGeom& V, float& mx, float& my,
                                                  int32_t& radius) {
  view_geom(G, C, V);
  radius = 0;
  mx = my = 0.f;
  if (!V.ok) return 0;
  const float rz = 1.0f / V.p[2];
  mx = C.fx * V.p[0] * rz + C.cx;
  my = C.fy * V.p[1] * rz + C.cy;
  const float half = 0.5f * (V.a - V.c);
  const float lam = 0.5f * (V.a + V.c) + sqrtf(fmaxf(half * half + V.b * V.b, 0.f));
  const float rr = fminf(kRadiusSigma * sqrtf(lam), kRadiusCap);
  radius = (int32_t)ceilf(rr);
  int32_t x0, x1, y0, y1;
  tile_rect(mx, my, radius, cs.tiles_x, cs.tiles_y, x0, x1, y0, y1);
  return (x1 - x0) * (y1 - y0);
}

// The record of a visible row: mean, conic, opacity, SH colour, depth,
// radius, tile count.
__device__ __forceinline__ void write_record(const Gauss& G, const CamK& C, const ViewGeom& V,
                                             float mx, float my, int32_t radius, int32_t tiles,
                                             const float sh[48], float4* rec) {
  float dir[3] = {G.mu[0] - C.campos[0], G.mu[1] - C.campos[1], G.mu[2] - C.campos[2]};
  const float il = 1.0f / sqrtf(dir[0] * dir[0] + dir[1] * dir[1] + dir[2] * dir[2]);
  float Y[16];
  sh_eval(dir[0] * il, dir[1] * il, dir[2] * il, Y);
  float col[3];
#pragma unroll
  for (int ch = 0; ch < 3; ++ch) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) acc += Y[k] * sh[3 * k + ch];
    col[ch] = fmaxf(acc + 0.5f, 0.f);
  }
  const float idet = 1.0f / V.det;
  rec[0] = make_float4(mx, my, V.c * idet, -V.b * idet);
  rec[1] = make_float4(V.a * idet, G.opacity, col[0], col[1]);
  rec[2] = make_float4(col[2], V.p[2], __int_as_float(radius), __int_as_float(tiles));
}

__global__ void __launch_bounds__(128, 5) project_fwd_kernel(int64_t n, const float* __restrict__ params,
                                                          const __grid_constant__ CamSet cs,
                                                          float4* __restrict__ out,
                                                          int32_t* __restrict__ counts) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n) return;
  Gauss G;
  load_gauss(params + g, n, G);
  float sh[48];
  bool have_sh = false;
  for (int v = 0; v < cs.n_views; ++v) {
    const CamK& C = cs.c[v];
    const int64_t row = (int64_t)v * n + g;
    float4* rec = out + 3 * row;
    ViewGeom V;
    float mx, my;
    int32_t radius;
    const int32_t tiles = view_footprint(G, C, cs, V, mx, my, radius);
    if (tiles == 0) {
      if (counts) counts[row] = 0;
      else rec[2] = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    if (!have_sh) {
#pragma unroll
      for (int k = 0; k < 48; ++k) sh[k] = __ldg(params + (11 + k) * n + g);
      have_sh = true;
    }
    write_record(G, C, V, mx, my, radius, tiles, sh, rec);
    if (counts) counts[row] = tiles;
  }
}

// Backward of one visible row (view camera C, row index row) into the
// Gaussian's geometric gradients (accumulated); Yo and gco receive the SH
// basis at the view direction and the colour gradient after the clamp, whose
// products are the row's SH-coefficient gradients.
__device__ __forceinline__ void view_backward(const Gauss& G, const CamK& C, int64_t row,
                                              const float4* __restrict__ splats,
                                              const float4* __restrict__ grads,
                                              const float* __restrict__ params, int64_t n,
                                              int64_t g, float g_mu[3], float g_ls[3],
                                              float g_q[4], float& g_logit, float Yo[16],
                                              float gco[3]) {
  // the colour from the row's record (its last 32 bytes); the conic is
  // recomputed with the projection's own arithmetic (bit for bit what it
  // stored), so the first 16 bytes are not read
  const float4 r1 = splats[3 * row + 1], r2 = splats[3 * row + 2];
  const float4 q0 = grads[3 * row], q1 = grads[3 * row + 1], q2 = grads[3 * row + 2];
  const float gm0 = q0.x, gm1 = q0.y, gA = q0.z, gB = q0.w, gC = q1.x, gop = q1.y;
  const float gcol[3] = {q1.z, q1.w, q2.x};
  const float col[3] = {r1.z, r1.w, r2.x};
  ViewGeom V;
  view_geom(G, C, V);
  const float* W = C.R;
  // opacity = sigmoid(logit)
  g_logit += gop * G.opacity * (1.f - G.opacity);
  // colour = max(sum_k Y_k sh_k + 0.5, 0): clamped channels pass nothing
  {
    float dir[3] = {G.mu[0] - C.campos[0], G.mu[1] - C.campos[1], G.mu[2] - C.campos[2]};
    const float il = 1.0f / sqrtf(dir[0] * dir[0] + dir[1] * dir[1] + dir[2] * dir[2]);
    const float d[3] = {dir[0] * il, dir[1] * il, dir[2] * il};
    float Y[16];
    sh_eval(d[0], d[1], d[2], Y);
    const float gc0 = col[0] > 0.f ? gcol[0] : 0.f;
    const float gc1 = col[1] > 0.f ? gcol[1] : 0.f;
    const float gc2 = col[2] > 0.f ? gcol[2] : 0.f;
    gco[0] = gc0;
    gco[1] = gc1;
    gco[2] = gc2;
    float e[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      Yo[k] = Y[k];
      e[k] = __ldg(params + (11 + 3 * k) * n + g) * gc0 +
             __ldg(params + (12 + 3 * k) * n + g) * gc1 +
             __ldg(params + (13 + 3 * k) * n + g) * gc2;
    }
    float gd[3];
    sh_grad_dot(d[0], d[1], d[2], e, gd);
    const float dd = d[0] * gd[0] + d[1] * gd[1] + d[2] * gd[2];
    for (int i = 0; i < 3; ++i) g_mu[i] += (gd[i] - d[i] * dd) * il;
  }
  const float x = V.p[0], y = V.p[1], z = V.p[2];
  const float rz = 1.0f / z, rz2 = rz * rz;
  float gp[3];
  // mean2d = (fx x/z + cx, fy y/z + cy)
  gp[0] = gm0 * C.fx * rz;
  gp[1] = gm1 * C.fy * rz;
  gp[2] = -(gm0 * C.fx * x + gm1 * C.fy * y) * rz2;
  // conic = cov2^-1: H = -K Gk K with Gk = [[gA, gB/2], [gB/2, gC]], K = conic
  const float idet = 1.0f / V.det;
  const float A = V.c * idet, B = -V.b * idet, Cc = V.a * idet;
  const float hB = 0.5f * gB;
  const float t00 = A * gA + B * hB, t01 = A * hB + B * gC;
  const float t10 = B * gA + Cc * hB, t11 = B * hB + Cc * gC;
  const float H00 = -(t00 * A + t01 * B);
  const float H01 = -(t00 * B + t01 * Cc);
  const float H11 = -(t10 * B + t11 * Cc);
  // cov2 = T Sigma T^T + 0.3 I: G_T = 2 H T Sigma, G_Sigma = T^T H T
  const float* S = G.S;
  const float* T = V.T;
  float TS[6];
  TS[0] = T[0] * S[0] + T[1] * S[1] + T[2] * S[2];
  TS[1] = T[0] * S[1] + T[1] * S[3] + T[2] * S[4];
  TS[2] = T[0] * S[2] + T[1] * S[4] + T[2] * S[5];
  TS[3] = T[3] * S[0] + T[4] * S[1] + T[5] * S[2];
  TS[4] = T[3] * S[1] + T[4] * S[3] + T[5] * S[4];
  TS[5] = T[3] * S[2] + T[4] * S[4] + T[5] * S[5];
  float GT[6];
  for (int j = 0; j < 3; ++j) {
    GT[j] = 2.f * (H00 * TS[j] + H01 * TS[3 + j]);
    GT[3 + j] = 2.f * (H01 * TS[j] + H11 * TS[3 + j]);
  }
  // G_Sigma = T^T H T (symmetric 3x3)
  float HT[6];  // H T, 2x3
  for (int j = 0; j < 3; ++j) {
    HT[j] = H00 * T[j] + H01 * T[3 + j];
    HT[3 + j] = H01 * T[j] + H11 * T[3 + j];
  }
  float GS[9];
  for (int a_ = 0; a_ < 3; ++a_)
    for (int b_ = 0; b_ < 3; ++b_) GS[3 * a_ + b_] = T[a_] * HT[b_] + T[3 + a_] * HT[3 + b_];
  // T = J W: G_J = G_T W^T (only the four non-constant entries of J)
  const float GJ00 = GT[0] * W[0] + GT[1] * W[1] + GT[2] * W[2];
  const float GJ02 = GT[0] * W[6] + GT[1] * W[7] + GT[2] * W[8];
  const float GJ11 = GT[3] * W[3] + GT[4] * W[4] + GT[5] * W[5];
  const float GJ12 = GT[3] * W[6] + GT[4] * W[7] + GT[5] * W[8];
  gp[2] += -(GJ00 * C.fx + GJ11 * C.fy) * rz2;
  // J02 = -fx tx / z^2 with tx = z clamp(x/z): x-derivative only when unclamped
  if (!V.clamped[0]) {
    gp[0] += GJ02 * (-C.fx * rz2);
    gp[2] += GJ02 * (2.f * C.fx * x * rz2 * rz);
  } else {
    gp[2] += GJ02 * (C.fx * V.tpos[0] * rz * rz2);
  }
  if (!V.clamped[1]) {
    gp[1] += GJ12 * (-C.fy * rz2);
    gp[2] += GJ12 * (2.f * C.fy * y * rz2 * rz);
  } else {
    gp[2] += GJ12 * (C.fy * V.tpos[1] * rz * rz2);
  }
  // p = W mu + t
  for (int i = 0; i < 3; ++i) g_mu[i] += W[i] * gp[0] + W[3 + i] * gp[1] + W[6 + i] * gp[2];
  // Sigma = M M^T, M = Rq diag(scale): G_M = 2 G_Sigma M
  float GM[9];
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j)
      GM[3 * i + j] = 2.f * (GS[3 * i] * G.M[j] + GS[3 * i + 1] * G.M[3 + j] +
                             GS[3 * i + 2] * G.M[6 + j]);
  float GR[9];
  for (int j = 0; j < 3; ++j) {
    const float gsj = G.Rq[j] * GM[j] + G.Rq[3 + j] * GM[3 + j] + G.Rq[6 + j] * GM[6 + j];
    g_ls[j] += gsj * G.scale[j];
    for (int i = 0; i < 3; ++i) GR[3 * i + j] = GM[3 * i + j] * G.scale[j];
  }
  // rotation matrix of the unit quaternion -> quaternion, then normalisation
  const float w = G.qn[0], qx = G.qn[1], qy = G.qn[2], qz = G.qn[3];
  float gqn[4];
  gqn[0] = 2.f * (-qz * GR[1] + qy * GR[2] + qz * GR[3] - qx * GR[5] - qy * GR[6] + qx * GR[7]);
  gqn[1] = 2.f * (qy * GR[1] + qz * GR[2] + qy * GR[3] - 2.f * qx * GR[4] - w * GR[5] +
                  qz * GR[6] + w * GR[7] - 2.f * qx * GR[8]);
  gqn[2] = 2.f * (-2.f * qy * GR[0] + qx * GR[1] + w * GR[2] + qx * GR[3] + qz * GR[5] -
                  w * GR[6] + qz * GR[7] - 2.f * qy * GR[8]);
  gqn[3] = 2.f * (-2.f * qz * GR[0] - w * GR[1] + qx * GR[2] + w * GR[3] - 2.f * qz * GR[4] +
                  qy * GR[5] + qx * GR[6] + qy * GR[7]);
  const float dq = w * gqn[0] + qx * gqn[1] + qy * gqn[2] + qz * gqn[3];
  for (int i = 0; i < 4; ++i) g_q[i] += (gqn[i] - G.qn[i] * dq) * G.qinv;
}

__global__ void __launch_bounds__(128, 5) project_bwd_kernel(int64_t n, const float* __restrict__ params,
                                                          const __grid_constant__ CamSet cs,
                                                          const float4* __restrict__ splats,
                                                          const int32_t* __restrict__ counts,
                                                          const float4* __restrict__ grads,
                                                          float* __restrict__ grad,
                                                          uint8_t* __restrict__ visible) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n) return;
  // the views in which the row is visible, all loads issued up front
  uint32_t vmask = 0;
  if (counts) {
#pragma unroll
    for (int v = 0; v < GS_MAX_VIEWS; ++v)
      if (v < cs.n_views && __ldg(counts + (int64_t)v * n + g) > 0) vmask |= 1u << v;
  } else {
#pragma unroll
    for (int v = 0; v < GS_MAX_VIEWS; ++v)
      if (v < cs.n_views && __float_as_int(splats[3 * ((int64_t)v * n + g) + 2].z) > 0)
        vmask |= 1u << v;
  }
  float* out = grad + g;
  if (!vmask) {  // seen by no view: a zero gradient column
#pragma unroll
    for (int i = 0; i < GS_NPARAM; ++i) out[i * n] = 0.f;
    if (visible) visible[g] = 0;
    return;
  }
  Gauss G;
  load_gauss(params + g, n, G);
  float g_mu[3] = {0.f, 0.f, 0.f}, g_ls[3] = {0.f, 0.f, 0.f}, g_q[4] = {0.f, 0.f, 0.f, 0.f};
  float g_logit = 0.f;
  __shared__ float s_gsh[48][128];  // this thread's SH gradient sums in column threadIdx.x
  float* g_sh_col = &s_gsh[0][threadIdx.x];
#pragma unroll
  for (int k = 0; k < 48; ++k) g_sh_col[128 * k] = 0.f;
  for (uint32_t vm = vmask; vm; vm &= vm - 1u) {
    const int v = __ffs(vm) - 1;
    const int64_t row = (int64_t)v * n + g;
    float Y[16], gc[3];
    view_backward(G, cs.c[v], row, splats, grads, params, n, g, g_mu, g_ls, g_q, g_logit, Y, gc);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      g_sh_col[128 * (3 * k)] += Y[k] * gc[0];
      g_sh_col[128 * (3 * k + 1)] += Y[k] * gc[1];
      g_sh_col[128 * (3 * k + 2)] += Y[k] * gc[2];
    }
  }
  for (int i = 0; i < 3; ++i) out[i * n] = g_mu[i];
  for (int i = 0; i < 3; ++i) out[(3 + i) * n] = g_ls[i];
  for (int i = 0; i < 4; ++i) out[(6 + i) * n] = g_q[i];
  out[10 * n] = g_logit;
#pragma unroll
  for (int k = 0; k < 48; ++k) out[(11 + k) * n] = g_sh_col[128 * k];
  if (visible) visible[g] = 1;
}

}  // namespace
}  // namespace gs

using namespace gs;

extern "C" gs_status gs_project(int64_t n, const float* params, const gs_camera* cams,
                                int32_t n_views, gs_splat* splats, int32_t* tile_counts,
                                void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || !cams_valid(cams, n_views)) return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  if (!params || !splats || !aligned16(splats) || !aligned4(tile_counts)) return GS_ERR_INVALID_ARG;
  const CamSet cs = make_camset(cams, n_views);
  const int threads = 128;
  cudaStream_t st = (cudaStream_t)stream;
  float4* sp = reinterpret_cast<float4*>(splats);
  project_fwd_kernel<<<(unsigned)div_up(n, threads), threads, 0, st>>>(n, params, cs, sp,
                                                                        tile_counts);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

extern "C" gs_status gs_project_bwd(int64_t n, const float* params, const gs_camera* cams,
                                    int32_t n_views, const gs_splat* splats,
                                    const int32_t* tile_counts, const gs_splat_grad* grads,
                                    float* grad, uint8_t* visible, void* stream) {
  if (n < 0 || n >= (int64_t(1) << 32) || !cams_valid(cams, n_views)) return GS_ERR_INVALID_ARG;
  if (n == 0) return GS_OK;
  if (!params || !splats || !grads || !grad || !aligned16(splats) || !aligned16(grads) ||
      !aligned4(tile_counts))
    return GS_ERR_INVALID_ARG;
  const CamSet cs = make_camset(cams, n_views);
  const int threads = 128;
  cudaStream_t st = (cudaStream_t)stream;
  const float4* sp = reinterpret_cast<const float4*>(splats);
  const float4* gr = reinterpret_cast<const float4*>(grads);
  project_bwd_kernel<<<(unsigned)div_up(n, threads), threads, 0, st>>>(n, params, cs, sp,
                                                                        tile_counts, gr, grad,
                                                                        visible);
  GS_CHECK_LAUNCH();
  return GS_OK;
}

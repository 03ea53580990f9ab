/*
 * gs_oracle.c -- plain CPU oracle of the 3DGS training step (fp64).
 *
 * TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use this file.  It is deliberately slow and literal: one
 * loop per definition, no tiling tricks beyond the tile lists the method
 * itself defines, no fused passes.  Compile with -ffp-contract=off so that the
 * fp32 steps (tile rectangle, sort key) round exactly as written.
 *
 * Sources (page title, section):
 *  - parameter record: "On Scaling Up 3D Gaussian Splatting Training", answer
 *    on the storage requirement (59 fp32: 48 SH, 3 xyz, 3 scale, 4 rotation,
 *    1 opacity);
 *  - per-tile sorted intersection lists: "AMD ROCm team open-sources
 *    distributed 3D Gaussian Splatting training", per-tile intersection bullet;
 *  - 16x16 pixel blocks that alter no pixel value: "On Scaling Up ...", answer
 *    (1) on the pixel block size;
 *  - opacity saturation depth (early termination): "On Scaling Up ...",
 *    comparison to RetinaGS;
 *  - forward and backward rasterization: "ByteSplat" abstract;
 *  - Adam: Kingma & Ba, cited in "A Scalable PyTorch Abstraction for
 *    Multi-GPU Gaussian Splatting", references; moments per the ROCm item.
 * The projection, SH colour and compositing formulas are the standard 3D
 * Gaussian Splatting model (Kerbl et al., cited in "A Scalable PyTorch
 * Abstraction ...", references); the pages name it but print none of its
 * equations, so each step below states the formula it evaluates.
 */
#include "gs_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* Method constants (readings where the pages are silent). */
static const double kDilation = 0.3;    /* added to the 2D covariance diagonal      */
static const double kClampFov = 1.3;    /* J is evaluated with x/z, y/z clamped     */
static const double kAlphaMax = 0.99;   /* alpha cap                                */
static const double kAlphaMin = 1.0 / 255.0; /* pairs below this alpha are skipped  */
static const double kTMin = 1e-4;       /* stop before transmittance drops below    */
static const double kRadiusSigma = 3.0; /* footprint radius in std deviations       */
static const double kRadiusCap = 1073741824.0; /* 2^30: keeps the int32 radius finite */

/* ------------------------------------------------------------------------ */
/* Real spherical harmonics, degree <= 3.  Order: l = 0..3, m = -l..l.
 * Convention: Y_{l,0} = complex Y_l^0; Y_{l,m>0} = sqrt(2) Re Y_l^m;
 * Y_{l,m<0} = sqrt(2) Im Y_l^{|m|}, with the Condon-Shortley phase inside
 * the complex Y_l^m.  Written out as polynomials of the unit direction. */
static void sh_consts(double k[10]) {
  const double pi = M_PI;
  k[0] = 0.5 * sqrt(1.0 / pi);          /* l=0                      */
  k[1] = sqrt(3.0 / (4.0 * pi));        /* l=1                      */
  k[2] = sqrt(15.0 / (4.0 * pi));       /* l=2, m=+-1, m=-2          */
  k[3] = sqrt(5.0 / (16.0 * pi));       /* l=2, m=0                  */
  k[4] = sqrt(15.0 / (16.0 * pi));      /* l=2, m=2                  */
  k[5] = sqrt(35.0 / (32.0 * pi));      /* l=3, m=+-3                */
  k[6] = sqrt(105.0 / (4.0 * pi));      /* l=3, m=-2                 */
  k[7] = sqrt(21.0 / (32.0 * pi));      /* l=3, m=+-1                */
  k[8] = sqrt(7.0 / (16.0 * pi));       /* l=3, m=0                  */
  k[9] = sqrt(105.0 / (16.0 * pi));     /* l=3, m=2                  */
}

void or_sh_basis(const double d[3], double Y[16]) {
  double k[10];
  sh_consts(k);
  const double x = d[0], y = d[1], z = d[2];
  Y[0] = k[0];
  Y[1] = -k[1] * y;
  Y[2] = k[1] * z;
  Y[3] = -k[1] * x;
  Y[4] = k[2] * x * y;
  Y[5] = -k[2] * y * z;
  Y[6] = k[3] * (2.0 * z * z - x * x - y * y);
  Y[7] = -k[2] * x * z;
  Y[8] = k[4] * (x * x - y * y);
  Y[9] = -k[5] * y * (3.0 * x * x - y * y);
  Y[10] = k[6] * x * y * z;
  Y[11] = -k[7] * y * (4.0 * z * z - x * x - y * y);
  Y[12] = k[8] * z * (2.0 * z * z - 3.0 * x * x - 3.0 * y * y);
  Y[13] = -k[7] * x * (4.0 * z * z - x * x - y * y);
  Y[14] = k[9] * z * (x * x - y * y);
  Y[15] = -k[5] * x * (x * x - 3.0 * y * y);
}

/* Partial derivatives of the 16 polynomials above w.r.t. (x, y, z):
 * dY[k][0..2]. */
static void sh_basis_grad(const double d[3], double dY[16][3]) {
  double k[10];
  sh_consts(k);
  const double x = d[0], y = d[1], z = d[2];
  memset(dY, 0, sizeof(double) * 48);
  /* l=1 */
  dY[1][1] = -k[1];
  dY[2][2] = k[1];
  dY[3][0] = -k[1];
  /* l=2 */
  dY[4][0] = k[2] * y;  dY[4][1] = k[2] * x;
  dY[5][1] = -k[2] * z; dY[5][2] = -k[2] * y;
  dY[6][0] = -2.0 * k[3] * x; dY[6][1] = -2.0 * k[3] * y; dY[6][2] = 4.0 * k[3] * z;
  dY[7][0] = -k[2] * z; dY[7][2] = -k[2] * x;
  dY[8][0] = 2.0 * k[4] * x; dY[8][1] = -2.0 * k[4] * y;
  /* l=3 */
  dY[9][0] = -6.0 * k[5] * x * y;
  dY[9][1] = -k[5] * (3.0 * x * x - 3.0 * y * y);
  dY[10][0] = k[6] * y * z; dY[10][1] = k[6] * x * z; dY[10][2] = k[6] * x * y;
  dY[11][0] = 2.0 * k[7] * x * y;
  dY[11][1] = -k[7] * (4.0 * z * z - x * x - 3.0 * y * y);
  dY[11][2] = -8.0 * k[7] * y * z;
  dY[12][0] = -6.0 * k[8] * x * z;
  dY[12][1] = -6.0 * k[8] * y * z;
  dY[12][2] = k[8] * (6.0 * z * z - 3.0 * x * x - 3.0 * y * y);
  dY[13][0] = -k[7] * (4.0 * z * z - 3.0 * x * x - y * y);
  dY[13][1] = 2.0 * k[7] * x * y;
  dY[13][2] = -8.0 * k[7] * x * z;
  dY[14][0] = 2.0 * k[9] * x * z; dY[14][1] = -2.0 * k[9] * y * z;
  dY[14][2] = k[9] * (x * x - y * y);
  dY[15][0] = -k[5] * (3.0 * x * x - 3.0 * y * y);
  dY[15][1] = 6.0 * k[5] * x * y;
}

/* ------------------------------------------------------------------------ */
/* Unit quaternion (w,x,y,z) -> rotation matrix (row-major). */
void or_quat_to_rot(const double q[4], double Rm[9]) {
  const double w = q[0], x = q[1], y = q[2], z = q[3];
  Rm[0] = 1.0 - 2.0 * (y * y + z * z);
  Rm[1] = 2.0 * (x * y - w * z);
  Rm[2] = 2.0 * (x * z + w * y);
  Rm[3] = 2.0 * (x * y + w * z);
  Rm[4] = 1.0 - 2.0 * (x * x + z * z);
  Rm[5] = 2.0 * (y * z - w * x);
  Rm[6] = 2.0 * (x * z - w * y);
  Rm[7] = 2.0 * (y * z + w * x);
  Rm[8] = 1.0 - 2.0 * (x * x + y * y);
}

/* Derivative of the matrix above w.r.t. each quaternion component, contracted
 * with the matrix gradient G: out[i] = sum_ab G[ab] dR[ab]/dq_i. */
static void quat_rot_vjp(const double q[4], const double G[9], double out[4]) {
  const double w = q[0], x = q[1], y = q[2], z = q[3];
  const double dw[9] = {0, -2 * z, 2 * y, 2 * z, 0, -2 * x, -2 * y, 2 * x, 0};
  const double dx[9] = {0, 2 * y, 2 * z, 2 * y, -4 * x, -2 * w, 2 * z, 2 * w, -4 * x};
  const double dy[9] = {-4 * y, 2 * x, 2 * w, 2 * x, 0, 2 * z, -2 * w, 2 * z, -4 * y};
  const double dz[9] = {-4 * z, -2 * w, 2 * x, 2 * w, -4 * z, 2 * y, 2 * x, 2 * y, 0};
  out[0] = out[1] = out[2] = out[3] = 0.0;
  for (int i = 0; i < 9; ++i) {
    out[0] += G[i] * dw[i];
    out[1] += G[i] * dx[i];
    out[2] += G[i] * dy[i];
    out[3] += G[i] * dz[i];
  }
}

/* ------------------------------------------------------------------------ */
/* Tile rectangle, evaluated in fp32 with one rounding per operation:
 *   x0 = clamp(floor((mx - r) / tile), 0, tiles_x)
 *   x1 = clamp(ceil ((mx + r) / tile), 0, tiles_x)   (same for y). */
void or_tile_rect(float mx, float my, int32_t radius, int32_t tile, int32_t tiles_x,
                  int32_t tiles_y, int32_t rect[4]) {
  const float fr = (float)radius;
  const float ft = (float)tile;
  float x0 = floorf((mx - fr) / ft);
  float x1 = ceilf((mx + fr) / ft);
  float y0 = floorf((my - fr) / ft);
  float y1 = ceilf((my + fr) / ft);
  x0 = fminf(fmaxf(x0, 0.0f), (float)tiles_x);
  x1 = fminf(fmaxf(x1, 0.0f), (float)tiles_x);
  y0 = fminf(fmaxf(y0, 0.0f), (float)tiles_y);
  y1 = fminf(fmaxf(y1, 0.0f), (float)tiles_y);
  rect[0] = (int32_t)x0;
  rect[1] = (int32_t)x1;
  rect[2] = (int32_t)y0;
  rect[3] = (int32_t)y1;
}

static int near_integer(double v, double tol) { return fabs(v - nearbyint(v)) < tol; }

/* ------------------------------------------------------------------------ */
/* One Gaussian in one view, all intermediate quantities kept for the
 * backward pass. */
typedef struct proj_state {
  int visible;
  double mu[3], p[3];
  double scale[3], qn[4], qnorm, Rq[9], M[9], Sigma[9];
  double lim[2], clamped[2], tpos[2];
  double J[6], T[6], cov2[3], det, conic[3];
  double mean2d[2], radius_real;
  int32_t radius, tiles;
  double dir[3], dnorm, d[3], Y[16], color_raw[3], color[3];
  double opacity;
  uint8_t flags;
} proj_state;

static void project_one(const double* params, int64_t n, int64_t g, const or_camera* cam,
                        int32_t tile, proj_state* s) {
  memset(s, 0, sizeof(*s));
  for (int i = 0; i < 3; ++i) s->mu[i] = params[i * n + g];
  const double* W = cam->R;
  /* 1. camera-space mean p = W mu + t */
  for (int i = 0; i < 3; ++i)
    s->p[i] = W[3 * i] * s->mu[0] + W[3 * i + 1] * s->mu[1] + W[3 * i + 2] * s->mu[2] + cam->t[i];
  const double x = s->p[0], y = s->p[1], z = s->p[2];
  if (fabs(z - cam->near_z) < 1e-4 * fabs(cam->near_z) ||
      (isfinite(cam->far_z) && fabs(z - cam->far_z) < 1e-4 * fabs(cam->far_z)))
    s->flags |= OR_FLAG_DEPTH;
  if (!(z >= cam->near_z) || z > cam->far_z) return;
  /* 2. 3D covariance Sigma = Rq S S^T Rq^T, S = diag(exp(log-scale)) */
  for (int i = 0; i < 3; ++i) s->scale[i] = exp(params[(3 + i) * n + g]);
  double q[4];
  for (int i = 0; i < 4; ++i) q[i] = params[(6 + i) * n + g];
  s->qnorm = sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
  for (int i = 0; i < 4; ++i) s->qn[i] = q[i] / s->qnorm;
  or_quat_to_rot(s->qn, s->Rq);
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j) s->M[3 * i + j] = s->Rq[3 * i + j] * s->scale[j];
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j) {
      double acc = 0.0;
      for (int k = 0; k < 3; ++k) acc += s->M[3 * i + k] * s->M[3 * j + k];
      s->Sigma[3 * i + j] = acc;
    }
  /* 3. EWA: J at the clamped position, cov2 = J W Sigma W^T J^T + 0.3 I */
  s->lim[0] = kClampFov * (0.5 * cam->width) / cam->fx;
  s->lim[1] = kClampFov * (0.5 * cam->height) / cam->fy;
  const double ratio[2] = {x / z, y / z};
  for (int a = 0; a < 2; ++a) {
    double u = ratio[a];
    if (fabs(fabs(u) - s->lim[a]) < 1e-4 * s->lim[a]) s->flags |= OR_FLAG_CLAMP;
    if (u < -s->lim[a]) { u = -s->lim[a]; s->clamped[a] = 1.0; }
    else if (u > s->lim[a]) { u = s->lim[a]; s->clamped[a] = 1.0; }
    s->tpos[a] = u * z;
  }
  const double fx = cam->fx, fy = cam->fy;
  s->J[0] = fx / z; s->J[1] = 0.0; s->J[2] = -fx * s->tpos[0] / (z * z);
  s->J[3] = 0.0;    s->J[4] = fy / z; s->J[5] = -fy * s->tpos[1] / (z * z);
  for (int i = 0; i < 2; ++i)
    for (int j = 0; j < 3; ++j) {
      double acc = 0.0;
      for (int k = 0; k < 3; ++k) acc += s->J[3 * i + k] * W[3 * k + j];
      s->T[3 * i + j] = acc;
    }
  double C2[4];
  for (int i = 0; i < 2; ++i)
    for (int j = 0; j < 2; ++j) {
      double acc = 0.0;
      for (int a = 0; a < 3; ++a)
        for (int b = 0; b < 3; ++b) acc += s->T[3 * i + a] * s->Sigma[3 * a + b] * s->T[3 * j + b];
      C2[2 * i + j] = acc;
    }
  s->cov2[0] = C2[0] + kDilation;
  s->cov2[1] = C2[1];
  s->cov2[2] = C2[3] + kDilation;
  /* 4. conic = inverse of the dilated 2D covariance */
  const double a = s->cov2[0], b = s->cov2[1], c = s->cov2[2];
  s->det = a * c - b * b;
  if (s->det < 1e-6 * a * c) s->flags |= OR_FLAG_DET;
  if (!(s->det > 0.0)) return;
  s->conic[0] = c / s->det;
  s->conic[1] = -b / s->det;
  s->conic[2] = a / s->det;
  s->mean2d[0] = fx * x / z + cam->cx;
  s->mean2d[1] = fy * y / z + cam->cy;
  /* 5. radius = ceil(3 sqrt(lambda_max)), tile rectangle */
  const double half = 0.5 * (a - c);
  const double lam = 0.5 * (a + c) + sqrt(fmax(half * half + b * b, 0.0));
  s->radius_real = fmin(kRadiusSigma * sqrt(lam), kRadiusCap);
  if (near_integer(s->radius_real, 1e-4 * fmax(1.0, s->radius_real))) s->flags |= OR_FLAG_RADIUS;
  s->radius = (int32_t)ceil(s->radius_real);
  const int32_t tiles_x = (cam->width + tile - 1) / tile;
  const int32_t tiles_y = (cam->height + tile - 1) / tile;
  int32_t rect[4];
  const float mxf = (float)s->mean2d[0], myf = (float)s->mean2d[1];
  or_tile_rect(mxf, myf, s->radius, tile, tiles_x, tiles_y, rect);
  {
    const double e[4] = {((double)mxf - s->radius) / tile, ((double)mxf + s->radius) / tile,
                         ((double)myf - s->radius) / tile, ((double)myf + s->radius) / tile};
    for (int i = 0; i < 4; ++i)
      if (near_integer(e[i], 1e-4 * fmax(1.0, fabs(e[i])))) s->flags |= OR_FLAG_RECT;
  }
  s->tiles = (rect[1] - rect[0]) * (rect[3] - rect[2]);
  if (s->tiles == 0) { s->radius = 0; return; }
  /* 6. view-dependent colour from SH degree 3 */
  double campos[3];
  for (int i = 0; i < 3; ++i)
    campos[i] = -(W[i] * cam->t[0] + W[3 + i] * cam->t[1] + W[6 + i] * cam->t[2]);
  for (int i = 0; i < 3; ++i) s->dir[i] = s->mu[i] - campos[i];
  s->dnorm = sqrt(s->dir[0] * s->dir[0] + s->dir[1] * s->dir[1] + s->dir[2] * s->dir[2]);
  for (int i = 0; i < 3; ++i) s->d[i] = s->dir[i] / s->dnorm;
  or_sh_basis(s->d, s->Y);
  for (int ch = 0; ch < 3; ++ch) {
    double acc = 0.0;
    for (int k = 0; k < 16; ++k) acc += s->Y[k] * params[(11 + 3 * k + ch) * n + g];
    s->color_raw[ch] = acc + 0.5;
    s->color[ch] = s->color_raw[ch] > 0.0 ? s->color_raw[ch] : 0.0;
    if (fabs(s->color_raw[ch]) < 1e-5) s->flags |= OR_FLAG_COLOR;
  }
  /* 7. opacity = sigmoid(logit) */
  s->opacity = 1.0 / (1.0 + exp(-params[10 * n + g]));
  s->visible = 1;
}

typedef struct proj_job {
  int64_t n, g0, g1;
  const double* params;
  int32_t n_views;
  const or_camera* cams;
  int32_t tile;
  double *mean2d, *conic, *depth, *color, *opacity;
  int32_t *radius, *tiles;
  uint8_t* flags;
} proj_job;

/* Projection of Gaussians g0 <= g < g1 into every view. */
static void project_range(const proj_job* j) {
  const int64_t n = j->n;
  double *mean2d = j->mean2d, *conic = j->conic, *depth = j->depth, *color = j->color,
         *opacity = j->opacity;
  int32_t *radius = j->radius, *tiles = j->tiles;
  uint8_t* flags = j->flags;
  proj_state s;
  for (int32_t v = 0; v < j->n_views; ++v)
    for (int64_t g = j->g0; g < j->g1; ++g) {
      const int64_t r = (int64_t)v * n + g;
      project_one(j->params, n, g, &j->cams[v], j->tile, &s);
      if (flags) flags[r] = s.flags;
      if (!s.visible) {
        mean2d[2 * r] = mean2d[2 * r + 1] = 0.0;
        conic[3 * r] = conic[3 * r + 1] = conic[3 * r + 2] = 0.0;
        color[3 * r] = color[3 * r + 1] = color[3 * r + 2] = 0.0;
        depth[r] = 0.0;
        opacity[r] = 0.0;
        radius[r] = 0;
        tiles[r] = 0;
        continue;
      }
      mean2d[2 * r] = s.mean2d[0];
      mean2d[2 * r + 1] = s.mean2d[1];
      for (int i = 0; i < 3; ++i) conic[3 * r + i] = s.conic[i];
      for (int i = 0; i < 3; ++i) color[3 * r + i] = s.color[i];
      depth[r] = s.p[2];
      opacity[r] = s.opacity;
      radius[r] = s.radius;
      tiles[r] = s.tiles;
    }
}

static void* project_thread(void* arg) {
  project_range((const proj_job*)arg);
  return NULL;
}

void or_project_mt(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                   int32_t tile, double* mean2d, double* conic, double* depth, double* color,
                   double* opacity, int32_t* radius, int32_t* tiles, uint8_t* flags,
                   int32_t threads) {
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  proj_job jobs[64];
  pthread_t tid[64];
  int started[64] = {0};
  for (int32_t t = 0; t < threads; ++t) {
    proj_job j = {n, n * t / threads, n * (t + 1) / threads, params, n_views, cams, tile,
                  mean2d, conic, depth, color, opacity, radius, tiles, flags};
    jobs[t] = j;
  }
  for (int32_t t = 1; t < threads; ++t)
    started[t] = pthread_create(&tid[t], NULL, project_thread, &jobs[t]) == 0;
  project_range(&jobs[0]);
  for (int32_t t = 1; t < threads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    else project_range(&jobs[t]);  /* no thread: do its share here */
  }
}

void or_project(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                int32_t tile, double* mean2d, double* conic, double* depth, double* color,
                double* opacity, int32_t* radius, int32_t* tiles, uint8_t* flags) {
  or_project_mt(n, params, n_views, cams, tile, mean2d, conic, depth, color, opacity, radius,
                tiles, flags, 1);
}

/* ------------------------------------------------------------------------ */
/* Binning and sort. */
typedef struct kv { uint64_t key; uint32_t val; } kv;

static int kv_cmp(const void* pa, const void* pb) {
  const kv* a = (const kv*)pa;
  const kv* b = (const kv*)pb;
  if (a->key != b->key) return a->key < b->key ? -1 : 1;
  if (a->val != b->val) return a->val < b->val ? -1 : 1;
  return 0;
}

int64_t or_count_isect(int64_t n_rows, const float* mean2d, const int32_t* radius,
                       int32_t tile, int32_t width, int32_t height) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  int64_t total = 0;
  int32_t rect[4];
  for (int64_t r = 0; r < n_rows; ++r) {
    if (radius[r] <= 0) continue;
    or_tile_rect(mean2d[2 * r], mean2d[2 * r + 1], radius[r], tile, tx, ty, rect);
    total += (int64_t)(rect[1] - rect[0]) * (rect[3] - rect[2]);
  }
  return total;
}

static uint32_t float_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof(u));
  return u;
}

void or_bin(int64_t n, int32_t n_views, const float* mean2d, const int32_t* radius,
            const float* depth, int32_t tile, int32_t width, int32_t height,
            uint64_t* keys, uint32_t* vals, int64_t* ranges) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t T = (int64_t)tx * ty;
  const int64_t n_rows = n * n_views;
  const int64_t total = or_count_isect(n_rows, mean2d, radius, tile, width, height);
  kv* items = (kv*)malloc(sizeof(kv) * (size_t)(total > 0 ? total : 1));
  int64_t w = 0;
  int32_t rect[4];
  for (int64_t r = 0; r < n_rows; ++r) {
    if (radius[r] <= 0) continue;
    const int64_t view = r / n, g = r % n;
    or_tile_rect(mean2d[2 * r], mean2d[2 * r + 1], radius[r], tile, tx, ty, rect);
    for (int32_t yy = rect[2]; yy < rect[3]; ++yy)
      for (int32_t xx = rect[0]; xx < rect[1]; ++xx) {
        const uint64_t flat = (uint64_t)(view * T + (int64_t)yy * tx + xx);
        items[w].key = (flat << 32) | (uint64_t)float_bits(depth[r]);
        items[w].val = (uint32_t)g;
        ++w;
      }
  }
  qsort(items, (size_t)total, sizeof(kv), kv_cmp);
  for (int64_t i = 0; i < n_views * T; ++i) ranges[2 * i] = ranges[2 * i + 1] = 0;
  for (int64_t i = 0; i < total; ++i) {
    keys[i] = items[i].key;
    vals[i] = items[i].val;
    const int64_t flat = (int64_t)(items[i].key >> 32);
    if (i == 0 || (int64_t)(items[i - 1].key >> 32) != flat) ranges[2 * flat] = i;
    ranges[2 * flat + 1] = i + 1;
  }
  free(items);
}

/* Thread split of or_bin.  The rows are split into contiguous chunks, one
 * per thread; each thread counts its chunk's pairs per flattened tile, the
 * counts give every (tile, chunk) its place, and each thread writes its
 * chunk's pairs there in row order.  Every tile's segment (keys sharing the
 * tile's high bits) is then sorted by (key, id) on its own.  The sort keys
 * are unique, so the result is the one of or_bin exactly. */
typedef struct bin_job {
  int64_t n, r0, r1, n_flat, f0, f1;
  int32_t tile, width, height, pass;
  const float *mean2d, *depth;
  const int32_t* radius;
  int64_t* counts;  /* [n_flat] of this chunk (pass 0); its cursors (pass 1) */
  kv* items;
  const int64_t* offsets;  /* [n_flat + 1] (pass 2) */
} bin_job;

static void* bin_thread(void* arg) {
  bin_job* j = (bin_job*)arg;
  const int32_t tx = (j->width + j->tile - 1) / j->tile, ty = (j->height + j->tile - 1) / j->tile;
  const int64_t T = (int64_t)tx * ty;
  int32_t rect[4];
  if (j->pass == 2) {  /* sort the segments of tiles f0 <= f < f1 */
    for (int64_t f = j->f0; f < j->f1; ++f)
      qsort(j->items + j->offsets[f], (size_t)(j->offsets[f + 1] - j->offsets[f]), sizeof(kv),
            kv_cmp);
    return NULL;
  }
  for (int64_t r = j->r0; r < j->r1; ++r) {
    if (j->radius[r] <= 0) continue;
    const int64_t view = r / j->n, g = r % j->n;
    or_tile_rect(j->mean2d[2 * r], j->mean2d[2 * r + 1], j->radius[r], j->tile, tx, ty, rect);
    for (int32_t yy = rect[2]; yy < rect[3]; ++yy)
      for (int32_t xx = rect[0]; xx < rect[1]; ++xx) {
        const int64_t flat = view * T + (int64_t)yy * tx + xx;
        if (j->pass == 0) {
          ++j->counts[flat];
        } else {
          kv* it = &j->items[j->counts[flat]++];
          it->key = ((uint64_t)flat << 32) | (uint64_t)float_bits(j->depth[r]);
          it->val = (uint32_t)g;
        }
      }
  }
  return NULL;
}

static void run_bin_jobs(bin_job* jobs, int32_t threads) {
  pthread_t tid[256];
  int started[256] = {0};
  for (int32_t t = 1; t < threads; ++t)
    started[t] = pthread_create(&tid[t], NULL, bin_thread, &jobs[t]) == 0;
  bin_thread(&jobs[0]);
  for (int32_t t = 1; t < threads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    else bin_thread(&jobs[t]);
  }
}

void or_bin_mt(int64_t n, int32_t n_views, const float* mean2d, const int32_t* radius,
               const float* depth, int32_t tile, int32_t width, int32_t height,
               uint64_t* keys, uint32_t* vals, int64_t* ranges, int32_t threads) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t n_flat = n_views * (int64_t)tx * ty;
  const int64_t n_rows = n * n_views;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  int64_t* counts = (int64_t*)calloc((size_t)(threads * n_flat), sizeof(int64_t));
  int64_t* offsets = (int64_t*)calloc((size_t)(n_flat + 1), sizeof(int64_t));
  bin_job jobs[256];
  for (int32_t t = 0; t < threads; ++t) {
    bin_job j = {n, n_rows * t / threads, n_rows * (t + 1) / threads, n_flat, 0, 0, tile, width,
                 height, 0, mean2d, depth, radius, counts + (int64_t)t * n_flat, NULL, offsets};
    jobs[t] = j;
  }
  run_bin_jobs(jobs, threads);
  /* offsets of the tiles; cursor of (tile, chunk) */
  for (int64_t f = 0; f < n_flat; ++f) {
    int64_t run = offsets[f];
    for (int32_t t = 0; t < threads; ++t) {
      const int64_t c = counts[(int64_t)t * n_flat + f];
      counts[(int64_t)t * n_flat + f] = run;
      run += c;
    }
    offsets[f + 1] = run;
  }
  const int64_t total = offsets[n_flat];
  kv* items = (kv*)malloc(sizeof(kv) * (size_t)(total > 0 ? total : 1));
  for (int32_t t = 0; t < threads; ++t) {
    jobs[t].pass = 1;
    jobs[t].items = items;
  }
  run_bin_jobs(jobs, threads);
  for (int32_t t = 0; t < threads; ++t) {  /* tile ranges of about total / threads pairs */
    int64_t f0 = 0, f1 = 0;
    while (f0 < n_flat && offsets[f0] < total * t / threads) ++f0;
    f1 = f0;
    while (f1 < n_flat && offsets[f1] < total * (t + 1) / threads) ++f1;
    if (t == threads - 1) f1 = n_flat;
    jobs[t].pass = 2;
    jobs[t].f0 = f0;
    jobs[t].f1 = f1;
  }
  run_bin_jobs(jobs, threads);
  for (int64_t f = 0; f < n_flat; ++f) {
    const int64_t a = offsets[f], b = offsets[f + 1];
    ranges[2 * f] = a < b ? a : 0;
    ranges[2 * f + 1] = a < b ? b : 0;
  }
  for (int64_t i = 0; i < total; ++i) {
    keys[i] = items[i].key;
    vals[i] = items[i].val;
  }
  free(items);
  free(counts);
  free(offsets);
}

typedef struct dk { uint32_t dbits; uint32_t id; } dk;

static int dk_cmp(const void* pa, const void* pb) {
  const dk* a = (const dk*)pa;
  const dk* b = (const dk*)pb;
  if (a->dbits != b->dbits) return a->dbits < b->dbits ? -1 : 1;
  if (a->id != b->id) return a->id < b->id ? -1 : 1;
  return 0;
}

/* Brute-force lists of selected tiles: every row of the tile's view whose
 * fp32 rectangle covers the tile, ordered by (depth bits, id). */
int64_t or_bin_select(int64_t n, int32_t n_views, const float* mean2d, const int32_t* radius,
                      const float* depth, int32_t tile, int32_t width, int32_t height,
                      const int64_t* tile_sel, int64_t n_sel, uint32_t* out_vals,
                      int64_t* out_ranges) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t T = (int64_t)tx * ty;
  int64_t total = 0;
  int32_t rect[4];
  (void)n_views;
  for (int64_t s = 0; s < n_sel; ++s) {
    const int64_t flat = tile_sel[s], view = flat / T, t = flat % T;
    const int32_t sx = (int32_t)(t % tx), sy = (int32_t)(t / tx);
    const int64_t begin = total;
    for (int64_t g = 0; g < n; ++g) {
      const int64_t r = view * n + g;
      if (radius[r] <= 0) continue;
      or_tile_rect(mean2d[2 * r], mean2d[2 * r + 1], radius[r], tile, tx, ty, rect);
      if (sx < rect[0] || sx >= rect[1] || sy < rect[2] || sy >= rect[3]) continue;
      if (out_vals) out_vals[total] = (uint32_t)g;
      ++total;
    }
    if (out_vals) {
      const int64_t m = total - begin;
      dk* items = (dk*)malloc(sizeof(dk) * (size_t)(m > 0 ? m : 1));
      for (int64_t i = 0; i < m; ++i) {
        items[i].dbits = float_bits(depth[view * n + out_vals[begin + i]]);
        items[i].id = out_vals[begin + i];
      }
      qsort(items, (size_t)m, sizeof(dk), dk_cmp);
      for (int64_t i = 0; i < m; ++i) out_vals[begin + i] = items[i].id;
      free(items);
      out_ranges[2 * s] = begin;
      out_ranges[2 * s + 1] = total;
    }
  }
  return total;
}

/* ------------------------------------------------------------------------ */
/* Compositing of one pair: returns the un-capped alpha o*exp(power) and the
 * power through *power_out. */
static double pair_alpha_raw(double px, double py, const double* m, const double* co, double o,
                             double* power_out, double* dx_out, double* dy_out) {
  const double dx = px - m[0], dy = py - m[1];
  const double power = -0.5 * (co[0] * dx * dx + co[2] * dy * dy) - co[1] * dx * dy;
  *power_out = power;
  *dx_out = dx;
  *dy_out = dy;
  return o * exp(power);
}

static double rel_dist(double v, double ref) { return fabs(v - ref) / ref; }

/* Forward compositing of one flattened tile (view * T + tile) of its sorted
 * list, pixel by pixel in the pages' order: front to back, skip alpha <
 * 1/255, stop before the transmittance drops below 1e-4. */
static void raster_fwd_tile(int64_t flat, int64_t n, int32_t width, int32_t height, int32_t tile,
                            const double* mean2d, const double* conic, const double* opacity,
                            const double* color, const uint32_t* vals, const int64_t* ranges,
                            const double bg[3], double* image, double* T_final,
                            int32_t* n_contrib, int64_t* pairs, int64_t* included,
                            double* margin, double* importance) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t T = (int64_t)tx * ty;
  const int64_t HW = (int64_t)width * height;
  const int64_t view = flat / T, t = flat % T;
  const int32_t tile_x = (int32_t)(t % tx), tile_y = (int32_t)(t / tx);
  const int64_t start = ranges[2 * flat], end = ranges[2 * flat + 1];
  for (int32_t yy = tile_y * tile; yy < (tile_y + 1) * tile && yy < height; ++yy)
    for (int32_t xx = tile_x * tile; xx < (tile_x + 1) * tile && xx < width; ++xx) {
      const double px = xx + 0.5, py = yy + 0.5;
      double Tr = 1.0, C[3] = {0.0, 0.0, 0.0};
      int32_t last = 0;
      int64_t tested = 0, composited = 0;
      double mg = INFINITY;
      for (int64_t i = start; i < end; ++i) {
        const int64_t r = view * n + vals[i];
        double power, dx, dy;
        ++tested;
        const double araw = pair_alpha_raw(px, py, &mean2d[2 * r], &conic[3 * r], opacity[r],
                                           &power, &dx, &dy);
        mg = fmin(mg, rel_dist(araw, kAlphaMin));
        mg = fmin(mg, rel_dist(araw, kAlphaMax));
        const double alpha = araw < kAlphaMax ? araw : kAlphaMax;
        if (alpha < kAlphaMin) continue;
        const double Tn = Tr * (1.0 - alpha);
        mg = fmin(mg, rel_dist(Tn, kTMin));
        if (Tn < kTMin) break;
        for (int ch = 0; ch < 3; ++ch) C[ch] += color[3 * r + ch] * alpha * Tr;
        if (importance && alpha * Tr > importance[r]) importance[r] = alpha * Tr;
        Tr = Tn;
        last = (int32_t)(i - start + 1);
        ++composited;
      }
      const int64_t pix = (int64_t)yy * width + xx;
      for (int ch = 0; ch < 3; ++ch) image[(view * 3 + ch) * HW + pix] = C[ch] + Tr * bg[ch];
      T_final[view * HW + pix] = Tr;
      n_contrib[view * HW + pix] = last;
      if (pairs) pairs[view * HW + pix] = tested;
      if (included) included[view * HW + pix] = composited;
      if (margin) margin[view * HW + pix] = mg;
    }
}

void or_raster_fwd(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                   const double* mean2d, const double* conic, const double* opacity,
                   const double* color, const uint32_t* vals, const int64_t* ranges,
                   const double bg[3], const int64_t* tile_sel, int64_t n_sel,
                   double* image, double* T_final, int32_t* n_contrib, int64_t* pairs,
                   int64_t* included, double* margin, double* importance) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t T = (int64_t)tx * ty;
  const int64_t n_tiles = tile_sel ? n_sel : n_views * T;
  for (int64_t it = 0; it < n_tiles; ++it)
    raster_fwd_tile(tile_sel ? tile_sel[it] : it, n, width, height, tile, mean2d, conic, opacity,
                    color, vals, ranges, bg, image, T_final, n_contrib, pairs, included, margin,
                    importance);
}

/* Thread split of or_raster_fwd: tile k of the work list goes to thread
 * k mod threads.  Tiles write disjoint pixels, so the outputs are those of
 * or_raster_fwd exactly (importance is not offered here: rows are shared
 * between tiles). */
typedef struct fwd_job {
  int64_t n, n_tiles;
  int32_t width, height, tile, threads, index;
  const double *mean2d, *conic, *opacity, *color;
  const uint32_t* vals;
  const int64_t *ranges, *tile_sel;
  const double* bg;
  double *image, *T_final, *margin;
  int32_t* n_contrib;
  int64_t *pairs, *included;
} fwd_job;

static void* raster_fwd_thread(void* arg) {
  const fwd_job* j = (const fwd_job*)arg;
  for (int64_t it = j->index; it < j->n_tiles; it += j->threads)
    raster_fwd_tile(j->tile_sel ? j->tile_sel[it] : it, j->n, j->width, j->height, j->tile,
                    j->mean2d, j->conic, j->opacity, j->color, j->vals, j->ranges, j->bg,
                    j->image, j->T_final, j->n_contrib, j->pairs, j->included, j->margin, NULL);
  return NULL;
}

void or_raster_fwd_mt(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                      const double* mean2d, const double* conic, const double* opacity,
                      const double* color, const uint32_t* vals, const int64_t* ranges,
                      const double bg[3], const int64_t* tile_sel, int64_t n_sel,
                      double* image, double* T_final, int32_t* n_contrib, int64_t* pairs,
                      int64_t* included, double* margin, int32_t threads) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t n_tiles = tile_sel ? n_sel : n_views * (int64_t)tx * ty;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  fwd_job jobs[256];
  pthread_t tid[256];
  int started[256] = {0};
  for (int32_t t = 0; t < threads; ++t) {
    fwd_job j = {n, n_tiles, width, height, tile, threads, t, mean2d, conic, opacity, color,
                 vals, ranges, tile_sel, bg, image, T_final, margin, n_contrib, pairs, included};
    jobs[t] = j;
  }
  for (int32_t t = 1; t < threads; ++t)
    started[t] = pthread_create(&tid[t], NULL, raster_fwd_thread, &jobs[t]) == 0;
  raster_fwd_thread(&jobs[0]);
  for (int32_t t = 1; t < threads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    else raster_fwd_thread(&jobs[t]);
  }
}

void or_raster_fwd_brute(int64_t n, int32_t n_views, int32_t width, int32_t height,
                         int32_t tile, const double* mean2d, const double* conic,
                         const double* opacity, const double* color, const double* depth,
                         const int32_t* radius, const double bg[3], double* image,
                         double* T_final) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t HW = (int64_t)width * height;
  dk* order = (dk*)malloc(sizeof(dk) * (size_t)(n > 0 ? n : 1));
  int32_t* rects = (int32_t*)malloc(sizeof(int32_t) * 4 * (size_t)(n > 0 ? n : 1));
  for (int32_t v = 0; v < n_views; ++v) {
    int64_t m = 0;
    for (int64_t g = 0; g < n; ++g) {
      const int64_t r = (int64_t)v * n + g;
      if (radius[r] <= 0) continue;
      order[m].dbits = float_bits((float)depth[r]);
      order[m].id = (uint32_t)g;
      ++m;
    }
    qsort(order, (size_t)m, sizeof(dk), dk_cmp);
    for (int64_t i = 0; i < m; ++i) {
      const int64_t r = (int64_t)v * n + order[i].id;
      or_tile_rect((float)mean2d[2 * r], (float)mean2d[2 * r + 1], radius[r], tile, tx, ty,
                   &rects[4 * i]);
    }
    for (int32_t yy = 0; yy < height; ++yy)
      for (int32_t xx = 0; xx < width; ++xx) {
        const int32_t ptx = xx / tile, pty = yy / tile;
        const double px = xx + 0.5, py = yy + 0.5;
        double Tr = 1.0, C[3] = {0.0, 0.0, 0.0};
        for (int64_t i = 0; i < m; ++i) {
          const int32_t* rc = &rects[4 * i];
          if (ptx < rc[0] || ptx >= rc[1] || pty < rc[2] || pty >= rc[3]) continue;
          const int64_t r = (int64_t)v * n + order[i].id;
          double power, dx, dy;
          const double araw = pair_alpha_raw(px, py, &mean2d[2 * r], &conic[3 * r], opacity[r],
                                             &power, &dx, &dy);
          const double alpha = araw < kAlphaMax ? araw : kAlphaMax;
          if (alpha < kAlphaMin) continue;
          const double Tn = Tr * (1.0 - alpha);
          if (Tn < kTMin) break;
          for (int ch = 0; ch < 3; ++ch) C[ch] += color[3 * r + ch] * alpha * Tr;
          Tr = Tn;
        }
        const int64_t pix = (int64_t)yy * width + xx;
        for (int ch = 0; ch < 3; ++ch) image[((int64_t)v * 3 + ch) * HW + pix] = C[ch] + Tr * bg[ch];
        T_final[(int64_t)v * HW + pix] = Tr;
      }
  }
  free(order);
  free(rects);
}

/* ------------------------------------------------------------------------ */
double or_loss_l1(int64_t n, const double* image, const double* target, double* dL_dimage) {
  double sum = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const double d = image[i] - target[i];
    sum += fabs(d);
    if (dL_dimage) dL_dimage[i] = (d > 0.0 ? 1.0 : (d < 0.0 ? -1.0 : 0.0)) / (double)n;
  }
  return sum / (double)n;
}

/* ------------------------------------------------------------------------ */
/* Scratch of one pixel's included pairs, front to back. */
typedef struct bwd_scratch {
  int64_t *row, *pos;
  double *alpha, *T, *raw, *dx, *dy;
} bwd_scratch;

static int bwd_scratch_alloc(bwd_scratch* b, int64_t len) {
  const size_t m = (size_t)(len > 0 ? len : 1);
  b->row = (int64_t*)malloc(sizeof(int64_t) * m);
  b->pos = (int64_t*)malloc(sizeof(int64_t) * m);
  b->alpha = (double*)malloc(sizeof(double) * m);
  b->T = (double*)malloc(sizeof(double) * m);
  b->raw = (double*)malloc(sizeof(double) * m);
  b->dx = (double*)malloc(sizeof(double) * m);
  b->dy = (double*)malloc(sizeof(double) * m);
  return b->row && b->pos && b->alpha && b->T && b->raw && b->dx && b->dy;
}

static void bwd_scratch_free(bwd_scratch* b) {
  free(b->row);
  free(b->pos);
  free(b->alpha);
  free(b->T);
  free(b->raw);
  free(b->dx);
  free(b->dy);
}

/* Backward compositing of one flattened tile.  For each pixel the forward is
 * run again (T_i as a running product), then its included pairs are walked
 * back to front with S = the colour composited behind the pair.  Gradients
 * are added at index row (by_pos == 0) or at the pair's list position minus
 * the tile's start (by_pos == 1, for a per-tile buffer). */
static void raster_bwd_tile(int64_t flat, int64_t n, int32_t width, int32_t height, int32_t tile,
                            const double* mean2d, const double* conic, const double* opacity,
                            const double* color, const uint32_t* vals, const int64_t* ranges,
                            const double bg[3], const double* dL_dimage, bwd_scratch* sc,
                            int by_pos, double* g_mean2d, double* g_conic, double* g_opacity,
                            double* g_color) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t T = (int64_t)tx * ty;
  const int64_t HW = (int64_t)width * height;
  const int64_t view = flat / T, t = flat % T;
  const int32_t tile_x = (int32_t)(t % tx), tile_y = (int32_t)(t / tx);
  const int64_t start = ranges[2 * flat], end = ranges[2 * flat + 1];
  for (int32_t yy = tile_y * tile; yy < (tile_y + 1) * tile && yy < height; ++yy)
    for (int32_t xx = tile_x * tile; xx < (tile_x + 1) * tile && xx < width; ++xx) {
      const double px = xx + 0.5, py = yy + 0.5;
      const int64_t pix = (int64_t)yy * width + xx;
      /* forward again: T_i as a running product */
      double Tr = 1.0;
      int64_t k = 0;
      for (int64_t i = start; i < end; ++i) {
        const int64_t r = view * n + vals[i];
        double power, dx, dy;
        const double araw = pair_alpha_raw(px, py, &mean2d[2 * r], &conic[3 * r], opacity[r],
                                           &power, &dx, &dy);
        const double alpha = araw < kAlphaMax ? araw : kAlphaMax;
        if (alpha < kAlphaMin) continue;
        const double Tn = Tr * (1.0 - alpha);
        if (Tn < kTMin) break;
        sc->row[k] = r;
        sc->pos[k] = i - start;
        sc->alpha[k] = alpha;
        sc->T[k] = Tr;
        sc->raw[k] = araw;
        sc->dx[k] = dx;
        sc->dy[k] = dy;
        ++k;
        Tr = Tn;
      }
      double gC[3];
      for (int ch = 0; ch < 3; ++ch) gC[ch] = dL_dimage[(view * 3 + ch) * HW + pix];
      /* S = colour composited behind the current pair, background included */
      double S[3] = {Tr * bg[0], Tr * bg[1], Tr * bg[2]};
      for (int64_t j = k - 1; j >= 0; --j) {
        const int64_t r = sc->row[j];
        const int64_t a = by_pos ? sc->pos[j] : r; /* where the sums go */
        const double alpha = sc->alpha[j], Ti = sc->T[j];
        const double* col = &color[3 * r];
        double dL_dalpha = 0.0;
        for (int ch = 0; ch < 3; ++ch) {
          g_color[3 * a + ch] += alpha * Ti * gC[ch];
          dL_dalpha += gC[ch] * (col[ch] * Ti - S[ch] / (1.0 - alpha));
        }
        for (int ch = 0; ch < 3; ++ch) S[ch] += col[ch] * alpha * Ti;
        if (sc->raw[j] >= kAlphaMax) continue; /* capped: alpha does not move */
        const double* co = &conic[3 * r];
        const double o = opacity[r];
        const double e = sc->raw[j] / o; /* exp(power) */
        const double dx = sc->dx[j], dy = sc->dy[j];
        g_opacity[a] += dL_dalpha * e;
        const double dL_dpower = dL_dalpha * sc->raw[j];
        g_mean2d[2 * a] += dL_dpower * (co[0] * dx + co[1] * dy);
        g_mean2d[2 * a + 1] += dL_dpower * (co[1] * dx + co[2] * dy);
        g_conic[3 * a] += dL_dpower * (-0.5 * dx * dx);
        g_conic[3 * a + 1] += dL_dpower * (-dx * dy);
        g_conic[3 * a + 2] += dL_dpower * (-0.5 * dy * dy);
      }
    }
}

static int64_t longest_list(int32_t n_views, int32_t width, int32_t height, int32_t tile,
                            const int64_t* ranges) {
  const int64_t T = (int64_t)((width + tile - 1) / tile) * ((height + tile - 1) / tile);
  int64_t max_len = 1;
  for (int64_t f = 0; f < n_views * T; ++f)
    if (ranges[2 * f + 1] - ranges[2 * f] > max_len) max_len = ranges[2 * f + 1] - ranges[2 * f];
  return max_len;
}

void or_raster_bwd(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                   const double* mean2d, const double* conic, const double* opacity,
                   const double* color, const uint32_t* vals, const int64_t* ranges,
                   const double bg[3], const double* dL_dimage, const int64_t* tile_sel,
                   int64_t n_sel, double* g_mean2d, double* g_conic, double* g_opacity,
                   double* g_color) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t T = (int64_t)tx * ty;
  const int64_t n_rows = n * n_views;
  memset(g_mean2d, 0, sizeof(double) * 2 * (size_t)n_rows);
  memset(g_conic, 0, sizeof(double) * 3 * (size_t)n_rows);
  memset(g_opacity, 0, sizeof(double) * (size_t)n_rows);
  memset(g_color, 0, sizeof(double) * 3 * (size_t)n_rows);
  bwd_scratch sc;
  if (!bwd_scratch_alloc(&sc, longest_list(n_views, width, height, tile, ranges))) {
    bwd_scratch_free(&sc);
    return;
  }
  const int64_t n_tiles = tile_sel ? n_sel : n_views * T;
  for (int64_t it = 0; it < n_tiles; ++it)
    raster_bwd_tile(tile_sel ? tile_sel[it] : it, n, width, height, tile, mean2d, conic, opacity,
                    color, vals, ranges, bg, dL_dimage, &sc, 0, g_mean2d, g_conic, g_opacity,
                    g_color);
  bwd_scratch_free(&sc);
}

/* Thread split of or_raster_bwd: tile k of the work list goes to thread
 * k mod threads, which sums the tile's gradients per list position (a row
 * occurs once in a tile's list) and then adds them to the rows under one
 * lock.  Equal to or_raster_bwd up to the order of the fp64 sums. */
typedef struct bwd_job {
  int64_t n, n_tiles, max_len;
  int32_t width, height, tile, threads, index;
  const double *mean2d, *conic, *opacity, *color, *bg, *dL_dimage;
  const uint32_t* vals;
  const int64_t *ranges, *tile_sel;
  double *g_mean2d, *g_conic, *g_opacity, *g_color;
  pthread_mutex_t* lock;
} bwd_job;

static void* raster_bwd_thread(void* arg) {
  const bwd_job* j = (const bwd_job*)arg;
  const int32_t tx = (j->width + j->tile - 1) / j->tile, ty = (j->height + j->tile - 1) / j->tile;
  const int64_t T = (int64_t)tx * ty;
  const size_t m = (size_t)j->max_len;
  bwd_scratch sc;
  double* lm = (double*)calloc(2 * m, sizeof(double));
  double* lc = (double*)calloc(3 * m, sizeof(double));
  double* lo = (double*)calloc(m, sizeof(double));
  double* lk = (double*)calloc(3 * m, sizeof(double));
  if (bwd_scratch_alloc(&sc, j->max_len) && lm && lc && lo && lk) {
    for (int64_t it = j->index; it < j->n_tiles; it += j->threads) {
      const int64_t flat = j->tile_sel ? j->tile_sel[it] : it;
      const int64_t start = j->ranges[2 * flat], len = j->ranges[2 * flat + 1] - start;
      memset(lm, 0, sizeof(double) * 2 * (size_t)len);
      memset(lc, 0, sizeof(double) * 3 * (size_t)len);
      memset(lo, 0, sizeof(double) * (size_t)len);
      memset(lk, 0, sizeof(double) * 3 * (size_t)len);
      raster_bwd_tile(flat, j->n, j->width, j->height, j->tile, j->mean2d, j->conic, j->opacity,
                      j->color, j->vals, j->ranges, j->bg, j->dL_dimage, &sc, 1, lm, lc, lo, lk);
      const int64_t view = flat / T;
      pthread_mutex_lock(j->lock);
      for (int64_t i = 0; i < len; ++i) {
        const int64_t r = view * j->n + j->vals[start + i];
        for (int c = 0; c < 2; ++c) j->g_mean2d[2 * r + c] += lm[2 * i + c];
        for (int c = 0; c < 3; ++c) j->g_conic[3 * r + c] += lc[3 * i + c];
        j->g_opacity[r] += lo[i];
        for (int c = 0; c < 3; ++c) j->g_color[3 * r + c] += lk[3 * i + c];
      }
      pthread_mutex_unlock(j->lock);
    }
  }
  bwd_scratch_free(&sc);
  free(lm);
  free(lc);
  free(lo);
  free(lk);
  return NULL;
}

void or_raster_bwd_mt(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                      const double* mean2d, const double* conic, const double* opacity,
                      const double* color, const uint32_t* vals, const int64_t* ranges,
                      const double bg[3], const double* dL_dimage, const int64_t* tile_sel,
                      int64_t n_sel, double* g_mean2d, double* g_conic, double* g_opacity,
                      double* g_color, int32_t threads) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t n_rows = n * n_views;
  memset(g_mean2d, 0, sizeof(double) * 2 * (size_t)n_rows);
  memset(g_conic, 0, sizeof(double) * 3 * (size_t)n_rows);
  memset(g_opacity, 0, sizeof(double) * (size_t)n_rows);
  memset(g_color, 0, sizeof(double) * 3 * (size_t)n_rows);
  const int64_t n_tiles = tile_sel ? n_sel : n_views * (int64_t)tx * ty;
  const int64_t max_len = longest_list(n_views, width, height, tile, ranges);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_mutex_t lock;
  pthread_mutex_init(&lock, NULL);
  bwd_job jobs[256];
  pthread_t tid[256];
  int started[256] = {0};
  for (int32_t t = 0; t < threads; ++t) {
    bwd_job j = {n, n_tiles, max_len, width, height, tile, threads, t, mean2d, conic, opacity,
                 color, bg, dL_dimage, vals, ranges, tile_sel, g_mean2d, g_conic, g_opacity,
                 g_color, &lock};
    jobs[t] = j;
  }
  for (int32_t t = 1; t < threads; ++t)
    started[t] = pthread_create(&tid[t], NULL, raster_bwd_thread, &jobs[t]) == 0;
  raster_bwd_thread(&jobs[0]);
  for (int32_t t = 1; t < threads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    else raster_bwd_thread(&jobs[t]);
  }
  pthread_mutex_destroy(&lock);
}

/* ------------------------------------------------------------------------ */
/* Projection backward of Gaussians g0 <= g < g1 (columns of grad and
 * entries of visible that the caller has zeroed). */
static void project_bwd_range(int64_t n, int64_t g0, int64_t g1, const double* params,
                              int32_t n_views, const or_camera* cams, int32_t tile,
                              const double* g_mean2d, const double* g_conic,
                              const double* g_opacity, const double* g_color, double* grad,
                              uint8_t* visible) {
  proj_state s;
  for (int64_t g = g0; g < g1; ++g) {
    double g_mu[3] = {0, 0, 0}, g_ls[3] = {0, 0, 0}, g_q[4] = {0, 0, 0, 0}, g_logit = 0.0;
    double g_sh[48];
    memset(g_sh, 0, sizeof(g_sh));
    for (int32_t v = 0; v < n_views; ++v) {
      const or_camera* cam = &cams[v];
      project_one(params, n, g, cam, tile, &s);
      if (!s.visible) continue;
      if (visible) visible[g] = 1;
      const int64_t r = (int64_t)v * n + g;
      const double* W = cam->R;
      /* opacity = sigmoid(logit) */
      g_logit += g_opacity[r] * s.opacity * (1.0 - s.opacity);
      /* colour = max(sum_k Y_k sh_k + 0.5, 0) */
      double g_d[3] = {0, 0, 0};
      {
        double dY[16][3];
        sh_basis_grad(s.d, dY);
        for (int ch = 0; ch < 3; ++ch) {
          if (!(s.color_raw[ch] > 0.0)) continue;
          const double gc = g_color[3 * r + ch];
          for (int k = 0; k < 16; ++k) {
            g_sh[3 * k + ch] += s.Y[k] * gc;
            const double shk = params[(11 + 3 * k + ch) * n + g];
            for (int i = 0; i < 3; ++i) g_d[i] += shk * gc * dY[k][i];
          }
        }
        /* d = dir / |dir|, dir = mu - campos */
        const double dd = s.d[0] * g_d[0] + s.d[1] * g_d[1] + s.d[2] * g_d[2];
        for (int i = 0; i < 3; ++i) g_mu[i] += (g_d[i] - s.d[i] * dd) / s.dnorm;
      }
      /* camera-space gradient g_p */
      const double x = s.p[0], y = s.p[1], z = s.p[2];
      const double fx = cam->fx, fy = cam->fy;
      double g_p[3] = {0, 0, 0};
      /* mean2d = (fx x/z + cx, fy y/z + cy) */
      {
        const double gm0 = g_mean2d[2 * r], gm1 = g_mean2d[2 * r + 1];
        g_p[0] += gm0 * fx / z;
        g_p[1] += gm1 * fy / z;
        g_p[2] += -gm0 * fx * x / (z * z) - gm1 * fy * y / (z * z);
      }
      /* conic = inverse(cov2): G_cov2 = -Conic G_Conic Conic, with the
       * off-diagonal conic entry counted once in the power */
      double H[4];
      {
        const double A = s.conic[0], B = s.conic[1], C = s.conic[2];
        const double Mc[4] = {A, B, B, C};
        const double Gc[4] = {g_conic[3 * r], 0.5 * g_conic[3 * r + 1], 0.5 * g_conic[3 * r + 1],
                              g_conic[3 * r + 2]};
        double tmp[4];
        for (int i = 0; i < 2; ++i)
          for (int j = 0; j < 2; ++j)
            tmp[2 * i + j] = Mc[2 * i] * Gc[j] + Mc[2 * i + 1] * Gc[2 + j];
        for (int i = 0; i < 2; ++i)
          for (int j = 0; j < 2; ++j)
            H[2 * i + j] = -(tmp[2 * i] * Mc[j] + tmp[2 * i + 1] * Mc[2 + j]);
      }
      /* cov2 = T Sigma T^T + 0.3 I, T = J W:  G_T = 2 H T Sigma,  G_Sigma = T^T H T */
      double G_T[6], G_Sigma[9];
      {
        double TS[6];
        for (int i = 0; i < 2; ++i)
          for (int j = 0; j < 3; ++j) {
            double acc = 0.0;
            for (int k = 0; k < 3; ++k) acc += s.T[3 * i + k] * s.Sigma[3 * k + j];
            TS[3 * i + j] = acc;
          }
        for (int i = 0; i < 2; ++i)
          for (int j = 0; j < 3; ++j)
            G_T[3 * i + j] = 2.0 * (H[2 * i] * TS[j] + H[2 * i + 1] * TS[3 + j]);
        for (int a = 0; a < 3; ++a)
          for (int b = 0; b < 3; ++b) {
            double acc = 0.0;
            for (int i = 0; i < 2; ++i)
              for (int j = 0; j < 2; ++j) acc += s.T[3 * i + a] * H[2 * i + j] * s.T[3 * j + b];
            G_Sigma[3 * a + b] = acc;
          }
      }
      /* T = J W: G_J = G_T W^T; J depends on (x, y, z) through the clamp */
      {
        double G_J[6];
        for (int i = 0; i < 2; ++i)
          for (int j = 0; j < 3; ++j) {
            double acc = 0.0;
            for (int k = 0; k < 3; ++k) acc += G_T[3 * i + k] * W[3 * j + k];
            G_J[3 * i + j] = acc;
          }
        g_p[2] += G_J[0] * (-fx / (z * z)) + G_J[4] * (-fy / (z * z));
        /* J02 = -fx tx / z^2 with tx = z clamp(x/z, -lim, lim) */
        if (s.clamped[0] == 0.0) {
          g_p[0] += G_J[2] * (-fx / (z * z));
          g_p[2] += G_J[2] * (2.0 * fx * x / (z * z * z));
        } else {
          const double u = s.tpos[0] / z;
          g_p[2] += G_J[2] * (fx * u / (z * z));
        }
        if (s.clamped[1] == 0.0) {
          g_p[1] += G_J[5] * (-fy / (z * z));
          g_p[2] += G_J[5] * (2.0 * fy * y / (z * z * z));
        } else {
          const double u = s.tpos[1] / z;
          g_p[2] += G_J[5] * (fy * u / (z * z));
        }
      }
      /* p = W mu + t */
      for (int i = 0; i < 3; ++i)
        g_mu[i] += W[i] * g_p[0] + W[3 + i] * g_p[1] + W[6 + i] * g_p[2];
      /* Sigma = M M^T, M = Rq diag(scale):  G_M = 2 G_Sigma M */
      {
        double G_M[9];
        for (int i = 0; i < 3; ++i)
          for (int j = 0; j < 3; ++j) {
            double acc = 0.0;
            for (int k = 0; k < 3; ++k) acc += G_Sigma[3 * i + k] * s.M[3 * k + j];
            G_M[3 * i + j] = 2.0 * acc;
          }
        double G_R[9];
        for (int j = 0; j < 3; ++j) {
          double gs = 0.0;
          for (int i = 0; i < 3; ++i) {
            gs += s.Rq[3 * i + j] * G_M[3 * i + j];
            G_R[3 * i + j] = G_M[3 * i + j] * s.scale[j];
          }
          g_ls[j] += gs * s.scale[j]; /* scale = exp(log-scale) */
        }
        double g_qn[4];
        quat_rot_vjp(s.qn, G_R, g_qn);
        const double dq = s.qn[0] * g_qn[0] + s.qn[1] * g_qn[1] + s.qn[2] * g_qn[2] +
                          s.qn[3] * g_qn[3];
        for (int i = 0; i < 4; ++i) g_q[i] += (g_qn[i] - s.qn[i] * dq) / s.qnorm;
      }
    }
    for (int i = 0; i < 3; ++i) grad[i * n + g] = g_mu[i];
    for (int i = 0; i < 3; ++i) grad[(3 + i) * n + g] = g_ls[i];
    for (int i = 0; i < 4; ++i) grad[(6 + i) * n + g] = g_q[i];
    grad[10 * n + g] = g_logit;
    for (int k = 0; k < 48; ++k) grad[(11 + k) * n + g] = g_sh[k];
  }
}

void or_project_bwd(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                    int32_t tile, const double* g_mean2d, const double* g_conic,
                    const double* g_opacity, const double* g_color, double* grad,
                    uint8_t* visible) {
  memset(grad, 0, sizeof(double) * OR_NPARAM * (size_t)n);
  if (visible) memset(visible, 0, (size_t)n);
  project_bwd_range(n, 0, n, params, n_views, cams, tile, g_mean2d, g_conic, g_opacity, g_color,
                    grad, visible);
}

/* Thread split of or_project_bwd by Gaussian (contiguous ranges); every
 * Gaussian's column is computed as in or_project_bwd, so the outputs are
 * identical. */
typedef struct pbwd_job {
  int64_t n, g0, g1;
  const double* params;
  int32_t n_views, tile;
  const or_camera* cams;
  const double *g_mean2d, *g_conic, *g_opacity, *g_color;
  double* grad;
  uint8_t* visible;
} pbwd_job;

static void* project_bwd_thread(void* arg) {
  const pbwd_job* j = (const pbwd_job*)arg;
  project_bwd_range(j->n, j->g0, j->g1, j->params, j->n_views, j->cams, j->tile, j->g_mean2d,
                    j->g_conic, j->g_opacity, j->g_color, j->grad, j->visible);
  return NULL;
}

void or_project_bwd_mt(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                       int32_t tile, const double* g_mean2d, const double* g_conic,
                       const double* g_opacity, const double* g_color, double* grad,
                       uint8_t* visible, int32_t threads) {
  memset(grad, 0, sizeof(double) * OR_NPARAM * (size_t)n);
  if (visible) memset(visible, 0, (size_t)n);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pbwd_job jobs[256];
  pthread_t tid[256];
  int started[256] = {0};
  for (int32_t t = 0; t < threads; ++t) {
    pbwd_job j = {n, n * t / threads, n * (t + 1) / threads, params, n_views, tile, cams,
                  g_mean2d, g_conic, g_opacity, g_color, grad, visible};
    jobs[t] = j;
  }
  for (int32_t t = 1; t < threads; ++t)
    started[t] = pthread_create(&tid[t], NULL, project_bwd_thread, &jobs[t]) == 0;
  project_bwd_thread(&jobs[0]);
  for (int32_t t = 1; t < threads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    else project_bwd_thread(&jobs[t]);
  }
}

/* ------------------------------------------------------------------------ */
/* Adam over columns c0 <= col < c1 of every row. */
static void adam_range(int64_t n_rows, int64_t n_cols, int64_t c0, int64_t c1, double* p,
                       const double* g, double* m, double* v, int64_t t, double lr, double beta1,
                       double beta2, double eps, const uint8_t* visible) {
  const double bc1 = 1.0 - pow(beta1, (double)t);
  const double bc2 = 1.0 - pow(beta2, (double)t);
  for (int64_t row = 0; row < n_rows; ++row)
    for (int64_t col = c0; col < c1; ++col) {
      if (visible && !visible[col]) continue;
      const int64_t i = row * n_cols + col;
      m[i] = beta1 * m[i] + (1.0 - beta1) * g[i];
      v[i] = beta2 * v[i] + (1.0 - beta2) * g[i] * g[i];
      const double mhat = m[i] / bc1;
      const double vhat = v[i] / bc2;
      p[i] -= lr * mhat / (sqrt(vhat) + eps);
    }
}

void or_adam(int64_t n_rows, int64_t n_cols, double* p, const double* g, double* m,
             double* v, int64_t t, double lr, double beta1, double beta2, double eps,
             const uint8_t* visible) {
  adam_range(n_rows, n_cols, 0, n_cols, p, g, m, v, t, lr, beta1, beta2, eps, visible);
}

/* Thread split of or_adam by column range: element-wise, identical results. */
typedef struct adam_job {
  int64_t n_rows, n_cols, c0, c1, t;
  double *p, *m, *v;
  const double* g;
  double lr, beta1, beta2, eps;
  const uint8_t* visible;
} adam_job;

static void* adam_thread(void* arg) {
  const adam_job* j = (const adam_job*)arg;
  adam_range(j->n_rows, j->n_cols, j->c0, j->c1, j->p, j->g, j->m, j->v, j->t, j->lr, j->beta1,
             j->beta2, j->eps, j->visible);
  return NULL;
}

void or_adam_mt(int64_t n_rows, int64_t n_cols, double* p, const double* g, double* m,
                double* v, int64_t t, double lr, double beta1, double beta2, double eps,
                const uint8_t* visible, int32_t threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  adam_job jobs[256];
  pthread_t tid[256];
  int started[256] = {0};
  for (int32_t k = 0; k < threads; ++k) {
    adam_job j = {n_rows, n_cols, n_cols * k / threads, n_cols * (k + 1) / threads, t, p, m, v,
                  g, lr, beta1, beta2, eps, visible};
    jobs[k] = j;
  }
  for (int32_t k = 1; k < threads; ++k)
    started[k] = pthread_create(&tid[k], NULL, adam_thread, &jobs[k]) == 0;
  adam_thread(&jobs[0]);
  for (int32_t k = 1; k < threads; ++k) {
    if (started[k]) pthread_join(tid[k], NULL);
    else adam_thread(&jobs[k]);
  }
}

/* ------------------------------------------------------------------------ */
/* Morton order ("A Scalable PyTorch Abstraction for Multi-GPU Gaussian
 * Splatting", references: Morton order).  The quantisation decides integers,
 * so it is done in fp32 with one rounding per operation, as the library
 * does; the interleave is a plain loop over the 21 bits. */
static uint32_t morton_q21(float v, float lo, float s) {
  float t = floorf((v - lo) * s);
  if (!(t >= 0.0f)) t = 0.0f;
  if (t > 2097151.0f) t = 2097151.0f;
  return (uint32_t)t;
}

void or_morton_codes(int64_t n, const float* params, uint64_t* codes) {
  float lo[3], hi[3], sc[3];
  for (int a = 0; a < 3; ++a) {
    lo[a] = hi[a] = n > 0 ? params[a * n] : 0.0f;
    for (int64_t i = 1; i < n; ++i) {
      const float v = params[a * n + i];
      if (v < lo[a]) lo[a] = v;
      if (v > hi[a]) hi[a] = v;
    }
    const float ext = hi[a] - lo[a];
    sc[a] = ext > 0.0f ? 2097152.0f / ext : 0.0f;
  }
  for (int64_t i = 0; i < n; ++i) {
    uint32_t q[3];
    for (int a = 0; a < 3; ++a) q[a] = morton_q21(params[a * n + i], lo[a], sc[a]);
    uint64_t code = 0;
    for (int b = 0; b < 21; ++b)
      for (int a = 0; a < 3; ++a) code |= (uint64_t)((q[a] >> b) & 1u) << (3 * b + a);
    codes[i] = code;
  }
}

void or_morton_order(int64_t n, const float* params, uint32_t* perm) {
  uint64_t* codes = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)(n > 0 ? n : 1));
  kv* items = (kv*)malloc(sizeof(kv) * (size_t)(n > 0 ? n : 1));
  or_morton_codes(n, params, codes);
  for (int64_t i = 0; i < n; ++i) {
    items[i].key = codes[i];
    items[i].val = (uint32_t)i;
  }
  qsort(items, (size_t)n, sizeof(kv), kv_cmp);
  for (int64_t i = 0; i < n; ++i) perm[i] = items[i].val;
  free(items);
  free(codes);
}

/* ------------------------------------------------------------------------ */
/* Pruning bounded by the per-tile working set ("ByteSplat" abstract:
 * pruning under rendering-quality and per-tile shared-memory constraints).
 * For each (view, tile): L = the largest n_contrib over its pixels (capped
 * at the list length); when L > K, theta = the K-th largest importance of
 * the entries at positions [0, L), and every entry there with importance <
 * theta and importance < tau marks its Gaussian.  importance is per row
 * (view * n + id), fp32 as the library receives it; mask is per Gaussian. */
static int desc_float_cmp(const void* pa, const void* pb) {
  const float a = *(const float*)pa, b = *(const float*)pb;
  return a > b ? -1 : (a < b ? 1 : 0);
}

void or_prune_mask(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                   const uint32_t* vals, const int64_t* ranges, const int32_t* n_contrib,
                   const float* importance, int64_t K, float tau, uint8_t* mask) {
  const int32_t tx = (width + tile - 1) / tile, ty = (height + tile - 1) / tile;
  const int64_t T = (int64_t)tx * ty, HW = (int64_t)width * height;
  for (int64_t g = 0; g < n; ++g) mask[g] = 0;
  for (int64_t flat = 0; flat < n_views * T; ++flat) {
    const int64_t view = flat / T, t = flat % T;
    const int32_t x0 = (int32_t)(t % tx) * tile, y0 = (int32_t)(t / tx) * tile;
    int64_t L = 0;
    for (int32_t y = y0; y < y0 + tile && y < height; ++y)
      for (int32_t x = x0; x < x0 + tile && x < width; ++x)
        if (n_contrib[view * HW + (int64_t)y * width + x] > L)
          L = n_contrib[view * HW + (int64_t)y * width + x];
    const int64_t start = ranges[2 * flat], len = ranges[2 * flat + 1] - start;
    if (L > len) L = len;
    if (L <= K) continue;
    float* v = (float*)malloc(sizeof(float) * (size_t)L);
    for (int64_t i = 0; i < L; ++i) {
      const float w = importance[view * n + vals[start + i]];
      v[i] = w > 0.0f ? w : 0.0f;
    }
    qsort(v, (size_t)L, sizeof(float), desc_float_cmp);
    const float theta = v[K - 1];
    free(v);
    for (int64_t i = 0; i < L; ++i) {
      const uint32_t g = vals[start + i];
      float w = importance[view * n + g];
      if (!(w > 0.0f)) w = 0.0f;
      if (w < theta && w < tau) mask[g] = 1;
    }
  }
}

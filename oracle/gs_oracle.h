/*
 * gs_oracle.h -- plain, slow CPU oracle for the 3D Gaussian Splatting
 * training step (single-threaded; the _mt variants only split the same loops
 * over POSIX threads).  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg may call it; the product path
 * never does.  It shares no code, header or constant table with the CUDA
 * library.
 *
 * What it computes is the standard 3DGS training step that every page of the
 * source material builds on but none prints:
 *   - 59 fp32 parameters per Gaussian: 3 mean, 3 log-scale, 4 quaternion,
 *     1 opacity logit, 48 SH-degree-3 colour coefficients
 *     ("On Scaling Up 3D Gaussian Splatting Training", rebuttal answer on the
 *     storage requirement);
 *   - Adam with two moment vectors ("AMD ROCm team open-sources distributed 3D
 *     Gaussian Splatting training", memory-footprint bullet; Kingma & Ba in the
 *     reference list of "A Scalable PyTorch Abstraction for Multi-GPU Gaussian
 *     Splatting");
 *   - per-tile depth-sorted intersection lists (ROCm news item, per-tile
 *     intersection bullet) over 16x16 pixel blocks whose size changes no pixel
 *     ("On Scaling Up ...", answer (1) on pixel block size);
 *   - front-to-back alpha compositing and its analytic backward (ByteSplat
 *     abstract: forward and backward rasterization).
 * Everything is computed in fp64 except the integer/bit decisions the method
 * defines on its fp32 projected values (tile rectangle, sort key), which are
 * evaluated in fp32 exactly as stated next to each function.
 *
 * Parameter layout: one row-major [59][n] array, row k holds parameter k of
 * every Gaussian: rows 0-2 mean, 3-5 log-scale, 6-9 quaternion (w,x,y,z),
 * 10 opacity logit, 11+3*j+c SH coefficient j (0..15) of channel c (0..2).
 * Projected rows are indexed r = view*n + g.
 */
#ifndef GS_ORACLE_H
#define GS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OR_NPARAM 59

typedef struct or_camera {
  double R[9];     /* world -> camera rotation, row-major */
  double t[3];     /* world -> camera translation: p_cam = R p + t */
  double fx, fy, cx, cy;
  int32_t width, height;
  double near_z, far_z;
} or_camera;

/* flags returned per projected row: the row sits close to a discontinuity of
 * the method, so an fp32 implementation may legitimately land on the other
 * side of it. */
#define OR_FLAG_RADIUS   1u  /* 3*sqrt(lambda_max) within 1e-4 (rel) of an integer */
#define OR_FLAG_RECT     2u  /* (mean -+ r)/16 within 1e-4 of an integer          */
#define OR_FLAG_CLAMP    4u  /* x/z or y/z within 1e-4 (rel) of the J clamp       */
#define OR_FLAG_DEPTH    8u  /* depth within 1e-4 (rel) of near/far plane          */
#define OR_FLAG_COLOR   16u  /* a colour channel within 1e-5 of the clamp at 0     */
#define OR_FLAG_DET     32u  /* dilated covariance nearly singular                  */

/* Real SH basis up to degree 3 at unit direction d: out[16]. */
void or_sh_basis(const double d[3], double out[16]);

/* Rotation matrix of the normalised quaternion q = (w,x,y,z): out row-major. */
void or_quat_to_rot(const double q[4], double out[9]);

/* Projection of every Gaussian into every view.
 * params: [59][n] (fp64 copy of the fp32 parameters)
 * outputs per row r = v*n + g: mean2d[r][2], conic[r][3], depth[r],
 *   color[r][3], opacity[r], radius[r], tiles[r], flags[r] (may be NULL).
 * Culled rows get radius 0, tiles 0 and zeros elsewhere. */
void or_project(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                int32_t tile, double* mean2d, double* conic, double* depth, double* color,
                double* opacity, int32_t* radius, int32_t* tiles, uint8_t* flags);

/* or_project split over `threads` POSIX threads by Gaussian index; the
 * outputs are identical for any thread count. */
void or_project_mt(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                   int32_t tile, double* mean2d, double* conic, double* depth, double* color,
                   double* opacity, int32_t* radius, int32_t* tiles, uint8_t* flags,
                   int32_t threads);

/* Tile rectangle of one projected row, evaluated in fp32:
 * [x0,x1) x [y0,y1) in tile units, clamped to the tile grid. */
void or_tile_rect(float mx, float my, int32_t radius, int32_t tile, int32_t tiles_x,
                  int32_t tiles_y, int32_t rect[4]);

/* Total intersections of the projected rows (sum of tile-rect areas of rows
 * with radius > 0). */
int64_t or_count_isect(int64_t n_rows, const float* mean2d, const int32_t* radius,
                       int32_t tile, int32_t width, int32_t height);

/* Binning: emit one (key, gaussian id) pair per (row, tile in its rect), with
 * key = (view*T + tile_index) << 32 | float_bits(depth), then sort by
 * (key, id) with the C library sort, then extract per-(view,tile) ranges
 * [start, end) into ranges[(view*T + tile)*2 + {0,1}] (empty = [0,0)).
 * keys/vals must hold or_count_isect() entries. */
void or_bin(int64_t n, int32_t n_views, const float* mean2d, const int32_t* radius,
            const float* depth, int32_t tile, int32_t width, int32_t height,
            uint64_t* keys, uint32_t* vals, int64_t* ranges);

/* or_bin with the rows and the per-tile sorts split over `threads` POSIX
 * threads; identical outputs. */
void or_bin_mt(int64_t n, int32_t n_views, const float* mean2d, const int32_t* radius,
               const float* depth, int32_t tile, int32_t width, int32_t height,
               uint64_t* keys, uint32_t* vals, int64_t* ranges, int32_t threads);

/* The sorted list of each selected flattened tile (view*T + tile) by brute
 * force: every row of that view whose tile rectangle covers it, ordered by
 * (float_bits(depth), id) -- the same lists or_bin produces for those tiles.
 * Returns the total length; with out_vals NULL it only counts.  Otherwise
 * out_vals receives the concatenated ids and out_ranges[2*s..2*s+1] the
 * [start, end) of selection s. */
int64_t or_bin_select(int64_t n, int32_t n_views, const float* mean2d, const int32_t* radius,
                      const float* depth, int32_t tile, int32_t width, int32_t height,
                      const int64_t* tile_sel, int64_t n_sel, uint32_t* out_vals,
                      int64_t* out_ranges);

/* Morton codes of the Gaussians' means (params: [59][n] fp32, rows 0-2):
 * q = clamp(floor((x - lo) * (2^21 / (hi - lo))), 0, 2^21 - 1) per axis in
 * fp32 over the means' bounding box [lo, hi] (0 when hi == lo); bit b of
 * q_x, q_y, q_z goes to code bit 3b, 3b+1, 3b+2. */
void or_morton_codes(int64_t n, const float* params, uint64_t* codes);

/* perm[k] = index of the k-th Gaussian in ascending (code, index) order. */
void or_morton_order(int64_t n, const float* params, uint32_t* perm);

/* Pruning mask bounded by the per-tile working set; see gs_oracle.c. */
void or_prune_mask(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                   const uint32_t* vals, const int64_t* ranges, const int32_t* n_contrib,
                   const float* importance, int64_t K, float tau, uint8_t* mask);

/* Forward compositing over the sorted per-tile lists (tiled mode).
 * features are fp64 arrays indexed by row; vals hold gaussian ids (row =
 * view*n + id).  tile_sel/n_sel restrict the work to selected flattened
 * (view*T + tile) indices (NULL = all tiles); untouched pixels are left as
 * they were.  Outputs: image[v][3][H][W], T_final[v][H][W],
 * n_contrib[v][H][W]; optional: pairs[v][H][W] (list entries tested before
 * the pixel stopped, the stopping entry included), included[v][H][W] (pairs
 * composited) and margin[v][H][W] = smallest relative distance of any
 * threshold decision of the pixel (alpha vs 1/255, alpha vs 0.99, next
 * transmittance vs 1e-4) from its cut-off; +inf when nothing was tested;
 * importance[row] (optional, caller-initialised) raised to the largest
 * blending weight alpha T of the row over the composited pixels. */
void or_raster_fwd(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                   const double* mean2d, const double* conic, const double* opacity,
                   const double* color, const uint32_t* vals, const int64_t* ranges,
                   const double bg[3], const int64_t* tile_sel, int64_t n_sel,
                   double* image, double* T_final, int32_t* n_contrib, int64_t* pairs,
                   int64_t* included, double* margin, double* importance);

/* or_raster_fwd with the tiles split over `threads` POSIX threads (tile k
 * of the work list on thread k mod threads); identical outputs, no
 * importance. */
void or_raster_fwd_mt(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                      const double* mean2d, const double* conic, const double* opacity,
                      const double* color, const uint32_t* vals, const int64_t* ranges,
                      const double bg[3], const int64_t* tile_sel, int64_t n_sel,
                      double* image, double* T_final, int32_t* n_contrib, int64_t* pairs,
                      int64_t* included, double* margin, int32_t threads);

/* Brute mode: per pixel, every row of the view with radius > 0 whose tile
 * rectangle holds the pixel's tile, visited in (float depth bits, id) order.
 * No intersection lists.  Same outputs as or_raster_fwd (n_contrib counts
 * position in that per-pixel order, so only image/T_final are comparable). */
void or_raster_fwd_brute(int64_t n, int32_t n_views, int32_t width, int32_t height,
                         int32_t tile, const double* mean2d, const double* conic,
                         const double* opacity, const double* color, const double* depth,
                         const int32_t* radius, const double bg[3], double* image,
                         double* T_final);

/* L1 loss mean |image - target| over n values and its gradient sign()/n. */
double or_loss_l1(int64_t n, const double* image, const double* target, double* dL_dimage);

/* Backward compositing: recomputes the forward per pixel (transmittance by
 * forward product) and accumulates per-row gradients (overwritten):
 * g_mean2d[r][2], g_conic[r][3], g_opacity[r], g_color[r][3].  tile_sel/n_sel
 * as in or_raster_fwd (NULL = all tiles). */
void or_raster_bwd(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                   const double* mean2d, const double* conic, const double* opacity,
                   const double* color, const uint32_t* vals, const int64_t* ranges,
                   const double bg[3], const double* dL_dimage, const int64_t* tile_sel,
                   int64_t n_sel, double* g_mean2d, double* g_conic, double* g_opacity,
                   double* g_color);

/* or_raster_bwd with the tiles split over `threads` POSIX threads: each
 * tile's gradients are summed per list position, then added to the rows
 * under a lock.  Equal to or_raster_bwd up to the order of fp64 sums. */
void or_raster_bwd_mt(int64_t n, int32_t n_views, int32_t width, int32_t height, int32_t tile,
                      const double* mean2d, const double* conic, const double* opacity,
                      const double* color, const uint32_t* vals, const int64_t* ranges,
                      const double bg[3], const double* dL_dimage, const int64_t* tile_sel,
                      int64_t n_sel, double* g_mean2d, double* g_conic, double* g_opacity,
                      double* g_color, int32_t threads);

/* Backward through projection and SH colour, summed over views:
 * grad[59][n] (overwritten); visible[n] (may be NULL) = 1 if radius > 0 in
 * any view. */
void or_project_bwd(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                    int32_t tile, const double* g_mean2d, const double* g_conic,
                    const double* g_opacity, const double* g_color, double* grad,
                    uint8_t* visible);

/* or_project_bwd split over `threads` POSIX threads by Gaussian; identical
 * outputs. */
void or_project_bwd_mt(int64_t n, const double* params, int32_t n_views, const or_camera* cams,
                       int32_t tile, const double* g_mean2d, const double* g_conic,
                       const double* g_opacity, const double* g_color, double* grad,
                       uint8_t* visible, int32_t threads);

/* Adam over a [rows][n_cols] array with bias correction at step t (t >= 1).
 * visible (may be NULL): per column; columns with visible == 0 keep p, m, v. */
void or_adam(int64_t n_rows, int64_t n_cols, double* p, const double* g, double* m,
             double* v, int64_t t, double lr, double beta1, double beta2, double eps,
             const uint8_t* visible);

/* or_adam split over `threads` POSIX threads by column; identical outputs. */
void or_adam_mt(int64_t n_rows, int64_t n_cols, double* p, const double* g, double* m,
                double* v, int64_t t, double lr, double beta1, double beta2, double eps,
                const uint8_t* visible, int32_t threads);

#ifdef __cplusplus
}
#endif
#endif

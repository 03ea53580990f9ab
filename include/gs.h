/*
 * gs.h -- C ABI of the GB300 3D Gaussian Splatting training-step library
 * (libgs103.so, CUDA kernels for sm_103a).
 *
 * One training step on one GPU is
 *   gs_project -> gs_bin_and_sort -> gs_tile_order -> gs_rasterize_fwd ->
 *   gs_loss_l1 -> gs_rasterize_bwd -> gs_project_bwd -> gs_adam_step
 * where gs_rasterize_fused may replace the three calls from gs_rasterize_fwd
 * to gs_rasterize_bwd, and gs_tile_order is optional (it only sets the order
 * in which the compositing CTAs start).  The fused call's zeroing of the
 * gradient records can be split off (gs_zero_grads on a second stream after
 * gs_project, then gs_rasterize_fused_acc), so that it runs beside the
 * binning.  Forward-only rendering is the calls up to gs_rasterize_fwd.
 *
 * Source pages (title, section) for what the step computes:
 *  [S1] "On Scaling Up 3D Gaussian Splatting Training": answer on the storage
 *       requirement (59 fp32 parameters per Gaussian: 3 xyz, 3 scale,
 *       4 rotation, 1 opacity, 48 SH); answer (1) on the 16x16 pixel blocks,
 *       whose size alters no pixel value; RetinaGS comparison (opacity
 *       saturation depth, i.e. early termination); independent-gradients
 *       answer (gradients averaged over the views of a batch).
 *  [S2] "AMD ROCm team open-sources distributed 3D Gaussian Splatting
 *       training": memory-footprint bullet (Adam, two moment vectors, SH
 *       degree 3, 708 B per Gaussian); per-tile intersection bullet (per-tile
 *       sorted lists of Gaussian-to-pixel intersections).
 *  [S3] "ByteSplat": abstract (forward and backward rasterization).
 *  [S4] "A Scalable PyTorch Abstraction for Multi-GPU Gaussian Splatting":
 *       references (Kerbl et al. 3D Gaussian Splatting, which defines the
 *       projection, SH colour and compositing model; Kingma & Ba, Adam;
 *       Merrill & Garland, single-pass prefix scan with decoupled look-back;
 *       Merrill & Grimshaw, radix sorting).
 *
 * Conventions for every call:
 *  - Ownership: the caller owns and allocates every buffer.  The library
 *    allocates no memory, host or device.
 *  - Pointers are DEVICE pointers unless marked (host).  Device buffers must
 *    be 16-byte aligned (any cudaMalloc / torch allocation is).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  Only gs_bin_and_sort (not its asynchronous
 *    variant), gs_bin_and_sort_static and gs_workspace_status
 *    synchronise the stream.
 *  - Errors: arguments are validated on the host before anything is
 *    enqueued; an invalid call returns GS_ERR_INVALID_ARG and launches
 *    nothing.  A failed launch returns GS_ERR_CUDA.  Errors the device
 *    detects (a bounded wait that ran out) are written to a status word in
 *    the binning workspace and returned by the next synchronising call.  No
 *    call prints, aborts or exits.
 *  - Cameras are passed by value from host memory (up to GS_MAX_VIEWS) and
 *    must all share one width and height.
 */
#ifndef GS_H
#define GS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GS_NPARAM 59     /* parameters per Gaussian [S1]                     */
#define GS_TILE 16       /* pixel block edge [S1]                             */
#define GS_MAX_VIEWS 16  /* cameras per call                                  */

typedef enum gs_status {
  GS_OK = 0,
  GS_ERR_INVALID_ARG = 1,  /* a pointer, size or camera failed validation      */
  GS_ERR_CAPACITY = 2,     /* intersections exceed the caller's capacity       */
  GS_ERR_TIMEOUT = 3,      /* a bounded device-side wait ran out               */
  GS_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed             */
  GS_ERR_DEVICE_CHECK = 5  /* a device-side consistency check failed           */
} gs_status;

/* Pinhole camera, OpenCV axes (+x right, +y down, +z forward).
 * p_cam = R p_world + t, R row-major.  Pixel (u, v) samples the image plane
 * at (u + 0.5, v + 0.5); mean2d = (fx x/z + cx, fy y/z + cy).
 * Gaussians with z < near_z or z > far_z are culled (far_z may be +inf). */
typedef struct gs_camera {
  float R[9];
  float t[3];
  float fx, fy, cx, cy;
  int32_t width, height;
  float near_z, far_z;
} gs_camera;

/* Projected Gaussian, one per (view, Gaussian) row r = view * n + g.
 * 48 bytes, so one record is three 16-byte vectors.  A culled row has
 * radius = 0 and tiles = 0 (its other fields are unspecified except
 * color_b = depth = 0), unless gs_project was given a tile-count array: then
 * a culled row's record is not written at all and the array says which rows
 * are culled (count 0).
 *
 * Tile counts.  gs_project can write, besides the records, an int32 array
 * tile_counts[n_views * n] holding each row's tile count (0 = culled).  The
 * calls that need to know which rows are visible (gs_bin_and_sort*,
 * gs_rasterize_bwd, gs_rasterize_fused, gs_project_bwd) take the same array
 * (4-byte aligned) or NULL.  With it, culled rows cost 4 bytes each instead
 * of a 48-byte record: written once by the projection, read by the binning,
 * the gradient zeroing and the projection backward, none of which touches a
 * culled row's record or gradient record.  With NULL, the records' radius
 * and tiles fields decide, and every record must have been written. */
typedef struct gs_splat {
  float mean_x, mean_y;     /* projected mean, pixels                          */
  float conic_a, conic_b;   /* inverse 2D covariance [[a, b], [b, c]]          */
  float conic_c, opacity;   /* opacity = sigmoid(logit)                        */
  float color_r, color_g;   /* SH degree-3 colour, clamped at 0                */
  float color_b, depth;     /* depth = camera-space z                          */
  int32_t radius;           /* ceil(3 sqrt(lambda_max)), 0 = culled            */
  int32_t tiles;            /* tiles in the footprint rectangle                */
} gs_splat;

/* Gradient of the loss w.r.t. one projected row, same row indexing.
 * 48 bytes; pad entries are written as 0. */
typedef struct gs_splat_grad {
  float mean_x, mean_y;
  float conic_a, conic_b;
  float conic_c, opacity;
  float color_r, color_g;
  float color_b, pad0, pad1, pad2;
} gs_splat_grad;

/* ---------------------------------------------------------------------- */
/* gs_project -- EWA projection of every Gaussian into every view, SH
 * degree-3 colour, sigmoid opacity, footprint radius and tile count, culling.
 * Defines the "3D-to-2D Gaussian transformations" of [S1] (rendering-speed
 * answer) with the model of [S4] (Kerbl et al.).
 *   n         Gaussians (>= 0, < 2^32)
 *   params    [59][n] fp32, row-major: rows 0-2 mean, 3-5 log-scale,
 *             6-9 quaternion (w,x,y,z), 10 opacity logit, 11+3k+c SH
 *             coefficient k of channel c  [S1]
 *   cams      (host) n_views cameras, 1 <= n_views <= GS_MAX_VIEWS
 *   splats    [n_views * n] output records
 *   tile_counts  [n_views * n] int32 output, or NULL (then every row's
 *             record is written, culled ones with radius = tiles = 0)
 * Returns GS_ERR_INVALID_ARG for bad sizes/cameras or NULL pointers with
 * n > 0. */
gs_status gs_project(int64_t n, const float* params, const gs_camera* cams, int32_t n_views,
                     gs_splat* splats, int32_t* tile_counts, void* stream);

/* ---------------------------------------------------------------------- */
/* Workspace for gs_bin_and_sort, in bytes, for n_rows = n_views * n
 * projected rows and room for `capacity` intersections. */
size_t gs_bin_workspace_bytes(int64_t n_rows, int64_t capacity);

/* Number of radix-sort key bits used for n_views views of a width x height
 * image: 32 depth bits plus the bits of the flattened (view, tile) index. */
int32_t gs_key_bits(int32_t n_views, int32_t width, int32_t height);

/* gs_bin_and_sort -- per-tile depth-sorted intersection lists [S2]:
 * one (key, id) pair per row and tile of its footprint rectangle, key =
 * (view * T + tile) << 32 | bits(depth), T = ceil(W/16) * ceil(H/16), in the
 * order of a stable sort of the keys emitted with rows in order and tiles
 * row-major (ties of equal depth fall back to Gaussian id); and
 * ranges[(view * T + tile)] = [first, last + 1) of each tile's pairs, [0, 0)
 * when empty.  Computed as:
 *  1. compaction of the visible rows (tile count > 0) in row order, single
 *     pass with decoupled look-back [S4 Merrill & Garland] -> totals I and R
 *     (read back to the host: the one synchronisation of the step);
 *  2. stable LSD radix sort of the R visible rows on their 32 depth bits,
 *     8 bits per pass, onesweep style [S4 Merrill & Grimshaw];
 *  3. emission of each row's tiles in that order (a second look-back scan
 *     gives the offsets);
 *  4. stable radix passes on the tile bits of gs_key_bits() (8 per pass);
 *  5. the ranges.
 *   splats     [n_views * n] from gs_project
 *   tile_counts  [n_views * n] from gs_project, or NULL
 *   workspace  ws_bytes >= gs_bin_workspace_bytes(n_views * n, capacity);
 *              its first 256 bytes (a status header) must be zero before the
 *              first call (e.g. cudaMemset once after allocation); calls keep
 *              it consistent afterwards
 *   capacity   length of keys/vals (<= 2^32 - 1)
 *   keys, vals [capacity] output: sorted keys and Gaussian ids (also used as
 *              scratch during the call)
 *   ranges     [n_views * T][2] int64 output
 *   n_isect    (host) receives I, also when I > capacity
 * Returns GS_ERR_CAPACITY (no result; ranges untouched, keys and vals
 * overwritten) when I > capacity; GS_ERR_TIMEOUT if a device wait ran out
 * (this call's compaction, or the previous call on this workspace);
 * GS_ERR_DEVICE_CHECK if a record's tile count did not match its rectangle
 * (that row is left out).  GS_ERR_INVALID_ARG unless n_views * n and
 * n_views * T are below 2^32 and ceil(W/16), ceil(H/16) <= 65535. */
gs_status gs_bin_and_sort(int64_t n, int32_t n_views, const gs_splat* splats,
                          const int32_t* tile_counts, int32_t width, int32_t height,
                          void* workspace, size_t ws_bytes, int64_t capacity, uint64_t* keys,
                          uint32_t* vals, int64_t* ranges, int64_t* n_isect, void* stream);

/* Synchronises `stream` and returns (and clears) the device status word of a
 * binning workspace: GS_OK, GS_ERR_TIMEOUT, GS_ERR_DEVICE_CHECK, or
 * GS_ERR_CAPACITY when the latest gs_bin_and_sort_async call exceeded its
 * capacity. */
gs_status gs_workspace_status(void* workspace, void* stream);

/* gs_bin_and_sort_async -- gs_bin_and_sort without synchronising the stream,
 * so that a whole training step can be captured once into a CUDA graph and
 * replayed.  Launch shapes follow n_views * n and `capacity` (not the counts,
 * which stay on the device); surplus work items exit at once.
 *   n_isect  (device) int64, receives I
 * When I > capacity nothing is emitted, ranges are all empty, and the
 * workspace status word carries the capacity bit: gs_workspace_status then
 * returns GS_ERR_CAPACITY, and gs_adam_step_dev / gs_step_advance given the
 * workspace skip their update.  The bit describes the latest call.  The first
 * call on a device should be made outside graph capture (it sets a kernel
 * attribute), as any gs_bin_and_sort call does. */
gs_status gs_bin_and_sort_async(int64_t n, int32_t n_views, const gs_splat* splats,
                                const int32_t* tile_counts, int32_t width, int32_t height,
                                void* workspace, size_t ws_bytes, int64_t capacity,
                                uint64_t* keys, uint32_t* vals, int64_t* ranges,
                                int64_t* n_isect, void* stream);

/* Self-test of the bounded device waits: runs one look-back partition whose
 * predecessor never publishes, so its wait runs out (about a second); the
 * kernel flags the error and returns, and the call synchronises and returns
 * GS_ERR_TIMEOUT (GS_OK would mean the bound failed).  The context stays
 * usable.  Needs ws_bytes >= gs_bin_workspace_bytes(1, 1); overwrites it. */
gs_status gs_selftest_lookback_timeout(void* workspace, size_t ws_bytes, void* stream);

/* gs_bin_and_sort_static -- gs_bin_and_sort for callers that cannot allocate
 * device memory: an application whose own allocator owns the whole GPU and
 * gives out no extra buffers, a frame loop that must not stall on an
 * allocation, or a plug-in that only receives its input and output buffers.
 * The scratch lives in one array inside the library (14 MiB, held by every
 * GPU that loads the library until the process exits); the call allocates
 * nothing.  The source pages have no counterpart to this entry point; it is
 * an interface convenience over gs_bin_and_sort, with the same arguments
 * minus the workspace and the same results.
 *   limits   n_views * n <= GS_BIN_STATIC_MAX_ROWS and
 *            capacity <= GS_BIN_STATIC_MAX_ISECT, else GS_ERR_INVALID_ARG
 *            (I > capacity still returns GS_ERR_CAPACITY)
 *   set-up   the first call on a device (with that device current) looks up
 *            the array's device address and zeroes its status header, with a
 *            device-wide synchronisation; make that first call before any
 *            stream capture
 *   sharing  every call uses the same array, which keeps the last call's
 *            contents: calls that overlap on the GPU (other streams, other
 *            host threads) race; serialise them */
#define GS_BIN_STATIC_MAX_ROWS 65536
#define GS_BIN_STATIC_MAX_ISECT 1048576
gs_status gs_bin_and_sort_static(int64_t n, int32_t n_views, const gs_splat* splats,
                                 const int32_t* tile_counts, int32_t width, int32_t height,
                                 int64_t capacity, uint64_t* keys, uint32_t* vals,
                                 int64_t* ranges, int64_t* n_isect, void* stream);

/* ---------------------------------------------------------------------- */
/* gs_tile_order -- the launch order for the compositing calls: the tiles
 * (view * T + tile) by descending floor(log2(list length)), empty tiles
 * last, ties in tile order (longest lists first: a tile's cost grows with
 * its list, and a long list started late leaves the other SMs idle at the
 * end).  Any permutation gives the same images; the gradients differ only by
 * the order of float atomics.
 *   ranges  [n_flat][2] from gs_bin_and_sort
 *   order   [n_flat] uint32 output (device) */
gs_status gs_tile_order(int64_t n_flat, const int64_t* ranges, uint32_t* order, void* stream);

/* gs_rasterize_fwd -- per-tile front-to-back alpha compositing [S3] over
 * the sorted lists.  Per pixel (centre (u+0.5, v+0.5)), for each pair of its
 * tile's list in order: power = -(a dx^2 + c dy^2)/2 - b dx dy,
 * alpha = min(0.99, opacity e^power); pairs with alpha < 1/255 are skipped;
 * the pair that would take transmittance below 1e-4 stops the pixel and is
 * excluded [S1 opacity saturation]; C = sum c alpha T + T_final bg.
 *   vals, ranges  from gs_bin_and_sort
 *   tile_order    [n_views * T] from gs_tile_order (the order in which the
 *                 tiles' CTAs start), or NULL for tile order; the same
 *                 argument in every gs_rasterize_* call
 *   bg            (host) background colour [3]
 *   image         [n_views][3][H][W]
 *   T_final       [n_views][H][W] final transmittance
 *   n_contrib     [n_views][H][W] 1 + list position of the last included
 *                 pair (0 = none) */
gs_status gs_rasterize_fwd(int64_t n, int32_t n_views, const gs_splat* splats, int32_t width,
                           int32_t height, const uint32_t* vals, const int64_t* ranges,
                           const uint32_t* tile_order, const float* bg, float* image,
                           float* T_final, int32_t* n_contrib, void* stream);

/* gs_rasterize_fwd_counted -- gs_rasterize_fwd with the same outputs that
 * also adds to counts[0] the pairs tested (per pixel: the list entries up to
 * and including the one that stopped it, or the whole list) and to counts[1]
 * the pairs composited.  Work accounting for the compositing roofline; not
 * part of the training step.
 *   counts        device uint64[2], accumulated (zero it first)
 *   pixel_counts  device int32 [2][n_views][H][W] or NULL: the same two
 *                 counts per pixel (plane 0 tested, plane 1 composited),
 *                 zeroed by this call */
gs_status gs_rasterize_fwd_counted(int64_t n, int32_t n_views, const gs_splat* splats,
                                   int32_t width, int32_t height, const uint32_t* vals,
                                   const int64_t* ranges, const uint32_t* tile_order,
                                   const float* bg, float* image, float* T_final,
                                   int32_t* n_contrib, uint64_t* counts, int32_t* pixel_counts,
                                   void* stream);

/* gs_loss_l1 -- L = mean |image - target| over `count` values and
 * dL/dimage = sign(image - target) / count (sign(0) = 0).  Helper beyond the
 * six step calls; the configs of the step use an L1 photometric loss.
 *   loss  device scalar, overwritten */
gs_status gs_loss_l1(const float* image, const float* target, int64_t count, float* loss,
                     float* dL_dimage, void* stream);

/* gs_rasterize_bwd -- analytic backward of gs_rasterize_fwd [S3]: each
 * pixel walks its list back to front from n_contrib, rebuilding
 * T_i = T_{i+1} / (1 - alpha_i) from T_final and the colour composited
 * behind each pair; per-pair gradients are reduced per warp before global
 * atomics.
 *   tile_counts  [n_views * n] from gs_project, or NULL
 *   grads  [n_views * n] output, zeroed by this call, then accumulated; with
 *          tile_counts, only the rows with a positive count are written, and
 *          the records are zeroed in pairs of rows (2k, 2k+1) of which one at
 *          least is visible (a culled row's record is either left as it was
 *          or zeroed) */
gs_status gs_rasterize_bwd(int64_t n, int32_t n_views, const gs_splat* splats,
                           const int32_t* tile_counts, int32_t width,
                           int32_t height, const uint32_t* vals, const int64_t* ranges,
                           const uint32_t* tile_order, const float* bg, const float* T_final,
                           const int32_t* n_contrib, const float* dL_dimage,
                           gs_splat_grad* grads, void* stream);

/* gs_rasterize_fused -- gs_rasterize_fwd, gs_loss_l1 and gs_rasterize_bwd
 * in one launch, one CTA per tile ([S3] abstract: forward and backward
 * rasterization fused into a single kernel that keeps intermediate results
 * on chip).  The forward's per-pixel results (transmittance, last
 * contributor, colour) and the L1 gradient stay on chip instead of passing
 * through T_final, n_contrib and dL/dimage in memory, and the batches the
 * forward leaves staged in shared memory are reused by the backward without
 * a new gather.  With a workspace the forward also records, per batch of 192
 * list entries and per 4x2 pixel block, which entries it composited (768 B
 * per batch), and the backward walks exactly those instead of every entry
 * whose footprint box meets the block.  Results equal those of the three
 * separate calls (the gradient up to the order of float atomics), with or
 * without the workspace.
 *   tile_counts  [n_views * n] from gs_project, or NULL (as gs_rasterize_bwd)
 *   target     [n_views][3][H][W] fp32, the images the L1 loss compares with
 *   image, T_final, n_contrib   outputs as gs_rasterize_fwd
 *   loss       device scalar, overwritten: mean |image - target| over
 *              n_views*3*H*W
 *   grads      [n_views * n] output, zeroed by this call, then accumulated;
 *              as gs_rasterize_bwd with dL/dimage = sign(image - target) /
 *              (n_views*3*H*W)
 *   workspace  NULL, or gs_rasterize_workspace_bytes(n_views, W, H, capacity)
 *              bytes (16-byte aligned, no initialisation) for lists of at
 *              most `capacity` entries in all; a tile whose records do not
 *              fit in ws_bytes falls back to the box walk */
size_t gs_rasterize_workspace_bytes(int32_t n_views, int32_t width, int32_t height,
                                    int64_t capacity);
gs_status gs_rasterize_fused(int64_t n, int32_t n_views, const gs_splat* splats,
                             const int32_t* tile_counts, int32_t width,
                             int32_t height, const uint32_t* vals, const int64_t* ranges,
                             const uint32_t* tile_order, const float* bg, const float* target,
                             float* image, float* T_final, int32_t* n_contrib, float* loss,
                             gs_splat_grad* grads, void* workspace, size_t ws_bytes,
                             void* stream);

/* gs_zero_grads -- the zeroing that gs_rasterize_bwd and gs_rasterize_fused
 * start with, as a call of its own: all n_views * n gradient records without
 * tile_counts; with tile_counts, the records of the pairs of rows (2k, 2k+1)
 * of which one at least has a positive count.  It reads nothing but the tile
 * counts, so it can run on a second stream while gs_bin_and_sort builds the
 * lists; gs_rasterize_fused_acc then adds the gradients.
 *   tile_counts  [n_views * n] from gs_project, or NULL
 *   grads        [n_views * n] output (16-byte aligned)
 *   beside       nonzero: launched to run beside other kernels (a grid of two
 *                CTAs per SM that strides over the rows, which leaves them
 *                room; slower alone on very large row counts); 0: one thread
 *                per pair of rows, the fastest form alone
 * GS_ERR_INVALID_ARG unless 0 <= n < 2^32 and 1 <= n_views <= GS_MAX_VIEWS. */
gs_status gs_zero_grads(int64_t n, int32_t n_views, const int32_t* tile_counts,
                        gs_splat_grad* grads, int32_t beside, void* stream);

/* gs_rasterize_fused_acc -- gs_rasterize_fused without its zeroing: the
 * gradients are added to `grads` as it stands, which gs_zero_grads (same
 * tile_counts) has zeroed before.  Arguments, checks and every other result
 * as gs_rasterize_fused. */
gs_status gs_rasterize_fused_acc(int64_t n, int32_t n_views, const gs_splat* splats,
                                 const int32_t* tile_counts, int32_t width, int32_t height,
                                 const uint32_t* vals, const int64_t* ranges,
                                 const uint32_t* tile_order, const float* bg, const float* target,
                                 float* image, float* T_final, int32_t* n_contrib, float* loss,
                                 gs_splat_grad* grads, void* workspace, size_t ws_bytes,
                                 void* stream);

/* gs_project_bwd -- chain rule from the per-row gradients back to the 59
 * parameters, summed over the views (the 1/n_views average of [S1] comes
 * from the loss normalisation):
 * colour -> SH coefficients and view direction -> mean; conic -> 2D
 * covariance -> (J, Sigma) -> (mean, quaternion, log-scale); opacity ->
 * logit.  The derivative is exact where the step is differentiable; through
 * an active clamp (alpha cap, colour at 0, the J field-of-view clamp) the
 * clamped quantity contributes 0.
 *   tile_counts  [n_views * n] from gs_project, or NULL; a row is read (its
 *            record and gradient record) only when visible
 *   grad     [59][n] output (overwritten)
 *   visible  [n] output or NULL: 1 if the Gaussian has radius > 0 in any
 *            view, else 0 */
gs_status gs_project_bwd(int64_t n, const float* params, const gs_camera* cams, int32_t n_views,
                         const gs_splat* splats, const int32_t* tile_counts,
                         const gs_splat_grad* grads, float* grad, uint8_t* visible,
                         void* stream);

/* gs_adam_step -- Adam [S4 Kingma & Ba; S2 two moments] over the [59][n]
 * parameters, fused in one pass:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p -= lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps),   t = step >= 1.
 * visible == NULL: dense, every column updated.  Otherwise sparse: columns
 * with visible[g] == 0 keep p, m and v unchanged (t stays global). */
gs_status gs_adam_step(int64_t n, float* params, const float* grad, float* m, float* v,
                       int64_t step, float lr, float beta1, float beta2, float eps,
                       const uint8_t* visible, void* stream);

/* gs_adam_step_dev -- gs_adam_step with the step number read from device
 * memory (*step >= 1, bias corrections computed on the device), for a step
 * captured once and replayed.  bin_workspace (or NULL): when its status word
 * carries the capacity bit of gs_bin_and_sort_async, nothing is updated. */
gs_status gs_adam_step_dev(int64_t n, float* params, const float* grad, float* m, float* v,
                           const int64_t* step, float lr, float beta1, float beta2, float eps,
                           const uint8_t* visible, const void* bin_workspace, void* stream);

/* gs_step_advance -- *step += 1 on the device (step: device int64), unless
 * bin_workspace (or NULL) carries the capacity bit. */
gs_status gs_step_advance(int64_t* step, const void* bin_workspace, void* stream);

/* ---------------------------------------------------------------------- */
/* Morton order of the Gaussians ([S4] references: Morton order), for the
 * locality of the id-indexed gathers of compositing.  A reorder permutes the
 * columns of every [rows][n] array consistently (parameters, Adam m and v,
 * with gs_gather_columns);
 * the step's results are those of the original scene with the Gaussians
 * renamed (equal-depth ties in a tile then break by the new ids).
 *
 * gs_morton_order -- perm[k] = index of the k-th Gaussian in Morton order.
 * Each mean is quantised to 21 bits per axis inside the means' bounding box,
 *   q = clamp(floor((x - lo) * (2^21 / (hi - lo))), 0, 2^21 - 1)  (fp32,
 *   one rounding per operation; 0 when hi == lo),
 * and code = sum_i bit_i(q_x) 2^(3i) + bit_i(q_y) 2^(3i+1) + bit_i(q_z)
 * 2^(3i+2); perm sorts (code, index) ascending (stable radix sort, 8 passes).
 *   params     [59][n] (rows 0-2 are read)
 *   workspace  gs_morton_workspace_bytes(n) bytes, 16-byte aligned; its
 *              first 256 bytes must be zero before the first use (device
 *              status word, as the binning workspace; gs_workspace_status
 *              reads it)
 *   perm       [n] uint32 output
 * Asynchronous; does not synchronise. */
size_t gs_morton_workspace_bytes(int64_t n);
gs_status gs_morton_order(int64_t n, const float* params, void* workspace, size_t ws_bytes,
                          uint32_t* perm, void* stream);

/* gs_gather_columns -- dst[r][i] = src[r][idx[i]] for r < rows, i < n_dst
 * (row-major fp32, src [rows][n_src], dst [rows][n_dst], distinct; idx
 * entries >= n_src are clamped to n_src - 1).  With idx = perm and n_dst =
 * n_src it applies a Morton order; with idx from gs_compact_index it drops
 * pruned Gaussians. */
gs_status gs_gather_columns(int64_t rows, int64_t n_src, int64_t n_dst, const float* src,
                            const uint32_t* idx, float* dst, void* stream);

/* ---------------------------------------------------------------------- */
/* Pruning bounded by the per-tile working set ([S3] abstract: pruning that
 * considers rendering quality and per-tile shared-memory constraints, so
 * that the fused forward + backward keeps its working set on chip).
 *
 * gs_rasterize_fwd_importance -- gs_rasterize_fwd that also records, per
 * projected row, the largest blending weight alpha T the Gaussian has in
 * any pixel (its importance).
 *   importance  [n_views * n] fp32 output (zeroed by this call). */
gs_status gs_rasterize_fwd_importance(int64_t n, int32_t n_views, const gs_splat* splats,
                                      int32_t width, int32_t height, const uint32_t* vals,
                                      const int64_t* ranges, const uint32_t* tile_order,
                                      const float* bg, float* image, float* T_final,
                                      int32_t* n_contrib, float* importance, void* stream);

/* gs_prune_mask -- for every (view, tile): L = the largest n_contrib over
 * its pixels (its working set is list positions [0, L)); when L > capacity,
 * theta = the capacity-th largest importance in the working set, and every
 * Gaussian there with importance < theta and importance < tau is marked.
 * tau is the quality floor (tau > 1 disables it).
 *   n_contrib   [n_views][H][W] from the forward over the same lists
 *   importance  [n_views * n] per-row importance (any non-negative score)
 *   mask        [n] uint8 output: 1 = prune, 0 = keep (zeroed by this call) */
gs_status gs_prune_mask(int64_t n, int32_t n_views, int32_t width, int32_t height,
                        const uint32_t* vals, const int64_t* ranges, const int32_t* n_contrib,
                        const float* importance, int64_t capacity, float tau, uint8_t* mask,
                        void* stream);

/* gs_compact_index -- idx[0..k) = the indices i with mask[i] == 0, in
 * order; *n_keep = k (device int64).  workspace: gs_compact_workspace_bytes(n)
 * bytes, no initialisation needed. */
size_t gs_compact_workspace_bytes(int64_t n);
gs_status gs_compact_index(int64_t n, const uint8_t* mask, void* workspace, size_t ws_bytes,
                           uint32_t* idx, int64_t* n_keep, void* stream);

/* ---------------------------------------------------------------------- */
/* Text of a status code (static storage; "unknown status" for other
 * values).  gs_status_str is the same function under a shorter name. */
const char* gs_status_string(gs_status status);
const char* gs_status_str(gs_status status);
int32_t gs_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GS_H */

/*
 * gm.h -- C ABI of libgm, a B300 (sm_103a) CUDA library for the tile-based
 * forward and backward rendering of scenes that hold both a triangle mesh
 * and 3D Gaussians.
 *
 * The method is the hybrid renderer of "A Lightweight and Differentiable
 * Renderer for Joint Mesh and 3D Gaussian Splat Scenes" (Design Details:
 * Mesh rasterizer items 1-3, Hybrid rendering).  By default each Gaussian is
 * depth-tested against the mesh (hard split) and the mesh layer is opaque and
 * not antialiased; options add the soft split at the mesh surface
 * (gm_opts.softness) and analytic edge antialiasing (gm_antialias and the
 * gm_aa_layer argument).  The renderer's call (rgb, depth, alpha from a mesh,
 * Gaussians and a camera pose) is split into seven steps; a forward pass is
 *
 *   gm_bin_triangles -> gm_zbuffer -> gm_interp_mesh          (mesh layer)
 *     (or gm_zbuffer_direct -> gm_interp_mesh: the same face ids, no lists)
 *     [-> gm_antialias, with gm_mesh_edges once per mesh]
 *   gm_project_gaussians -> gm_bin_sort_gaussians             (Gaussians)
 *   gm_composite_hybrid_fwd                                   (image)
 *
 * and gm_composite_hybrid_bwd returns the gradients of a loss with respect to
 * the projected Gaussians and to the mesh's vertex positions and colours
 * (with antialiasing through gm_antialias_bwd and gm_interp_mesh_bwd);
 * gm_project_gaussians_bwd carries the Gaussians' to their 3D parameters.
 *
 * Conventions shared by every call
 *   - Camera: pinhole, world -> camera  X_c = R X_w + t  (R row-major),
 *     OpenCV axes (x right, y down, z forward).  Pixel (i, j) has its centre
 *     at (i + 0.5, j + 0.5).  Images are row-major [height][width]; colour
 *     images interleave RGB ([height][width][3]).  Tiles are 16 x 16 pixels,
 *     tile id = ty * ceil(width / 16) + tx.
 *   - Memory: every pointer argument is a device pointer (memory the caller
 *     allocated with cudaMalloc or an equivalent), except the gm_camera /
 *     gm_opts structs and *K_host, which are host memory.  The library never
 *     allocates, frees or keeps caller memory; scratch memory comes from the
 *     caller's workspace (see the *_workspace_size calls).  Arrays marked
 *     "16-byte aligned" are read or written with 16-byte vector accesses.
 *   - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *     Every call only enqueues work on it and returns, unless K_host is given
 *     (then it waits for that stream once, at the end).
 *   - Errors: every call returns a gm_status.  GM_ERR_INVALID_ARG is returned
 *     before any work is enqueued.  GM_ERR_CUDA means a launch failed; the
 *     stream may hold partial work.  gm_last_error() returns a message for
 *     the calling thread's last failure.  Gradient outputs are accumulated
 *     (+=); the caller zeroes them.
 *   - Sizes: counts (N, nV, nF, capacities) are int32 and must be >= 0; the
 *     number of (primitive, tile) entries must stay below 2^30.
 */
#ifndef GM_H
#define GM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GM_TILE 16
#define GM_SPLAT_STRIDE 12 /* floats per projected-Gaussian record */

typedef enum gm_status {
    GM_OK = 0,
    GM_ERR_INVALID_ARG = 1, /* null / misaligned pointer, negative size, bad camera */
    GM_ERR_CAPACITY = 2,    /* more entries than the caller's capacity (needed K in *K_host) */
    GM_ERR_CUDA = 3,        /* a kernel launch or CUDA runtime call failed */
    GM_ERR_TIMEOUT = 4,     /* a bounded inter-block wait in the sort gave up (see counters) */
    GM_ERR_INTERNAL = 5
} gm_status;

/* counters: a caller-owned device int32[4] written by the two binning calls */
enum { GM_CNT_K = 0,        /* entries needed (after the occlusion cull) */
       GM_CNT_K_PRECULL = 1,/* entries before the cull (Gaussians only) */
       GM_CNT_FLAGS = 2 };  /* bit 0: capacity overflow, bit 1: wait timeout */
#define GM_FLAG_OVERFLOW 1
#define GM_FLAG_TIMEOUT 2

typedef struct gm_camera {
    int32_t width, height;          /* pixels, > 0 */
    float fx, fy, cx, cy;           /* focal lengths and principal point, pixels */
    float near_plane, far_plane;    /* camera-z range, 0 < near < far */
    float R[9];                     /* world -> camera rotation, row-major */
    float t[3];                     /* world -> camera translation */
} gm_camera;

typedef struct gm_opts {
    float bg[3];            /* background colour behind uncovered pixels */
    int32_t cull_occluded;  /* 1: drop Gaussians hidden behind fully covered tiles */
    int32_t sh_degree;      /* -1: colours are RGB [N][3]; 0..3: SH coefficients [N][(d+1)^2][3] */
    int32_t tile_test;      /* 1: also drop a (Gaussian, tile) pair when no pixel centre of the tile
                               can reach alpha >= 1/255 (see gm_bin_sort_gaussians) */
    float softness;         /* 0: hard depth test; > 0: soft split of each Gaussian at the mesh
                               (see gm_composite_hybrid_fwd) with this width factor */
    int32_t soft_split;     /* form of the split's front fraction f(x): GM_SPLIT_PHI (the
                               standard normal CDF) or GM_SPLIT_LOGISTIC (1 / (1 + exp(-1.702 x))) */
} gm_opts;

#define GM_SPLIT_PHI 0
#define GM_SPLIT_LOGISTIC 1

/* The antialiased mesh layer (gm_antialias) and the buffers of the chain of
 * Gaussians composited behind it, for gm_composite_hybrid_fwd / _bwd.  All
 * images row-major [H][W], device memory owned by the caller. */
typedef struct gm_aa_layer {
    const float* cov;  /* [H][W] coverage a in [0, 1]; the call's mesh_rgb is then the
                          premultiplied colour M = a c and mesh_depth the split depth */
    float* back;       /* [H][W][4], 16-byte aligned: colour and depth composited behind the
                          layer (written by the forward, read by the backward) */
    float* T_back;     /* [H][W]: that chain's transmittance (forward out, backward in) */
    int32_t* n_back;   /* [H][W]: 1 + list position of its last composited Gaussian */
    float* v_cov;      /* [H][W] backward out: dL/da */
    float* v_rgb;      /* [H][W][3] backward out: dL/dM */
} gm_aa_layer;

/* Staged records of the Gaussian tile lists (Hybrid rendering, the
 * compositing kernel): one record per list position, the compositing's form
 * of that position's splat (mean, conic pre-scaled for exp2, opacity, colour,
 * depth, the Gaussian's id and the exponent bound of alpha >= 1/255; with the
 * soft split also its depth model; with the hard split instead, for each of
 * the tile's 8 x 4 pixel blocks, which records of each batch reach it).
 * gm_composite_hybrid_fwd writes the records (and the hard split's hit lists)
 * of every batch it stages; gm_composite_hybrid_bwd then reads the records
 * instead of gathering the splats through the ids: with the hard split each
 * warp loads the records its hit lists name, with the soft split each batch
 * of a tile's list comes into shared memory by bulk copies.  With the hard
 * split it takes the forward's hit lists instead of testing the records
 * again.  recs: device memory of
 * gm_staged_bytes(cap, opts->softness) bytes, 16-byte aligned, owned by the
 * caller, contents private to the library; cap >= the number of entries the
 * tile ranges address.  The backward call must get the records its forward
 * call wrote, for the same tile lists, splats and options. */
typedef struct gm_staged {
    float* recs;
    int32_t cap;
} gm_staged;

/* bytes of a staged-record buffer for cap list positions: 56 per position,
 * 64 with the soft split (softness > 0) */
size_t gm_staged_bytes(int32_t cap, float softness);

/* gm_get_copy_status -- the bulk copies of gm_composite_hybrid_bwd (soft
 * split, staged records) wait for their data at most about one second; a wait that gives up stops that CTA
 * (its gradients are then incomplete) and sets bit 0 of a device status word.
 * *flags (host) receives the word; clear != 0 resets it.  Synchronous. */
int gm_get_copy_status(uint32_t* flags, int32_t clear);

/*
 * Projected-Gaussian record ("splat"), GM_SPLAT_STRIDE floats, 16-byte aligned:
 *   [0] mean2d x  [1] mean2d y      (pixels)
 *   [2] conic a   [3] conic b   [4] conic c   (inverse 2D covariance:
 *        sigma(d) = (a dx^2 + c dy^2) / 2 + b dx dy)
 *   [5] opacity   [6..8] RGB    [9] camera-space depth of the centre
 *   [10] the soft split's hide depth z_c - R - t sigma_z softness (written by
 *        gm_project_gaussians when opts->softness > 0; 0 otherwise): beyond it
 *        the mesh hides the Gaussian (the soft occlusion cull reads it; 0
 *        disables that cull)
 *   [11] reserved (0)
 * Gradient buffers of the same layout hold dL/d of each field.
 */

/* ------------------------------------------------------------------------
 * gm_bin_triangles -- Mesh rasterizer, item 1 (triangles binned into 16x16
 * tiles).  A triangle is drawn when every vertex is strictly beyond the near
 * plane (no clipping; Mesh rasterizer, last paragraph), its projected area
 * is non-zero and its box of pixel centres meets the image; it is binned to
 * every tile that box touches.
 *   V [nV][3] f32 world positions; F [nF][3] i32 vertex indices (checked
 *   against nV: an out-of-range index drops the face and sets no error).
 *   tile_range [T][2] i32 out: [first, last) entries of each tile in tri_ids.
 *   tri_ids [cap] i32 out: face ids, tile-major, ascending within a tile.
 *   counters [4] i32 out (device): GM_CNT_K = entries needed; flags.
 *   K_host: NULL, or a host int32 that receives the needed K after a stream
 *   synchronisation; then GM_ERR_CAPACITY is returned when K > cap.  With
 *   K_host == NULL nothing waits: when K > cap the outputs are invalid
 *   (GM_FLAG_OVERFLOW is set in counters) but no write leaves the buffers.
 *   ws / ws_bytes: workspace of at least gm_bin_triangles_workspace_size().
 * ---------------------------------------------------------------------- */
size_t gm_bin_triangles_workspace_size(int32_t nF, int32_t cap, int32_t width, int32_t height);
int gm_bin_triangles(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                     int32_t* tile_range, int32_t* tri_ids, int32_t cap, int32_t* counters,
                     int32_t* K_host, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * gm_zbuffer -- Mesh rasterizer, item 1 (nearest triangle at each pixel
 * centre; the only non-differentiable step).  Over the tile's triangles: a
 * pixel centre is covered when it lies in the triangle's pixel-centre box and
 * every edge function has the sign of the area (edges inclusive, both
 * windings).  The nearest perspective-correct depth wins; equal depths go to
 * the smaller face id.
 *   tile_range / tri_ids: from gm_bin_triangles (ids outside [0, nF) are
 *   skipped).  face_id [H][W] i32 out (-1 = uncovered).
 * ---------------------------------------------------------------------- */
int gm_zbuffer(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
               const int32_t* tile_range, const int32_t* tri_ids, int32_t* face_id, void* stream);

/* ------------------------------------------------------------------------
 * gm_zbuffer_direct -- gm_zbuffer without triangle lists: the same coverage,
 * depth and tie rules over every (triangle, box pixel) pair, the nearest
 * surface kept per pixel with an atomic minimum of (reciprocal depth, face
 * id).  face_id equals gm_zbuffer's bit for bit (for the lists
 * gm_bin_triangles builds of the same mesh).  No gm_bin_triangles call is
 * needed.  Triangles that a vertex puts at or in front of the near plane, of
 * zero area or outside the image are skipped, as by gm_bin_triangles.
 *   face_id [H][W] i32 out (-1 = uncovered).
 *   ws: gm_zbuffer_direct_workspace_size(nF, width, height) bytes, 16-byte
 *   aligned (8 bytes per pixel plus 100 bytes per face); nothing else may
 *   use it during the call.
 * ---------------------------------------------------------------------- */
size_t gm_zbuffer_direct_workspace_size(int32_t nF, int32_t width, int32_t height);
int gm_zbuffer_direct(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                      int32_t* face_id, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * gm_interp_mesh -- Mesh rasterizer, item 2 (depth and vertex colours
 * recomputed from the face ids with perspective-correct interpolation).
 *   l_k = e_k / area (screen barycentrics), D = 1 / sum_k l_k / z_k,
 *   w_k = (l_k / z_k) D, colour = sum_k w_k vcol_k.
 *   vcol [nV][3] f32.  mesh_depth [H][W] f32 out (+inf where uncovered);
 *   mesh_rgb [H][W][3] f32 out (0 where uncovered).
 *   tile_far [T] f32 out: largest mesh depth of a fully covered tile, +inf
 *   otherwise; tile_full [T] u8 out: 1 when every in-image pixel of the tile
 *   is covered.  Both feed the occlusion cull of gm_bin_sort_gaussians.
 * ---------------------------------------------------------------------- */
int gm_interp_mesh(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                   const float* vcol, const int32_t* face_id, float* mesh_depth, float* mesh_rgb,
                   float* tile_far, uint8_t* tile_full, void* stream);

/* ------------------------------------------------------------------------
 * gm_mesh_edges -- edge adjacency for the antialiasing (Mesh rasterizer,
 * item 3: internal edges of a connected surface are left untouched).
 *   adj [nF][3] i32 out: the face that shares edge k of face f (edge k joins
 *   corners k+1 and k+2 mod 3, the edge opposite corner k), -1 when no other
 *   face does, -2 when more than one does.  Depends on F only (compute once
 *   per mesh topology).  Vertex ids must lie in [0, nV).
 *   ws / ws_bytes: device scratch of at least gm_mesh_edges_workspace_size(nF)
 *   bytes; counters: device int32[4] (flags: a sort wait that gave up sets
 *   GM_FLAG_TIMEOUT).
 * ---------------------------------------------------------------------- */
size_t gm_mesh_edges_workspace_size(int32_t nF);
int gm_mesh_edges(const int32_t* F, int32_t nF, int32_t nV, int32_t* adj, int32_t* counters, void* ws,
                  size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * gm_antialias -- Mesh rasterizer, item 3: analytic edge antialiasing (as in
 * nvdiffrast; Limitations: a per-axis 1D approximation, exact for straight
 * edges away from corners).  For each pair of neighbouring pixels (along x
 * and y) that see different faces, the nearer surface (smaller mesh_depth,
 * none when equal) is followed from its pixel's centre towards the other
 * centre through its faces -- across internal edges: one face across, lying
 * on the other side of the edge in the image -- until it leaves by a
 * silhouette edge (no face across, more than one, or one folded onto the
 * same side), at most 8 faces; a pair along x only takes an edge more
 * vertical than horizontal in the image, a pair along y the others.  The
 * crossing t (0 at the nearer pixel's centre, 1 at the other's) gives the
 * weight w = |t - 0.5|, which moves the layer (a, M) of one pixel towards the
 * other pixel's (coverage 1 and colour c where the mesh covers a pixel, 0
 * elsewhere): the other pixel when t >= 0.5 (the surface reaches into it),
 * the nearer one when t < 0.5 (the surface leaves part of it).  Weights add
 * up per pixel; a is clamped to [0, 1].  A pixel the mesh does not cover and
 * a surface reaches takes that surface pixel's depth as its split depth.
 *   Inputs: face_id / mesh_depth / mesh_rgb of gm_zbuffer + gm_interp_mesh,
 *   adj of gm_mesh_edges.  Outputs [H][W]: cov (a), rgb_aa [H][W][3] (M),
 *   depth_aa (split depth, +inf where no mesh), and per tile tile_far (the
 *   largest split depth) / tile_full (every pixel has a = 1), which replace
 *   those of gm_interp_mesh for the occlusion cull.
 *   Decisions are taken in fp32 with the z-buffer's operations; the crossing
 *   t in double-float arithmetic (pairs of fp32 values, ~48 bits).
 * ---------------------------------------------------------------------- */
int gm_antialias(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                 const int32_t* adj, const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb,
                 float* cov, float* rgb_aa, float* depth_aa, float* tile_far, uint8_t* tile_full, void* stream);

/* ------------------------------------------------------------------------
 * gm_antialias_bwd -- gradients of gm_antialias: from dL/d(cov, rgb_aa,
 * depth_aa) (v_cov, v_rgb_aa, v_depth_aa [H][W], [H][W][3], [H][W], e.g. the
 * layer gradients of gm_composite_hybrid_bwd), given the forward call's cov
 * and depth_aa, to
 *   v_mesh_rgb [H][W][3], v_mesh_depth [H][W] (written): dL/d the
 *   interpolated colour and depth of each pixel, for gm_interp_mesh_bwd;
 *   v_verts [nV][3] (+=): dL/d the world positions of the silhouette edges'
 *   vertices through the crossings t (the weights' other dependence).
 *   Same mesh inputs as the forward call.  A weight that falls on a pixel
 *   whose coverage was clamped carries no coverage gradient.
 * ---------------------------------------------------------------------- */
int gm_antialias_bwd(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                     const int32_t* adj, const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb,
                     const float* cov, const float* depth_aa, const float* v_cov, const float* v_rgb_aa,
                     const float* v_depth_aa, float* v_mesh_rgb, float* v_mesh_depth, float* v_verts, void* stream);

/* ------------------------------------------------------------------------
 * gm_interp_mesh_bwd -- backward of gm_interp_mesh for given per-pixel
 * gradients v_mesh_rgb [H][W][3] and v_mesh_depth [H][W] of the interpolated
 * colour and depth (face ids held fixed): v_verts, v_vcol [nV][3] (+=).
 * ---------------------------------------------------------------------- */
int gm_interp_mesh_bwd(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                       const float* vcol, const int32_t* face_id, const float* v_mesh_rgb,
                       const float* v_mesh_depth, float* v_verts, float* v_vcol, void* stream);

/* ------------------------------------------------------------------------
 * gm_project_gaussians -- EWA projection and colour of each Gaussian
 * (Hybrid rendering; the 3DGS projection and SH kernels).  Inputs in the
 * stored parameterisation: means [N][3], log_scales [N][3], quats [N][4]
 * (w, x, y, z; normalised here), logits [N] (opacity = sigmoid), colors
 * [N][3] RGB (opts->sh_degree = -1) or [N][(d+1)^2][3] real SH coefficients
 * (rgb = max(0, sum Y_lm(view dir) c_lm + 0.5)).
 *   splats [N][12] f32 out, 16-byte aligned (layout above; all zero for a
 *   culled Gaussian).  radii [N] i32 out: ceil(3 sqrt(largest eigenvalue of
 *   the 2D covariance)), 0 = culled (behind near / beyond far, or its tile
 *   rectangle misses the image).  tiles_touched [N] i32 out: tiles in the
 *   rectangle [floor((m - r)/16), ceil((m + r)/16)) per axis, clamped.
 *   depth_model [N][4] f32 out, 16-byte aligned, or NULL: the soft split's
 *   depth model (g_u, g_v, sigma_z, R) of each Gaussian (Hybrid rendering:
 *   the depth given the pixel p is Gaussian with mean z*(p) = z_c + g .
 *   (p - mean2d) and standard deviation sigma_z); with the camera-frame
 *   covariance Sigma_c and the splat's Jacobian J, g = (J Sigma_c J^T +
 *   0.3 I)^-1 J Sigma_c e_z and sigma_z^2 = e_z^T Sigma_c e_z - (J Sigma_c
 *   e_z) . g, floored at 1e-12 (0.3: the splat's low-pass).  R >= 0, the
 *   reach, bounds g . (p - mean2d) over the pixels where the Gaussian's
 *   alpha can reach 1/255 (sqrt(2 ln(255 opacity) g^T Sigma2 g), with a
 *   margin); the compositing uses it only to skip Gaussians hidden behind
 *   the mesh (a depth model made elsewhere must bound the same, or hold
 *   +inf there).
 * ---------------------------------------------------------------------- */
int gm_project_gaussians(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* means,
                         const float* log_scales, const float* quats, const float* logits,
                         const float* colors, float* splats, int32_t* radii, int32_t* tiles_touched,
                         float* depth_model, void* stream);

/* ------------------------------------------------------------------------
 * gm_project_gaussians_bwd -- backward of gm_project_gaussians (Hybrid
 * rendering: everything is differentiable; the page's Gaussian kernels are
 * adapted from gsplat).  Given dL/d of each projected record, the chain rule
 * through the EWA projection and the SH colour:
 *   inputs: the same camera, opts, N and parameters as the forward call;
 *   radii [N] i32 from that call (radius 0 = culled: zero gradients);
 *   v_splats [N][12] f32, 16-byte aligned: dL/d record, e.g. the output of
 *   gm_composite_hybrid_bwd (the two padding floats are ignored).
 *   v_depth_model [N][4] f32, 16-byte aligned, or NULL: dL/d of the soft
 *   split's depth model (g_u, g_v, sigma_z, -), chained through g and
 *   sigma_z into the same parameters (no gradient where sigma_z^2 sits at
 *   its floor).
 *   v_means [N][3], v_log_scales [N][3], v_quats [N][4] (16-byte aligned),
 *   v_logits [N], v_colors (the layout of colors; 16-byte aligned for SH
 *   degree 1 and 3) f32 out: dL/d of each parameter, written when
 *   accumulate = 0, added (+=) when accumulate != 0 (e.g. over views).
 * Non-smooth points take these one-sided choices: a colour clamped at 0
 * passes no gradient; past the Jacobian's direction clamp the clamped
 * component is constant; the quaternion gradient is orthogonal to q (the
 * projection depends on q / |q| only).
 * ---------------------------------------------------------------------- */
int gm_project_gaussians_bwd(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* means,
                             const float* log_scales, const float* quats, const float* logits, const float* colors,
                             const int32_t* radii, const float* v_splats, const float* v_depth_model,
                             int32_t accumulate, float* v_means, float* v_log_scales, float* v_quats,
                             float* v_logits, float* v_colors, void* stream);

/* ------------------------------------------------------------------------
 * gm_bin_sort_gaussians -- tile intersection and sort (Hybrid rendering;
 * Limitations: Gaussians ordered by centre depth) with the per-tile cull
 * (Hybrid rendering, cull_occluded bullet: Gaussians certainly hidden behind
 * the mesh in fully covered tiles are removed; the image does not change).
 * Every (Gaussian, tile) pair of a rectangle gets the 64-bit key
 *   (tile id << 32) | bits(depth)
 * and the Gaussian id as value; with opts->cull_occluded a pair is dropped
 * when tile_full[tile] and depth >= tile_far[tile] (under the soft split,
 * opts->softness > 0: when the record's hide depth, field 10, exceeds
 * tile_far[tile] by more than 4e-6 relative -- the bound the soft
 * compositing itself skips by); with opts->tile_test a
 * pair is dropped when the smallest sigma over the tile's square of pixel
 * centres exceeds ln(255 opacity) by a margin (0.1 % + 1e-4): the Gaussian
 * cannot reach alpha >= 1/255 at any of those pixels, so the image and the
 * gradients do not change.  Keys are sorted ascending by a stable LSD radix
 * sort, so equal depths keep ascending ids.
 *   splats / radii: from gm_project_gaussians.  tile_far / tile_full: from
 *   gm_interp_mesh (read only when cull_occluded).
 *   keys [cap] u64 out, gids [cap] i32 out, tile_range [T][2] i32 out.
 *   counters [4] i32 out (device): GM_CNT_K, GM_CNT_K_PRECULL, flags.
 *   K_host, cap, ws: as for gm_bin_triangles.  GM_ERR_TIMEOUT is returned
 *   (K_host != NULL) when a bounded inter-block wait of the sort gave up.
 * ---------------------------------------------------------------------- */
size_t gm_bin_sort_gaussians_workspace_size(int32_t N, int32_t cap, int32_t width, int32_t height);
int gm_bin_sort_gaussians(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* splats,
                          const int32_t* radii, const float* tile_far, const uint8_t* tile_full,
                          uint64_t* keys, int32_t* gids, int32_t* tile_range, int32_t cap,
                          int32_t* counters, int32_t* K_host, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * gm_sort_gaussians_by_depth + gm_bin_gaussians -- gm_bin_sort_gaussians in
 * two halves, for callers that overlap the first with the mesh layer: the
 * depth pre-sort of the Gaussians (centre depth, ascending; ids break ties;
 * Gaussians whose tile rectangle is empty last), their tile rectangles and
 * the per-tile ellipse test need only splats / radii; the occlusion cull,
 * emission and tile sort need tile_far / tile_full.
 * Call both, in this order, with the same N, cap and workspace (nothing else
 * may use the workspace in between); the results equal gm_bin_sort_gaussians'.
 * gm_sort_gaussians_by_depth zeroes counters; gm_bin_gaussians reports the
 * entry count and flags there (and in K_host, as gm_bin_sort_gaussians).
 * ---------------------------------------------------------------------- */
int gm_sort_gaussians_by_depth(const gm_camera* cam, int32_t N, const float* splats, const int32_t* radii,
                               int32_t cap, int32_t* counters, void* ws, size_t ws_bytes, void* stream);
int gm_bin_gaussians(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* splats,
                     const int32_t* radii, const float* tile_far, const uint8_t* tile_full, uint64_t* keys,
                     int32_t* gids, int32_t* tile_range, int32_t cap, int32_t* counters, int32_t* K_host,
                     void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * gm_composite_hybrid_fwd -- Hybrid rendering, compositing with a hard
 * split: per pixel, front to back over its tile's sorted Gaussians, each
 * drawn only where its centre depth is in front of the mesh (z < D);
 *   sigma = (a dx^2 + c dy^2)/2 + b dx dy, d = pixel centre - mean (skip
 *   sigma < 0); alpha = min(0.99, opacity exp(-sigma)) (skip alpha < 1/255);
 *   stop before a Gaussian that would bring T to 1e-4 or below;
 *   C += alpha T rgb, Z += alpha T z, T *= 1 - alpha.
 * The opaque mesh is the terminal layer (covered = face_id >= 0):
 *   out_rgb = C + T (covered ? mesh_rgb : bg), out_depth = Z + T covered D,
 *   out_alpha = 1 - T (1 - covered).
 *   N: number of splat records; tile_range / gids come from
 *   gm_bin_sort_gaussians over the same splats (an id outside [0, N) is
 *   treated as an entry that draws nothing).
 *   Saved for the backward pass: T_final [H][W] f32 and n_contrib [H][W]
 *   i32 (1 + position in the tile's list of the last composited Gaussian).
 *   stats: NULL, or a device uint64[2] incremented by the number of
 *   (pixel, Gaussian) pairs evaluated [0] and composited [1] (profiling
 *   counts; the caller zeroes them).
 *   staged: NULL, or the staged-record buffer (gm_staged) this call fills
 *   for the backward pass; positions past staged->cap are neither written
 *   nor composited.
 * Soft split (opts->softness > 0; Hybrid rendering, the split at the mesh
 * surface): at a covered pixel there is no hard test; each Gaussian's part
 * in front of the mesh, f = Phi((D - z*(p)) / (sigma_z softness)) with
 * z*(p) = z + g . (p - mean2d) from depth_model [N][4] (gm_project_gaussians,
 * required, 16-byte aligned), scales its alpha: alpha f replaces alpha in the
 * skip, the stop and the sums (the back parts lie behind the opaque mesh).
 * Uncovered pixels are unchanged.  depth_model is ignored when softness = 0.
 * Antialiased layer (aa != NULL, aa->cov given; Hybrid rendering, the
 * two-layer equation): the mesh layer has coverage a = aa->cov in [0, 1],
 * premultiplied colour M = mesh_rgb and split depth D = mesh_depth (the
 * outputs of gm_antialias); Gaussians split at D composite in front of it
 * (the chain above) and, where 0 < a < 1, behind it in a second chain C_b,
 * Z_b, T_b (hard split: those at or behind D; soft split: alpha (1 - f)):
 *   out_rgb = C + T (M + (1 - a)(C_b + T_b bg)), out_depth = Z + T (a D +
 *   (1 - a) Z_b), out_alpha = 1 - T (1 - a) T_b.
 *   aa->back / T_back / n_back receive the back chain (read only where
 *   0 < a < 1 and D is finite).  face_id is not read.
 * opts->soft_split picks f = Phi (GM_SPLIT_PHI) or the logistic 1 / (1 +
 * exp(-1.702 x)) (GM_SPLIT_LOGISTIC) as the front fraction.
 * Each warp's 8 x 4 pixel block passes over the Gaussians with z_c - R -
 * t sigma_z softness beyond the largest mesh depth of its pixels (all
 * covered), t = 2.75 for Phi and 3.5 for the logistic: f(-t) puts alpha f
 * below 1/255 at each of them.
 * ---------------------------------------------------------------------- */
int gm_composite_hybrid_fwd(const gm_camera* cam, const gm_opts* opts, int32_t N,
                            const int32_t* tile_range, const int32_t* gids, const float* splats,
                            const float* depth_model, const float* mesh_depth, const float* mesh_rgb,
                            const int32_t* face_id, float* out_rgb, float* out_depth, float* out_alpha,
                            float* T_final, int32_t* n_contrib, const gm_aa_layer* aa, const gm_staged* staged,
                            uint64_t* stats, void* stream);

/* ------------------------------------------------------------------------
 * gm_composite_hybrid_bwd -- Hybrid rendering ("everything is
 * differentiable"): gradients of L = sum g_rgb . out_rgb + g_depth out_depth
 * + g_alpha out_alpha, given the saved T_final / n_contrib of the forward
 * pass over the same inputs.
 *   v_splats [N][12] f32 (+=, 16-byte aligned): dL/d mean2d, conic, opacity,
 *   rgb, depth of each Gaussian (the hard depth test, the skips and the sort
 *   carry no gradient; alpha clamped at 0.99 has none w.r.t. opacity/conic).
 *   Sums are added with 16-byte vector atomics; the two padding floats of a
 *   row receive += 0.  Summation order varies between runs (last-bit noise).
 *   v_verts [nV][3], v_vcol [nV][3] f32 (+=): dL/d vertex world position and
 *   colour through the interpolated mesh depth and colour of covered pixels
 *   (face ids held fixed).  V / F / vcol / v_verts / v_vcol may all be NULL
 *   (with nV = nF = 0) to skip the mesh gradients.
 *   stats: NULL, or a device uint64[2] incremented by the number of (pixel,
 *   Gaussian) pairs evaluated [0] and given gradient terms [1] (profiling).
 *   staged: NULL (each batch of a tile's list is gathered through gids), or
 *   the buffer the forward call filled (gm_staged): with the hard split each
 *   warp then loads the records of its hit lists (the next group's loads in
 *   flight while it works on the current one); with the soft split each batch
 *   arrives by bulk copies, the next one in flight while the current one is
 *   worked on.  The Gaussian part reads it; the mesh part does not.
 *   Soft split (opts->softness > 0): depth_model as for the forward pass;
 *   v_depth_model [N][4] f32 (+=, 16-byte aligned, required with v_splats):
 *   dL/d(g_u, g_v, sigma_z, -); v_mesh_depth [H][W] f32 (required with the
 *   mesh gradients): dL/dD through the split, written by the Gaussian part
 *   (v_splats != NULL) and read by the mesh part (v_verts != NULL), so a
 *   call with only the mesh part must follow one with the Gaussian part.
 *   Antialiased layer (aa as for the forward, with aa->back / T_back / n_back
 *   as the forward wrote them): the Gaussian gradients of both chains; the
 *   layer's gradients aa->v_cov (dL/da), aa->v_rgb (dL/dM) and, in
 *   v_mesh_depth (required), dL/dD (the depth output and the soft split) --
 *   the input of gm_antialias_bwd; the mesh arguments must then be NULL
 *   (the mesh gradients come from gm_antialias_bwd and gm_interp_mesh_bwd).
 * ---------------------------------------------------------------------- */
int gm_composite_hybrid_bwd(const gm_camera* cam, const gm_opts* opts, int32_t N,
                            const int32_t* tile_range, const int32_t* gids, const float* splats,
                            const float* depth_model, const float* mesh_depth, const float* mesh_rgb,
                            const int32_t* face_id, const float* T_final, const int32_t* n_contrib,
                            const float* g_rgb, const float* g_depth, const float* g_alpha, float* v_splats,
                            float* v_depth_model, float* v_mesh_depth, const float* V, int32_t nV,
                            const int32_t* F, int32_t nF, const float* vcol, float* v_verts,
                            float* v_vcol, const gm_aa_layer* aa, const gm_staged* staged, uint64_t* stats,
                            void* stream);

/* ------------------------------------------------------------------------
 * Batched views (several cameras of one scene, e.g. the views of a training
 * batch): the projection and its backward for V cameras in one call.  Each
 * thread takes one Gaussian through every view, so its parameters are read
 * from memory once, and the backward sums the views' gradients in registers
 * (in view order, the order in which per-view calls with accumulate = 1
 * would add them) before writing once.  The per-view steps between the two
 * (binning, z-buffer, compositing) take one view's slice of these arrays.
 *   cams [V] host array, 1 <= V <= GM_MAX_VIEWS.
 *   gm_project_gaussians_views: as gm_project_gaussians for every view;
 *   splats [V][N][12], radii [V][N], tiles_touched [V][N], depth_model
 *   [V][N][4] (or NULL) out (view v at offset v N).
 *   gm_project_gaussians_bwd_views: as gm_project_gaussians_bwd with radii
 *   [V][N] and v_splats [V][N][12] from the views; the parameter gradients
 *   are the sum over the views (written, or added when accumulate != 0),
 *   summed in view order within each group of 8 views, the groups added in
 *   order (so up to 8 views the result is that of per-view calls).
 * ---------------------------------------------------------------------- */
#define GM_MAX_VIEWS 64
int gm_project_gaussians_views(const gm_camera* cams, int32_t V, const gm_opts* opts, int32_t N, const float* means,
                               const float* log_scales, const float* quats, const float* logits, const float* colors,
                               float* splats, int32_t* radii, int32_t* tiles_touched, float* depth_model,
                               void* stream);
int gm_project_gaussians_bwd_views(const gm_camera* cams, int32_t V, const gm_opts* opts, int32_t N,
                                   const float* means, const float* log_scales, const float* quats,
                                   const float* logits, const float* colors, const int32_t* radii,
                                   const float* v_splats, const float* v_depth_model, int32_t accumulate,
                                   float* v_means, float* v_log_scales, float* v_quats, float* v_logits,
                                   float* v_colors, void* stream);

/* ------------------------------------------------------------------------
 * gm_bin_triangles_noalloc -- gm_bin_triangles for callers that may not
 * allocate device memory at all (a plugin or engine inside a host
 * application that owns all device memory through its own pool and budget,
 * so a library cudaMalloc would fail against that budget or stall the
 * device).  The paper has no counterpart: this is a packaging of the same
 * triangle binning.  The caller still passes V, F and the outputs; the
 * scratch memory is a static device array of GM_NOALLOC_TRI_SCRATCH_BYTES
 * that every GPU loading libgm holds until the process exits.  Calls whose
 * gm_bin_triangles_workspace_size(nF, cap, ...) exceeds that size are
 * rejected with GM_ERR_INVALID_ARG (message in gm_last_error).  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress,
 * then cached per device), so make that first call before any stream
 * capture.  All calls share the one array (each call clears what must start
 * at zero): calls that overlap on the GPU -- concurrent streams or host
 * threads -- race and corrupt each other's results.  The cached address
 * belongs to the device's context at the first call: it does not survive
 * cudaDeviceReset (or any reset of the primary context), after which this
 * entry point must not be called again in the same process.  Everything else as
 * gm_bin_triangles; no cudaMalloc / cudaFree or allocating library call.
 * ---------------------------------------------------------------------- */
#define GM_NOALLOC_TRI_SCRATCH_BYTES (32u << 20)
int gm_bin_triangles_noalloc(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F,
                             int32_t nF, int32_t* tile_range, int32_t* tri_ids, int32_t cap,
                             int32_t* counters, int32_t* K_host, void* stream);

/* ----------------------------------------------------------------------
 * gm_set_wait_limit / gm_get_wait_limit -- the bound on the inter-block waits
 * of the scans and radix sorts (the decoupled look-back of gm_bin_triangles,
 * gm_bin_sort_gaussians, gm_sort_gaussians_by_depth, gm_bin_gaussians and
 * gm_mesh_edges).  A waiting block polls its predecessor's descriptor at
 * most `polls` times (default GM_WAIT_LIMIT_DEFAULT), then sets
 * GM_FLAG_TIMEOUT in the call's counters and carries on with a prefix that is
 * at most the true one, so every write stays inside the caller's buffers;
 * the call's result is then not a valid sort (GM_ERR_TIMEOUT with K_host).
 * The pages have no counterpart: this exists to test the failure path (a
 * limit of 0 makes any block that finds its predecessor unpublished give up).
 * The setting is process-wide, holds until changed and is read when a call
 * enqueues its kernels (a captured CUDA graph keeps the value it was captured
 * with).  Host-only, no device work.  Errors: GM_ERR_INVALID_ARG for a NULL
 * `polls`.
 * ---------------------------------------------------------------------- */
#define GM_WAIT_LIMIT_DEFAULT (1u << 22)
int gm_set_wait_limit(uint32_t polls);
int gm_get_wait_limit(uint32_t* polls);

/* Message describing the calling thread's last failure ("" if none). */
const char* gm_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* GM_H */

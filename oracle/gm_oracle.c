/*
 * gm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU restatement of the hybrid mesh + 3D Gaussian renderer
 * described on the page "A Lightweight and Differentiable Renderer for Joint
 * Mesh and 3D Gaussian Splat Scenes" (Design Details: Mesh rasterizer,
 * Hybrid rendering; Limitations and Todos).  Only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark load it; the CUDA library never
 * does, and the two share no code.
 *
 * What it computes, step by step, with no tiling, fusion or reordering
 * beyond what each definition states:
 *   - triangle tile bins and a brute-force z-buffer that tests every pixel
 *     centre against every triangle (Mesh rasterizer, item 1);
 *   - perspective-correct depth and vertex colour at each pixel from its
 *     face id (Mesh rasterizer, item 2);
 *   - EWA projection of each Gaussian, SH colour (Hybrid rendering; the
 *     projection / SH kernels the page says are adapted from gsplat);
 *   - Gaussian tile bins, sorted by (tile, centre depth, id), with the
 *     per-tile occlusion cull (Hybrid rendering, cull_occluded bullet;
 *     Limitations: Gaussians sorted by centre depth);
 *   - per-pixel front-to-back compositing over the full, fully sorted list
 *     of Gaussians whose tile rectangle holds the pixel, each depth-tested
 *     against the mesh, the mesh colour as the terminal layer (Hybrid
 *     rendering, compositing equation with a hard split);
 *   - gradients by central finite differences in double precision, with
 *     every discrete decision (face ids, tile lists, skips, clamps, the
 *     transmittance cut-off, the depth test) held fixed, and any parameter
 *     whose perturbation flips one of them reported instead of used.
 *
 * Precision.  Every integer the method decides from floating point (face
 * ids, coverage, tile rectangles, radii, skips, the transmittance stop) is
 * decided in fp32, the precision the renderer works in, one correctly
 * rounded operation at a time in the order the formula is written (build
 * with -ffp-contract=off: no fused multiply-add).  Continuous values that
 * feed no decision (interpolated depth and colour, conics, means, colours,
 * colour and depth sums) are computed in double.  The compositing routine
 * runs in either mode: "f32" rounds sigma, alpha and transmittance to fp32
 * after every operation (an fp32 result of +, -, *, / or sqrt computed in
 * double and rounded once is the correctly rounded fp32 result), "f64"
 * keeps everything in double for finite differences.
 *
 * Parity unpinned (the page fixes none of these; each is a stated reading):
 * the gsplat constants (0.3 px low-pass, 1.3 x half-FOV clamp of the
 * Jacobian, 3-sigma radius), the real-SH sign convention, the depth/alpha
 * output definitions and the camera axes.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TILE 16
#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif
#ifndef M_SQRT1_2
#define M_SQRT1_2 0.70710678118654752440
#endif

typedef struct {
    int32_t width, height;
    float fx, fy, cx, cy, near_plane, far_plane;
    float R[9]; /* world -> camera rotation, row-major (OpenCV axes) */
    float t[3];
} orc_camera;

static int n_tiles_x(const orc_camera* c) { return (c->width + TILE - 1) / TILE; }
static int n_tiles_y(const orc_camera* c) { return (c->height + TILE - 1) / TILE; }

/* splat record: the projected 2D Gaussian, 12 floats */
enum { S_MX = 0, S_MY, S_CA, S_CB, S_CC, S_OP, S_R, S_G, S_B, S_Z, S_STRIDE = 12 };

/* ========================================================================
 * Mesh rasterizer, item 1: triangle bins and the z-buffer (fp32 decisions)
 * ====================================================================== */

/* X_c = R X + t, each row summed left to right, one rounding per operation */
static void world_to_cam_f32(const orc_camera* c, const float* X, float* xc)
{
    for (int r = 0; r < 3; ++r) {
        float s = c->R[3 * r + 0] * X[0];
        s = s + c->R[3 * r + 1] * X[1];
        s = s + c->R[3 * r + 2] * X[2];
        xc[r] = s + c->t[r];
    }
}

/* edge function of the directed edge a->b at point p:
 *   (ub - ua)(py - va) - (vb - va)(px - ua)                                */
static float edge_f32(float ua, float va, float ub, float vb, float px, float py)
{
    float p = (ub - ua) * (py - va);
    float q = (vb - va) * (px - ua);
    return p - q;
}

typedef struct {
    float u[3], v[3], z[3];
    float area; /* edge function of v0->v1 at v2: twice the signed area */
    int x0, x1, y0, y1; /* inclusive pixel-centre box, clamped to the image */
} tri32;

/* Returns 1 when the triangle is drawn: every vertex strictly beyond the near
 * plane (triangles with a vertex in front of it are skipped, no clipping:
 * Mesh rasterizer, last paragraph; Limitations), a non-zero area, and a
 * non-empty box of pixel centres (i + 0.5, j + 0.5) inside the image.   */
static int tri_setup_f32(const orc_camera* c, const float* V, const int32_t* F, int f, tri32* t)
{
    for (int k = 0; k < 3; ++k) {
        float xc[3];
        world_to_cam_f32(c, V + 3 * (int64_t)F[3 * f + k], xc);
        if (!(xc[2] > c->near_plane))
            return 0;
        t->z[k] = xc[2];
        t->u[k] = (c->fx * xc[0]) / xc[2] + c->cx;
        t->v[k] = (c->fy * xc[1]) / xc[2] + c->cy;
    }
    t->area = edge_f32(t->u[0], t->v[0], t->u[1], t->v[1], t->u[2], t->v[2]);
    if (!(t->area != 0.0f))
        return 0;
    float umin = fminf(fminf(t->u[0], t->u[1]), t->u[2]);
    float umax = fmaxf(fmaxf(t->u[0], t->u[1]), t->u[2]);
    float vmin = fminf(fminf(t->v[0], t->v[1]), t->v[2]);
    float vmax = fmaxf(fmaxf(t->v[0], t->v[1]), t->v[2]);
    float x0 = fmaxf(ceilf(umin - 0.5f), 0.0f);
    float x1 = fminf(floorf(umax - 0.5f), (float)(c->width - 1));
    float y0 = fmaxf(ceilf(vmin - 0.5f), 0.0f);
    float y1 = fminf(floorf(vmax - 0.5f), (float)(c->height - 1));
    if (!(x0 <= x1) || !(y0 <= y1))
        return 0;
    t->x0 = (int)x0; t->x1 = (int)x1; t->y0 = (int)y0; t->y1 = (int)y1;
    return 1;
}

/* coverage of pixel (i, j) and, when covered, its depth D = 1 / sum_k (l_k / z_k)
 * with screen barycentrics l_k = e_k / area.  Inclusive edges, both windings. */
static int tri_cover_f32(const tri32* t, int i, int j, float* D)
{
    if (i < t->x0 || i > t->x1 || j < t->y0 || j > t->y1)
        return 0;
    float px = (float)i + 0.5f, py = (float)j + 0.5f;
    float e0 = edge_f32(t->u[1], t->v[1], t->u[2], t->v[2], px, py);
    float e1 = edge_f32(t->u[2], t->v[2], t->u[0], t->v[0], px, py);
    float e2 = edge_f32(t->u[0], t->v[0], t->u[1], t->v[1], px, py);
    int in = t->area > 0.0f ? (e0 >= 0.0f && e1 >= 0.0f && e2 >= 0.0f)
                            : (e0 <= 0.0f && e1 <= 0.0f && e2 <= 0.0f);
    if (!in)
        return 0;
    float l0 = e0 / t->area, l1 = e1 / t->area, l2 = e2 / t->area;
    float s = l0 / t->z[0];
    s = s + l1 / t->z[1];
    s = s + l2 / t->z[2];
    *D = 1.0f / s;
    return 1;
}

/* Triangle tile bins: tile (tx, ty) holds every drawn triangle whose pixel-
 * centre box meets it; within a tile, face ids ascend.  Returns the number of
 * (triangle, tile) entries; fills tile_count[T] and, when ids != NULL and the
 * total fits in cap, the tile-major list of face ids.                      */
int64_t orc_bin_triangles(const orc_camera* c, const float* V, const int32_t* F, int32_t nF,
                          int32_t* tile_count, int32_t* ids, int64_t cap)
{
    int TW = n_tiles_x(c), TH = n_tiles_y(c);
    int64_t T = (int64_t)TW * TH;
    memset(tile_count, 0, sizeof(int32_t) * T);
    int64_t total = 0;
    for (int f = 0; f < nF; ++f) {
        tri32 t;
        if (!tri_setup_f32(c, V, F, f, &t))
            continue;
        for (int ty = t.y0 / TILE; ty <= t.y1 / TILE; ++ty)
            for (int tx = t.x0 / TILE; tx <= t.x1 / TILE; ++tx) {
                tile_count[(int64_t)ty * TW + tx]++;
                total++;
            }
    }
    if (!ids || total > cap)
        return total;
    int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (T + 1));
    fill[0] = 0;
    for (int64_t k = 0; k < T; ++k)
        fill[k + 1] = fill[k] + tile_count[k];
    for (int f = 0; f < nF; ++f) {
        tri32 t;
        if (!tri_setup_f32(c, V, F, f, &t))
            continue;
        for (int ty = t.y0 / TILE; ty <= t.y1 / TILE; ++ty)
            for (int tx = t.x0 / TILE; tx <= t.x1 / TILE; ++tx)
                ids[fill[(int64_t)ty * TW + tx]++] = f;
    }
    free(fill);
    (void)TH;
    return total;
}

/* Brute-force z-buffer: every listed pixel (all pixels when pixels == NULL)
 * against every triangle.  The nearest depth wins, equal depths go to the
 * smaller face id.  Also returns the nearest depth and the nearest depth of
 * any other covering face (+inf if none), so near-ties can be reported.   */
void orc_zbuffer(const orc_camera* c, const float* V, const int32_t* F, int32_t nF,
                 const int32_t* pixels, int64_t n_pixels,
                 int32_t* face_id, float* best_depth, float* second_depth)
{
    tri32* tris = (tri32*)malloc(sizeof(tri32) * (nF > 0 ? nF : 1));
    uint8_t* ok = (uint8_t*)malloc(nF > 0 ? nF : 1);
    for (int f = 0; f < nF; ++f)
        ok[f] = (uint8_t)tri_setup_f32(c, V, F, f, &tris[f]);
    int64_t np = pixels ? n_pixels : (int64_t)c->width * c->height;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t k = 0; k < np; ++k) {
        int64_t pix = pixels ? pixels[k] : k;
        int i = (int)(pix % c->width), j = (int)(pix / c->width);
        int best = -1;
        float bd = INFINITY, sd = INFINITY;
        for (int f = 0; f < nF; ++f) {
            float D;
            if (!ok[f] || !tri_cover_f32(&tris[f], i, j, &D))
                continue;
            if (best < 0 || D < bd) {
                if (best >= 0) sd = fminf(sd, bd);
                bd = D;
                best = f;
            } else {
                sd = fminf(sd, D);
            }
        }
        face_id[k] = best;
        best_depth[k] = bd;
        second_depth[k] = sd;
    }
    free(tris);
    free(ok);
}

/* ========================================================================
 * Mesh rasterizer, item 2: perspective-correct depth and colour (double)
 * ====================================================================== */

typedef struct {
    double u[3], v[3], z[3];
} tri64;

static void tri_setup_f64(const orc_camera* c, const double X[3][3], tri64* t)
{
    for (int k = 0; k < 3; ++k) {
        double xc[3];
        for (int r = 0; r < 3; ++r)
            xc[r] = (double)c->R[3 * r + 0] * X[k][0] + (double)c->R[3 * r + 1] * X[k][1] +
                    (double)c->R[3 * r + 2] * X[k][2] + (double)c->t[r];
        t->z[k] = xc[2];
        t->u[k] = (double)c->fx * xc[0] / xc[2] + (double)c->cx;
        t->v[k] = (double)c->fy * xc[1] / xc[2] + (double)c->cy;
    }
}

static double edge_f64(double ua, double va, double ub, double vb, double px, double py)
{
    return (ub - ua) * (py - va) - (vb - va) * (px - ua);
}

/* depth D and weights w_k at pixel centre (px, py) of a triangle given by its
 * camera-space vertices:  l_k = e_k / area,  D = 1 / sum_k l_k / z_k,
 * w_k = (l_k / z_k) D, so the colour is sum_k w_k c_k.                     */
static void interp_f64(const tri64* t, double px, double py, double* D, double w[3])
{
    double area = edge_f64(t->u[0], t->v[0], t->u[1], t->v[1], t->u[2], t->v[2]);
    double e[3];
    e[0] = edge_f64(t->u[1], t->v[1], t->u[2], t->v[2], px, py);
    e[1] = edge_f64(t->u[2], t->v[2], t->u[0], t->v[0], px, py);
    e[2] = edge_f64(t->u[0], t->v[0], t->u[1], t->v[1], px, py);
    double q[3], s = 0.0;
    for (int k = 0; k < 3; ++k) {
        q[k] = (e[k] / area) / t->z[k];
        s += q[k];
    }
    *D = 1.0 / s;
    for (int k = 0; k < 3; ++k)
        w[k] = q[k] / s;
}

static void load_tri(const float* V, const int32_t* F, int f, double X[3][3])
{
    for (int k = 0; k < 3; ++k)
        for (int d = 0; d < 3; ++d)
            X[k][d] = V[3 * (int64_t)F[3 * f + k] + d];
}

/* Interpolated mesh depth and colour for the listed pixels (all when NULL).
 * Uncovered pixels: depth +inf, colour 0.  Per tile (only tiles whose pixels
 * are all listed, tile_flags[t] = 1 on input): tile_full = every in-image
 * pixel covered, tile_far = the largest fp32 mesh depth over the tile.     */
void orc_interp_mesh(const orc_camera* c, const float* V, const int32_t* F, const float* vcol,
                     const int32_t* pixels, int64_t n_pixels, const int32_t* face_id,
                     float* mesh_depth, float* mesh_rgb)
{
    int64_t np = pixels ? n_pixels : (int64_t)c->width * c->height;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < np; ++k) {
        int64_t pix = pixels ? pixels[k] : k;
        int i = (int)(pix % c->width), j = (int)(pix / c->width);
        int f = face_id[k];
        if (f < 0) {
            mesh_depth[k] = INFINITY;
            mesh_rgb[3 * k] = mesh_rgb[3 * k + 1] = mesh_rgb[3 * k + 2] = 0.0f;
            continue;
        }
        double X[3][3], D, w[3];
        tri64 t;
        load_tri(V, F, f, X);
        tri_setup_f64(c, X, &t);
        interp_f64(&t, i + 0.5, j + 0.5, &D, w);
        mesh_depth[k] = (float)D;
        for (int ch = 0; ch < 3; ++ch) {
            double s = 0.0;
            for (int v = 0; v < 3; ++v)
                s += w[v] * vcol[3 * (int64_t)F[3 * f + v] + ch];
            mesh_rgb[3 * k + ch] = (float)s;
        }
    }
}

/* tile_full / tile_far from a full-frame mesh depth image (fp32 values). */
void orc_tile_depth_bounds(const orc_camera* c, const float* mesh_depth, float* tile_far,
                           uint8_t* tile_full)
{
    int TW = n_tiles_x(c), TH = n_tiles_y(c);
    for (int ty = 0; ty < TH; ++ty)
        for (int tx = 0; tx < TW; ++tx) {
            float far = -INFINITY;
            int full = 1;
            for (int j = ty * TILE; j < ty * TILE + TILE && j < c->height; ++j)
                for (int i = tx * TILE; i < tx * TILE + TILE && i < c->width; ++i) {
                    float d = mesh_depth[(int64_t)j * c->width + i];
                    if (!(d < INFINITY)) full = 0;
                    if (d > far) far = d;
                }
            tile_far[ty * TW + tx] = full ? far : INFINITY;
            tile_full[ty * TW + tx] = (uint8_t)full;
        }
}

/* ========================================================================
 * Mesh rasterizer, item 3: analytic edge antialiasing at silhouettes
 * ====================================================================== */

/* Edge k of face f joins its corners k+1 and k+2 (mod 3), the edge opposite
 * corner k (the edge function e_k of the coverage test).  adj[3 f + k] is the
 * other face with the same two vertices, -1 when there is none, -2 when more
 * than two faces share them.                                              */
typedef struct {
    uint64_t key;
    int32_t fe;
} edge_rec;

static int edge_rec_cmp(const void* a, const void* b)
{
    const edge_rec* x = (const edge_rec*)a;
    const edge_rec* y = (const edge_rec*)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return (x->fe > y->fe) - (x->fe < y->fe);
}

void orc_mesh_edges(const int32_t* F, int32_t nF, int32_t* adj)
{
    int64_t n = 3 * (int64_t)nF;
    edge_rec* e = (edge_rec*)malloc(sizeof(edge_rec) * (n > 0 ? n : 1));
    for (int f = 0; f < nF; ++f)
        for (int k = 0; k < 3; ++k) {
            uint32_t a = (uint32_t)F[3 * f + (k + 1) % 3], b = (uint32_t)F[3 * f + (k + 2) % 3];
            uint32_t lo = a < b ? a : b, hi = a < b ? b : a;
            e[3 * f + k].key = ((uint64_t)lo << 32) | hi;
            e[3 * f + k].fe = 3 * f + k;
        }
    qsort(e, (size_t)n, sizeof(edge_rec), edge_rec_cmp);
    for (int64_t i = 0; i < n;) {
        int64_t j = i;
        while (j < n && e[j].key == e[i].key) ++j;
        for (int64_t q = i; q < j; ++q)
            adj[e[q].fe] = j - i == 1 ? -1 : (j - i == 2 ? e[i + j - 1 - q].fe / 3 : -2);
        i = j;
    }
    free(e);
}

/* The mesh as the antialiasing sees it: vertices (one of them optionally
 * moved by delta along one axis, for finite differences), faces, adjacency,
 * the z-buffer's face ids, and the interpolated depth and colour per pixel
 * (fp32 images, with optional double values overriding a sorted pixel set). */
typedef struct {
    const orc_camera* c;
    const float* V;
    const int32_t* F;
    const int32_t* adj;
    const int32_t* face_id;
    const float* depth;
    const float* rgb;
    int pvid, pfield;
    double pdelta;
    const int64_t* ov_pix;
    const double* ov_depth;
    const double* ov_rgb;
    int64_t n_ov;
} aa_view;

static int64_t aa_find(const aa_view* w, int64_t pix)
{
    int64_t lo = 0, hi = w->n_ov;
    while (lo < hi) {
        int64_t mid = (lo + hi) / 2;
        if (w->ov_pix[mid] < pix) lo = mid + 1;
        else hi = mid;
    }
    return lo < w->n_ov && w->ov_pix[lo] == pix ? lo : -1;
}

static double aa_depth(const aa_view* w, int64_t pix)
{
    int64_t k = w->n_ov ? aa_find(w, pix) : -1;
    return k >= 0 ? w->ov_depth[k] : (double)w->depth[pix];
}

static void aa_rgb(const aa_view* w, int64_t pix, double c[3])
{
    int64_t k = w->n_ov ? aa_find(w, pix) : -1;
    for (int ch = 0; ch < 3; ++ch) c[ch] = k >= 0 ? w->ov_rgb[3 * k + ch] : (double)w->rgb[3 * pix + ch];
}

/* screen position (u, v) of vertex vid: fp32 one rounding per operation in
 * the rasterizer's order (f32 = 1; the vertex must be unmoved), or double.
 * Returns 0 when the vertex is not beyond the near plane.                */
static int aa_vertex(const aa_view* w, int f32, int vid, double* u, double* v)
{
    const orc_camera* c = w->c;
    if (f32) {
        float xc[3];
        world_to_cam_f32(c, w->V + 3 * (int64_t)vid, xc);
        if (!(xc[2] > c->near_plane)) return 0;
        *u = (float)((c->fx * xc[0]) / xc[2] + c->cx);
        *v = (float)((c->fy * xc[1]) / xc[2] + c->cy);
        return 1;
    }
    double X[3];
    for (int d = 0; d < 3; ++d)
        X[d] = (double)w->V[3 * (int64_t)vid + d] + (vid == w->pvid && d == w->pfield ? w->pdelta : 0.0);
    double xc[3];
    for (int r = 0; r < 3; ++r)
        xc[r] = (double)c->R[3 * r] * X[0] + (double)c->R[3 * r + 1] * X[1] + (double)c->R[3 * r + 2] * X[2] +
                (double)c->t[r];
    if (!(xc[2] > (double)c->near_plane)) return 0;
    *u = (double)c->fx * xc[0] / xc[2] + (double)c->cx;
    *v = (double)c->fy * xc[1] / xc[2] + (double)c->cy;
    return 1;
}

static double aa_edge(int f32, double ua, double va, double ub, double vb, double px, double py)
{
    if (f32) return edge_f32((float)ua, (float)va, (float)ub, (float)vb, (float)px, (float)py);
    return edge_f64(ua, va, ub, vb, px, py);
}

/* faces the walk below may cross before it gives up */
#define AA_WALK 8

/* One pair of neighbouring pixels p and q (Mesh rasterizer, item 3): where
 * they see different faces, the nearer of the two surfaces (smaller mesh
 * depth; none when equal) is the occluder o, whose face A covers o's centre.
 * The segment from o's centre to the other centre is followed through the
 * surface: it leaves the current face through the edge with the smallest
 * crossing t_k = e_k(o) / (e_k(o) - e_k(other)) among those its far end lies
 * outside of (ties: smaller k; the edge it entered by is skipped); across an
 * internal edge -- one other face shares it and lies on the other side of
 * the edge in the image -- it goes on into that face (at most AA_WALK faces);
 * at a silhouette edge -- no other face, more than one, or one folded onto
 * the same side -- it stops, and the crossing t in [0, 1] gives the weight
 * w = |t - 0.5| on one pixel: the other one when t >= 0.5 (the surface
 * reaches into it), o when t < 0.5 (it leaves part of o).  A pair along x
 * only takes a silhouette edge more vertical than horizontal in the image
 * (|dv| > |du|), a pair along y only the others (the per-axis 1D model counts
 * each edge along one axis).  Decisions are taken in fp32 (f32 = 1) or
 * double; the returned t is evaluated in double.  Returns 0 (nothing), else
 * 1 with *occ = o's pixel, *t and a code naming the silhouette edge and the
 * side.                                                                   */
static int aa_pair(const aa_view* w, int f32, int64_t pp, int64_t pq, int64_t* occ, double* t_out, int* code)
{
    const orc_camera* c = w->c;
    int fp = w->face_id[pp], fq = w->face_id[pq];
    if (fp == fq) return 0;
    double Dp = fp >= 0 ? aa_depth(w, pp) : INFINITY, Dq = fq >= 0 ? aa_depth(w, pq) : INFINITY;
    if (f32) {
        Dp = (float)Dp;
        Dq = (float)Dq;
    }
    int64_t o, nb;
    if (Dp < Dq) { o = pp; nb = pq; }
    else if (Dq < Dp) { o = pq; nb = pp; }
    else return 0;
    double ox = (double)(o % c->width) + 0.5, oy = (double)(o / c->width) + 0.5;
    double nx = (double)(nb % c->width) + 0.5, ny = (double)(nb / c->width) + 0.5;
    int X = w->face_id[o], entry = -1, exit_k = -1;
    double u[3], v[3], best = INFINITY;
    for (int step = 0;; ++step) {
        if (step == AA_WALK) return 0;
        for (int k = 0; k < 3; ++k)
            if (!aa_vertex(w, f32, w->F[3 * X + k], &u[k], &v[k])) return 0;
        double area = aa_edge(f32, u[0], v[0], u[1], v[1], u[2], v[2]);
        double sgn = area > 0.0 ? 1.0 : -1.0;
        exit_k = -1;
        best = INFINITY;
        for (int k = 0; k < 3; ++k) {
            if (k == entry) continue;
            int a = (k + 1) % 3, b = (k + 2) % 3;
            double eo = aa_edge(f32, u[a], v[a], u[b], v[b], ox, oy);
            double en = aa_edge(f32, u[a], v[a], u[b], v[b], nx, ny);
            if (step == 0 && sgn * eo < 0.0) return 0; /* A no longer covers o's centre */
            if (!(sgn * en < 0.0)) continue;
            if (sgn * eo < 0.0) return 0; /* the segment misses this face */
            double tk = f32 ? (double)((float)eo / ((float)eo - (float)en)) : eo / (eo - en);
            if (tk < best) {
                best = tk;
                exit_k = k;
            }
        }
        if (exit_k < 0) return 0; /* the other centre lies on the surface */
        int a = (exit_k + 1) % 3, b = (exit_k + 2) % 3;
        int nf = w->adj[3 * X + exit_k];
        if (nf < 0) break;
        int va_ = w->F[3 * X + a], vb_ = w->F[3 * X + b], third = -1, back = -1;
        for (int k = 0; k < 3; ++k) {
            int vk = w->F[3 * nf + k];
            if (vk != va_ && vk != vb_) { third = vk; back = k; }
        }
        double u3, v3;
        if (third < 0 || !aa_vertex(w, f32, third, &u3, &v3)) break;
        double sX = aa_edge(f32, u[a], v[a], u[b], v[b], u[exit_k], v[exit_k]);
        double sN = aa_edge(f32, u[a], v[a], u[b], v[b], u3, v3);
        if (!(sX * sN < 0.0)) break; /* folded onto the same side: a silhouette */
        X = nf;                       /* the surface goes on across the edge */
        entry = back;
    }
    int a = (exit_k + 1) % 3, b = (exit_k + 2) % 3;
    {
        double du = f32 ? (double)((float)u[b] - (float)u[a]) : u[b] - u[a];
        double dv = f32 ? (double)((float)v[b] - (float)v[a]) : v[b] - v[a];
        int along_x = (o / c->width) == (nb / c->width);
        if (along_x != (fabs(dv) > fabs(du))) return 0;
    }
    /* the crossing in double */
    double ud[3], vd[3];
    for (int k = 0; k < 3; ++k)
        if (!aa_vertex(w, 0, w->F[3 * X + k], &ud[k], &vd[k])) return 0;
    double eo = edge_f64(ud[a], vd[a], ud[b], vd[b], ox, oy);
    double en = edge_f64(ud[a], vd[a], ud[b], vd[b], nx, ny);
    double t = eo / (eo - en);
    t = t < 0.0 ? 0.0 : (t > 1.0 ? 1.0 : t);
    *occ = o;
    *t_out = t;
    *code = 2 * (3 * X + exit_k + 1) + (best >= 0.5 ? 1 : 0);
    return 1;
}

/* The antialiased mesh layer of pixel (i, j): coverage a, premultiplied colour
 * M and the depth D the Gaussians are split at.  Without antialiasing the
 * layer is a0 = covered, M0 = a0 c, D.  Each of the pixel's four pairs whose
 * weight falls on it moves the layer towards the other pixel's by w (colours
 * and coverage of both as they were before any pair):
 *   onto the occluder o:   (a, M) += w ((a0, M0)(other) - (1, c_o)),
 *   onto the other pixel:  (a, M) += w ((1, c_o) - (a0, M0)(other)),
 * and a pixel the mesh does not cover takes the depth of the nearest
 * occluder that reaches into it (w > 0).  a is clamped to [0, 1] (two pairs
 * can act on one pixel near corners).  codes (optional) get each pair's
 * decision code (left, right, up, down), 0 when it does nothing here.     */
static void aa_pixel(const aa_view* w, int f32, int i, int j, double* a_out, double M[3], double* D_out,
                     int codes[4])
{
    const orc_camera* c = w->c;
    int64_t pp = (int64_t)j * c->width + i;
    int cov = w->face_id[pp] >= 0;
    double cp[3];
    aa_rgb(w, pp, cp);
    double a = cov ? 1.0 : 0.0;
    for (int ch = 0; ch < 3; ++ch) M[ch] = cov ? cp[ch] : 0.0;
    double Dp = cov ? aa_depth(w, pp) : INFINITY, Dnear = INFINITY;
    const int di[4] = {-1, 1, 0, 0}, dj[4] = {0, 0, -1, 1};
    for (int s = 0; s < 4; ++s) {
        if (codes) codes[s] = 0;
        int qi = i + di[s], qj = j + dj[s];
        if (qi < 0 || qj < 0 || qi >= c->width || qj >= c->height) continue;
        int64_t pq = (int64_t)qj * c->width + qi, o;
        double t;
        int code;
        if (!aa_pair(w, f32, pp, pq, &o, &t, &code)) continue;
        int onto_other = (code & 1) != 0;
        int onto_me = onto_other ? o != pp : o == pp;
        if (!onto_me) continue;
        if (codes) codes[s] = code;
        double wgt = fabs(t - 0.5);
        int64_t other = o == pp ? pq : pp;
        int cov_o = 1, cov_n = w->face_id[other] >= 0;
        double co[3], cn[3];
        aa_rgb(w, o, co);
        aa_rgb(w, other, cn);
        if (o == pp) { /* A leaves part of this pixel: towards the other pixel's layer */
            a += wgt * ((cov_n ? 1.0 : 0.0) - 1.0);
            for (int ch = 0; ch < 3; ++ch) M[ch] += wgt * ((cov_n ? cn[ch] : 0.0) - co[ch]);
        } else { /* A reaches into this pixel */
            a += wgt * (1.0 - (cov ? 1.0 : 0.0));
            for (int ch = 0; ch < 3; ++ch) M[ch] += wgt * (co[ch] - (cov ? cp[ch] : 0.0));
            if (!cov && wgt > 0.0) Dnear = fmin(Dnear, aa_depth(w, o));
        }
        (void)cov_o;
    }
    *a_out = a < 0.0 ? 0.0 : (a > 1.0 ? 1.0 : a);
    *D_out = cov ? Dp : Dnear;
}

/* Antialiased mesh layer for the listed pixels (all when NULL): cov [H*W],
 * premultiplied colour rgb_aa [H*W*3], split depth depth_aa [H*W], written at
 * the listed pixels.  face_id / mesh_depth / mesh_rgb are full-frame images
 * (the pixels' 4-neighbours are read).                                    */
void orc_antialias(const orc_camera* c, const float* V, const int32_t* F, const int32_t* adj,
                   const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb,
                   const int32_t* pixels, int64_t n_pixels, float* cov, float* rgb_aa, float* depth_aa,
                   int32_t* codes)
{
    aa_view w = {c, V, F, adj, face_id, mesh_depth, mesh_rgb, -1, 0, 0.0, NULL, NULL, NULL, 0};
    int64_t np = pixels ? n_pixels : (int64_t)c->width * c->height;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < np; ++k) {
        int64_t pix = pixels ? pixels[k] : k;
        int i = (int)(pix % c->width), j = (int)(pix / c->width);
        double a, M[3], D;
        int cd[4];
        aa_pixel(&w, 1, i, j, &a, M, &D, cd);
        cov[pix] = (float)a;
        for (int ch = 0; ch < 3; ++ch) rgb_aa[3 * pix + ch] = (float)M[ch];
        depth_aa[pix] = (float)D;
        if (codes)
            for (int s = 0; s < 4; ++s) codes[4 * pix + s] = cd[s];
    }
}

/* tile_full / tile_far over an antialiased layer: full = every in-image pixel
 * fully covered (a = 1), far = the largest split depth over the tile.     */
void orc_tile_bounds_cov(const orc_camera* c, const float* cov, const float* depth, float* tile_far,
                         uint8_t* tile_full)
{
    int TW = n_tiles_x(c), TH = n_tiles_y(c);
    for (int ty = 0; ty < TH; ++ty)
        for (int tx = 0; tx < TW; ++tx) {
            float far = -INFINITY;
            int full = 1;
            for (int j = ty * TILE; j < ty * TILE + TILE && j < c->height; ++j)
                for (int i = tx * TILE; i < tx * TILE + TILE && i < c->width; ++i) {
                    int64_t p = (int64_t)j * c->width + i;
                    if (!(cov[p] >= 1.0f)) full = 0;
                    if (depth[p] > far) far = depth[p];
                }
            tile_far[ty * TW + tx] = full ? far : INFINITY;
            tile_full[ty * TW + tx] = (uint8_t)full;
        }
}

/* ========================================================================
 * EWA projection and SH colour of the Gaussians
 * ====================================================================== */

/* real spherical harmonics Y_lm, m = -l..l, index l*l + l + m, from the
 * associated Legendre functions without the Condon-Shortley phase:
 *   Y_l0 = K_l0 P_l(cos t),  Y_lm = sqrt2 K_lm cos(m p) P_l^m,  Y_l-m = sqrt2 K_lm sin(m p) P_l^m,
 *   K_lm = sqrt((2l+1)/(4 pi) (l-m)!/(l+m)!).                             */
static double fact(int n)
{
    double r = 1.0;
    for (int k = 2; k <= n; ++k) r *= k;
    return r;
}

static double legendre_p(int l, int m, double x)
{
    /* P_m^m = (2m-1)!! (1-x^2)^(m/2); P_{m+1}^m = x (2m+1) P_m^m;
     * (l-m) P_l^m = x (2l-1) P_{l-1}^m - (l+m-1) P_{l-2}^m */
    double pmm = 1.0, sx = sqrt(fmax(0.0, 1.0 - x * x));
    for (int k = 1; k <= m; ++k)
        pmm *= (2.0 * k - 1.0) * sx;
    if (l == m) return pmm;
    double pm1 = x * (2.0 * m + 1.0) * pmm;
    if (l == m + 1) return pm1;
    double pl = 0.0;
    for (int ll = m + 2; ll <= l; ++ll) {
        pl = (x * (2.0 * ll - 1.0) * pm1 - (ll + m - 1.0) * pmm) / (ll - m);
        pmm = pm1;
        pm1 = pl;
    }
    return pl;
}

void orc_sh_basis(int deg, const double* dir, double* Y)
{
    double x = dir[0], y = dir[1], z = dir[2];
    double ct = fmax(-1.0, fmin(1.0, z));
    double ph = atan2(y, x);
    for (int l = 0; l <= deg; ++l)
        for (int m = -l; m <= l; ++m) {
            int am = m < 0 ? -m : m;
            double K = sqrt((2.0 * l + 1.0) / (4.0 * M_PI) * fact(l - am) / fact(l + am));
            double P = legendre_p(l, am, ct);
            double v;
            if (m == 0) v = K * P;
            else if (m > 0) v = sqrt(2.0) * K * cos(am * ph) * P;
            else v = sqrt(2.0) * K * sin(am * ph) * P;
            Y[l * l + l + m] = v;
        }
}

/* The rectangle of tiles a projected Gaussian is binned to (fp32):
 *   [floor((mx - r)/16), ceil((mx + r)/16)) x [floor((my - r)/16), ceil((my + r)/16)),
 * clamped to the tile grid.  Returns its area (0 = not binned).           */
static int64_t gauss_rect(const orc_camera* c, float mx, float my, int32_t r, int rect[4])
{
    if (r <= 0) return 0;
    float fr = (float)r, TW = (float)n_tiles_x(c), TH = (float)n_tiles_y(c);
    float x0 = floorf((mx - fr) / 16.0f), x1 = ceilf((mx + fr) / 16.0f);
    float y0 = floorf((my - fr) / 16.0f), y1 = ceilf((my + fr) / 16.0f);
    x0 = fminf(fmaxf(x0, 0.0f), TW); x1 = fminf(fmaxf(x1, 0.0f), TW);
    y0 = fminf(fmaxf(y0, 0.0f), TH); y1 = fminf(fmaxf(y1, 0.0f), TH);
    rect[0] = (int)x0; rect[1] = (int)y0; rect[2] = (int)x1; rect[3] = (int)y1;
    if (rect[2] <= rect[0] || rect[3] <= rect[1]) return 0;
    return (int64_t)(rect[2] - rect[0]) * (rect[3] - rect[1]);
}

/* Depth model of the soft split (Hybrid rendering): under the same local
 * affine map as the splat, (u, v, z) of a point of the Gaussian are jointly
 * Gaussian with covariance M Sigma_c M^T, M = [J; e_z^T]; the depth given
 * the pixel p is Gaussian with mean z*(p) = z_c + g . (p - mean2d) and
 * standard deviation sigma_z, where
 *   g = (Sigma_uv + eps I)^-1 Sigma_uv,z,   sigma_z^2 = Sigma_zz - Sigma_z,uv g,
 * Sigma_uv = J Sigma_c J^T, Sigma_uv,z = J Sigma_c e_z, Sigma_zz = e_z^T Sigma_c e_z.
 * eps = 0.3 px^2, the low-pass of the splat (reading: Sigma_uv + eps I is the
 * 2D covariance whose inverse is the conic); sigma_z^2 is floored at 1e-12.
 * JS = J Sigma_c (2 x 3), S2 = Sigma_uv + eps I, Sc = Sigma_c.
 * dm = (g_u, g_v, sigma_z).                                               */
static void depth_model_f64(const double JS[2][3], const double S2[2][2], const double Sc[3][3], double dm[3])
{
    double det = S2[0][0] * S2[1][1] - S2[0][1] * S2[1][0];
    double bu = JS[0][2], bv = JS[1][2];
    double gu = (S2[1][1] * bu - S2[0][1] * bv) / det;
    double gv = (-S2[1][0] * bu + S2[0][0] * bv) / det;
    double var = Sc[2][2] - (bu * gu + bv * gv);
    dm[0] = gu;
    dm[1] = gv;
    dm[2] = sqrt(fmax(var, 1e-12));
}

/* Projection of one Gaussian (EWA splatting as in the 3DGS projection the
 * page says was adapted from gsplat):
 *   t = R mu + t_cw; culled when t_z <= near or t_z > far;
 *   Sigma = M M^T with M = R(q) diag(exp(log_s)), q = (w, x, y, z) normalised;
 *   J = [[fx/tz, 0, -fx tx'/tz^2], [0, fy/tz, -fy ty'/tz^2]], where
 *       tx'/tz, ty'/tz are clamped to 1.3 x the tangent of the half field of
 *       view on each side of the principal point;
 *   Sigma2 = J R_cw Sigma R_cw^T J^T + 0.3 I;  conic = Sigma2^-1 as (a, b, c);
 *   radius = ceil(3 sqrt(lambda_max)), lambda_max = m + sqrt(h^2 + b^2),
 *       m = (a + c)/2, h = (a - c)/2 of Sigma2 (fp32, decides the bins);
 *   mean2d = (fx tx/tz + cx, fy ty/tz + cy);  opacity = sigmoid(logit);
 *   colour = given RGB (sh_degree < 0) or max(0, sum_lm Y_lm(d) coef_lm + 0.5)
 *       with d = normalize(mu - camera centre).
 * margin[g] = distance of 3 sqrt(lambda_max) (double) to the nearest integer,
 * relative to its value (a radius decided within rounding of it is a tie). */
void orc_project_gaussians(const orc_camera* c, int32_t sh_degree, int32_t N,
                           const float* means, const float* log_scales, const float* quats,
                           const float* logits, const float* colors,
                           float* splats, int32_t* radii, int32_t* tiles_touched, double* margin,
                           float* depth_model)
{
    int ncoef = sh_degree >= 0 ? (sh_degree + 1) * (sh_degree + 1) : 1;
    double Rc[3][3], cam_pos[3];
    for (int r = 0; r < 3; ++r)
        for (int k = 0; k < 3; ++k)
            Rc[r][k] = c->R[3 * r + k];
    for (int k = 0; k < 3; ++k)
        cam_pos[k] = -(Rc[0][k] * c->t[0] + Rc[1][k] * c->t[1] + Rc[2][k] * c->t[2]);
    double limx_pos = 1.3 * (c->width - (double)c->cx) / c->fx;
    double limx_neg = 1.3 * (double)c->cx / c->fx;
    double limy_pos = 1.3 * (c->height - (double)c->cy) / c->fy;
    double limy_neg = 1.3 * (double)c->cy / c->fy;

#pragma omp parallel for schedule(static)
    for (int64_t g = 0; g < N; ++g) {
        float* s = splats + S_STRIDE * g;
        for (int k = 0; k < S_STRIDE; ++k) s[k] = 0.0f;
        if (depth_model)
            for (int k = 0; k < 4; ++k) depth_model[4 * g + k] = 0.0f;
        radii[g] = 0;
        tiles_touched[g] = 0;
        margin[g] = INFINITY;
        const float* mu = means + 3 * g;
        double t[3];
        for (int r = 0; r < 3; ++r)
            t[r] = Rc[r][0] * mu[0] + Rc[r][1] * mu[1] + Rc[r][2] * mu[2] + c->t[r];
        float tz32 = (float)t[2];
        if (!(tz32 > c->near_plane) || tz32 > c->far_plane)
            continue;
        /* rotation of the quaternion and the 3D covariance */
        const float* qq = quats + 4 * g;
        double qn = sqrt((double)qq[0] * qq[0] + (double)qq[1] * qq[1] + (double)qq[2] * qq[2] +
                         (double)qq[3] * qq[3]);
        double w = qq[0] / qn, x = qq[1] / qn, y = qq[2] / qn, z = qq[3] / qn;
        double Rq[3][3] = {
            {1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)},
            {2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)},
            {2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)}};
        double sc[3], M[3][3], S3[3][3], Sc[3][3], Tmp[3][3];
        for (int k = 0; k < 3; ++k) sc[k] = exp((double)log_scales[3 * g + k]);
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) M[r][k] = Rq[r][k] * sc[k];
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) {
                S3[r][k] = 0;
                for (int m = 0; m < 3; ++m) S3[r][k] += M[r][m] * M[k][m];
            }
        /* camera-frame covariance R_cw Sigma R_cw^T */
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) {
                Tmp[r][k] = 0;
                for (int m = 0; m < 3; ++m) Tmp[r][k] += Rc[r][m] * S3[m][k];
            }
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) {
                Sc[r][k] = 0;
                for (int m = 0; m < 3; ++m) Sc[r][k] += Tmp[r][m] * Rc[k][m];
            }
        /* Jacobian of the pinhole projection with the clamped direction */
        double tx = t[2] * fmin(limx_pos, fmax(-limx_neg, t[0] / t[2]));
        double ty = t[2] * fmin(limy_pos, fmax(-limy_neg, t[1] / t[2]));
        double J[2][3] = {{c->fx / t[2], 0.0, -c->fx * tx / (t[2] * t[2])},
                          {0.0, c->fy / t[2], -c->fy * ty / (t[2] * t[2])}};
        double JS[2][3], S2[2][2];
        for (int r = 0; r < 2; ++r)
            for (int k = 0; k < 3; ++k) {
                JS[r][k] = 0;
                for (int m = 0; m < 3; ++m) JS[r][k] += J[r][m] * Sc[m][k];
            }
        for (int r = 0; r < 2; ++r)
            for (int k = 0; k < 2; ++k) {
                S2[r][k] = 0;
                for (int m = 0; m < 3; ++m) S2[r][k] += JS[r][m] * J[k][m];
            }
        S2[0][0] += 0.3;
        S2[1][1] += 0.3;
        /* fp32 decisions: positive determinant, radius */
        float a32 = (float)S2[0][0], b32 = (float)S2[0][1], c32 = (float)S2[1][1];
        float det32 = a32 * c32 - b32 * b32;
        if (!(det32 > 0.0f))
            continue;
        float m32 = 0.5f * (a32 + c32);
        float h32 = 0.5f * (a32 - c32);
        float lam32 = m32 + sqrtf(h32 * h32 + b32 * b32);
        float r32 = ceilf(3.0f * sqrtf(lam32));
        double lam64 = 0.5 * (S2[0][0] + S2[1][1]) +
                       sqrt(0.25 * (S2[0][0] - S2[1][1]) * (S2[0][0] - S2[1][1]) + S2[0][1] * S2[0][1]);
        double ext = 3.0 * sqrt(lam64);
        int32_t r = (int32_t)r32;
        double mx = c->fx * t[0] / t[2] + c->cx;
        double my = c->fy * t[1] / t[2] + c->cy;
        int rect[4];
        int64_t area = gauss_rect(c, (float)mx, (float)my, r, rect);
        if (area <= 0)
            continue;
        margin[g] = fabs(ext - nearbyint(ext)) / ext;
        double det = S2[0][0] * S2[1][1] - S2[0][1] * S2[0][1];
        s[S_MX] = (float)mx;
        s[S_MY] = (float)my;
        s[S_CA] = (float)(S2[1][1] / det);
        s[S_CB] = (float)(-S2[0][1] / det);
        s[S_CC] = (float)(S2[0][0] / det);
        s[S_OP] = (float)(1.0 / (1.0 + exp(-(double)logits[g])));
        if (sh_degree < 0) {
            for (int ch = 0; ch < 3; ++ch) s[S_R + ch] = colors[3 * g + ch];
        } else {
            double d[3], dn = 0.0, Y[16];
            for (int k = 0; k < 3; ++k) {
                d[k] = mu[k] - cam_pos[k];
                dn += d[k] * d[k];
            }
            dn = sqrt(dn);
            for (int k = 0; k < 3; ++k) d[k] /= dn;
            orc_sh_basis(sh_degree, d, Y);
            for (int ch = 0; ch < 3; ++ch) {
                double v = 0.5;
                for (int k = 0; k < ncoef; ++k)
                    v += Y[k] * colors[((int64_t)g * ncoef + k) * 3 + ch];
                s[S_R + ch] = (float)fmax(0.0, v);
            }
        }
        s[S_Z] = (float)t[2];
        radii[g] = r;
        tiles_touched[g] = (int32_t)area;
        if (depth_model) {
            double dm[3];
            depth_model_f64(JS, S2, Sc, dm);
            for (int k = 0; k < 3; ++k) depth_model[4 * g + k] = (float)dm[k];
        }
    }
}

/* ========================================================================
 * Gaussian tile bins, sorted by (tile, centre depth, id), with the cull
 * ====================================================================== */

typedef struct {
    uint64_t key;
    int32_t gid;
} kv;

static int kv_cmp(const void* a, const void* b)
{
    const kv* x = (const kv*)a;
    const kv* y = (const kv*)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return (x->gid > y->gid) - (x->gid < y->gid);
}

static uint32_t fbits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* Emits key = (tile << 32) | bits(depth), value = Gaussian id, for every tile
 * of every binned Gaussian's rectangle, except (cull != 0) tiles that are
 * fully covered by the mesh and whose farthest mesh depth is not beyond the
 * Gaussian's centre depth (depth >= tile_far): such a Gaussian fails the
 * depth test at every pixel of the tile, so dropping it changes nothing
 * (Hybrid rendering, cull_occluded bullet).  Sorted ascending by key, then
 * id.  Returns the number of entries after the cull; *pre gets the number
 * before it.  keys/gids are written when non-NULL and the total fits cap.  */
int64_t orc_bin_gaussians_masked(const orc_camera* c, int32_t N, const float* splats, const int32_t* radii,
                                 const float* tile_far, const uint8_t* tile_full, int32_t cull,
                                 const uint8_t* tile_mask, uint64_t* keys, int32_t* gids, int64_t cap,
                                 int64_t* pre);

int64_t orc_bin_gaussians(const orc_camera* c, int32_t N, const float* splats, const int32_t* radii,
                          const float* tile_far, const uint8_t* tile_full, int32_t cull,
                          uint64_t* keys, int32_t* gids, int64_t cap, int64_t* pre)
{
    return orc_bin_gaussians_masked(c, N, splats, radii, tile_far, tile_full, cull, NULL, keys, gids, cap, pre);
}

/* As orc_bin_gaussians, restricted to the tiles with tile_mask[t] != 0 (all
 * tiles when tile_mask is NULL): the same entries, fewer tiles.            */
int64_t orc_bin_gaussians_masked(const orc_camera* c, int32_t N, const float* splats, const int32_t* radii,
                                 const float* tile_far, const uint8_t* tile_full, int32_t cull,
                                 const uint8_t* tile_mask, uint64_t* keys, int32_t* gids, int64_t cap,
                                 int64_t* pre)
{
    int TW = n_tiles_x(c);
    int64_t total = 0, before = 0;
    for (int pass = 0; pass < 2; ++pass) {
        kv* out = NULL;
        if (pass == 1) {
            if (!keys || total > cap) break;
            out = (kv*)malloc(sizeof(kv) * (total > 0 ? total : 1));
        }
        int64_t n = 0;
        for (int32_t g = 0; g < N; ++g) {
            int rect[4];
            const float* s = splats + S_STRIDE * (int64_t)g;
            if (gauss_rect(c, s[S_MX], s[S_MY], radii[g], rect) <= 0)
                continue;
            for (int ty = rect[1]; ty < rect[3]; ++ty)
                for (int tx = rect[0]; tx < rect[2]; ++tx) {
                    int64_t tile = (int64_t)ty * TW + tx;
                    if (tile_mask && !tile_mask[tile]) continue;
                    if (pass == 0) before++;
                    if (cull && tile_full[tile] && s[S_Z] >= tile_far[tile])
                        continue;
                    if (pass == 1) {
                        out[n].key = ((uint64_t)tile << 32) | fbits(s[S_Z]);
                        out[n].gid = g;
                    }
                    n++;
                }
        }
        if (pass == 0) {
            total = n;
        } else {
            qsort(out, (size_t)n, sizeof(kv), kv_cmp);
            for (int64_t k = 0; k < n; ++k) {
                keys[k] = out[k].key;
                gids[k] = out[k].gid;
            }
            free(out);
        }
    }
    if (pre) *pre = before;
    return total;
}

/* Full per-tile candidate lists for compositing (no cull): tile t holds every
 * binned Gaussian whose rectangle contains it, ordered by (depth, id); only
 * tiles with tile_mask[t] != 0 get entries when a mask is given.
 * tile_start[T+1] is filled always; entries when non-NULL and K fits cap. */
int64_t orc_tile_lists(const orc_camera* c, int32_t N, const float* splats, const int32_t* radii,
                       const uint8_t* tile_mask, int64_t* tile_start, int32_t* entries, int64_t cap)
{
    int TW = n_tiles_x(c), TH = n_tiles_y(c);
    int64_t T = (int64_t)TW * TH;
    int64_t K = orc_bin_gaussians_masked(c, N, splats, radii, NULL, NULL, 0, tile_mask, NULL, NULL, 0, NULL);
    if (!entries || K > cap) {
        /* counts only */
        memset(tile_start, 0, sizeof(int64_t) * (T + 1));
        for (int32_t g = 0; g < N; ++g) {
            int rect[4];
            const float* s = splats + S_STRIDE * (int64_t)g;
            if (gauss_rect(c, s[S_MX], s[S_MY], radii[g], rect) <= 0) continue;
            for (int ty = rect[1]; ty < rect[3]; ++ty)
                for (int tx = rect[0]; tx < rect[2]; ++tx)
                    if (!tile_mask || tile_mask[(int64_t)ty * TW + tx]) tile_start[(int64_t)ty * TW + tx + 1]++;
        }
        for (int64_t t = 0; t < T; ++t) tile_start[t + 1] += tile_start[t];
        return K;
    }
    uint64_t* keys = (uint64_t*)malloc(sizeof(uint64_t) * (K > 0 ? K : 1));
    orc_bin_gaussians_masked(c, N, splats, radii, NULL, NULL, 0, tile_mask, keys, entries, K, NULL);
    for (int64_t t = 0; t <= T; ++t) tile_start[t] = 0;
    for (int64_t k = 0; k < K; ++k) tile_start[(keys[k] >> 32) + 1]++;
    for (int64_t t = 0; t < T; ++t) tile_start[t + 1] += tile_start[t];
    free(keys);
    return K;
}

/* ========================================================================
 * Hybrid compositing (hard split, mesh colour as the terminal layer)
 * ====================================================================== */

#define ALPHA_MAX 0.99
#define ALPHA_MIN (1.0 / 255.0)
#define T_STOP 1e-4

enum { TR_DEPTH = 1, TR_SIGMA = 2, TR_ALPHA = 3, TR_BLEND = 4, TR_BLEND_CLAMPED = 5, TR_STOP = 6 };

typedef struct {
    int gid, field;
    double delta;
} pert_t;

/* Soft split (Hybrid rendering): the depth model [N][4] = (g_u, g_v,
 * sigma_z, -) of each Gaussian (see depth_model_f64), the softness and the
 * form of the front fraction (the exported calls take it as `split`).
 * Perturbation fields F_GU, F_GV, F_SZ address the depth model.          */
typedef struct {
    const float* dm;
    double softness;
    int logistic; /* 0: f = Phi(x); 1: f = 1 / (1 + exp(-1.702 x)) */
} soft_t;

/* The split's front fraction: the standard normal CDF, or its logistic
 * approximation with slope 1.702 (the two agree within 0.01 everywhere). */
static inline double split_front(double x, int logistic)
{
    return logistic ? 1.0 / (1.0 + exp(-1.702 * x)) : 0.5 * erfc(-x * M_SQRT1_2);
}
enum { F_GU = 12, F_GV = 13, F_SZ = 14 };

static inline double dmfield(const soft_t* sm, int g, int k, const pert_t* p)
{
    double v = sm->dm[4 * (int64_t)g + k];
    if (p && p->gid == g && p->field == F_GU + k) v += p->delta;
    return v;
}

typedef struct {
    double rgb[3], depth, alpha, T;
    int32_t n_contrib;
    /* smallest relative distance of a decision operand to its threshold */
    double m_depth, m_alpha, m_clamp, m_stop, m_sigma;
    /* the watched Gaussian: its trace code (0 = not reached) and the smallest
     * margin of its own decisions */
    int self_code;
    double m_self;
} pix_t;

static inline double rnd(double x, int f32) { return f32 ? (double)(float)x : x; }

static inline double sfield(const float* splats, int g, int f, const pert_t* p)
{
    double v = splats[S_STRIDE * (int64_t)g + f];
    if (p && p->gid == g && p->field == f) v += p->delta;
    return v;
}

/* One pixel, front to back over its tile's sorted list, onto a mesh layer of
 * coverage a, premultiplied colour M (= a c_mesh) and depth D (+inf where no
 * mesh reaches the pixel).  Each Gaussian i:
 *   d = p - mu_i,  sigma = 1/2 (a dx^2 + c dy^2) + b dx dy  (skip sigma < 0);
 *   alpha = min(0.99, o_i exp(-sigma));
 * and is split at the mesh (Hybrid rendering) into a front part, composited
 * over the layer, and a back part, composited behind it:
 *   hard split: front = alpha if z_i < D (else 0), back = alpha - front;
 *   soft split (sm != NULL, D finite): front = alpha f, back = alpha (1 - f),
 *     f = Phi((D - z*(p)) / (sigma_z softness)) or its logistic
 *     approximation (split_front), z*(p) = z_i + g . d.
 * Each of the two chains (front; back) composites its parts on its own:
 *   skip a part below 1/255; stop the chain before a part that would bring
 *   its T to 1e-4 or below; C += part T c_i, Z += part T z_i, T *= 1 - part.
 * With the back chain (C_b, Z_b, T_b), the page's two-layer equation:
 *   rgb = C + T (M + (1 - a)(C_b + T_b bg));  depth = Z + T (a D + (1 - a) Z_b);
 *   alpha = 1 - T (1 - a) T_b.
 * The back chain is evaluated only where it is seen (a < 1 and D finite):
 * with a in {0, 1} (no antialiasing) it never is, and the pixel reduces to
 * the one-layer form rgb = C + T (covered ? c_mesh : bg).
 * trace[k] (optional) records the decision taken on list entry k: the front
 * chain's code in bits 0-2, the back chain's in bits 3-5.               */
#define SET_CODE(c)                      \
    do {                                 \
        if (trace) trace[k] = (c);       \
        if (g == watch) o->self_code = (c); \
    } while (0)

typedef struct {
    double T, C[3], Z;
    int on;
} chain_t;

/* one part (alpha already split) into one chain; returns the trace code */
static int chain_add(chain_t* ch, int f32, double part, double amin, double tstop, int clamped,
                     const float* splats, int g, const pert_t* p, pix_t* o, int watch, double ma)
{
    o->m_alpha = fmin(o->m_alpha, ma);
    if (g == watch) o->m_self = fmin(o->m_self, ma);
    if (part < amin) return TR_ALPHA;
    double Tn = rnd(ch->T * rnd(1.0 - part, f32), f32);
    double mt = fabs(Tn - tstop) / tstop;
    o->m_stop = fmin(o->m_stop, mt);
    if (g == watch) o->m_self = fmin(o->m_self, mt);
    if (Tn <= tstop) {
        ch->on = 0;
        return TR_STOP;
    }
    double w = rnd(part * ch->T, f32);
    for (int c = 0; c < 3; ++c) ch->C[c] += w * sfield(splats, g, S_R + c, p);
    ch->Z += w * sfield(splats, g, S_Z, p);
    ch->T = Tn;
    return clamped ? TR_BLEND_CLAMPED : TR_BLEND;
}

static void composite_pixel(int f32, double px, double py, const int32_t* list, int64_t n,
                            const float* splats, const soft_t* sm, double D, double acov, const double M[3],
                            const double bg[3], const pert_t* p, pix_t* o, uint8_t* trace,
                            int64_t* trace_len, int watch)
{
    chain_t fr = {1.0, {0, 0, 0}, 0.0, 1}, bk = {1.0, {0, 0, 0}, 0.0, 0};
    int32_t last = 0;
    const double amax = rnd(ALPHA_MAX, f32), amin = rnd(ALPHA_MIN, f32), tstop = rnd(T_STOP, f32);
    const int has_mesh = D < INFINITY;
    const int soft = sm && has_mesh;
    bk.on = has_mesh && acov < 1.0;
    o->m_depth = o->m_alpha = o->m_clamp = o->m_stop = o->m_sigma = INFINITY;
    o->self_code = 0;
    o->m_self = INFINITY;
    int64_t k;
    for (k = 0; k < n && (fr.on || bk.on); ++k) {
        int g = list[k];
        double z = sfield(splats, g, S_Z, p);
        int code_f = 0, code_b = 0;
        int in_front = 1, in_back = 0; /* hard split: which chain takes the Gaussian */
        if (!soft) {
            if (has_mesh) {
                double m = fabs(z - D) / D;
                o->m_depth = fmin(o->m_depth, m);
                if (g == watch) o->m_self = fmin(o->m_self, m);
            }
            in_front = z < D;
            in_back = !in_front;
            if ((in_front && !fr.on) || (in_back && !bk.on)) {
                if (in_back) SET_CODE(TR_DEPTH);
                else SET_CODE(0);
                continue;
            }
        }
        double dx = rnd(px - sfield(splats, g, S_MX, p), f32);
        double dy = rnd(py - sfield(splats, g, S_MY, p), f32);
        double ca = sfield(splats, g, S_CA, p), cb = sfield(splats, g, S_CB, p),
               cc = sfield(splats, g, S_CC, p);
        double qa = rnd(ca * rnd(dx * dx, f32), f32);
        double qc = rnd(cc * rnd(dy * dy, f32), f32);
        double half = rnd(0.5 * rnd(qa + qc, f32), f32);
        double cross = rnd(rnd(cb * dx, f32) * dy, f32);
        double sigma = rnd(half + cross, f32);
        double ms = fabs(sigma) / (fabs(half) + fabs(cross) + 1e-30);
        o->m_sigma = fmin(o->m_sigma, ms);
        if (g == watch) o->m_self = fmin(o->m_self, ms);
        if (sigma < 0.0) {
            SET_CODE(TR_SIGMA | (bk.on && (soft || in_back) ? TR_SIGMA << 3 : 0));
            continue;
        }
        double G = rnd(exp(-sigma), f32);
        double oG = rnd(sfield(splats, g, S_OP, p) * G, f32);
        double mc = fabs(oG - amax) / amax;
        o->m_clamp = fmin(o->m_clamp, mc);
        if (g == watch) o->m_self = fmin(o->m_self, mc);
        int clamped = oG > amax;
        double alpha = clamped ? amax : oG;
        double pf = alpha, pb = alpha;             /* the front and back parts */
        double mf = fabs(alpha - amin) / amin, mb = mf; /* their skip margins */
        if (soft) {
            double zs = rnd(z + rnd(rnd(dmfield(sm, g, 0, p) * dx, f32) + rnd(dmfield(sm, g, 1, p) * dy, f32), f32),
                            f32);
            double band = rnd(dmfield(sm, g, 2, p) * sm->softness, f32);
            double xa = rnd(rnd(D - zs, f32) / band, f32);
            double f = rnd(split_front(xa, sm->logistic), f32);
            pf = rnd(alpha * f, f32);
            pb = rnd(alpha * rnd(1.0 - f, f32), f32);
            /* an fp32 evaluation of x = (D - z*) / band in another order lands within
             * about 4 eps ((|D| + |z*|) / band + |x|) of this one: the skip margin of
             * each part is that of its whole interval (negative: either side possible) */
            double ex = 4.0 * FLT_EPSILON * ((fabs(D) + fabs(zs)) / band + fabs(xa));
            double flo = split_front(xa - ex, sm->logistic), fhi = split_front(xa + ex, sm->logistic);
            double lo = alpha * flo, hi = alpha * fhi;
            mf = hi < amin ? (amin - hi) / amin : (lo >= amin ? (lo - amin) / amin : -1.0);
            lo = alpha * (1.0 - fhi);
            hi = alpha * (1.0 - flo);
            mb = hi < amin ? (amin - hi) / amin : (lo >= amin ? (lo - amin) / amin : -1.0);
        }
        if (fr.on && in_front) {
            code_f = chain_add(&fr, f32, pf, amin, tstop, clamped, splats, g, p, o, watch, mf);
            if (code_f == TR_BLEND || code_f == TR_BLEND_CLAMPED) last = (int32_t)(k + 1);
        }
        if (bk.on && (soft || in_back))
            code_b = chain_add(&bk, f32, pb, amin, tstop, clamped, splats, g, p, o, watch, mb);
        if (trace) trace[k] = (uint8_t)(code_f | (code_b << 3));
        if (g == watch) o->self_code = code_f ? code_f : code_b;
    }
    if (trace_len) *trace_len = k;
    const double ua = 1.0 - acov;
    for (int ch = 0; ch < 3; ++ch) {
        double behind = ua > 0.0 ? ua * (bk.C[ch] + bk.T * bg[ch]) : 0.0;
        o->rgb[ch] = fr.C[ch] + fr.T * (M[ch] + behind);
    }
    o->depth = fr.Z + fr.T * ((acov > 0.0 ? acov * D : 0.0) + (ua > 0.0 ? ua * bk.Z : 0.0));
    o->alpha = 1.0 - fr.T * ua * bk.T;
    o->T = fr.T;
    o->n_contrib = last;
}

/* the mesh layer of one pixel: the antialiased one (coverage image given,
 * colour premultiplied) or the binary one of the z-buffer */
static double mesh_layer(const float* mesh_cov, const float* mesh_rgb, const int32_t* face_id, int64_t pix,
                         double M[3])
{
    double a = mesh_cov ? (double)mesh_cov[pix] : (face_id[pix] >= 0 ? 1.0 : 0.0);
    for (int ch = 0; ch < 3; ++ch) M[ch] = mesh_cov || a > 0.0 ? (double)mesh_rgb[3 * pix + ch] : 0.0;
    return a;
}

/* Full-frame compositing (tiles listed, or all).  The mesh layer is
 * (mesh_cov, mesh_rgb premultiplied, mesh_depth) when mesh_cov is given (the
 * antialiased layer), else coverage face_id >= 0 with colour mesh_rgb.     */
void orc_composite_fwd(const orc_camera* c, const float* bg, const float* splats,
                       const int64_t* tile_start, const int32_t* entries,
                       const float* mesh_depth, const float* mesh_rgb, const int32_t* face_id,
                       const float* mesh_cov, const int32_t* tiles, int32_t n_tiles_req,
                       float* out_rgb, float* out_depth, float* out_alpha, float* T_final,
                       int32_t* n_contrib, double* margins, const float* depth_model, double softness, int32_t split)
{
    soft_t smv = {depth_model, softness, split != 0};
    const soft_t* sm = depth_model && softness > 0.0 ? &smv : NULL;
    int TW = n_tiles_x(c), TH = n_tiles_y(c);
    int32_t nt = tiles ? n_tiles_req : TW * TH;
    double bgd[3] = {bg[0], bg[1], bg[2]};
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t q = 0; q < nt; ++q) {
        int32_t tile = tiles ? tiles[q] : q;
        int tx = tile % TW, ty = tile / TW;
        const int32_t* list = entries + tile_start[tile];
        int64_t n = tile_start[tile + 1] - tile_start[tile];
        for (int j = ty * TILE; j < ty * TILE + TILE && j < c->height; ++j)
            for (int i = tx * TILE; i < tx * TILE + TILE && i < c->width; ++i) {
                int64_t pix = (int64_t)j * c->width + i;
                double M[3];
                double a = mesh_layer(mesh_cov, mesh_rgb, face_id, pix, M);
                pix_t o;
                composite_pixel(1, i + 0.5, j + 0.5, list, n, splats, sm, (double)mesh_depth[pix], a, M,
                                bgd, NULL, &o, NULL, NULL, -1);
                for (int ch = 0; ch < 3; ++ch) out_rgb[3 * pix + ch] = (float)o.rgb[ch];
                out_depth[pix] = (float)o.depth;
                out_alpha[pix] = (float)o.alpha;
                T_final[pix] = (float)o.T;
                n_contrib[pix] = o.n_contrib;
                if (margins) {
                    margins[5 * pix + 0] = o.m_depth;
                    margins[5 * pix + 1] = o.m_alpha;
                    margins[5 * pix + 2] = o.m_clamp;
                    margins[5 * pix + 3] = o.m_stop;
                    margins[5 * pix + 4] = o.m_sigma;
                }
            }
    }
    (void)TH;
}

/* ========================================================================
 * Gradients by central finite differences (double), decisions held fixed
 * ====================================================================== */

enum { FD_OK = 0, FD_FLIP = 1, FD_PRECISION = 2, FD_TIE = 3, FD_ORDER = 4, FD_UNUSED = 5, FD_NONSMOOTH = 6 };

/* Central differences at steps h and h/2 combined by Richardson's rule
 * (error O(h^4)).  Where the two differ by more than 1% the loss is too
 * curved at this scale for either to be trusted: FD_NONSMOOTH.            */
static int richardson(double lp, double lm, double lp2, double lm2, double h, double* g)
{
    double g1 = (lp - lm) / (2.0 * h);
    double g2 = (lp2 - lm2) / h;
    *g = g2 + (g2 - g1) / 3.0;
    return fabs(g1 - g2) <= 1e-2 * fabs(g2) + 1e-7 ? FD_OK : FD_NONSMOOTH;
}

static double pixel_loss(const pix_t* o, const float* g_rgb, const float* g_depth,
                         const float* g_alpha, int64_t pix)
{
    return g_rgb[3 * pix] * o->rgb[0] + g_rgb[3 * pix + 1] * o->rgb[1] + g_rgb[3 * pix + 2] * o->rgb[2] +
           g_depth[pix] * o->depth + g_alpha[pix] * o->alpha;
}

static int same_trace(const uint8_t* a, int64_t na, const uint8_t* b, int64_t nb)
{
    return na == nb && memcmp(a, b, (size_t)na) == 0;
}

static int tie_pixel(const pix_t* o, double band)
{
    return o->m_alpha < band || o->m_clamp < band || o->m_stop < band || o->m_sigma < band;
}

/* dL/d(splat field) for the requested (Gaussian, field) pairs, L = sum over
 * pixels of g_rgb . rgb + g_depth depth + g_alpha alpha.  Only pixels of the
 * tiles in the Gaussian's rectangle can change; the tile lists stay fixed.
 * status: FD_OK; FD_FLIP a decision differs between +h and -h;
 * FD_PRECISION the double and fp32 evaluations decide differently at h = 0;
 * FD_TIE an fp32 decision margin is below tie_band where it matters;
 * FD_ORDER a depth step would reorder the list; FD_NONSMOOTH the steps h and
 * h/2 disagree (see richardson).  Decisions are compared at +-h, which
 * brackets the +-h/2 evaluations.                                        */
void orc_composite_fd(const orc_camera* c, const float* bg, const float* splats, const int32_t* radii,
                      const int64_t* tile_start, const int32_t* entries,
                      const float* mesh_depth, const float* mesh_rgb, const int32_t* face_id,
                      const float* mesh_cov, const float* g_rgb, const float* g_depth, const float* g_alpha,
                      int32_t n_req, const int32_t* req_gid, const int32_t* req_field,
                      const double* req_h, double tie_band, double* grad, int32_t* status,
                      const float* depth_model, double softness, int32_t split)
{
    soft_t smv = {depth_model, softness, split != 0};
    const soft_t* sm = depth_model && softness > 0.0 ? &smv : NULL;
    int TW = n_tiles_x(c);
    double bgd[3] = {bg[0], bg[1], bg[2]};
    int64_t maxlist = 1;
    for (int64_t t = 0; t < (int64_t)TW * n_tiles_y(c); ++t)
        if (tile_start[t + 1] - tile_start[t] > maxlist) maxlist = tile_start[t + 1] - tile_start[t];
#pragma omp parallel
    {
        uint8_t* tr[4];
        for (int k = 0; k < 4; ++k) tr[k] = (uint8_t*)malloc((size_t)maxlist);
#pragma omp for schedule(dynamic, 1)
        for (int32_t q = 0; q < n_req; ++q) {
            int g = req_gid[q], field = req_field[q];
            double h = req_h[q];
            int rect[4];
            const float* s = splats + S_STRIDE * (int64_t)g;
            grad[q] = 0.0;
            status[q] = FD_OK;
            if (gauss_rect(c, s[S_MX], s[S_MY], radii[g], rect) <= 0) {
                status[q] = FD_UNUSED;
                continue;
            }
            pert_t pp = {g, field, h}, pm = {g, field, -h}, pp2 = {g, field, 0.5 * h}, pm2 = {g, field, -0.5 * h};
            double lp = 0.0, lm = 0.0, lp2 = 0.0, lm2 = 0.0;
            int st = FD_OK;
            for (int ty = rect[1]; ty < rect[3] && st == FD_OK; ++ty)
                for (int tx = rect[0]; tx < rect[2] && st == FD_OK; ++tx) {
                    int64_t tile = (int64_t)ty * TW + tx;
                    const int32_t* list = entries + tile_start[tile];
                    int64_t n = tile_start[tile + 1] - tile_start[tile];
                    if (field == S_Z) {
                        for (int64_t k = 0; k < n; ++k) {
                            if (list[k] != g) continue;
                            double z = s[S_Z];
                            if (k > 0 && !(splats[S_STRIDE * (int64_t)list[k - 1] + S_Z] < z - h)) st = FD_ORDER;
                            if (k + 1 < n && !(z + h < splats[S_STRIDE * (int64_t)list[k + 1] + S_Z])) st = FD_ORDER;
                        }
                        if (st != FD_OK) break;
                    }
                    for (int j = ty * TILE; j < ty * TILE + TILE && j < c->height && st == FD_OK; ++j)
                        for (int i = tx * TILE; i < tx * TILE + TILE && i < c->width; ++i) {
                            int64_t pix = (int64_t)j * c->width + i;
                            double D = mesh_depth[pix];
                            double cm[3];
                            double cov = mesh_layer(mesh_cov, mesh_rgb, face_id, pix, cm);
                            pix_t o32, o0, op, om;
                            int64_t n32, n0, np_, nm;
                            composite_pixel(1, i + 0.5, j + 0.5, list, n, splats, sm, D, cov, cm, bgd, NULL, &o32, tr[0], &n32, g);
                            composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, D, cov, cm, bgd, NULL, &o0, tr[1], &n0, g);
                            composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, D, cov, cm, bgd, &pp, &op, tr[2], &np_, g);
                            composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, D, cov, cm, bgd, &pm, &om, tr[3], &nm, g);
                            /* a decision within rounding of its threshold matters where this
                             * Gaussian is composited (every decision of the pixel enters its
                             * gradient) or in its own decisions */
                            int blended = o32.self_code == TR_BLEND || o32.self_code == TR_BLEND_CLAMPED;
                            if ((blended && tie_pixel(&o32, tie_band)) || o32.m_self < tie_band) { st = FD_TIE; break; }
                            if (!same_trace(tr[0], n32, tr[1], n0)) { st = FD_PRECISION; break; }
                            if (!same_trace(tr[1], n0, tr[2], np_) || !same_trace(tr[1], n0, tr[3], nm)) {
                                st = FD_FLIP;
                                break;
                            }
                            lp += pixel_loss(&op, g_rgb, g_depth, g_alpha, pix);
                            lm += pixel_loss(&om, g_rgb, g_depth, g_alpha, pix);
                            composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, D, cov, cm, bgd, &pp2, &op, NULL, NULL, -1);
                            composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, D, cov, cm, bgd, &pm2, &om, NULL, NULL, -1);
                            lp2 += pixel_loss(&op, g_rgb, g_depth, g_alpha, pix);
                            lm2 += pixel_loss(&om, g_rgb, g_depth, g_alpha, pix);
                        }
                }
            double gv = 0.0;
            if (st == FD_OK) st = richardson(lp, lm, lp2, lm2, h, &gv);
            status[q] = st;
            grad[q] = st == FD_OK ? gv : 0.0;
        }
        for (int k = 0; k < 4; ++k) free(tr[k]);
    }
}

/* dL/d(vertex position or colour) through the interpolated mesh depth and
 * colour (face ids held fixed) and, with antialiasing (adj given), through the
 * silhouette crossings.  req_field 0..2 = world x, y, z of the vertex, 3..5 =
 * its r, g, b.  Re-evaluated: the depth and colour (in double, from the moved
 * mesh) of the pixels whose face uses the vertex, the antialiased layer of
 * every pixel within 2 px of the image box of such a face, and the composite
 * (double) of every such pixel.  The fp32 reference decisions use mesh_depth / mesh_rgb as
 * given.  Status codes as for orc_composite_fd; the antialiasing decisions
 * (occluder, exit edge, silhouette, side) count as decisions.             */
static int cmp_i64(const void* a, const void* b)
{
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

void orc_mesh_fd(const orc_camera* c, const float* bg, const float* V, int32_t nV, const int32_t* F,
                 int32_t nF, const float* vcol, const int32_t* face_id, const int32_t* adj, const float* splats,
                 const int64_t* tile_start, const int32_t* entries, const float* mesh_depth,
                 const float* mesh_rgb, const float* g_rgb, const float* g_depth, const float* g_alpha,
                 int32_t n_req, const int32_t* req_vid, const int32_t* req_field, const double* req_h,
                 double tie_band, double* grad, int32_t* status, const float* depth_model, double softness, int32_t split)
{
    soft_t smv = {depth_model, softness, split != 0};
    const soft_t* sm = depth_model && softness > 0.0 ? &smv : NULL;
    int TW = n_tiles_x(c);
    int64_t P = (int64_t)c->width * c->height;
    double bgd[3] = {bg[0], bg[1], bg[2]};
    /* pixels of each face (CSR) */
    int64_t* fstart = (int64_t*)calloc((size_t)nF + 1, sizeof(int64_t));
    for (int64_t p = 0; p < P; ++p)
        if (face_id[p] >= 0) fstart[face_id[p] + 1]++;
    for (int f = 0; f < nF; ++f) fstart[f + 1] += fstart[f];
    int64_t* fpix = (int64_t*)malloc(sizeof(int64_t) * (fstart[nF] > 0 ? fstart[nF] : 1));
    int64_t* ffill = (int64_t*)malloc(sizeof(int64_t) * (nF > 0 ? nF : 1));
    for (int f = 0; f < nF; ++f) ffill[f] = fstart[f];
    for (int64_t p = 0; p < P; ++p)
        if (face_id[p] >= 0) fpix[ffill[face_id[p]]++] = p;
    /* faces of each vertex (CSR) */
    int64_t* vstart = (int64_t*)calloc((size_t)nV + 1, sizeof(int64_t));
    for (int f = 0; f < nF; ++f)
        for (int k = 0; k < 3; ++k) vstart[F[3 * f + k] + 1]++;
    for (int v = 0; v < nV; ++v) vstart[v + 1] += vstart[v];
    int32_t* vface = (int32_t*)malloc(sizeof(int32_t) * (vstart[nV] > 0 ? vstart[nV] : 1));
    int64_t* vfill = (int64_t*)malloc(sizeof(int64_t) * (nV > 0 ? nV : 1));
    for (int v = 0; v < nV; ++v) vfill[v] = vstart[v];
    for (int f = 0; f < nF; ++f)
        for (int k = 0; k < 3; ++k) vface[vfill[F[3 * f + k]]++] = f;
    int64_t maxlist = 1;
    for (int64_t t = 0; t < (int64_t)TW * n_tiles_y(c); ++t)
        if (tile_start[t + 1] - tile_start[t] > maxlist) maxlist = tile_start[t + 1] - tile_start[t];

#pragma omp parallel
    {
        uint8_t* tr[4];
        for (int k = 0; k < 4; ++k) tr[k] = (uint8_t*)malloc((size_t)maxlist);
#pragma omp for schedule(dynamic, 1)
        for (int32_t q = 0; q < n_req; ++q) {
            int vid = req_vid[q], field = req_field[q];
            double h = req_h[q];
            const double steps[5] = {0.0, h, -h, 0.5 * h, -0.5 * h};
            /* P1: the pixels of the vertex's faces, sorted */
            int64_t n1 = 0;
            for (int64_t fk = vstart[vid]; fk < vstart[vid + 1]; ++fk)
                n1 += fstart[vface[fk] + 1] - fstart[vface[fk]];
            int64_t* p1 = (int64_t*)malloc(sizeof(int64_t) * (n1 > 0 ? n1 : 1));
            n1 = 0;
            for (int64_t fk = vstart[vid]; fk < vstart[vid + 1]; ++fk)
                for (int64_t pk = fstart[vface[fk]]; pk < fstart[vface[fk] + 1]; ++pk) p1[n1++] = fpix[pk];
            qsort(p1, (size_t)n1, sizeof(int64_t), cmp_i64);
            int64_t u1 = 0; /* a face that names the vertex twice lists its pixels twice */
            for (int64_t k = 0; k < n1; ++k)
                if (k == 0 || p1[k] != p1[k - 1]) p1[u1++] = p1[k];
            n1 = u1;
            /* depth and colour of P1 at each step, in double */
            double* ovd = (double*)malloc(sizeof(double) * 5 * (n1 > 0 ? n1 : 1));
            double* ovc = (double*)malloc(sizeof(double) * 15 * (n1 > 0 ? n1 : 1));
            for (int64_t k = 0; k < n1; ++k) {
                int64_t pix = p1[k];
                int f = face_id[pix];
                int i = (int)(pix % c->width), j = (int)(pix / c->width);
                for (int sgn = 0; sgn < 5; ++sgn) {
                    double X[3][3], C3[3][3], D, w[3];
                    load_tri(V, F, f, X);
                    for (int kk = 0; kk < 3; ++kk)
                        for (int d = 0; d < 3; ++d) C3[kk][d] = vcol[3 * (int64_t)F[3 * f + kk] + d];
                    for (int kk = 0; kk < 3; ++kk) {
                        if (F[3 * f + kk] != vid) continue;
                        if (field < 3) X[kk][field] += steps[sgn];
                        else C3[kk][field - 3] += steps[sgn];
                    }
                    tri64 t;
                    tri_setup_f64(c, X, &t);
                    interp_f64(&t, i + 0.5, j + 0.5, &D, w);
                    ovd[sgn * n1 + k] = D;
                    for (int ch = 0; ch < 3; ++ch)
                        ovc[3 * (sgn * n1 + k) + ch] = w[0] * C3[0][ch] + w[1] * C3[1][ch] + w[2] * C3[2][ch];
                }
            }
            /* P2: P1 and, with antialiasing, every pixel within 2 px of the image
             * box of a face that uses the vertex (a pair's segment may cross such a
             * face -- also one that covers no pixel centre -- on its way to a
             * silhouette edge, or end at one of its edges) */
            int64_t n2 = n1;
            int box[64][4];
            int nbox = 0;
            if (adj) {
                for (int64_t fk = vstart[vid]; fk < vstart[vid + 1] && nbox < 64; ++fk) {
                    int f = vface[fk];
                    double X[3][3];
                    load_tri(V, F, f, X);
                    tri64 t;
                    tri_setup_f64(c, X, &t);
                    int ok = 1;
                    for (int kk = 0; kk < 3; ++kk) ok &= t.z[kk] > (double)c->near_plane;
                    if (!ok) continue;
                    double u0 = fmin(fmin(t.u[0], t.u[1]), t.u[2]), u1 = fmax(fmax(t.u[0], t.u[1]), t.u[2]);
                    double v0 = fmin(fmin(t.v[0], t.v[1]), t.v[2]), v1 = fmax(fmax(t.v[0], t.v[1]), t.v[2]);
                    int b[4] = {(int)fmax(floor(u0) - 2, 0), (int)fmax(floor(v0) - 2, 0),
                                (int)fmin(ceil(u1) + 2, c->width - 1), (int)fmin(ceil(v1) + 2, c->height - 1)};
                    if (b[0] > b[2] || b[1] > b[3]) continue;
                    for (int kk = 0; kk < 4; ++kk) box[nbox][kk] = b[kk];
                    n2 += (int64_t)(b[2] - b[0] + 1) * (b[3] - b[1] + 1);
                    nbox++;
                }
            }
            int64_t* p2 = (int64_t*)malloc(sizeof(int64_t) * (n2 > 0 ? n2 : 1));
            n2 = 0;
            for (int64_t k = 0; k < n1; ++k) p2[n2++] = p1[k];
            for (int bq = 0; bq < nbox; ++bq)
                for (int j = box[bq][1]; j <= box[bq][3]; ++j)
                    for (int i = box[bq][0]; i <= box[bq][2]; ++i) p2[n2++] = (int64_t)j * c->width + i;
            qsort(p2, (size_t)n2, sizeof(int64_t), cmp_i64);
            int64_t u2 = 0;
            for (int64_t k = 0; k < n2; ++k)
                if (k == 0 || p2[k] != p2[k - 1]) p2[u2++] = p2[k];
            n2 = u2;
            double lp = 0.0, lm = 0.0, lp2 = 0.0, lm2 = 0.0;
            int st = FD_OK, any = n1 > 0;
            for (int64_t k = 0; k < n2 && st == FD_OK; ++k) {
                int64_t pix = p2[k];
                int i = (int)(pix % c->width), j = (int)(pix / c->width);
                int64_t tile = (int64_t)(j / TILE) * TW + i / TILE;
                const int32_t* list = entries + tile_start[tile];
                int64_t n = tile_start[tile + 1] - tile_start[tile];
                /* the mesh layer: fp32 reference (as given) and at each step */
                double a32, M32[3], D32, a[5], M[5][3], Dl[5];
                int cd32[4] = {0, 0, 0, 0}, cd[5][4];
                if (adj) {
                    aa_view w32 = {c, V, F, adj, face_id, mesh_depth, mesh_rgb, -1, 0, 0.0, NULL, NULL, NULL, 0};
                    aa_pixel(&w32, 1, i, j, &a32, M32, &D32, cd32);
                    for (int sgn = 0; sgn < 5; ++sgn) {
                        aa_view wd = {c, V, F, adj, face_id, mesh_depth, mesh_rgb, field < 3 ? vid : -1, field,
                                      steps[sgn], p1, ovd + sgn * n1, ovc + 3 * sgn * n1, n1};
                        aa_pixel(&wd, 0, i, j, &a[sgn], M[sgn], &Dl[sgn], cd[sgn]);
                    }
                } else {
                    int64_t kk = k; /* P2 = P1 */
                    a32 = 1.0;
                    D32 = mesh_depth[pix];
                    for (int ch = 0; ch < 3; ++ch) M32[ch] = mesh_rgb[3 * pix + ch];
                    for (int sgn = 0; sgn < 5; ++sgn) {
                        a[sgn] = 1.0;
                        Dl[sgn] = ovd[sgn * n1 + kk];
                        for (int ch = 0; ch < 3; ++ch) M[sgn][ch] = ovc[3 * (sgn * n1 + kk) + ch];
                        for (int s4 = 0; s4 < 4; ++s4) cd[sgn][s4] = 0;
                    }
                }
                if (memcmp(cd32, cd[0], sizeof(cd32)) != 0) { st = FD_PRECISION; break; }
                if (memcmp(cd[0], cd[1], sizeof(cd32)) != 0 || memcmp(cd[0], cd[2], sizeof(cd32)) != 0) {
                    st = FD_FLIP;
                    break;
                }
                pix_t o32, o0, op, om;
                int64_t n32, n0, np_, nm;
                composite_pixel(1, i + 0.5, j + 0.5, list, n, splats, sm, D32, a32, M32, bgd, NULL, &o32, tr[0], &n32, -1);
                composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, Dl[0], a[0], M[0], bgd, NULL, &o0, tr[1], &n0, -1);
                composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, Dl[1], a[1], M[1], bgd, NULL, &op, tr[2], &np_, -1);
                composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, Dl[2], a[2], M[2], bgd, NULL, &om, tr[3], &nm, -1);
                /* depth-test decisions: the PRECISION check below compares them
                 * exactly; alpha / stop / sigma decisions within rounding: a tie */
                if (tie_pixel(&o32, tie_band)) { st = FD_TIE; break; }
                if (!same_trace(tr[0], n32, tr[1], n0)) { st = FD_PRECISION; break; }
                if (!same_trace(tr[1], n0, tr[2], np_) || !same_trace(tr[1], n0, tr[3], nm)) {
                    st = FD_FLIP;
                    break;
                }
                lp += pixel_loss(&op, g_rgb, g_depth, g_alpha, pix);
                lm += pixel_loss(&om, g_rgb, g_depth, g_alpha, pix);
                composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, Dl[3], a[3], M[3], bgd, NULL, &op, NULL, NULL, -1);
                composite_pixel(0, i + 0.5, j + 0.5, list, n, splats, sm, Dl[4], a[4], M[4], bgd, NULL, &om, NULL, NULL, -1);
                lp2 += pixel_loss(&op, g_rgb, g_depth, g_alpha, pix);
                lm2 += pixel_loss(&om, g_rgb, g_depth, g_alpha, pix);
            }
            free(p1); free(p2); free(ovd); free(ovc);
            if (st == FD_OK && !any) st = FD_UNUSED;
            double gv = 0.0;
            if (st == FD_OK) st = richardson(lp, lm, lp2, lm2, h, &gv);
            status[q] = st;
            grad[q] = st == FD_OK ? gv : 0.0;
        }
        for (int k = 0; k < 4; ++k) free(tr[k]);
    }
    free(fstart); free(fpix); free(ffill); free(vstart); free(vface); free(vfill);
}

/* Single-pixel composite, exported for closed-form checks of the routine
 * itself (list of Gaussian ids into splats, f32 = 1 for the fp32 mode) over
 * a mesh layer of coverage cov, premultiplied colour M and depth D.
 * out: rgb[3], depth, alpha, T, n_contrib.                                */
void orc_composite_one(int32_t f32, double px, double py, const int32_t* list, int64_t n,
                       const float* splats, double D, double cov, const double* M,
                       const double* bg, double* out, const float* depth_model, double softness, int32_t split)
{
    soft_t smv = {depth_model, softness, split != 0};
    const soft_t* sm = depth_model && softness > 0.0 ? &smv : NULL;
    pix_t o;
    composite_pixel(f32, px, py, list, n, splats, sm, D, cov, M, bg, NULL, &o, NULL, NULL, -1);
    out[0] = o.rgb[0]; out[1] = o.rgb[1]; out[2] = o.rgb[2];
    out[3] = o.depth; out[4] = o.alpha; out[5] = o.T; out[6] = o.n_contrib;
}

/* ========================================================================
 * Gradients of the projection (the projection / SH backward: dL/d of the
 * 3D parameters), for L = sum over the record fields of v . record, by
 * central differences in double
 * ====================================================================== */

/* Parameters of one Gaussian as one double vector:
 *   p[0..2] mean, p[3..5] log-scales, p[6..9] quaternion (w, x, y, z),
 *   p[10] opacity logit, p[11 + 3 k + ch] colour coefficient k of channel
 *   ch (k < (d+1)^2 for SH degree d; k = 0 = plain RGB when d < 0).      */
#define PROJ_NPAR(deg) (11 + 3 * ((deg) >= 0 ? ((deg) + 1) * ((deg) + 1) : 1))

static void proj_load(int sh_degree, int64_t g, const float* means, const float* log_scales, const float* quats,
                      const float* logits, const float* colors, double* p)
{
    int ncoef = sh_degree >= 0 ? (sh_degree + 1) * (sh_degree + 1) : 1;
    for (int k = 0; k < 3; ++k) p[k] = means[3 * g + k];
    for (int k = 0; k < 3; ++k) p[3 + k] = log_scales[3 * g + k];
    for (int k = 0; k < 4; ++k) p[6 + k] = quats[4 * g + k];
    p[10] = logits[g];
    for (int k = 0; k < 3 * ncoef; ++k) p[11 + k] = colors[(int64_t)g * 3 * ncoef + k];
}

/* The record of one Gaussian (fields S_MX .. S_Z) from double parameters,
 * every value in double, by the definitions orc_project_gaussians states.
 * The decisions that make the map non-smooth go to trace: [0] culled (near
 * / far, determinant, empty tile rectangle -- decided in fp32 as the
 * forward decides them), [1] [2] the x / y clamps of the Jacobian
 * direction, [3..5] the colour clamps at 0.  A culled Gaussian's record is
 * all zeros.                                                              */
static void proj_record_f64(const orc_camera* c, int sh_degree, const double* p, double rec[13], uint8_t trace[6])
{
    int ncoef = sh_degree >= 0 ? (sh_degree + 1) * (sh_degree + 1) : 1;
    double Rc[3][3], cam_pos[3], t[3];
    for (int k = 0; k < 13; ++k) rec[k] = 0.0;
    for (int k = 0; k < 6; ++k) trace[k] = 0;
    for (int r = 0; r < 3; ++r)
        for (int k = 0; k < 3; ++k) Rc[r][k] = c->R[3 * r + k];
    for (int k = 0; k < 3; ++k)
        cam_pos[k] = -(Rc[0][k] * c->t[0] + Rc[1][k] * c->t[1] + Rc[2][k] * c->t[2]);
    for (int r = 0; r < 3; ++r) t[r] = Rc[r][0] * p[0] + Rc[r][1] * p[1] + Rc[r][2] * p[2] + c->t[r];
    float tz32 = (float)t[2];
    if (!(tz32 > c->near_plane) || tz32 > c->far_plane) {
        trace[0] = 1;
        return;
    }
    double qn = sqrt(p[6] * p[6] + p[7] * p[7] + p[8] * p[8] + p[9] * p[9]);
    double w = p[6] / qn, x = p[7] / qn, y = p[8] / qn, z = p[9] / qn;
    double Rq[3][3] = {
        {1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)},
        {2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)},
        {2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)}};
    double sc[3], M[3][3], S3[3][3], Tmp[3][3], Sc[3][3];
    for (int k = 0; k < 3; ++k) sc[k] = exp(p[3 + k]);
    for (int r = 0; r < 3; ++r)
        for (int k = 0; k < 3; ++k) M[r][k] = Rq[r][k] * sc[k];
    for (int r = 0; r < 3; ++r)
        for (int k = 0; k < 3; ++k) {
            S3[r][k] = 0;
            for (int m = 0; m < 3; ++m) S3[r][k] += M[r][m] * M[k][m];
        }
    for (int r = 0; r < 3; ++r)
        for (int k = 0; k < 3; ++k) {
            Tmp[r][k] = 0;
            for (int m = 0; m < 3; ++m) Tmp[r][k] += Rc[r][m] * S3[m][k];
        }
    for (int r = 0; r < 3; ++r)
        for (int k = 0; k < 3; ++k) {
            Sc[r][k] = 0;
            for (int m = 0; m < 3; ++m) Sc[r][k] += Tmp[r][m] * Rc[k][m];
        }
    double limx_pos = 1.3 * (c->width - (double)c->cx) / c->fx, limx_neg = 1.3 * (double)c->cx / c->fx;
    double limy_pos = 1.3 * (c->height - (double)c->cy) / c->fy, limy_neg = 1.3 * (double)c->cy / c->fy;
    double rx = t[0] / t[2], ry = t[1] / t[2];
    trace[1] = rx > limx_pos || rx < -limx_neg;
    trace[2] = ry > limy_pos || ry < -limy_neg;
    double tx = t[2] * fmin(limx_pos, fmax(-limx_neg, rx));
    double ty = t[2] * fmin(limy_pos, fmax(-limy_neg, ry));
    double J[2][3] = {{c->fx / t[2], 0.0, -c->fx * tx / (t[2] * t[2])},
                      {0.0, c->fy / t[2], -c->fy * ty / (t[2] * t[2])}};
    double JS[2][3], S2[2][2];
    for (int r = 0; r < 2; ++r)
        for (int k = 0; k < 3; ++k) {
            JS[r][k] = 0;
            for (int m = 0; m < 3; ++m) JS[r][k] += J[r][m] * Sc[m][k];
        }
    for (int r = 0; r < 2; ++r)
        for (int k = 0; k < 2; ++k) {
            S2[r][k] = 0;
            for (int m = 0; m < 3; ++m) S2[r][k] += JS[r][m] * J[k][m];
        }
    S2[0][0] += 0.3;
    S2[1][1] += 0.3;
    /* the cull decisions, in fp32 as the forward takes them */
    float a32 = (float)S2[0][0], b32 = (float)S2[0][1], c32 = (float)S2[1][1];
    float det32 = a32 * c32 - b32 * b32;
    double mx = c->fx * t[0] / t[2] + c->cx, my = c->fy * t[1] / t[2] + c->cy;
    int rect[4];
    if (!(det32 > 0.0f)) {
        trace[0] = 1;
        return;
    }
    float m32 = 0.5f * (a32 + c32), h32 = 0.5f * (a32 - c32);
    float lam32 = m32 + sqrtf(h32 * h32 + b32 * b32);
    if (gauss_rect(c, (float)mx, (float)my, (int32_t)ceilf(3.0f * sqrtf(lam32)), rect) <= 0) {
        trace[0] = 1;
        return;
    }
    double det = S2[0][0] * S2[1][1] - S2[0][1] * S2[0][1];
    rec[S_MX] = mx;
    rec[S_MY] = my;
    rec[S_CA] = S2[1][1] / det;
    rec[S_CB] = -S2[0][1] / det;
    rec[S_CC] = S2[0][0] / det;
    rec[S_OP] = 1.0 / (1.0 + exp(-p[10]));
    if (sh_degree < 0) {
        for (int ch = 0; ch < 3; ++ch) rec[S_R + ch] = p[11 + ch];
    } else {
        double d[3], dn = 0.0, Y[16];
        for (int k = 0; k < 3; ++k) {
            d[k] = p[k] - cam_pos[k];
            dn += d[k] * d[k];
        }
        dn = sqrt(dn);
        for (int k = 0; k < 3; ++k) d[k] /= dn;
        orc_sh_basis(sh_degree, d, Y);
        for (int ch = 0; ch < 3; ++ch) {
            double v = 0.5;
            for (int k = 0; k < ncoef; ++k) v += Y[k] * p[11 + 3 * k + ch];
            trace[3 + ch] = v < 0.0;
            rec[S_R + ch] = fmax(0.0, v);
        }
    }
    rec[S_Z] = t[2];
    depth_model_f64(JS, S2, Sc, rec + 10);
}

/* L = v . record (+ vd . depth model when vd is given) */
static double proj_loss(const orc_camera* c, int sh_degree, const double* p, const float* v, const float* vd,
                        uint8_t trace[6])
{
    double rec[13];
    proj_record_f64(c, sh_degree, p, rec, trace);
    double L = 0.0;
    for (int f = 0; f < 10; ++f) L += (double)v[f] * rec[f];
    if (vd)
        for (int f = 0; f < 3; ++f) L += (double)vd[f] * rec[10 + f];
    return L;
}

/* dL/d p[param] of Gaussian gid for the requested pairs, L = sum_f
 * v_splats[gid][f] record_f (central differences at h and h/2, Richardson).
 * status: FD_OK; FD_FLIP a decision in the trace differs anywhere in
 * [-h, +h]; FD_NONSMOOTH the two step sizes disagree.  A Gaussian culled
 * throughout gets 0 with FD_OK.                                           */
void orc_project_fd(const orc_camera* c, int32_t sh_degree, const float* means, const float* log_scales,
                    const float* quats, const float* logits, const float* colors, const float* v_splats,
                    const float* v_depth_model, int32_t n, const int32_t* gids, const int32_t* params,
                    const double* hs, double* grad, int32_t* status)
{
    int np = PROJ_NPAR(sh_degree);
#pragma omp parallel for schedule(dynamic, 4)
    for (int32_t i = 0; i < n; ++i) {
        double p[PROJ_NPAR(3)], q[PROJ_NPAR(3)];
        int64_t g = gids[i];
        int k = params[i];
        double h = hs[i];
        const float* v = v_splats + S_STRIDE * g;
        const float* vd = v_depth_model ? v_depth_model + 4 * g : NULL;
        grad[i] = 0.0;
        status[i] = FD_OK;
        if (k < 0 || k >= np) {
            status[i] = FD_UNUSED;
            continue;
        }
        proj_load(sh_degree, g, means, log_scales, quats, logits, colors, p);
        uint8_t t0[6], tp[6], tm[6], tp2[6], tm2[6];
        proj_loss(c, sh_degree, p, v, vd, t0);
        memcpy(q, p, sizeof(double) * np);
        q[k] = p[k] + h;
        double lp = proj_loss(c, sh_degree, q, v, vd, tp);
        q[k] = p[k] - h;
        double lm = proj_loss(c, sh_degree, q, v, vd, tm);
        q[k] = p[k] + 0.5 * h;
        double lp2 = proj_loss(c, sh_degree, q, v, vd, tp2);
        q[k] = p[k] - 0.5 * h;
        double lm2 = proj_loss(c, sh_degree, q, v, vd, tm2);
        if (memcmp(t0, tp, 6) || memcmp(t0, tm, 6) || memcmp(t0, tp2, 6) || memcmp(t0, tm2, 6)) {
            status[i] = FD_FLIP;
            continue;
        }
        if (t0[0]) continue; /* culled throughout: zero gradient */
        status[i] = richardson(lp, lm, lp2, lm2, h, &grad[i]);
    }
}

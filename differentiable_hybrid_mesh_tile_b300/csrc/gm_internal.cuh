// Internal definitions shared by the libgm CUDA sources (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gm.h"

namespace gm {

constexpr int TILE = GM_TILE;
constexpr int TILE_PIX = TILE * TILE;

// Camera as passed to kernels (by value).
struct Cam {
    int W, H, TW, TH;
    float fx, fy, cx, cy, znear, zfar;
    float R[9];
    float t[3];
};

inline Cam make_cam(const gm_camera& c)
{
    Cam k;
    k.W = c.width;
    k.H = c.height;
    k.TW = (c.width + TILE - 1) / TILE;
    k.TH = (c.height + TILE - 1) / TILE;
    k.fx = c.fx; k.fy = c.fy; k.cx = c.cx; k.cy = c.cy;
    k.znear = c.near_plane; k.zfar = c.far_plane;
    for (int i = 0; i < 9; ++i) k.R[i] = c.R[i];
    for (int i = 0; i < 3; ++i) k.t[i] = c.t[i];
    return k;
}

// ---------------------------------------------------------------------------
// Coverage arithmetic.  Face ids and triangle bins are integers decided from
// fp32 arithmetic; these helpers evaluate each formula one correctly rounded
// operation at a time, in the written order, with no fused multiply-add, so
// the decisions are reproducible by any IEEE fp32 evaluation of the same
// formulas:
//   X_c = ((R0 X + R1 Y) + R2 Z) + t per row;   u = (fx x) / z + cx;
//   e(a -> b, p) = (ub - ua)(py - va) - (vb - va)(px - ua).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float cam_row_rn(const Cam& c, int r, float X, float Y, float Z)
{
    float s = __fmul_rn(c.R[3 * r + 0], X);
    s = __fadd_rn(s, __fmul_rn(c.R[3 * r + 1], Y));
    s = __fadd_rn(s, __fmul_rn(c.R[3 * r + 2], Z));
    return __fadd_rn(s, c.t[r]);
}

__device__ __forceinline__ float edge_rn(float ua, float va, float ub, float vb, float px, float py)
{
    float p = __fmul_rn(__fsub_rn(ub, ua), __fsub_rn(py, va));
    float q = __fmul_rn(__fsub_rn(vb, va), __fsub_rn(px, ua));
    return __fsub_rn(p, q);
}

struct Tri {
    float u[3], v[3], z[3];
    float area;          // edge function of v0 -> v1 at v2 (twice the signed area)
    int x0, x1, y0, y1;  // inclusive pixel-centre box, clamped to the image
};

// Projects face f; returns false when it is not drawn: a vertex index out of
// range, a vertex at or in front of the near plane (no clipping), zero area,
// or a pixel-centre box that misses the image.
__device__ __forceinline__ bool tri_setup(const Cam& c, const float* __restrict__ V, int nV,
                                          const int32_t* __restrict__ F, int f, Tri& t)
{
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        int vi = __ldg(F + 3 * (int64_t)f + k);
        if (vi < 0 || vi >= nV) return false;
        float X = __ldg(V + 3 * (int64_t)vi), Y = __ldg(V + 3 * (int64_t)vi + 1), Z = __ldg(V + 3 * (int64_t)vi + 2);
        float x = cam_row_rn(c, 0, X, Y, Z);
        float y = cam_row_rn(c, 1, X, Y, Z);
        float z = cam_row_rn(c, 2, X, Y, Z);
        if (!(z > c.znear)) return false;
        t.z[k] = z;
        t.u[k] = __fadd_rn(__fdiv_rn(__fmul_rn(c.fx, x), z), c.cx);
        t.v[k] = __fadd_rn(__fdiv_rn(__fmul_rn(c.fy, y), z), c.cy);
    }
    t.area = edge_rn(t.u[0], t.v[0], t.u[1], t.v[1], t.u[2], t.v[2]);
    if (!(t.area != 0.0f)) return false;
    float umin = fminf(fminf(t.u[0], t.u[1]), t.u[2]);
    float umax = fmaxf(fmaxf(t.u[0], t.u[1]), t.u[2]);
    float vmin = fminf(fminf(t.v[0], t.v[1]), t.v[2]);
    float vmax = fmaxf(fmaxf(t.v[0], t.v[1]), t.v[2]);
    float x0 = fmaxf(ceilf(__fsub_rn(umin, 0.5f)), 0.0f);
    float x1 = fminf(floorf(__fsub_rn(umax, 0.5f)), (float)(c.W - 1));
    float y0 = fmaxf(ceilf(__fsub_rn(vmin, 0.5f)), 0.0f);
    float y1 = fminf(floorf(__fsub_rn(vmax, 0.5f)), (float)(c.H - 1));
    if (!(x0 <= x1) || !(y0 <= y1)) return false;
    t.x0 = (int)x0; t.x1 = (int)x1; t.y0 = (int)y0; t.y1 = (int)y1;
    return true;
}

// q = t / w and r = t % w for t >= 0 and w >= 1, below 2^21 with one fp32 multiply:
// (t + 0.5) / w lies at least 0.5 / w from every integer, far more than the
// rounding error of (t + 0.5) * rn(1 / w).  (Integer division by a variable
// costs tens of instructions.)
__device__ __forceinline__ void divmod_small(int t, int w, float inv_w, int& q, int& r)
{
    q = t < (1 << 21) ? (int)(((float)t + 0.5f) * inv_w) : t / w;
    r = t - q * w;
}

// Tile rectangle [x0, x1) x [y0, y1) of a projected Gaussian of radius r:
// floor((m - r) / 16) .. ceil((m + r) / 16), clamped to the tile grid.
__device__ __forceinline__ bool gauss_rect(const Cam& c, float mx, float my, int r, int& x0, int& y0,
                                           int& x1, int& y1)
{
    if (r <= 0) return false;
    float fr = (float)r;
    float fx0 = floorf(__fdiv_rn(__fsub_rn(mx, fr), 16.0f));
    float fx1 = ceilf(__fdiv_rn(__fadd_rn(mx, fr), 16.0f));
    float fy0 = floorf(__fdiv_rn(__fsub_rn(my, fr), 16.0f));
    float fy1 = ceilf(__fdiv_rn(__fadd_rn(my, fr), 16.0f));
    float TW = (float)c.TW, TH = (float)c.TH;
    fx0 = fminf(fmaxf(fx0, 0.0f), TW); fx1 = fminf(fmaxf(fx1, 0.0f), TW);
    fy0 = fminf(fmaxf(fy0, 0.0f), TH); fy1 = fminf(fmaxf(fy1, 0.0f), TH);
    x0 = (int)fx0; x1 = (int)fx1; y0 = (int)fy0; y1 = (int)fy1;
    return x1 > x0 && y1 > y0;
}

// ---------------------------------------------------------------------------
// Sort / scan (gm_sort.cu)
// ---------------------------------------------------------------------------
constexpr int SCAN_THREADS = 256;
constexpr int SCAN_IPT = 16;
constexpr int SCAN_PART = SCAN_THREADS * SCAN_IPT;
constexpr int SORT_THREADS = 256;
constexpr int SORT_IPT = 8;
constexpr int SORT_PART = SORT_THREADS * SORT_IPT;
constexpr int SORT_MAX_PASSES = 8;

// bounded inter-block wait: polls before a waiting block gives up
constexpr uint32_t SPIN_LIMIT = GM_WAIT_LIMIT_DEFAULT;

struct ScanWs {
    uint32_t* desc;    // [parts]
    uint32_t* ticket;  // [1]
    int parts;
};

struct SortWs {
    uint64_t* keys_alt;  // [cap]
    int32_t* vals_alt;   // [cap]
    uint32_t* hist;      // [SORT_MAX_PASSES][256]
    uint32_t* desc;      // [passes][max_parts][256]
    uint32_t* tickets;   // [SORT_MAX_PASSES]
    int max_parts;
};

size_t scan_ws_bytes(int64_t n);
size_t sort_ws_bytes(int64_t cap);
// carve workspaces out of a byte buffer; returns bytes used (256-aligned pieces)
size_t carve_scan_ws(void* base, int64_t n, ScanWs& ws);
size_t carve_sort_ws(void* base, int64_t cap, SortWs& ws);
// bytes of ws that must be zero before each use (they start at the carve base)
size_t scan_zero_bytes(const ScanWs& ws);

// exclusive scan of counts[idx[i]] (counts[i] when idx is NULL) into
// offsets[i], i < n; total -> counters[GM_CNT_K]
cudaError_t exclusive_scan(const int32_t* counts, const int32_t* idx, int32_t* offsets, int n, int32_t* counters,
                           const ScanWs& ws, cudaStream_t s);
// Sort (keys, values) ascending by key bits [begin_bit, end_bit), stable.
// The count is min(*n_dev, cap), read on the device; a bounded wait that gives
// up sets GM_FLAG_TIMEOUT in counters.  Input is in (k0, v0); the result is
// in (k0, v0) when the number of passes is even and in the alternate buffers
// otherwise -- sort_passes() tells which.
// have_hist: the caller counted every pass's digit histogram into ws.hist
// (zeroed first by clear_sort_hist, which also resets the passes' tickets) and
// zeroed the passes' look-back descriptors (for pass p, the n_parts * 256 words
// at ws.desc + p * ws.max_parts * 256, n_parts = ceil(n / SORT_PART)); else the
// sort does both itself.
int sort_passes(int begin_bit, int end_bit);
cudaError_t radix_sort(uint64_t* k0, int32_t* v0, uint64_t* k1, int32_t* v1, int cap, int begin_bit,
                       int end_bit, const int32_t* n_dev, int32_t* counters, const SortWs& ws, cudaStream_t s,
                       bool have_hist = false);
cudaError_t clear_sort_hist(const SortWs& ws, cudaStream_t s);
// tile_range[T][2] from sorted keys (tile id in the high 32 bits); range zeroed first
cudaError_t tile_ranges(const uint64_t* keys, int cap, const int32_t* counters, int32_t* tile_range,
                        int n_tiles, cudaStream_t s);

int num_sms();
int set_last_error(int code, const char* fmt, ...);
// the bounded waits' poll limit (gm_set_wait_limit), process-wide; each launch
// that waits takes the value current when it is enqueued
void set_wait_limit(uint32_t polls);
uint32_t wait_limit();

// ---------------------------------------------------------------------------
// Host launchers of the path's steps (enqueue on stream s, no synchronisation)
// ---------------------------------------------------------------------------
size_t tri_bin_ws_bytes(int nF, int cap);
cudaError_t tri_bin(const Cam& c, const float* V, int nV, const int32_t* F, int nF, int32_t* tile_range,
                    int32_t* tri_ids, int cap, int32_t* counters, void* ws, cudaStream_t s);
size_t zbuffer_direct_ws_bytes(int nF, int W, int H);
cudaError_t zbuffer_direct(const Cam& c, const float* V, int nV, const int32_t* F, int nF, int32_t* face_id,
                           void* ws, cudaStream_t s);
cudaError_t zbuffer(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const int32_t* tile_range,
                    const int32_t* tri_ids, int32_t* face_id, cudaStream_t s);
cudaError_t interp(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const float* vcol,
                   const int32_t* face_id, float* mesh_depth, float* mesh_rgb, float* tile_far, uint8_t* tile_full,
                   cudaStream_t s);
cudaError_t mesh_bwd(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const float* vcol,
                     const int32_t* face_id, const float* T_final, const float* g_rgb, const float* g_depth,
                     const float* v_mesh_depth, float* v_verts, float* v_vcol, cudaStream_t s);

// softness > 0 (split 0: Phi, 1: logistic): record field 10 receives the soft
// split's hide depth for the occlusion cull
cudaError_t project(const Cam& c, int sh_degree, float softness, int split, int N, const float* means,
                    const float* log_scales, const float* quats, const float* logits, const float* colors,
                    float* splats, int32_t* radii, int32_t* tiles_touched, float* depth_model, cudaStream_t s);
cudaError_t project_views(const Cam* cams, int V, int sh_degree, float softness, int split, int N,
                          const float* means, const float* log_scales, const float* quats, const float* logits,
                          const float* colors, float* splats, int32_t* radii, int32_t* tiles_touched,
                          float* depth_model, cudaStream_t s);
cudaError_t project_bwd_views(const Cam* cams, int V, int sh_degree, int N, const float* means,
                              const float* log_scales, const float* quats, const float* logits, const float* colors,
                              const int32_t* radii, const float* v_splats, const float* v_depth_model,
                              bool accumulate, float* v_means, float* v_log_scales, float* v_quats, float* v_logits,
                              float* v_colors, cudaStream_t s);
cudaError_t project_bwd(const Cam& c, int sh_degree, int N, const float* means, const float* log_scales,
                        const float* quats, const float* logits, const float* colors, const int32_t* radii,
                        const float* v_splats, const float* v_depth_model, bool accumulate, float* v_means,
                        float* v_log_scales, float* v_quats, float* v_logits, float* v_colors, cudaStream_t s);
size_t gauss_bin_ws_bytes(int N, int cap);
// the two halves of gauss_bin_sort (same workspace, in this order, with nothing
// else using the workspace in between): the depth pre-sort needs no mesh
cudaError_t gauss_depth_sort(const Cam& c, int N, const float* splats, const int32_t* radii, int cap,
                             int32_t* counters, void* ws, cudaStream_t s);
cudaError_t gauss_bin(const Cam& c, bool cull, bool soft, bool tile_test, int N, const float* splats,
                      const int32_t* radii,
                      const float* tile_far, const uint8_t* tile_full, uint64_t* keys, int32_t* gids,
                      int32_t* tile_range, int cap, int32_t* counters, void* ws, cudaStream_t s);
cudaError_t gauss_bin_sort(const Cam& c, bool cull, bool soft, bool tile_test, int N, const float* splats,
                           const int32_t* radii,
                           const float* tile_far, const uint8_t* tile_full, uint64_t* keys, int32_t* gids,
                           int32_t* tile_range, int cap, int32_t* counters, void* ws, cudaStream_t s);

// The antialiased mesh layer and the buffers of its back chain (Hybrid
// rendering, two-layer equation).  cov == nullptr: coverage is face_id >= 0
// and the compositing is the one-layer form.
struct AaLayer {
    const float* cov;  // [H][W] coverage a; mesh_rgb is then premultiplied, mesh_depth the split depth
    float4* back;      // [H][W] colour and depth composited behind the layer (forward out, backward in)
    float* T_back;     // [H][W] transmittance of that chain
    int32_t* n_back;   // [H][W] 1 + list position of its last composited Gaussian
    float* v_cov;      // [H][W] backward out: dL/da
    float* v_rgb;      // [H][W][3] backward out: dL/dM
};

size_t mesh_edges_ws_bytes(int nF);
cudaError_t mesh_edges(const int32_t* F, int nF, int nV, int32_t* adj, int32_t* counters, void* ws, cudaStream_t s);
cudaError_t antialias(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const int32_t* adj,
                      const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb, float* cov,
                      float* rgb_aa, float* depth_aa, float* tile_far, uint8_t* tile_full, cudaStream_t s);
cudaError_t antialias_bwd(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const int32_t* adj,
                          const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb, const float* cov,
                          const float* depth_aa, const float* v_cov, const float* v_rgb_aa, const float* v_depth_aa,
                          float* v_mesh_rgb, float* v_mesh_depth, float* v_verts, cudaStream_t s);
cudaError_t interp_bwd(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const float* vcol,
                       const int32_t* face_id, const float* v_mesh_rgb, const float* v_mesh_depth, float* v_verts,
                       float* v_vcol, cudaStream_t s);

cudaError_t composite_fwd(const Cam& c, const float bg[3], int N, float softness, int split, const int32_t* tile_range,
                          const int32_t* gids, const float* splats, const float* depth_model, const float* mesh_depth,
                          const float* mesh_rgb, const int32_t* face_id, float* out_rgb, float* out_depth,
                          float* out_alpha, float* T_final, int32_t* n_contrib, const AaLayer& aa, float* staged,
                          int staged_cap, uint64_t* stats, cudaStream_t s);
cudaError_t composite_bwd(const Cam& c, const float bg[3], int N, float softness, int split, const int32_t* tile_range,
                          const int32_t* gids, const float* splats, const float* depth_model, const float* mesh_depth,
                          const float* mesh_rgb, const int32_t* face_id, const float* T_final,
                          const int32_t* n_contrib, const float* g_rgb, const float* g_depth, const float* g_alpha,
                          float* v_splats, float* v_depth_model, float* v_mesh_depth, const AaLayer& aa,
                          const float* staged, int staged_cap, uint64_t* stats, cudaStream_t s);
// bytes of a staged-record buffer of cap list positions (48 each, 64 with the soft split)
size_t staged_bytes(int cap, bool soft);
// the bulk-copy wait status (bit 0: a wait gave up), optionally cleared
cudaError_t copy_status(uint32_t* flags, bool clear);

}  // namespace gm

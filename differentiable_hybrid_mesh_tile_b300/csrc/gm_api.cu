// extern "C" entry points of libgm (declared in include/gm.h): argument
// checks, workspace carving, launches on the caller's stream, status codes.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "gm_internal.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* where)
{
    return fail(GM_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

gm::AaLayer layer_of(const gm_aa_layer* aa)
{
    gm::AaLayer l{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    if (aa && aa->cov) {
        l.cov = aa->cov;
        l.back = reinterpret_cast<float4*>(aa->back);
        l.T_back = aa->T_back;
        l.n_back = aa->n_back;
        l.v_cov = aa->v_cov;
        l.v_rgb = aa->v_rgb;
    }
    return l;
}

int check_cam(const gm_camera* cam)
{
    if (!cam) return fail(GM_ERR_INVALID_ARG, "camera is NULL");
    if (cam->width <= 0 || cam->height <= 0) return fail(GM_ERR_INVALID_ARG, "image size %dx%d", cam->width, cam->height);
    if (cam->width > (1 << 20) || cam->height > (1 << 20))
        return fail(GM_ERR_INVALID_ARG, "image size %dx%d too large", cam->width, cam->height);
    const float v[6] = {cam->fx, cam->fy, cam->cx, cam->cy, cam->near_plane, cam->far_plane};
    for (float x : v)
        if (!isfinite(x)) return fail(GM_ERR_INVALID_ARG, "camera intrinsics must be finite");
    if (!(cam->fx > 0.0f) || !(cam->fy > 0.0f)) return fail(GM_ERR_INVALID_ARG, "focal lengths must be > 0");
    if (!(cam->near_plane > 0.0f) || !(cam->far_plane > cam->near_plane))
        return fail(GM_ERR_INVALID_ARG, "need 0 < near < far");
    for (int i = 0; i < 9; ++i)
        if (!isfinite(cam->R[i])) return fail(GM_ERR_INVALID_ARG, "R must be finite");
    for (int i = 0; i < 3; ++i)
        if (!isfinite(cam->t[i])) return fail(GM_ERR_INVALID_ARG, "t must be finite");
    int64_t tiles = (int64_t)((cam->width + GM_TILE - 1) / GM_TILE) * ((cam->height + GM_TILE - 1) / GM_TILE);
    if (tiles > (1 << 24)) return fail(GM_ERR_INVALID_ARG, "too many tiles");
    return GM_OK;
}

#define GM_REQUIRE(cond, ...)                                   \
    do {                                                        \
        if (!(cond)) return fail(GM_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

// after the launches: optional host read-back of the counters
int finish_binning(int32_t* counters, int32_t* K_host, int32_t cap, cudaStream_t s)
{
    if (!K_host) return GM_OK;
    int32_t h[4];
    cudaError_t e = cudaMemcpyAsync(h, counters, sizeof(h), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading counters");
    *K_host = h[GM_CNT_K];
    if (h[GM_CNT_FLAGS] & GM_FLAG_TIMEOUT) return fail(GM_ERR_TIMEOUT, "a bounded inter-block wait gave up");
    if (h[GM_CNT_K] > cap) return fail(GM_ERR_CAPACITY, "need %d entries, capacity %d", h[GM_CNT_K], cap);
    return GM_OK;
}

}  // namespace

namespace gm {
// Records a message for gm_last_error() and returns code (used by entry
// points defined in other files).
int set_last_error(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}
}  // namespace gm

extern "C" {

const char* gm_last_error(void) { return g_err; }

size_t gm_staged_bytes(int32_t cap, float softness) { return gm::staged_bytes(cap, softness > 0.0f); }

int gm_get_copy_status(uint32_t* flags, int32_t clear)
{
    GM_REQUIRE(flags, "flags is NULL");
    cudaError_t e = gm::copy_status(flags, clear != 0);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_get_copy_status");
}

int gm_set_wait_limit(uint32_t polls)
{
    gm::set_wait_limit(polls);
    return GM_OK;
}

int gm_get_wait_limit(uint32_t* polls)
{
    GM_REQUIRE(polls, "polls is NULL");
    *polls = gm::wait_limit();
    return GM_OK;
}

size_t gm_bin_triangles_workspace_size(int32_t nF, int32_t cap, int32_t width, int32_t height)
{
    (void)width;
    (void)height;
    return gm::tri_bin_ws_bytes(nF < 0 ? 0 : nF, cap < 0 ? 0 : cap);
}

int gm_bin_triangles(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                     int32_t* tile_range, int32_t* tri_ids, int32_t cap, int32_t* counters, int32_t* K_host, void* ws,
                     size_t ws_bytes, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(nV >= 0 && nF >= 0 && cap >= 0, "negative size");
    GM_REQUIRE(nV == 0 || V, "V is NULL");
    GM_REQUIRE(nF == 0 || F, "F is NULL");
    GM_REQUIRE(tile_range && counters, "tile_range / counters is NULL");
    GM_REQUIRE(cap == 0 || tri_ids, "tri_ids is NULL");
    const size_t need = gm::tri_bin_ws_bytes(nF, cap);
    GM_REQUIRE(ws && ws_bytes >= need, "workspace of %zu bytes needed", need);
    GM_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = gm::tri_bin(gm::make_cam(*cam), V, nV, F, nF, tile_range, tri_ids, cap, counters, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "gm_bin_triangles");
    return finish_binning(counters, K_host, cap, s);
}

int gm_zbuffer(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
               const int32_t* tile_range, const int32_t* tri_ids, int32_t* face_id, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(nV >= 0 && nF >= 0, "negative size");
    GM_REQUIRE(nV == 0 || V, "V is NULL");
    GM_REQUIRE(nF == 0 || F, "F is NULL");
    GM_REQUIRE(tile_range && face_id, "tile_range / face_id is NULL");
    GM_REQUIRE(tri_ids || nF == 0, "tri_ids is NULL");
    cudaError_t e = gm::zbuffer(gm::make_cam(*cam), V, nV, F, nF, tile_range, tri_ids, face_id, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_zbuffer");
}

size_t gm_zbuffer_direct_workspace_size(int32_t nF, int32_t width, int32_t height)
{
    return gm::zbuffer_direct_ws_bytes(nF, width > 0 ? width : 0, height > 0 ? height : 0);
}

int gm_zbuffer_direct(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                      int32_t* face_id, void* ws, size_t ws_bytes, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(nV >= 0 && nF >= 0, "negative size");
    GM_REQUIRE(nV == 0 || V, "V is NULL");
    GM_REQUIRE(nF == 0 || F, "F is NULL");
    GM_REQUIRE(face_id, "face_id is NULL");
    const size_t need = gm::zbuffer_direct_ws_bytes(nF, cam->width, cam->height);
    GM_REQUIRE(ws && ws_bytes >= need, "workspace of %zu bytes needed", need);
    GM_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    cudaError_t e = gm::zbuffer_direct(gm::make_cam(*cam), V, nV, F, nF, face_id, ws, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_zbuffer_direct");
}

int gm_interp_mesh(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF, const float* vcol,
                   const int32_t* face_id, float* mesh_depth, float* mesh_rgb, float* tile_far, uint8_t* tile_full,
                   void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(nV >= 0 && nF >= 0, "negative size");
    GM_REQUIRE(nV == 0 || (V && vcol), "V / vcol is NULL");
    GM_REQUIRE(nF == 0 || F, "F is NULL");
    GM_REQUIRE(face_id && mesh_depth && mesh_rgb && tile_far && tile_full, "an output is NULL");
    cudaError_t e = gm::interp(gm::make_cam(*cam), V, nV, F, nF, vcol, face_id, mesh_depth, mesh_rgb, tile_far,
                               tile_full, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_interp_mesh");
}

int gm_project_gaussians(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* means,
                         const float* log_scales, const float* quats, const float* logits, const float* colors,
                         float* splats, int32_t* radii, int32_t* tiles_touched, float* depth_model, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(N >= 0, "negative N");
    GM_REQUIRE(opts->sh_degree >= -1 && opts->sh_degree <= 3, "sh_degree %d not in -1..3", opts->sh_degree);
    if (N > 0) {
        GM_REQUIRE(means && log_scales && quats && logits && colors, "an input is NULL");
        GM_REQUIRE(splats && radii && tiles_touched, "an output is NULL");
        GM_REQUIRE(aligned16(quats) && aligned16(splats), "quats / splats must be 16-byte aligned");
        if (opts->sh_degree == 1 || opts->sh_degree == 3)
            GM_REQUIRE(aligned16(colors), "SH coefficients must be 16-byte aligned");
    }
    GM_REQUIRE(!depth_model || aligned16(depth_model), "depth_model must be 16-byte aligned");
    cudaError_t e = gm::project(gm::make_cam(*cam), opts->sh_degree, opts->softness, opts->soft_split, N, means,
                                log_scales, quats, logits, colors, splats,
                                radii, tiles_touched, depth_model, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_project_gaussians");
}

int gm_project_gaussians_bwd(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* means,
                             const float* log_scales, const float* quats, const float* logits, const float* colors,
                             const int32_t* radii, const float* v_splats, const float* v_depth_model,
                             int32_t accumulate, float* v_means, float* v_log_scales, float* v_quats,
                             float* v_logits, float* v_colors, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(N >= 0, "negative N");
    GM_REQUIRE(opts->sh_degree >= -1 && opts->sh_degree <= 3, "sh_degree %d not in -1..3", opts->sh_degree);
    if (N > 0) {
        GM_REQUIRE(means && log_scales && quats && logits && colors && radii && v_splats, "an input is NULL");
        GM_REQUIRE(v_means && v_log_scales && v_quats && v_logits && v_colors, "an output is NULL");
        GM_REQUIRE(aligned16(quats) && aligned16(v_splats) && aligned16(v_quats),
                   "quats / v_splats / v_quats must be 16-byte aligned");
        if (opts->sh_degree == 1 || opts->sh_degree == 3)
            GM_REQUIRE(aligned16(colors) && aligned16(v_colors), "SH coefficients and their gradient must be "
                       "16-byte aligned");
    }
    GM_REQUIRE(!v_depth_model || aligned16(v_depth_model), "v_depth_model must be 16-byte aligned");
    cudaError_t e = gm::project_bwd(gm::make_cam(*cam), opts->sh_degree, N, means, log_scales, quats, logits, colors,
                                    radii, v_splats, v_depth_model, accumulate != 0, v_means, v_log_scales, v_quats,
                                    v_logits, v_colors, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_project_gaussians_bwd");
}

int gm_project_gaussians_views(const gm_camera* cams, int32_t V, const gm_opts* opts, int32_t N, const float* means,
                               const float* log_scales, const float* quats, const float* logits, const float* colors,
                               float* splats, int32_t* radii, int32_t* tiles_touched, float* depth_model,
                               void* stream)
{
    g_err[0] = 0;
    GM_REQUIRE(cams && V >= 1 && V <= GM_MAX_VIEWS, "cams is NULL or V = %d not in 1..%d", V, GM_MAX_VIEWS);
    GM_REQUIRE(!depth_model || aligned16(depth_model), "depth_model must be 16-byte aligned");
    for (int v = 0; v < V; ++v)
        if (int st = check_cam(cams + v)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(N >= 0, "negative N");
    GM_REQUIRE(opts->sh_degree >= -1 && opts->sh_degree <= 3, "sh_degree %d not in -1..3", opts->sh_degree);
    if (N > 0) {
        GM_REQUIRE(means && log_scales && quats && logits && colors, "an input is NULL");
        GM_REQUIRE(splats && radii && tiles_touched, "an output is NULL");
        GM_REQUIRE(aligned16(quats) && aligned16(splats), "quats / splats must be 16-byte aligned");
        if (opts->sh_degree == 1 || opts->sh_degree == 3)
            GM_REQUIRE(aligned16(colors), "SH coefficients must be 16-byte aligned");
    }
    gm::Cam c[GM_MAX_VIEWS];
    for (int v = 0; v < V; ++v) c[v] = gm::make_cam(cams[v]);
    cudaError_t e = gm::project_views(c, V, opts->sh_degree, opts->softness, opts->soft_split, N, means, log_scales,
                                      quats, logits, colors, splats, radii,
                                      tiles_touched, depth_model, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_project_gaussians_views");
}

int gm_project_gaussians_bwd_views(const gm_camera* cams, int32_t V, const gm_opts* opts, int32_t N,
                                   const float* means, const float* log_scales, const float* quats,
                                   const float* logits, const float* colors, const int32_t* radii,
                                   const float* v_splats, const float* v_depth_model, int32_t accumulate,
                                   float* v_means, float* v_log_scales, float* v_quats, float* v_logits,
                                   float* v_colors, void* stream)
{
    g_err[0] = 0;
    GM_REQUIRE(cams && V >= 1 && V <= GM_MAX_VIEWS, "cams is NULL or V = %d not in 1..%d", V, GM_MAX_VIEWS);
    for (int v = 0; v < V; ++v)
        if (int st = check_cam(cams + v)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(N >= 0, "negative N");
    GM_REQUIRE(opts->sh_degree >= -1 && opts->sh_degree <= 3, "sh_degree %d not in -1..3", opts->sh_degree);
    if (N > 0) {
        GM_REQUIRE(means && log_scales && quats && logits && colors && radii && v_splats, "an input is NULL");
        GM_REQUIRE(v_means && v_log_scales && v_quats && v_logits && v_colors, "an output is NULL");
        GM_REQUIRE(aligned16(quats) && aligned16(v_splats) && aligned16(v_quats),
                   "quats / v_splats / v_quats must be 16-byte aligned");
        if (opts->sh_degree == 1 || opts->sh_degree == 3)
            GM_REQUIRE(aligned16(colors) && aligned16(v_colors), "SH coefficients and their gradient must be "
                       "16-byte aligned");
    }
    gm::Cam c[GM_MAX_VIEWS];
    for (int v = 0; v < V; ++v) c[v] = gm::make_cam(cams[v]);
    GM_REQUIRE(!v_depth_model || aligned16(v_depth_model), "v_depth_model must be 16-byte aligned");
    cudaError_t e = gm::project_bwd_views(c, V, opts->sh_degree, N, means, log_scales, quats, logits, colors, radii,
                                          v_splats, v_depth_model, accumulate != 0, v_means, v_log_scales, v_quats,
                                          v_logits, v_colors, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_project_gaussians_bwd_views");
}

size_t gm_bin_sort_gaussians_workspace_size(int32_t N, int32_t cap, int32_t width, int32_t height)
{
    (void)width;
    (void)height;
    return gm::gauss_bin_ws_bytes(N < 0 ? 0 : N, cap < 0 ? 0 : cap);
}

int gm_sort_gaussians_by_depth(const gm_camera* cam, int32_t N, const float* splats, const int32_t* radii,
                               int32_t cap, int32_t* counters, void* ws, size_t ws_bytes, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(N >= 0 && cap >= 0, "negative size");
    GM_REQUIRE(N == 0 || (splats && radii), "splats / radii is NULL");
    GM_REQUIRE(N == 0 || aligned16(splats), "splats must be 16-byte aligned");
    GM_REQUIRE(counters, "counters is NULL");
    const size_t need = gm::gauss_bin_ws_bytes(N, cap);
    GM_REQUIRE(ws && ws_bytes >= need, "workspace of %zu bytes needed", need);
    GM_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    cudaError_t e = gm::gauss_depth_sort(gm::make_cam(*cam), N, splats, radii, cap, counters, ws,
                                         (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_sort_gaussians_by_depth");
}

int gm_bin_gaussians(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* splats,
                     const int32_t* radii, const float* tile_far, const uint8_t* tile_full, uint64_t* keys,
                     int32_t* gids, int32_t* tile_range, int32_t cap, int32_t* counters, int32_t* K_host,
                     void* ws, size_t ws_bytes, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(N >= 0 && cap >= 0, "negative size");
    GM_REQUIRE(N == 0 || (splats && radii), "splats / radii is NULL");
    GM_REQUIRE(N == 0 || aligned16(splats), "splats must be 16-byte aligned");
    GM_REQUIRE(!opts->cull_occluded || (tile_far && tile_full), "cull_occluded needs tile_far and tile_full");
    GM_REQUIRE(tile_range && counters, "tile_range / counters is NULL");
    GM_REQUIRE(cap == 0 || (keys && gids), "keys / gids is NULL");
    const size_t need = gm::gauss_bin_ws_bytes(N, cap);
    GM_REQUIRE(ws && ws_bytes >= need, "workspace of %zu bytes needed", need);
    GM_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    // the soft split culls on the record's hide depth (field 10, from gm_project_gaussians)
    const bool cull = opts->cull_occluded != 0, soft = opts->softness > 0.0f;
    cudaError_t e = gm::gauss_bin(gm::make_cam(*cam), cull, soft, opts->tile_test != 0, N, splats, radii, tile_far,
                                  tile_full, keys, gids, tile_range, cap, counters, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "gm_bin_gaussians");
    return finish_binning(counters, K_host, cap, s);
}

int gm_bin_sort_gaussians(const gm_camera* cam, const gm_opts* opts, int32_t N, const float* splats,
                          const int32_t* radii, const float* tile_far, const uint8_t* tile_full, uint64_t* keys,
                          int32_t* gids, int32_t* tile_range, int32_t cap, int32_t* counters, int32_t* K_host,
                          void* ws, size_t ws_bytes, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(N >= 0 && cap >= 0, "negative size");
    GM_REQUIRE(N == 0 || (splats && radii), "splats / radii is NULL");
    GM_REQUIRE(N == 0 || aligned16(splats), "splats must be 16-byte aligned");
    GM_REQUIRE(!opts->cull_occluded || (tile_far && tile_full), "cull_occluded needs tile_far and tile_full");
    GM_REQUIRE(tile_range && counters, "tile_range / counters is NULL");
    GM_REQUIRE(cap == 0 || (keys && gids), "keys / gids is NULL");
    const size_t need = gm::gauss_bin_ws_bytes(N, cap);
    GM_REQUIRE(ws && ws_bytes >= need, "workspace of %zu bytes needed", need);
    GM_REQUIRE(aligned16(ws), "workspace must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    // the soft split lets a Gaussian behind the mesh show through a little: no cull
    // the soft split culls on the record's hide depth (field 10, from gm_project_gaussians)
    const bool cull = opts->cull_occluded != 0, soft = opts->softness > 0.0f;
    cudaError_t e = gm::gauss_bin_sort(gm::make_cam(*cam), cull, soft, opts->tile_test != 0, N, splats,
                                       radii, tile_far,
                                       tile_full, keys, gids, tile_range, cap, counters, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "gm_bin_sort_gaussians");
    return finish_binning(counters, K_host, cap, s);
}

size_t gm_mesh_edges_workspace_size(int32_t nF)
{
    return nF < 0 ? 0 : gm::mesh_edges_ws_bytes(nF);
}

int gm_mesh_edges(const int32_t* F, int32_t nF, int32_t nV, int32_t* adj, int32_t* counters, void* ws,
                  size_t ws_bytes, void* stream)
{
    g_err[0] = 0;
    GM_REQUIRE(nF >= 0 && nV >= 0, "negative size");
    GM_REQUIRE(nF == 0 || (F && adj), "F / adj is NULL");
    GM_REQUIRE(counters, "counters is NULL");
    GM_REQUIRE(nF <= (1 << 29), "too many faces");
    GM_REQUIRE(nF == 0 || (ws && ws_bytes >= gm::mesh_edges_ws_bytes(nF)), "workspace too small");
    cudaError_t e = gm::mesh_edges(F, nF, nV, adj, counters, ws, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_mesh_edges");
}

int gm_antialias(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                 const int32_t* adj, const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb,
                 float* cov, float* rgb_aa, float* depth_aa, float* tile_far, uint8_t* tile_full, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(nV >= 0 && nF >= 0, "negative size");
    GM_REQUIRE(nF == 0 || (V && F && adj), "V / F / adj is NULL");
    GM_REQUIRE(face_id && mesh_depth && mesh_rgb, "an input is NULL");
    GM_REQUIRE(cov && rgb_aa && depth_aa && tile_far && tile_full, "an output is NULL");
    cudaError_t e = gm::antialias(gm::make_cam(*cam), V, nV, F, nF, adj, face_id, mesh_depth, mesh_rgb, cov, rgb_aa,
                                  depth_aa, tile_far, tile_full, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_antialias");
}

int gm_antialias_bwd(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                     const int32_t* adj, const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb,
                     const float* cov, const float* depth_aa, const float* v_cov, const float* v_rgb_aa,
                     const float* v_depth_aa, float* v_mesh_rgb, float* v_mesh_depth, float* v_verts, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(nV >= 0 && nF >= 0, "negative size");
    GM_REQUIRE(nF == 0 || (V && F && adj), "V / F / adj is NULL");
    GM_REQUIRE(face_id && mesh_depth && mesh_rgb && cov && depth_aa && v_cov && v_rgb_aa && v_depth_aa,
               "an input is NULL");
    GM_REQUIRE(v_mesh_rgb && v_mesh_depth && (v_verts || nV == 0), "an output is NULL");
    cudaError_t e = gm::antialias_bwd(gm::make_cam(*cam), V, nV, F, nF, adj, face_id, mesh_depth, mesh_rgb, cov,
                                      depth_aa, v_cov, v_rgb_aa, v_depth_aa, v_mesh_rgb, v_mesh_depth, v_verts,
                                      (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_antialias_bwd");
}

int gm_interp_mesh_bwd(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                       const float* vcol, const int32_t* face_id, const float* v_mesh_rgb,
                       const float* v_mesh_depth, float* v_verts, float* v_vcol, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(nV >= 0 && nF >= 0, "negative size");
    GM_REQUIRE(nF == 0 || (V && F && vcol), "V / F / vcol is NULL");
    GM_REQUIRE(face_id && v_mesh_rgb && v_mesh_depth, "an input is NULL");
    GM_REQUIRE(nV == 0 || (v_verts && v_vcol), "an output is NULL");
    if (nF == 0) return GM_OK;
    cudaError_t e = gm::interp_bwd(gm::make_cam(*cam), V, nV, F, nF, vcol, face_id, v_mesh_rgb, v_mesh_depth, v_verts,
                                   v_vcol, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_interp_mesh_bwd");
}

int gm_composite_hybrid_fwd(const gm_camera* cam, const gm_opts* opts, int32_t N, const int32_t* tile_range,
                            const int32_t* gids, const float* splats, const float* depth_model,
                            const float* mesh_depth, const float* mesh_rgb, const int32_t* face_id, float* out_rgb,
                            float* out_depth, float* out_alpha, float* T_final, int32_t* n_contrib,
                            const gm_aa_layer* aa, const gm_staged* staged, uint64_t* stats, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(opts->softness >= 0.0f, "negative softness");
    GM_REQUIRE(opts->soft_split == GM_SPLIT_PHI || opts->soft_split == GM_SPLIT_LOGISTIC, "soft_split %d unknown",
               opts->soft_split);
    const bool aa_on = aa && aa->cov;
    GM_REQUIRE(tile_range && mesh_depth && mesh_rgb && (face_id || aa_on), "an input is NULL");
    GM_REQUIRE(out_rgb && out_depth && out_alpha && T_final && n_contrib, "an output is NULL");
    if (aa_on)
        GM_REQUIRE(aa->back && aligned16(aa->back) && aa->T_back && aa->n_back,
                   "the antialiased layer needs back (16-byte aligned), T_back and n_back");
    GM_REQUIRE(N >= 0, "negative N");
    GM_REQUIRE(N == 0 || (splats && gids), "splats / gids is NULL");
    GM_REQUIRE(!splats || aligned16(splats), "splats must be 16-byte aligned");
    const bool soft = opts->softness > 0.0f;
    GM_REQUIRE(!soft || N == 0 || (depth_model && aligned16(depth_model)),
               "the soft split needs a 16-byte aligned depth_model");
    if (staged) GM_REQUIRE(staged->recs && aligned16(staged->recs) && staged->cap >= 0,
                           "staged records need a 16-byte aligned buffer and a capacity >= 0");
    cudaError_t e = gm::composite_fwd(gm::make_cam(*cam), opts->bg, N, opts->softness, opts->soft_split, tile_range,
                                      gids, splats,
                                      depth_model, mesh_depth, mesh_rgb, face_id, out_rgb, out_depth, out_alpha,
                                      T_final, n_contrib, layer_of(aa), staged ? staged->recs : nullptr,
                                      staged ? staged->cap : 0, stats, (cudaStream_t)stream);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_composite_hybrid_fwd");
}

int gm_composite_hybrid_bwd(const gm_camera* cam, const gm_opts* opts, int32_t N, const int32_t* tile_range,
                            const int32_t* gids, const float* splats, const float* depth_model,
                            const float* mesh_depth, const float* mesh_rgb, const int32_t* face_id,
                            const float* T_final, const int32_t* n_contrib, const float* g_rgb, const float* g_depth,
                            const float* g_alpha, float* v_splats, float* v_depth_model, float* v_mesh_depth,
                            const float* V, int32_t nV, const int32_t* F, int32_t nF, const float* vcol,
                            float* v_verts, float* v_vcol, const gm_aa_layer* aa, const gm_staged* staged,
                            uint64_t* stats, void* stream)
{
    g_err[0] = 0;
    if (int st = check_cam(cam)) return st;
    GM_REQUIRE(opts, "opts is NULL");
    GM_REQUIRE(opts->softness >= 0.0f, "negative softness");
    GM_REQUIRE(opts->soft_split == GM_SPLIT_PHI || opts->soft_split == GM_SPLIT_LOGISTIC, "soft_split %d unknown",
               opts->soft_split);
    const bool soft = opts->softness > 0.0f;
    if (soft && v_splats && N > 0)
        GM_REQUIRE(depth_model && aligned16(depth_model) && v_depth_model && aligned16(v_depth_model),
                   "the soft split needs 16-byte aligned depth_model and v_depth_model");
    const bool aa_on = aa && aa->cov;
    GM_REQUIRE(tile_range && mesh_depth && mesh_rgb && (face_id || aa_on) && T_final && n_contrib,
               "an input is NULL");
    if (aa_on) {
        GM_REQUIRE(aa->back && aligned16(aa->back) && aa->T_back && aa->n_back && aa->v_cov && aa->v_rgb,
                   "the antialiased layer needs back (16-byte aligned), T_back, n_back, v_cov and v_rgb");
        GM_REQUIRE(v_mesh_depth, "the antialiased layer's gradient needs v_mesh_depth");
        GM_REQUIRE(!V && !F && !vcol && !v_verts && !v_vcol,
                   "with the antialiased layer the mesh gradients come from gm_antialias_bwd");
    }
    GM_REQUIRE(g_rgb && g_depth && g_alpha, "an upstream gradient is NULL");
    GM_REQUIRE(!splats || aligned16(splats), "splats must be 16-byte aligned");
    GM_REQUIRE(!v_splats || aligned16(v_splats), "v_splats must be 16-byte aligned");
    if (staged) GM_REQUIRE(staged->recs && aligned16(staged->recs) && staged->cap >= 0,
                           "staged records need a 16-byte aligned buffer and a capacity >= 0");
    GM_REQUIRE(nV >= 0 && nF >= 0 && N >= 0, "negative size");
    GM_REQUIRE(N == 0 || !v_splats || (splats && gids), "splats / gids is NULL");
    const bool mesh_grads = v_verts || v_vcol;
    if (mesh_grads) GM_REQUIRE(v_verts && v_vcol && (nF == 0 || (F && V && vcol)), "mesh gradient arguments incomplete");
    if (soft && mesh_grads) GM_REQUIRE(v_mesh_depth, "the soft split's mesh gradients need v_mesh_depth");
    cudaStream_t s = (cudaStream_t)stream;
    const gm::Cam c = gm::make_cam(*cam);
    cudaError_t e = cudaSuccess;
    if (v_splats)
        e = gm::composite_bwd(c, opts->bg, N, opts->softness, opts->soft_split, tile_range, gids, splats, depth_model,
                              mesh_depth,
                              mesh_rgb, face_id, T_final, n_contrib, g_rgb, g_depth, g_alpha, v_splats, v_depth_model,
                              soft || aa_on ? v_mesh_depth : nullptr, layer_of(aa), staged ? staged->recs : nullptr,
                              staged ? staged->cap : 0, stats, s);
    if (e == cudaSuccess && mesh_grads && nF > 0)
        e = gm::mesh_bwd(c, V, nV, F, nF, vcol, face_id, T_final, g_rgb, g_depth, soft ? v_mesh_depth : nullptr,
                         v_verts, v_vcol, s);
    return e == cudaSuccess ? GM_OK : cuda_fail(e, "gm_composite_hybrid_bwd");
}

}  // extern "C"

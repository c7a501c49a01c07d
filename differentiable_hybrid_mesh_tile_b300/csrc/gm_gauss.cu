// Gaussian side of the hybrid renderer ("A Lightweight and Differentiable
// Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Hybrid rendering):
// EWA projection with SH colour, and the tile binning by 64-bit
// (tile | depth) keys with the per-tile occlusion cull.
#include <algorithm>

#include "gm_internal.cuh"
#include "gm_lookback.cuh"
#include "gm_proj.cuh"

namespace gm {
namespace {

// The record, radius and tile count of Gaussian g seen by camera c.
// DEG < 0: colours are RGB [N][3]; else SH coefficients [N][(DEG+1)^2][3].
// sh_row: the Gaussian's SH row staged in shared memory (ShStage), or null.
template <int DEG>
__device__ __forceinline__ void project_gaussian(const Cam& c, const ProjConsts& pc, int g,
                                                 const float* __restrict__ means,
                                                 const float* __restrict__ log_scales,
                                                 const float4* __restrict__ quats, const float* __restrict__ logits,
                                                 const float* __restrict__ colors, float4& o0, float4& o1, float4& o2,
                                                 float4& dm, int& rad, int& touched, const float4* sh_row = nullptr)
{
    o0 = make_float4(0.f, 0.f, 0.f, 0.f);
    o1 = o0;
    o2 = o0;
    dm = o0;
    rad = 0;
    touched = 0;
    if (DEG >= 1 && !sh_row) {
        // the SH row is read only after the culling tests and the covariance: ask
        // for its cache lines now (a row of 3 (DEG + 1)^2 floats spans at most two
        // 128-byte lines), so that its loads later find them in L2
        constexpr int ROW = 3 * (DEG + 1) * (DEG + 1);
        const float* row = colors + (int64_t)g * ROW;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + ROW - 1));
    }
    const float mx = __ldg(means + 3 * (int64_t)g), my = __ldg(means + 3 * (int64_t)g + 1),
                mz = __ldg(means + 3 * (int64_t)g + 2);
    // every per-Gaussian input is requested before the tests that may not need it,
    // so that the loads overlap
    const float4 q = __ldg(quats + g);
    float s[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) s[k] = __ldg(log_scales + 3 * (int64_t)g + k);
    const float logit = __ldg(logits + g);
    const float tx = fmaf(c.R[0], mx, fmaf(c.R[1], my, fmaf(c.R[2], mz, c.t[0])));
    const float ty = fmaf(c.R[3], mx, fmaf(c.R[4], my, fmaf(c.R[5], mz, c.t[1])));
    const float tz = fmaf(c.R[6], mx, fmaf(c.R[7], my, fmaf(c.R[8], mz, c.t[2])));
    if (tz > c.znear && tz <= c.zfar) {
        // M = R(q) diag(exp(log_s)); camera-frame factor WM = R_cw M
        const float qi = 1.0f / sqrtf(q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
        const float w = q.x * qi, x = q.y * qi, y = q.z * qi, z = q.w * qi;
        const float Rq[3][3] = {{1.f - 2.f * (y * y + z * z), 2.f * (x * y - w * z), 2.f * (x * z + w * y)},
                                {2.f * (x * y + w * z), 1.f - 2.f * (x * x + z * z), 2.f * (y * z - w * x)},
                                {2.f * (x * z - w * y), 2.f * (y * z + w * x), 1.f - 2.f * (x * x + y * y)}};
#pragma unroll
        for (int k = 0; k < 3; ++k) s[k] = expf(s[k]);
        float WM[3][3];
#pragma unroll
        for (int r = 0; r < 3; ++r)
#pragma unroll
            for (int k = 0; k < 3; ++k)
                WM[r][k] = (c.R[3 * r] * Rq[0][k] + c.R[3 * r + 1] * Rq[1][k] + c.R[3 * r + 2] * Rq[2][k]) * s[k];
        // Jacobian of the pinhole map at the clamped direction; G = J WM, Sigma2 = G G^T + 0.3 I
        const float iz = 1.0f / tz;
        const float txc = tz * fminf(pc.limx_pos, fmaxf(-pc.limx_neg, tx * iz));
        const float tyc = tz * fminf(pc.limy_pos, fmaxf(-pc.limy_neg, ty * iz));
        const float j00 = c.fx * iz, j02 = -c.fx * txc * iz * iz;
        const float j11 = c.fy * iz, j12 = -c.fy * tyc * iz * iz;
        float G0[3], G1[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            G0[k] = fmaf(j00, WM[0][k], j02 * WM[2][k]);
            G1[k] = fmaf(j11, WM[1][k], j12 * WM[2][k]);
        }
        const float a = G0[0] * G0[0] + G0[1] * G0[1] + G0[2] * G0[2] + 0.3f;
        const float b = G0[0] * G1[0] + G0[1] * G1[1] + G0[2] * G1[2];
        const float cc = G1[0] * G1[0] + G1[1] * G1[1] + G1[2] * G1[2] + 0.3f;
        const float det = a * cc - b * b;
        if (det > 0.0f) {
            const float m = 0.5f * (a + cc), h = 0.5f * (a - cc);
            const float lam = m + sqrtf(h * h + b * b);
            rad = (int)ceilf(3.0f * sqrtf(lam));
            const float u = fmaf(c.fx * tx, iz, c.cx);
            const float v = fmaf(c.fy * ty, iz, c.cy);
            int x0, y0, x1, y1;
            if (gauss_rect(c, u, v, rad, x0, y0, x1, y1)) {
                touched = (x1 - x0) * (y1 - y0);
                const float idet = 1.0f / det;
                const float op = 1.0f / (1.0f + expf(-logit));
                float rgb[3];
                if (DEG < 0) {
#pragma unroll
                    for (int ch = 0; ch < 3; ++ch) rgb[ch] = __ldg(colors + 3 * (int64_t)g + ch);
                } else {
                    constexpr int K = (DEG < 0 ? 1 : (DEG + 1) * (DEG + 1));
                    float dx = mx - pc.cpx, dy = my - pc.cpy, dz = mz - pc.cpz;
                    const float dn = 1.0f / sqrtf(dx * dx + dy * dy + dz * dz);
                    dx *= dn; dy *= dn; dz *= dn;
                    float Y[16];
                    sh_basis<DEG>(dx, dy, dz, Y);
                    float acc[3] = {0.5f, 0.5f, 0.5f};
                    const float* cf = colors + (int64_t)g * (3 * K);
                    if ((3 * K) % 4 == 0) {
                        const float4* cf4 = reinterpret_cast<const float4*>(cf);
#pragma unroll
                        for (int v4 = 0; v4 < 3 * K / 4; ++v4) {
                            const float4 e = sh_row ? sh_row[v4] : __ldg(cf4 + v4);
                            const float ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
                            for (int l = 0; l < 4; ++l) {
                                const int idx = 4 * v4 + l;
                                acc[idx % 3] = fmaf(Y[idx / 3], ev[l], acc[idx % 3]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int idx = 0; idx < 3 * K; ++idx) acc[idx % 3] = fmaf(Y[idx / 3], __ldg(cf + idx), acc[idx % 3]);
                    }
#pragma unroll
                    for (int ch = 0; ch < 3; ++ch) rgb[ch] = fmaxf(acc[ch], 0.0f);
                }
                o0 = make_float4(u, v, cc * idet, -b * idet);
                o1 = make_float4(a * idet, op, rgb[0], rgb[1]);
                o2 = make_float4(rgb[2], tz, 0.0f, 0.0f);
                // depth model of the soft split: with Sigma_c = WM WM^T, Sigma_uv,z =
                // J Sigma_c e_z = G WM_2^T and Sigma_zz = |WM_2|^2; g = conic Sigma_uv,z
                // (the conic is (Sigma_uv + 0.3 I)^-1), sigma_z^2 = Sigma_zz - Sigma_uv,z . g
                const float bu = G0[0] * WM[2][0] + G0[1] * WM[2][1] + G0[2] * WM[2][2];
                const float bv = G1[0] * WM[2][0] + G1[1] * WM[2][1] + G1[2] * WM[2][2];
                const float szz = WM[2][0] * WM[2][0] + WM[2][1] * WM[2][1] + WM[2][2] * WM[2][2];
                const float gu = (cc * bu - b * bv) * idet, gv = (a * bv - b * bu) * idet;
                const float quad = bu * gu + bv * gv;  // g^T (Sigma_uv + 0.3 I) g
                const float var = szz - quad;
                // reach: over the ellipse where alpha can reach 1/255 (sigma <= ln(255 o),
                // with the tile test's margins), g . d <= sqrt(2 ln(255 o) g^T Sigma2 g)
                const float L = fmaf(fmaxf(logf(255.0f * op), 0.0f), 1.001f, 1e-4f);
                const float reach = sqrtf(2.0f * L * fmaxf(quad, 0.0f)) * 1.002f;
                dm = make_float4(gu, gv, sqrtf(fmaxf(var, 1e-12f)), reach);
            } else {
                rad = 0;
            }
        }
    }
}

// The record's field 10 under the soft split: the depth beyond which the
// mesh hides the Gaussian (z_c - R - tail sigma_z softness, less a rounding
// margin; the compositing's own bound, computed from the same stored values).
// 0 under the hard split (the occlusion cull then uses the centre depth).
struct SoftCull {
    float softness, tail;  // softness 0: hard split
};

__device__ __forceinline__ float hide_depth(const SoftCull& sc, float z, const float4& dm)
{
    const float band = dm.z * sc.softness;
    return z - fmaf(sc.tail, band, dm.w) * 1.0001f - 2e-6f * fabsf(z);
}

template <int DEG>
__global__ void __launch_bounds__(PROJ_THREADS)
k_project(Cam c, ProjConsts pc, SoftCull sc, int N, const float* __restrict__ means, const float* __restrict__ log_scales,
          const float4* __restrict__ quats, const float* __restrict__ logits, const float* __restrict__ colors,
          float4* __restrict__ splats, int32_t* __restrict__ radii, int32_t* __restrict__ tiles_touched,
          float4* __restrict__ depth_model)
{
    constexpr int ROW4 = ShStage<DEG>::ROW4;
    __shared__ float4 s_sh[ROW4 ? PROJ_THREADS * ShStage<DEG>::STRIDE : 1];
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if constexpr (ROW4 > 0) {
        stage_sh_rows<DEG>(colors, blockIdx.x * blockDim.x, N, s_sh);
        __syncthreads();
    }
    if (g >= N) return;
    float4 o0, o1, o2, dm;
    int rad, touched;
    project_gaussian<DEG>(c, pc, g, means, log_scales, quats, logits, colors, o0, o1, o2, dm, rad, touched,
                          ROW4 ? s_sh + threadIdx.x * ShStage<DEG>::STRIDE : nullptr);
    if (sc.softness > 0.0f && rad > 0) o2.z = hide_depth(sc, o2.y, dm);
    splats[3 * (int64_t)g] = o0;
    splats[3 * (int64_t)g + 1] = o1;
    splats[3 * (int64_t)g + 2] = o2;
    radii[g] = rad;
    tiles_touched[g] = touched;
    if (depth_model) depth_model[g] = dm;
}

// Several views in one launch: each thread takes one Gaussian through every
// view of the batch, so its parameters come from DRAM once (its SH row staged
// in shared memory for all views, the rest found in L1 / L2 by later views);
// outputs are [view][N] arrays.
template <int DEG>
__global__ void __launch_bounds__(PROJ_THREADS)
k_project_views(ViewBatch vb, SoftCull sc, int N, const float* __restrict__ means, const float* __restrict__ log_scales,
                const float4* __restrict__ quats, const float* __restrict__ logits, const float* __restrict__ colors,
                float4* __restrict__ splats, int32_t* __restrict__ radii, int32_t* __restrict__ tiles_touched,
                float4* __restrict__ depth_model)
{
    constexpr int ROW4 = ShStage<DEG>::ROW4;
    __shared__ float4 s_sh[ROW4 ? PROJ_THREADS * ShStage<DEG>::STRIDE : 1];
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if constexpr (ROW4 > 0) {
        stage_sh_rows<DEG>(colors, blockIdx.x * blockDim.x, N, s_sh);
        __syncthreads();
    }
    if (g >= N) return;
    for (int v = 0; v < vb.n; ++v) {
        float4 o0, o1, o2, dm;
        int rad, touched;
        project_gaussian<DEG>(vb.cam[v], vb.pc[v], g, means, log_scales, quats, logits, colors, o0, o1, o2, dm, rad,
                              touched, ROW4 ? s_sh + threadIdx.x * ShStage<DEG>::STRIDE : nullptr);
        if (sc.softness > 0.0f && rad > 0) o2.z = hide_depth(sc, o2.y, dm);
        const int64_t i = (int64_t)v * N + g;
        splats[3 * i] = o0;
        splats[3 * i + 1] = o1;
        splats[3 * i + 2] = o2;
        radii[i] = rad;
        tiles_touched[i] = touched;
        if (depth_model) depth_model[i] = dm;
    }
}

// ------------------------------------------------------------- binning ----

// Which tiles of a Gaussian's rectangle get an entry.
struct BinRule {
    bool cull;        // drop tiles where the mesh hides the Gaussian (tile_full, depth >= tile_far)
    bool soft;        // soft split: hidden when the record's field 10 (hide depth) lies beyond tile_far
    bool tile_test;   // drop tiles no pixel centre of which the Gaussian reaches with alpha >= 1/255
    const float* __restrict__ tile_far;
    const uint8_t* __restrict__ tile_full;
    int TW;
};

// What the per-tile tests need of one Gaussian.
struct BinShape {
    float mx, my, a, b, c;  // mean and conic: sigma(d) = (a dx^2 + c dy^2) / 2 + b dx dy
    float nba, nbc;         // -b / a, -b / c: vertex of sigma along a line of constant v / u
    float smax;             // alpha >= 1/255 needs sigma <= ln(255 o); smax adds a margin
    float depth;
    float hide;             // record field 10: hide depth under the soft split (0: none)
    bool degenerate;        // conic not positive definite: every tile is kept
};

__device__ __forceinline__ BinShape bin_shape(const float4* __restrict__ splats, int g)
{
    const float4 s0 = splats[3 * (int64_t)g], s1 = splats[3 * (int64_t)g + 1];
    BinShape b;
    b.mx = s0.x; b.my = s0.y; b.a = s0.z; b.b = s0.w; b.c = s1.x;
    b.degenerate = !(b.a > 0.0f) || !(b.a * b.c - b.b * b.b > 0.0f);
    b.nba = b.degenerate ? 0.0f : -b.b / b.a;
    b.nbc = b.degenerate ? 0.0f : -b.b / b.c;
    // 0.1 % + 1e-4 above ln(255 o): the fp32 evaluation of sigma at a pixel centre
    // (compositing) can never keep a pair this test drops
    const float thr = logf(255.0f * s1.y);
    b.smax = thr + 1e-3f * fabsf(thr) + 1e-4f;
    const float4 s2 = splats[3 * (int64_t)g + 2];
    b.depth = s2.y;
    b.hide = s2.z;
    return b;
}

__device__ __forceinline__ BinShape shfl_shape(const BinShape& s, int j)
{
    BinShape o;
    o.mx = __shfl_sync(0xffffffffu, s.mx, j); o.my = __shfl_sync(0xffffffffu, s.my, j);
    o.a = __shfl_sync(0xffffffffu, s.a, j); o.b = __shfl_sync(0xffffffffu, s.b, j);
    o.c = __shfl_sync(0xffffffffu, s.c, j); o.smax = __shfl_sync(0xffffffffu, s.smax, j);
    o.nba = __shfl_sync(0xffffffffu, s.nba, j); o.nbc = __shfl_sync(0xffffffffu, s.nbc, j);
    o.depth = __shfl_sync(0xffffffffu, s.depth, j);
    o.hide = __shfl_sync(0xffffffffu, s.hide, j);
    o.degenerate = __shfl_sync(0xffffffffu, (int)s.degenerate, j) != 0;
    return o;
}

// Smallest sigma over the pixel centres of tile (tx, ty), relaxed to the
// tile's 15 x 15 px square of centres: 0 when it holds the mean, else on an
// edge, where sigma is a 1D parabola minimised at a clamped vertex.  A
// degenerate conic gives -inf (the tile is kept).
__device__ __forceinline__ float tile_min_sigma(const BinShape& s, int tx, int ty)
{
    if (s.degenerate) return -INFINITY;
    const float u0 = (float)(tx * TILE) + 0.5f - s.mx, u1 = u0 + (float)(TILE - 1);
    const float v0 = (float)(ty * TILE) + 0.5f - s.my, v1 = v0 + (float)(TILE - 1);
    if (u0 <= 0.0f && u1 >= 0.0f && v0 <= 0.0f && v1 >= 0.0f) return 0.0f;
    float best = INFINITY;
    {   // edges u = u0, u1: v* = -b u / c
        const float va = fminf(fmaxf(s.nbc * u0, v0), v1), vb = fminf(fmaxf(s.nbc * u1, v0), v1);
        best = fminf(best, 0.5f * (s.a * u0 * u0 + s.c * va * va) + s.b * u0 * va);
        best = fminf(best, 0.5f * (s.a * u1 * u1 + s.c * vb * vb) + s.b * u1 * vb);
    }
    {   // edges v = v0, v1: u* = -b v / a
        const float ua = fminf(fmaxf(s.nba * v0, u0), u1), ub = fminf(fmaxf(s.nba * v1, u0), u1);
        best = fminf(best, 0.5f * (s.a * ua * ua + s.c * v0 * v0) + s.b * ua * v0);
        best = fminf(best, 0.5f * (s.a * ub * ub + s.c * v1 * v1) + s.b * ub * v1);
    }
    return best;
}

// Whether the mesh hides the Gaussian (centre depth, hide depth) in tile t.
__device__ __forceinline__ bool tile_hidden(const BinRule& r, int t, float depth, float hide)
{
    if (!r.cull || !__ldg(r.tile_full + t)) return false;
    const float far = __ldg(r.tile_far + t);
    // the soft split's per-pixel skip takes the same bound against each pixel's depth
    return r.soft ? hide > far + 4e-6f * fabsf(far) : depth >= far;
}

__device__ __forceinline__ bool keep_tile(const BinRule& r, const BinShape& s, int tx, int ty)
{
    if (tile_hidden(r, ty * r.TW + tx, s.depth, s.hide)) return false;
    return !r.tile_test || tile_min_sigma(s, tx, ty) <= s.smax;
}

// Rectangles up to this many tiles are walked by their own thread; larger ones
// (near-camera Gaussians) by the whole warp, 32 tiles at a time, so one large
// Gaussian does not hold up the other 31 lanes.
constexpr int SMALL_RECT = 16;

// Depth keys of the pre-sort: the centre depth's bits for a Gaussian whose tile
// rectangle is not empty, all ones otherwise (it emits nothing and sorts last);
// ids as values.  Needs no mesh, so it can run before the mesh layer exists.
__global__ void __launch_bounds__(256)
// The keys' digit histograms of the four 8-bit passes of the depth sort are
// counted here (block sums in shared memory, then global atomics), and the
// passes' look-back descriptors cleared (desc_words words from desc): the sort
// needs no histogram pass over the keys.
k_gauss_depth_keys(Cam c, int N, const float4* __restrict__ splats, const int32_t* __restrict__ radii,
                   uint64_t* __restrict__ dkey, int32_t* __restrict__ dval, int32_t* n_dev,
                   uint32_t* __restrict__ hist, uint32_t* __restrict__ desc, int max_parts)
{
    __shared__ uint32_t s_hist[4][256];
    for (int t = threadIdx.x; t < 4 * 256; t += blockDim.x) (&s_hist[0][0])[t] = 0u;
    // the passes' descriptors: pass p uses ceil(N / SORT_PART) * 256 words at p * max_parts * 256
    const int64_t parts = ((int64_t)N + SORT_PART - 1) / SORT_PART, per = parts * 256;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < 4 * per;
         t += (int64_t)gridDim.x * blockDim.x)
        desc[(t / per) * (int64_t)max_parts * 256 + t % per] = 0u;
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) *n_dev = N;
    // a grid of a few CTAs per SM, each over many Gaussians, so that the block sums
    // reach the global histograms with few atomics
    for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < N; g += gridDim.x * blockDim.x) {
        const int r = radii[g];
        bool vis = false;
        float depth = 0.0f;
        if (r > 0) {
            const float4 s0 = splats[3 * (int64_t)g];
            depth = splats[3 * (int64_t)g + 2].y;
            int x0, y0, x1, y1;
            vis = gauss_rect(c, s0.x, s0.y, r, x0, y0, x1, y1);
        }
        const uint32_t key = vis ? __float_as_uint(depth) : 0xffffffffu;
        dkey[g] = (uint64_t)key;
        dval[g] = g;
#pragma unroll
        for (int p = 0; p < 4; ++p) atomicAdd(&s_hist[p][(key >> (8 * p)) & 0xffu], 1u);
    }
    __syncthreads();
    for (int t = threadIdx.x; t < 4 * 256; t += blockDim.x) {
        const uint32_t v = (&s_hist[0][0])[t];
        if (v) atomicAdd(hist + t, v);
    }
}

// What the binning keeps of a Gaussian, one record per position of the depth
// order: a = (x0, y0, rectangle width, Gaussian id), b = (rectangle area in
// tiles, tile mask, centre-depth bits, hide-depth bits).  For a rectangle of
// at most SMALL_RECT tiles the mask holds the tiles (row-major bit order) the
// per-tile ellipse test keeps; larger rectangles are tested tile by tile when
// they are binned.  An empty rectangle or an invalid id has area 0.
struct GaussRec {
    int4 a, b;
};

// Per position i of the depth order: the Gaussian's tile rectangle and the
// ellipse test of its tiles.  Needs no mesh, so it runs before the mesh layer
// exists; only the occlusion cull waits for it.
__global__ void __launch_bounds__(256)
k_gauss_shape(Cam c, int N, const float4* __restrict__ splats, const int32_t* __restrict__ radii,
              const int32_t* __restrict__ order, GaussRec* __restrict__ rec, int32_t* counters)
{
    __shared__ int s_pre[8];
    __shared__ BinShape s_shape[256];
    __shared__ int4 s_rect[256];  // x0, y0, width, 1 / width bits
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const int wbase = threadIdx.x & ~31;
    int g = -1, pre = 0, x0 = 0, y0 = 0, x1 = 0, y1 = 0;
    BinShape sh = {};
    if (i < N) {
        const int gi = order[i];
        if (gi >= 0 && gi < N) {
            const int r = radii[gi];
            if (r > 0) {
                sh = bin_shape(splats, gi);
                if (gauss_rect(c, sh.mx, sh.my, r, x0, y0, x1, y1)) {
                    pre = (x1 - x0) * (y1 - y0);
                    g = gi;
                }
            }
        }
    }
    BinRule rule = {};
    rule.tile_test = true;
    rule.TW = c.TW;
    // the (Gaussian, tile) pairs of the warp's small rectangles, flattened so that
    // each lane tests one pair per round whatever the rectangle sizes
    uint32_t mask = 0;
    const int a = pre <= SMALL_RECT ? pre : 0;
    int o = a;  // inclusive prefix sum over the lanes
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, o, d);
        if (lane >= d) o += y;
    }
    const int total = __shfl_sync(0xffffffffu, o, 31);
    o -= a;  // exclusive
    s_shape[threadIdx.x] = sh;
    s_rect[threadIdx.x] = make_int4(x0, y0, x1 - x0, __float_as_int(__frcp_rn((float)max(x1 - x0, 1))));
    __syncwarp();
    for (int base = 0; base < total; base += 32) {
        const int p = base + lane;
        // owner of pair p: the last lane whose first pair is at or before p (all
        // lanes take part in the search; lanes past the last pair test nothing)
        int j = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
            const int oj = __shfl_sync(0xffffffffu, o, j + step);
            if (oj <= p) j += step;
        }
        const int oj = __shfl_sync(0xffffffffu, o, j);
        bool keep = false;
        if (p < total) {
            const int4 rc = s_rect[wbase + j];
            const int t_in = p - oj;
            int row, col;
            divmod_small(t_in, rc.z, __int_as_float(rc.w), row, col);
            keep = keep_tile(rule, s_shape[wbase + j], rc.x + col, rc.y + row);
        }
        const uint32_t km = __ballot_sync(0xffffffffu, keep);
        // this lane's own pairs in the round: positions [lo, hi) of km
        const int lo = max(o, base) - base, hi = min(o + a, base + 32) - base;
        if (lo < hi) {
            const uint32_t bits = (hi - lo == 32 ? km : (km >> lo) & ((1u << (hi - lo)) - 1u));
            mask |= bits << (lo + base - o);
        }
    }
    if (i < N) {
        rec[i].a = make_int4(x0, y0, x1 - x0, g);
        rec[i].b = make_int4(pre, (int)mask, __float_as_int(sh.depth), __float_as_int(sh.hide));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, d);
    if (lane == 0) s_pre[threadIdx.x >> 5] = pre;
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0;
        for (int w = 0; w < 8; ++w) t += s_pre[w];
        if (t) atomicAdd(counters + GM_CNT_K_PRECULL, t);
    }
}

// Per position i of the depth order: the tiles the Gaussian is binned to now
// that the mesh's tile bounds exist -- for a small rectangle its ellipse-kept
// tiles less those the mesh hides, for a large one every tile of the rectangle
// tested again by the whole warp -- as a count and, for a small rectangle, the
// kept mask (for the emission); and per CTA the sum of its counts.
__global__ void __launch_bounds__(256)
k_gauss_cull(Cam c, BinRule rule, int N, const float4* __restrict__ splats, const GaussRec* __restrict__ rec,
             int32_t* __restrict__ counts, uint32_t* __restrict__ kept, int32_t* __restrict__ block_sums)
{
    __shared__ int s_sum[8];
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    int4 ra = make_int4(0, 0, 0, -1), rb = make_int4(0, 0, 0, 0);
    if (i < N) {
        ra = rec[i].a;
        rb = rec[i].b;
    }
    const int area = rb.x;
    uint32_t mask = 0;
    int post = 0;
    if (area > 0 && area <= SMALL_RECT) {
        mask = rule.tile_test ? (uint32_t)rb.y : ((1u << area) - 1u);
        if (rule.cull) {
            const float depth = __int_as_float(rb.z), hide = __int_as_float(rb.w);
            const float inv = __frcp_rn((float)ra.z);
            for (uint32_t m = mask; m; m &= m - 1) {
                const int pos = __ffs(m) - 1;
                int row, col;
                divmod_small(pos, ra.z, inv, row, col);
                if (tile_hidden(rule, (ra.y + row) * c.TW + ra.x + col, depth, hide)) mask &= ~(1u << pos);
            }
        }
        post = __popc(mask);
    }
    // large rectangles (near-camera Gaussians): the whole warp, 32 tiles at a time
    BinShape sh = {};
    if (area > SMALL_RECT) sh = bin_shape(splats, ra.w);
    uint32_t big = __ballot_sync(0xffffffffu, area > SMALL_RECT);
    while (big) {
        const int j = __ffs(big) - 1;
        big &= big - 1;
        const int jx0 = __shfl_sync(0xffffffffu, ra.x, j), jy0 = __shfl_sync(0xffffffffu, ra.y, j);
        const int jw = __shfl_sync(0xffffffffu, ra.z, j), jarea = __shfl_sync(0xffffffffu, area, j);
        const BinShape js = shfl_shape(sh, j);
        const float jinv = __frcp_rn((float)jw);
        int cnt = 0;
        for (int t = lane; t < jarea; t += 32) {
            int row, col;
            divmod_small(t, jw, jinv, row, col);
            cnt += keep_tile(rule, js, jx0 + col, jy0 + row);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        if (lane == j) post = cnt;
    }
    if (i < N) {
        counts[i] = post;
        kept[i] = mask;
    }
    int sum = post;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
    if (lane == 0) s_sum[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0;
        for (int w = 0; w < 8; ++w) t += s_sum[w];
        block_sums[blockIdx.x] = t;
    }
}

// The CTAs' count sums (one per 256 positions of the depth order) into their
// exclusive prefixes, in place, and the total into counters[GM_CNT_K]: the
// emission adds a CTA's prefix to the scan of its own counts.  One CTA.
constexpr int PREFIX_THREADS = 1024;

__global__ void __launch_bounds__(PREFIX_THREADS)
k_block_prefix(int32_t* __restrict__ sums, int nb, int32_t* counters)
{
    __shared__ uint32_t s_warp[PREFIX_THREADS / 32];
    const int per = (nb + PREFIX_THREADS - 1) / PREFIX_THREADS;
    const int b0 = threadIdx.x * per;
    uint32_t local = 0;
    for (int k = 0; k < per && b0 + k < nb; ++k) local += (uint32_t)sums[b0 + k];
    uint32_t total;
    uint32_t run = block_excl_scan<PREFIX_THREADS>(local, s_warp, total);
    for (int k = 0; k < per && b0 + k < nb; ++k) {
        const uint32_t v = (uint32_t)sums[b0 + k];
        sums[b0 + k] = (int32_t)run;
        run += v;
    }
    if (threadIdx.x == 0) counters[GM_CNT_K] = (int32_t)min(total, (uint32_t)INT32_MAX);
}

// Emits the (tile << 32 | depth bits, id) entries of the Gaussian at position
// i of the depth order, in ascending (depth, id) order, at its offset (the
// CTA's prefix plus the scan of the CTA's counts): entries
// come out depth-sorted, so a stable sort on the tile bits alone completes the
// (tile, depth, id) order.  The tiles kept are exactly those k_gauss_cull
// counted: its mask for small rectangles, the same predicate for large ones.
__global__ void __launch_bounds__(256)
k_gauss_emit(Cam c, BinRule rule, int N, const float4* __restrict__ splats, const GaussRec* __restrict__ rec,
             const int32_t* __restrict__ counts, const uint32_t* __restrict__ kept,
             const int32_t* __restrict__ block_prefix, int cap, int32_t* counters, uint64_t* __restrict__ keys,
             int32_t* __restrict__ vals)
{
    __shared__ int4 s_a[256];   // x0, y0, width, Gaussian id
    __shared__ int2 s_b[256];   // depth bits, first output slot
    __shared__ uint32_t s_m[256];
    __shared__ uint32_t s_warp[8];
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31;
    const int wbase = threadIdx.x & ~31;
    if (i == 0 && counters[GM_CNT_K] > cap) atomicOr(counters + GM_CNT_FLAGS, GM_FLAG_OVERFLOW);
    int4 ra = make_int4(0, 0, 0, -1);
    int area = 0, dbits = 0;
    BinShape sh = {};
    uint32_t mask = 0;
    const int cnt_i = i < N ? counts[i] : 0;
    uint32_t cta_total;
    const int64_t o = (int64_t)block_prefix[blockIdx.x] + block_excl_scan<256>((uint32_t)cnt_i, s_warp, cta_total);
    if (i < N) {
        const int4 rb = rec[i].b;
        if (rb.x > 0 && cnt_i > 0) {
            ra = rec[i].a;
            area = rb.x;
            dbits = rb.z;
            mask = kept[i];
            if (area > SMALL_RECT) sh = bin_shape(splats, ra.w);  // the big-rectangle path tests again
        }
    }
    {
        // the kept tiles of the warp's small rectangles, flattened: one entry per
        // lane per round, consecutive lanes writing consecutive slots
        const uint32_t m = (area > 0 && area <= SMALL_RECT) ? mask : 0u;
        const int a = __popc(m);
        int p0 = a;  // inclusive prefix sum over the lanes
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, p0, d);
            if (lane >= d) p0 += y;
        }
        const int total = __shfl_sync(0xffffffffu, p0, 31);
        p0 -= a;
        s_a[threadIdx.x] = ra;
        s_b[threadIdx.x] = make_int2(dbits, (int)o);
        s_m[threadIdx.x] = m;
        __syncwarp();
        for (int base = 0; base < total; base += 32) {
            const int p = base + lane;
            int j = 0;
#pragma unroll
            for (int step = 16; step > 0; step >>= 1) {
                const int pj = __shfl_sync(0xffffffffu, p0, j + step);
                if (pj <= p) j += step;
            }
            const int pj = __shfl_sync(0xffffffffu, p0, j);
            if (p < total) {
                const int r = p - pj;  // the r-th kept tile of lane j's rectangle
                const uint32_t mj = s_m[wbase + j];
                int pos = 0, rr = r;
#pragma unroll
                for (int st = 8; st > 0; st >>= 1) {
                    const int cnt = __popc((mj >> pos) & ((1u << st) - 1u));
                    if (cnt <= rr) {
                        rr -= cnt;
                        pos += st;
                    }
                }
                const int4 qa = s_a[wbase + j];
                const int2 qb = s_b[wbase + j];
                const int64_t dst = (int64_t)qb.y + r;
                if (dst >= 0 && dst < cap) {
                    int row, col;
                    divmod_small(pos, qa.z, __frcp_rn((float)qa.z), row, col);
                    const int t = (qa.y + row) * c.TW + qa.x + col;
                    keys[dst] = ((uint64_t)(uint32_t)t << 32) | (uint32_t)qb.x;
                    vals[dst] = qa.w;
                }
            }
        }
    }
    uint32_t big = __ballot_sync(0xffffffffu, area > SMALL_RECT);
    while (big) {
        const int j = __ffs(big) - 1;
        big &= big - 1;
        const int jx0 = __shfl_sync(0xffffffffu, ra.x, j), jy0 = __shfl_sync(0xffffffffu, ra.y, j);
        const int jw = __shfl_sync(0xffffffffu, ra.z, j), jarea = __shfl_sync(0xffffffffu, area, j);
        const int jg = __shfl_sync(0xffffffffu, ra.w, j);
        const BinShape js = shfl_shape(sh, j);
        const uint32_t jbits = __float_as_uint(js.depth);
        const float jinv = __frcp_rn((float)jw);
        int64_t jo = __shfl_sync(0xffffffffu, o, j);
        for (int base = 0; base < jarea; base += 32) {
            const int t_in = base + lane;
            int tx = 0, ty = 0;
            bool keep = false;
            if (t_in < jarea) {
                int row, col;
                divmod_small(t_in, jw, jinv, row, col);
                tx = jx0 + col;
                ty = jy0 + row;
                keep = keep_tile(rule, js, tx, ty);
            }
            const uint32_t km = __ballot_sync(0xffffffffu, keep);
            const int64_t dst = jo + __popc(km & ((1u << lane) - 1u));
            if (keep && dst >= 0 && dst < cap) {
                keys[dst] = ((uint64_t)(uint32_t)(ty * c.TW + tx) << 32) | jbits;
                vals[dst] = jg;
            }
            jo += __popc(km);
        }
    }
}

int tile_bits(int n_tiles) { return n_tiles > 1 ? 32 - __builtin_clz((unsigned)(n_tiles - 1)) : 0; }

size_t a256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

static SoftCull soft_cull(float softness, int split)
{
    // the compositing's tail bound of the front fraction: Phi(-2.75), logistic at -3.5
    return SoftCull{softness > 0.0f ? softness : 0.0f, split == 1 ? 3.5f : 2.75f};
}

cudaError_t project(const Cam& c, int sh_degree, float softness, int split, int N, const float* means,
                    const float* log_scales, const float* quats, const float* logits, const float* colors,
                    float* splats, int32_t* radii, int32_t* tiles_touched, float* depth_model, cudaStream_t s)
{
    if (N <= 0) return cudaSuccess;
    const ProjConsts pc = make_proj_consts(c);
    const SoftCull sc = soft_cull(softness, split);
    const int grid = (N + PROJ_THREADS - 1) / PROJ_THREADS;
    auto* q4 = reinterpret_cast<const float4*>(quats);
    auto* s4 = reinterpret_cast<float4*>(splats);
    auto* dm4 = reinterpret_cast<float4*>(depth_model);
#define GM_PROJ(D) k_project<D><<<grid, PROJ_THREADS, 0, s>>>(c, pc, sc, N, means, log_scales, q4, logits, colors, \
                                                              s4, radii, tiles_touched, dm4)
    switch (sh_degree) {
        case -1: GM_PROJ(-1); break;
        case 0: GM_PROJ(0); break;
        case 1: GM_PROJ(1); break;
        case 2: GM_PROJ(2); break;
        case 3: GM_PROJ(3); break;
        default: return cudaErrorInvalidValue;
    }
#undef GM_PROJ
    return cudaGetLastError();
}

cudaError_t project_views(const Cam* cams, int V, int sh_degree, float softness, int split, int N,
                          const float* means, const float* log_scales, const float* quats, const float* logits,
                          const float* colors, float* splats, int32_t* radii, int32_t* tiles_touched,
                          float* depth_model, cudaStream_t s)
{
    if (N <= 0) return cudaSuccess;
    const SoftCull sc = soft_cull(softness, split);
    const int grid = (N + PROJ_THREADS - 1) / PROJ_THREADS;
    auto* q4 = reinterpret_cast<const float4*>(quats);
    for (int v0 = 0; v0 < V; v0 += MAX_VIEWS) {
        ViewBatch vb;
        vb.n = std::min(MAX_VIEWS, V - v0);
        for (int v = 0; v < vb.n; ++v) {
            vb.cam[v] = cams[v0 + v];
            vb.pc[v] = make_proj_consts(cams[v0 + v]);
        }
        const int64_t off = (int64_t)v0 * N;
        auto* s4 = reinterpret_cast<float4*>(splats + 12 * off);
        auto* dm4 = depth_model ? reinterpret_cast<float4*>(depth_model + 4 * off) : nullptr;
#define GM_PROJ_V(D)                                                                                       \
    k_project_views<D><<<grid, PROJ_THREADS, 0, s>>>(vb, sc, N, means, log_scales, q4, logits, colors, s4,      \
                                                     radii + off, tiles_touched + off, dm4)
        switch (sh_degree) {
            case -1: GM_PROJ_V(-1); break;
            case 0: GM_PROJ_V(0); break;
            case 1: GM_PROJ_V(1); break;
            case 2: GM_PROJ_V(2); break;
            case 3: GM_PROJ_V(3); break;
            default: return cudaErrorInvalidValue;
        }
#undef GM_PROJ_V
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t gauss_bin_ws_bytes(int N, int cap)
{
    int64_t n = N > 0 ? N : 1, k = cap > 0 ? cap : 1;
    return scan_ws_bytes(n) + 3 * a256(sizeof(int32_t) * n) + 2 * a256(sizeof(uint64_t) * n) +
           2 * a256(sizeof(int32_t) * n) + a256(sizeof(GaussRec) * n) + 256 + sort_ws_bytes(n > k ? n : k);
}

// Tile binning of the Gaussians.  The entries' order (tile, depth, id) is
// reached in two stable LSD sorts: the N Gaussians by depth (32 bits), then,
// after emitting each Gaussian's tiles in that order, the K entries by tile
// only (ceil(log2 T) bits) -- instead of one 32 + log2 T bit sort of K keys.
// The first half (depth sort, rectangles and ellipse tests, one record per
// position of the depth order) needs no mesh; the second (occlusion cull,
// scan, emission, tile sort) reads the records in order, with no gathers.
struct GaussWs {
    ScanWs sw;
    int32_t *counts, *offsets;
    uint32_t* kept;
    uint64_t *dkey, *dkey_alt;
    int32_t *dval, *dval_alt, *n_dev;
    GaussRec* rec;
    SortWs so;
};

static GaussWs carve_gauss_ws(void* ws, int N, int cap)
{
    int64_t n = N > 0 ? N : 1, k = cap > 0 ? cap : 1;
    GaussWs w;
    uint8_t* b = (uint8_t*)ws;
    b += carve_scan_ws(b, n, w.sw);
    w.counts = (int32_t*)b;
    b += a256(sizeof(int32_t) * n);
    w.offsets = (int32_t*)b;
    b += a256(sizeof(int32_t) * n);
    w.kept = (uint32_t*)b;
    b += a256(sizeof(uint32_t) * n);
    w.dkey = (uint64_t*)b;
    b += a256(sizeof(uint64_t) * n);
    w.dkey_alt = (uint64_t*)b;
    b += a256(sizeof(uint64_t) * n);
    w.dval = (int32_t*)b;
    b += a256(sizeof(int32_t) * n);
    w.dval_alt = (int32_t*)b;
    b += a256(sizeof(int32_t) * n);
    w.rec = (GaussRec*)b;
    b += a256(sizeof(GaussRec) * n);
    w.n_dev = (int32_t*)b;
    b += 256;
    carve_sort_ws(b, n > k ? n : k, w.so);
    return w;
}

cudaError_t gauss_depth_sort(const Cam& c, int N, const float* splats, const int32_t* radii, int cap,
                             int32_t* counters, void* ws, cudaStream_t s)
{
    GaussWs w = carve_gauss_ws(ws, N, cap);
    cudaError_t e = cudaMemsetAsync(counters, 0, 4 * sizeof(int32_t), s);
    if (e != cudaSuccess || N <= 0) return e;
    if ((e = clear_sort_hist(w.so, s)) != cudaSuccess) return e;
    const int kgrid = (int)std::min<int64_t>(((int64_t)N + 255) / 256, (int64_t)num_sms() * 4);
    k_gauss_depth_keys<<<kgrid, 256, 0, s>>>(c, N, reinterpret_cast<const float4*>(splats), radii, w.dkey, w.dval,
                                             w.n_dev, w.so.hist, w.so.desc, w.so.max_parts);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4 passes: even, the result is back in dkey / dval
    e = radix_sort(w.dkey, w.dval, w.dkey_alt, w.dval_alt, N, 0, 32, w.n_dev, counters, w.so, s, true);
    if (e != cudaSuccess) return e;
    k_gauss_shape<<<(N + 255) / 256, 256, 0, s>>>(c, N, reinterpret_cast<const float4*>(splats), radii, w.dval,
                                                   w.rec, counters);
    return cudaGetLastError();
}

cudaError_t gauss_bin(const Cam& c, bool cull, bool soft, bool tile_test, int N, const float* splats,
                      const int32_t* radii,
                      const float* tile_far, const uint8_t* tile_full, uint64_t* keys, int32_t* gids,
                      int32_t* tile_range, int cap, int32_t* counters, void* ws, cudaStream_t s)
{
    GaussWs w = carve_gauss_ws(ws, N, cap);
    cudaError_t e = cudaSuccess;
    const int T = c.TW * c.TH;
    const int tb = tile_bits(T);
    const int passes = sort_passes(32, 32 + tb);
    uint64_t* ek = passes % 2 ? w.so.keys_alt : keys;
    int32_t* ev = passes % 2 ? w.so.vals_alt : gids;
    if (N > 0) {
        auto* s4 = reinterpret_cast<const float4*>(splats);
        const int grid = (N + 255) / 256;
        BinRule rule;
        rule.cull = cull;
        rule.soft = soft;
        rule.tile_test = tile_test;
        rule.tile_far = tile_far;
        rule.tile_full = tile_full;
        rule.TW = c.TW;
        // the offsets: per-CTA count sums (cull), their prefixes (one CTA), then each
        // emission CTA's own scan -- no inter-block waits
        k_gauss_cull<<<grid, 256, 0, s>>>(c, rule, N, s4, w.rec, w.counts, w.kept, w.offsets);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_block_prefix<<<1, PREFIX_THREADS, 0, s>>>(w.offsets, grid, counters);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_gauss_emit<<<grid, 256, 0, s>>>(c, rule, N, s4, w.rec, w.counts, w.kept, w.offsets, cap, counters, ek,
                                          ev);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (tb > 0) {
            if (passes % 2)
                e = radix_sort(w.so.keys_alt, w.so.vals_alt, keys, gids, cap, 32, 32 + tb, counters + GM_CNT_K,
                               counters, w.so, s);
            else
                e = radix_sort(keys, gids, w.so.keys_alt, w.so.vals_alt, cap, 32, 32 + tb, counters + GM_CNT_K,
                               counters, w.so, s);
            if (e != cudaSuccess) return e;
        }
    }
    return tile_ranges(keys, N > 0 ? cap : 0, counters, tile_range, T, s);
}

cudaError_t gauss_bin_sort(const Cam& c, bool cull, bool soft, bool tile_test, int N, const float* splats,
                           const int32_t* radii, const float* tile_far, const uint8_t* tile_full, uint64_t* keys,
                           int32_t* gids, int32_t* tile_range, int cap, int32_t* counters, void* ws, cudaStream_t s)
{
    cudaError_t e = gauss_depth_sort(c, N, splats, radii, cap, counters, ws, s);
    if (e != cudaSuccess) return e;
    return gauss_bin(c, cull, soft, tile_test, N, splats, radii, tile_far, tile_full, keys, gids, tile_range, cap,
                     counters, ws, s);
}

}  // namespace gm

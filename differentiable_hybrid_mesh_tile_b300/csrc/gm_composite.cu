// Hybrid compositing ("A Lightweight and Differentiable Renderer for Joint
// Mesh and 3D Gaussian Splat Scenes", Hybrid rendering) with a hard depth
// test: every Gaussian is tested against the mesh depth at the pixel, and the
// opaque mesh is the terminal layer.  Forward and backward, one CTA per
// 16 x 16 tile, one thread per pixel; the tile's sorted records are staged in
// shared memory in batches of 256.
#include "gm_internal.cuh"

namespace gm {
namespace {

constexpr float ALPHA_MAX = 0.99f;
constexpr float ALPHA_MIN = 1.0f / 255.0f;
constexpr float T_STOP = 1e-4f;

// sigma, exp(-sigma) and alpha of one splat at pixel centre (px, py).  Both
// passes call this one routine with explicit roundings so that they take the
// same skip / clamp decisions bit for bit.
struct Eval {
    float dx, dy, sigma, G, alpha;
    bool clamped;
};

__device__ __forceinline__ Eval eval_splat(const float4& A, const float4& B, float px, float py)
{
    Eval e;
    e.dx = __fsub_rn(px, A.x);
    e.dy = __fsub_rn(py, A.y);
    const float q = __fmaf_rn(A.z, __fmul_rn(e.dx, e.dx), __fmul_rn(B.x, __fmul_rn(e.dy, e.dy)));
    e.sigma = __fmaf_rn(0.5f, q, __fmul_rn(A.w, __fmul_rn(e.dx, e.dy)));
    e.G = __expf(-e.sigma);
    const float oG = __fmul_rn(B.y, e.G);
    e.clamped = oG > ALPHA_MAX;
    e.alpha = e.clamped ? ALPHA_MAX : oG;
    return e;
}

// adds a per-thread count over the block to *stats (one atomic per block)
__device__ __forceinline__ void block_count(uint32_t v, unsigned long long* stats)
{
    unsigned long long x = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0 && x) atomicAdd(stats, x);
}

__global__ void __launch_bounds__(TILE_PIX)
k_composite_fwd(Cam c, float3 bg, int N, const int2* __restrict__ tile_range, const int32_t* __restrict__ gids,
                const float4* __restrict__ splats, const float* __restrict__ mesh_depth,
                const float* __restrict__ mesh_rgb, const int32_t* __restrict__ face_id, float* __restrict__ out_rgb,
                float* __restrict__ out_depth, float* __restrict__ out_alpha, float* __restrict__ T_final,
                int32_t* __restrict__ n_contrib, unsigned long long* __restrict__ stats)
{
    __shared__ float4 sA[TILE_PIX], sB[TILE_PIX], sC[TILE_PIX];
    const int tile = blockIdx.x;
    const int tx = tile % c.TW, ty = tile / c.TW;
    const int i = tx * TILE + (threadIdx.x & (TILE - 1));
    const int j = ty * TILE + (threadIdx.x >> 4);
    const bool inside = i < c.W && j < c.H;
    const int64_t pix = (int64_t)j * c.W + i;
    const float px = (float)i + 0.5f, py = (float)j + 0.5f;
    float D = -INFINITY;
    bool cov = false;
    if (inside) {
        D = mesh_depth[pix];
        cov = face_id[pix] >= 0;
    }
    float T = 1.0f, Cr = 0.0f, Cg = 0.0f, Cb = 0.0f, Z = 0.0f;
    int last = 0;
    uint32_t visited = 0;
    bool done = !inside;
    const int2 r = tile_range[tile];
    for (int b = r.x; b < r.y; b += TILE_PIX) {
        if (__syncthreads_count(done) == TILE_PIX) break;
        const int n = min(TILE_PIX, r.y - b);
        if ((int)threadIdx.x < n) {
            const int64_t g = gids[b + threadIdx.x];
            if (g >= 0 && g < N) {
                sA[threadIdx.x] = splats[3 * g];
                sB[threadIdx.x] = splats[3 * g + 1];
                sC[threadIdx.x] = splats[3 * g + 2];
            } else {  // an id outside [0, N): an entry that draws nothing
                sA[threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
                sB[threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
                sC[threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        __syncthreads();
        if (!done) {
            int k = 0;
            for (; k < n; ++k) {
                const float4 C3 = sC[k];
                // sorted by depth: once a Gaussian is not in front of the mesh, none after it is
                if (!(C3.y < D)) {
                    done = true;
                    break;
                }
                const float4 A = sA[k], B = sB[k];
                const Eval e = eval_splat(A, B, px, py);
                if (e.sigma < 0.0f || e.alpha < ALPHA_MIN) continue;
                const float Tn = __fmul_rn(T, __fsub_rn(1.0f, e.alpha));
                if (Tn <= T_STOP) {
                    done = true;
                    break;
                }
                const float w = e.alpha * T;
                Cr = fmaf(w, B.z, Cr);
                Cg = fmaf(w, B.w, Cg);
                Cb = fmaf(w, C3.x, Cb);
                Z = fmaf(w, C3.y, Z);
                T = Tn;
                last = b - r.x + k + 1;
            }
            visited += (uint32_t)min(k + 1, n);
        }
        __syncthreads();
    }
    if (stats) block_count(visited, stats);
    if (inside) {
        float tr, tg, tb;
        if (cov) {
            tr = mesh_rgb[3 * pix]; tg = mesh_rgb[3 * pix + 1]; tb = mesh_rgb[3 * pix + 2];
        } else {
            tr = bg.x; tg = bg.y; tb = bg.z;
        }
        out_rgb[3 * pix] = fmaf(T, tr, Cr);
        out_rgb[3 * pix + 1] = fmaf(T, tg, Cg);
        out_rgb[3 * pix + 2] = fmaf(T, tb, Cb);
        out_depth[pix] = cov ? fmaf(T, D, Z) : Z;
        out_alpha[pix] = cov ? 1.0f : 1.0f - T;
        T_final[pix] = T;
        n_contrib[pix] = last;
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int NGRAD = 10;

__global__ void __launch_bounds__(TILE_PIX)
k_composite_bwd(Cam c, float3 bg, int N, const int2* __restrict__ tile_range, const int32_t* __restrict__ gids,
                const float4* __restrict__ splats, const float* __restrict__ mesh_depth,
                const float* __restrict__ mesh_rgb, const int32_t* __restrict__ face_id,
                const float* __restrict__ T_final, const int32_t* __restrict__ n_contrib,
                const float* __restrict__ g_rgb, const float* __restrict__ g_depth, const float* __restrict__ g_alpha,
                float* __restrict__ v_splats, unsigned long long* __restrict__ stats)
{
    __shared__ float4 sA[TILE_PIX], sB[TILE_PIX], sC[TILE_PIX];
    __shared__ int sG[TILE_PIX];
    __shared__ float sAcc[TILE_PIX][NGRAD + 1];
    __shared__ int s_max_last;
    const int tile = blockIdx.x;
    const int tx = tile % c.TW, ty = tile / c.TW;
    const int i = tx * TILE + (threadIdx.x & (TILE - 1));
    const int j = ty * TILE + (threadIdx.x >> 4);
    const int lane = threadIdx.x & 31;
    const bool inside = i < c.W && j < c.H;
    const int64_t pix = (int64_t)j * c.W + i;
    const float px = (float)i + 0.5f, py = (float)j + 0.5f;

    float D = -INFINITY, T = 1.0f, gr = 0.f, gg = 0.f, gb = 0.f, gz = 0.f, ga = 0.f;
    int last = 0;
    float BCr = 0.f, BCg = 0.f, BCb = 0.f, BZ = 0.f, aterm = 0.f;
    if (inside) {
        D = mesh_depth[pix];
        const bool cov = face_id[pix] >= 0;
        T = T_final[pix];
        last = n_contrib[pix];
        gr = g_rgb[3 * pix]; gg = g_rgb[3 * pix + 1]; gb = g_rgb[3 * pix + 2];
        gz = g_depth[pix];
        ga = g_alpha[pix];
        // the terminal layer, everything behind the last composited Gaussian
        if (cov) {
            BCr = T * mesh_rgb[3 * pix]; BCg = T * mesh_rgb[3 * pix + 1]; BCb = T * mesh_rgb[3 * pix + 2];
            BZ = T * D;
        } else {
            BCr = T * bg.x; BCg = T * bg.y; BCb = T * bg.z;
            aterm = ga * T;  // out_alpha = 1 - T_final when uncovered
        }
    }
    if (threadIdx.x == 0) s_max_last = 0;
    __syncthreads();
    if (last > 0) atomicMax(&s_max_last, last);
    __syncthreads();
    const int2 r = tile_range[tile];
    const int end = r.x + s_max_last;
    if (stats) block_count(inside ? (uint32_t)last : 0u, stats);
    for (int b_end = end; b_end > r.x; b_end -= TILE_PIX) {
        const int b0 = max(r.x, b_end - TILE_PIX);
        const int n = b_end - b0;
        if ((int)threadIdx.x < n) {
            int g = gids[b0 + threadIdx.x];
            if (g < 0 || g >= N) g = -1;  // an entry that draws nothing and gets no gradient
            sG[threadIdx.x] = g;
            const int64_t gg = g < 0 ? 0 : g;
            sA[threadIdx.x] = g < 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : splats[3 * gg];
            sB[threadIdx.x] = g < 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : splats[3 * gg + 1];
            sC[threadIdx.x] = g < 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : splats[3 * gg + 2];
#pragma unroll
            for (int q = 0; q < NGRAD; ++q) sAcc[threadIdx.x][q] = 0.0f;
        }
        __syncthreads();
        for (int k = n - 1; k >= 0; --k) {
            const int pos = b0 - r.x + k;
            bool on = inside && pos < last;
            float v[NGRAD];
#pragma unroll
            for (int q = 0; q < NGRAD; ++q) v[q] = 0.0f;
            if (on) {
                const float4 A = sA[k], B = sB[k], C3 = sC[k];
                const Eval e = eval_splat(A, B, px, py);
                on = C3.y < D && !(e.sigma < 0.0f) && !(e.alpha < ALPHA_MIN);
                if (on) {
                    const float om = 1.0f - e.alpha;
                    const float Tp = T / om;  // transmittance in front of this Gaussian
                    const float w = e.alpha * Tp;
                    v[6] = w * gr;
                    v[7] = w * gg;
                    v[8] = w * gb;
                    v[9] = w * gz;
                    const float front = B.z * gr + B.w * gg + C3.x * gb + C3.y * gz;
                    const float behind = BCr * gr + BCg * gg + BCb * gb + BZ * gz;
                    const float dLda = Tp * front + (aterm - behind) / om;
                    BCr = fmaf(w, B.z, BCr);
                    BCg = fmaf(w, B.w, BCg);
                    BCb = fmaf(w, C3.x, BCb);
                    BZ = fmaf(w, C3.y, BZ);
                    T = Tp;
                    if (!e.clamped) {
                        v[5] = dLda * e.G;
                        const float dLds = -dLda * e.alpha;
                        v[2] = dLds * 0.5f * e.dx * e.dx;
                        v[3] = dLds * e.dx * e.dy;
                        v[4] = dLds * 0.5f * e.dy * e.dy;
                        v[0] = -dLds * (A.z * e.dx + A.w * e.dy);
                        v[1] = -dLds * (A.w * e.dx + B.x * e.dy);
                    }
                }
            }
            if (__any_sync(0xffffffffu, on)) {
#pragma unroll
                for (int q = 0; q < NGRAD; ++q) v[q] = warp_sum(v[q]);
                if (lane == 0) {
#pragma unroll
                    for (int q = 0; q < NGRAD; ++q) atomicAdd(&sAcc[k][q], v[q]);
                }
            }
        }
        __syncthreads();
        if ((int)threadIdx.x < n && sG[threadIdx.x] >= 0) {
            float* dst = v_splats + 12 * (int64_t)sG[threadIdx.x];
#pragma unroll
            for (int q = 0; q < NGRAD; ++q) {
                const float a = sAcc[threadIdx.x][q];
                if (a != 0.0f) atomicAdd(dst + q, a);
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t composite_fwd(const Cam& c, const float bg[3], int N, const int32_t* tile_range, const int32_t* gids,
                          const float* splats, const float* mesh_depth, const float* mesh_rgb,
                          const int32_t* face_id, float* out_rgb, float* out_depth, float* out_alpha,
                          float* T_final, int32_t* n_contrib, uint64_t* stats, cudaStream_t s)
{
    k_composite_fwd<<<c.TW * c.TH, TILE_PIX, 0, s>>>(
        c, make_float3(bg[0], bg[1], bg[2]), N, reinterpret_cast<const int2*>(tile_range), gids,
        reinterpret_cast<const float4*>(splats), mesh_depth, mesh_rgb, face_id, out_rgb, out_depth, out_alpha,
        T_final, n_contrib, reinterpret_cast<unsigned long long*>(stats));
    return cudaGetLastError();
}

cudaError_t composite_bwd(const Cam& c, const float bg[3], int N, const int32_t* tile_range, const int32_t* gids,
                          const float* splats, const float* mesh_depth, const float* mesh_rgb,
                          const int32_t* face_id, const float* T_final, const int32_t* n_contrib,
                          const float* g_rgb, const float* g_depth, const float* g_alpha, float* v_splats,
                          uint64_t* stats, cudaStream_t s)
{
    k_composite_bwd<<<c.TW * c.TH, TILE_PIX, 0, s>>>(
        c, make_float3(bg[0], bg[1], bg[2]), N, reinterpret_cast<const int2*>(tile_range), gids,
        reinterpret_cast<const float4*>(splats), mesh_depth, mesh_rgb, face_id, T_final, n_contrib, g_rgb, g_depth,
        g_alpha, v_splats, reinterpret_cast<unsigned long long*>(stats));
    return cudaGetLastError();
}

}  // namespace gm

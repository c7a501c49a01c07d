// Hybrid compositing ("A Lightweight and Differentiable Renderer for Joint
// Mesh and 3D Gaussian Splat Scenes", Hybrid rendering) with a hard depth
// test: every Gaussian is tested against the mesh depth at the pixel, and the
// opaque mesh is the terminal layer.  Forward and backward, two CTAs of four
// warps per 16 x 16 tile (each CTA one 16 x 8 half), one thread per pixel,
// each warp an 8 x 4 pixel block; the tile's sorted records are staged in
// shared memory in batches of 128.
//
// Each warp first asks, per staged record, whether the Gaussian's ellipse of
// alpha >= 1/255 meets its 8 x 4 pixel block, lists those records in shared
// memory, and then visits only them (the other pairs would be skipped anyway),
// every lane evaluating every listed record and keeping, by selects rather than
// branches, what applies to its pixel.  With staged records the forward pass
// also writes each warp's lists out, and each warp of the backward pass (hard
// split) then works through its own lists, back to front, loading the listed
// records from the staged buffer itself, with no barrier across the CTA.
//
// Half-tile CTAs: the warps of a CTA wait for one another at every batch and
// at exit, so the slowest 8 x 4 block holds the CTA; four blocks per CTA
// instead of eight lose less to that imbalance than staging the list twice
// per tile costs.
#include <stdlib.h>

#include "gm_internal.cuh"

namespace gm {
namespace {

constexpr float ALPHA_MAX = 0.99f;
constexpr float ALPHA_MIN = 1.0f / 255.0f;
constexpr float T_STOP = 1e-4f;
constexpr float LOG2E = 1.4426950408889634f;

constexpr int CTA_WARPS = 4;                  // 8 x 4 blocks per CTA: half a tile
constexpr int CTA_THREADS = 32 * CTA_WARPS;   // = staging batch
constexpr int CTAS_PER_TILE = 8 / CTA_WARPS;
constexpr uint8_t NO_HIT = 0xff;              // padding of a warp's hit list

// Staged records of a tile list (one per list position, three float4 arrays,
// a fourth with the soft split's depth model): written by the forward pass,
// read by the backward pass (loaded per group of listed records with the hard
// split, bulk-copied into shared memory per batch with the soft split).
// A == nullptr: none.
// With the hard split the space of the fourth array holds instead each warp's
// hit lists: for warp w of a tile (0..7) and a batch starting at list position
// b, the staged indices of the batch's records that reach the warp's block, in
// list order, at L[w * cap + b ..], then NO_HIT up to the batch's end.
struct Staged {
    float4* A;
    float4* B;
    float4* C;
    float4* D;
    uint8_t* L;
    int cap;  // list positions the arrays hold
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Staged record, three float4.  The conic is stored pre-multiplied so that
// exp(-sigma) = 2^l, l = a2 dx^2 + b2 dx dy + c2 dy^2, a2 = -a log2e / 2,
// b2 = -b log2e, c2 = -c log2e / 2 (a2, c2 < 0 for a positive definite conic):
//   A = (mx, my, a2, b2), B = (c2, opacity, r, g), C = (b, depth, id, lmin),
// id the Gaussian's index (its int bits; -1 for an entry that draws nothing)
// and lmin = -log2(255 o): alpha >= 1/255 needs l >= lmin (-inf for a
// degenerate conic, every pixel evaluated; +inf when alpha never reaches 1/255).
__device__ __forceinline__ void stage_rec(const float4* __restrict__ splats, int g, float4& A, float4& B, float4& C)
{
    if (g < 0) {
        A = make_float4(0.f, 0.f, 0.f, 0.f);
        B = make_float4(0.f, 0.f, 0.f, 0.f);
        C = make_float4(0.f, 0.f, __int_as_float(-1), INFINITY);
        return;
    }
    const float4 s0 = splats[3 * (int64_t)g], s1 = splats[3 * (int64_t)g + 1], s2 = splats[3 * (int64_t)g + 2];
    // s0 = (mx, my, a, b), s1 = (c, o, r, g), s2 = (b, depth, 0, 0)
    A = make_float4(s0.x, s0.y, -0.5f * LOG2E * s0.z, -LOG2E * s0.w);
    B = make_float4(-0.5f * LOG2E * s1.x, s1.y, s1.z, s1.w);
    const float o255 = 255.0f * s1.y;
    const float det = s0.z * s1.x - s0.w * s0.w;
    float lmin;
    if (!(det > 0.0f) || !(s0.z > 0.0f)) {
        lmin = -INFINITY;  // degenerate conic: every pixel is evaluated
    } else if (!(o255 >= 1.0f)) {
        lmin = INFINITY;   // exp(-sigma) <= 1: never reaches 1/255
    } else {
        // lowered by 0.1 % + 1e-4 so that rounding in the block test and the
        // approximate logarithm (absolute error near 1e-6 here) never drop a pixel
        // the exact evaluation keeps
        lmin = -__log2f(o255) * 1.001f - 1e-4f;
    }
    C = make_float4(s2.x, s2.y, __int_as_float(g), lmin);
}

__device__ __forceinline__ int rec_id(const float4& C) { return __float_as_int(C.z); }

// Whether the Gaussian can reach alpha >= 1/255 at any pixel centre of the
// warp's 8 x 4 block (centres x0 .. x0 + 7, y0 .. y0 + 3): the maximum of the
// concave l over that rectangle is 0 when it holds the mean, else it lies on
// an edge, where l is a 1D parabola maximised at a clamped vertex.  The
// vertices need -1 / (2 a2) and -1 / (2 c2); an approximate quotient moves a
// vertex by a few ulp, which changes l there far less than lmin's margin.
__device__ __forceinline__ bool block_hits(const float4& A, const float4& B, float lmin, float x0, float y0)
{
    if (!(lmin <= 0.0f)) return false;      // invisible
    if (lmin == -INFINITY) return true;      // degenerate: evaluate
    const float u0 = x0 - A.x, u1 = u0 + 7.0f, v0 = y0 - A.y, v1 = v0 + 3.0f;
    if (u0 <= 0.0f && u1 >= 0.0f && v0 <= 0.0f && v1 >= 0.0f) return true;
    const float a2 = A.z, b2 = A.w, c2 = B.x;
    const float ka = __fdividef(-0.5f, a2), kc = __fdividef(-0.5f, c2);
    float best = -INFINITY;
    {   // edges u = u0, u1: v* = b2 u kc
        const float va = fminf(fmaxf(b2 * u0 * kc, v0), v1), vb = fminf(fmaxf(b2 * u1 * kc, v0), v1);
        best = fmaxf(best, fmaf(fmaf(a2, u0, b2 * va), u0, c2 * va * va));
        best = fmaxf(best, fmaf(fmaf(a2, u1, b2 * vb), u1, c2 * vb * vb));
    }
    {   // edges v = v0, v1: u* = b2 v ka
        const float ua = fminf(fmaxf(b2 * v0 * ka, u0), u1), ub = fminf(fmaxf(b2 * v1 * ka, u0), u1);
        best = fmaxf(best, fmaf(fmaf(c2, v0, b2 * ua), v0, a2 * ua * ua));
        best = fmaxf(best, fmaf(fmaf(c2, v1, b2 * ub), v1, a2 * ub * ub));
    }
    return best >= lmin;
}

// alpha of one staged record at pixel centre (px, py).  Both passes call this
// one routine with explicit roundings, so they take the same skip / clamp
// decisions bit for bit.
struct Eval {
    float dx, dy, G, alpha;
    bool skip, clamped;
};

__device__ __forceinline__ Eval eval_splat(const float4& A, const float4& B, float px, float py)
{
    Eval e;
    e.dx = __fsub_rn(px, A.x);
    e.dy = __fsub_rn(py, A.y);
    const float q = __fmaf_rn(B.x, __fmul_rn(e.dy, e.dy), __fmul_rn(A.w, __fmul_rn(e.dx, e.dy)));
    const float l = __fmaf_rn(A.z, __fmul_rn(e.dx, e.dx), q);  // = -sigma log2(e)
    e.G = ex2(l);
    const float oG = __fmul_rn(B.y, e.G);
    e.clamped = oG > ALPHA_MAX;
    e.alpha = e.clamped ? ALPHA_MAX : oG;
    e.skip = l > 0.0f || e.alpha < ALPHA_MIN;  // sigma < 0, or alpha below 1/255
    return e;
}

// adds a per-thread count over the block to *stats (one atomic per warp)
__device__ __forceinline__ void block_count(uint32_t v, unsigned long long* stats)
{
    unsigned long long x = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0 && x) atomicAdd(stats, x);
}

struct PixelMap {
    int i, j;      // this thread's pixel
    float x0, y0;  // centre of the warp block's first pixel
};

// CTA b covers half b % 2 of tile b / 2; warp w of the tile (w = 4 half + warp
// of the CTA) covers the 8 x 4 block at (8 (w % 2), 4 (w / 2))
__device__ __forceinline__ PixelMap pixel_of(const Cam& c, int& tile)
{
    tile = blockIdx.x / CTAS_PER_TILE;
    const int tx = tile % c.TW, ty = tile / c.TW;
    const int warp = (blockIdx.x % CTAS_PER_TILE) * CTA_WARPS + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int bx = tx * TILE + (warp & 1) * 8, by = ty * TILE + (warp >> 1) * 4;
    PixelMap m;
    m.i = bx + (lane & 7);
    m.j = by + (lane >> 3);
    m.x0 = (float)bx + 0.5f;
    m.y0 = (float)by + 0.5f;
    return m;
}

// The standard normal distribution function by the rational approximation of
// Abramowitz and Stegun, Handbook of Mathematical Functions, formula 26.2.17:
// for x >= 0, Phi(x) = 1 - phi(x) t (b1 + b2 t + b3 t^2 + b4 t^3 + b5 t^4) with
// t = 1 / (1 + p x) and phi the normal density, |error| < 7.5e-8; Phi(-x) =
// 1 - Phi(x).  The tail below 0 is formed directly (no cancellation).
__device__ __forceinline__ float normal_cdf(float x)
{
    constexpr float P = 0.2316419f;
    constexpr float B1 = 0.319381530f, B2 = -0.356563782f, B3 = 1.781477937f, B4 = -1.821255978f,
                    B5 = 1.330274429f;
    const float ax = fabsf(x);
    const float t = __fdividef(1.0f, fmaf(P, ax, 1.0f));
    const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, B5, B4), B3), B2), B1);
    const float q = 0.3989422804014327f * ex2(-0.5f * LOG2E * ax * ax) * poly;  // 1 - Phi(|x|)
    return x >= 0.0f ? 1.0f - q : q;
}

// The soft split: its width factor and the form of the front fraction f(x),
// Phi(x) or the logistic 1 / (1 + exp(-1.702 x)).  Past x <= -tail, f(x) <=
// 0.0030 (Phi(-2.75)) or 0.0026 (logistic at -3.5), so alpha f <= 0.99 f <
// 1/255 and the Gaussian is skipped at that pixel.
struct Split {
    float softness;
    int logistic;
    __device__ __forceinline__ float tail() const { return logistic ? 3.5f : 2.75f; }
    __device__ __forceinline__ float front(float x) const
    {
        return logistic ? 1.0f / (1.0f + __expf(-1.702f * x)) : normal_cdf(x);
    }
    // df/dx, given f = front(x)
    __device__ __forceinline__ float density(float x, float f) const
    {
        return logistic ? 1.702f * f * (1.0f - f) : 0.3989422804014327f * __expf(-0.5f * x * x);
    }
};

// Staged depth model of the soft split: (g_u, g_v, kappa = 1 / (sigma_z
// softness), z_hide); f = f((D - z*) kappa), z* = z_c + g . (p - mean2d).
// With the reach R (z* >= z_c - R wherever alpha can reach 1/255), a mesh depth
// D < z_hide = z_c - R - tail sigma_z softness (less a rounding margin) puts x
// below -tail: the Gaussian is hidden at every such pixel.
__device__ __forceinline__ float4 stage_depth_model(const float4* __restrict__ depth_model, int64_t g,
                                                    const Split& sp, float z)
{
    const float4 m = depth_model[g];
    const float band = m.z * sp.softness;
    const float hide = z - fmaf(sp.tail(), band, m.w) * 1.0001f - 2e-6f * fabsf(z);
    return make_float4(m.x, m.y, 1.0f / band, hide);
}

// The largest mesh depth over this warp's covered pixels (+inf if one of its
// pixels in the image is not covered: there every Gaussian is seen whole), with
// a rounding margin; Gaussians whose z_hide lies beyond it draw nothing here.
__device__ __forceinline__ float warp_hide_depth(bool inside, bool cov, float D)
{
    float k = !inside ? -INFINITY : (cov ? D : INFINITY);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) k = fmaxf(k, __shfl_xor_sync(0xffffffffu, k, o));
    return isinf(k) ? k : k + 4e-6f * fabsf(k);
}

// A tile's range clamped to the staged-record buffer [0, cap) (the ranges come
// from a sort that may have given up a bounded wait; the backward reads the
// records by range, so they must stay inside the buffer).
__device__ __forceinline__ int2 clamp_range(int2 r, int cap)
{
    r.x = min(max(r.x, 0), cap);
    r.y = min(max(r.y, r.x), cap);
    return r;
}

template <bool STATS, bool SOFT>
__global__ void __launch_bounds__(CTA_THREADS)
k_composite_fwd(Cam c, float3 bg, int N, Split sp, const int2* __restrict__ tile_range,
                const int32_t* __restrict__ gids, const float4* __restrict__ splats,
                const float4* __restrict__ depth_model, const float* __restrict__ mesh_depth,
                const float* __restrict__ mesh_rgb, const int32_t* __restrict__ face_id, float* __restrict__ out_rgb,
                float* __restrict__ out_depth, float* __restrict__ out_alpha, float* __restrict__ T_final,
                int32_t* __restrict__ n_contrib, const float* __restrict__ aa_cov, Staged rec,
                unsigned long long* __restrict__ stats)
{
    __shared__ float4 sA[CTA_THREADS], sB[CTA_THREADS], sC[CTA_THREADS];
    __shared__ float4 sD[SOFT ? CTA_THREADS : 1];
    __shared__ uint8_t sList[CTA_WARPS][CTA_THREADS + 2];  // each warp's hits of the current batch
    int tile;
    const PixelMap pm = pixel_of(c, tile);
    const int lane = threadIdx.x & 31;
    const bool inside = pm.i < c.W && pm.j < c.H;
    const int64_t pix = (int64_t)pm.j * c.W + pm.i;
    const float px = (float)pm.i + 0.5f, py = (float)pm.j + 0.5f;
    float D = -INFINITY;
    bool cov = false;
    if (inside) {
        D = mesh_depth[pix];
        // the antialiased layer has a split depth wherever any mesh reaches the pixel
        cov = aa_cov ? D < INFINITY : face_id[pix] >= 0;
    }
    // soft split at this pixel: covered by the mesh (elsewhere D = +inf, f = 1)
    const bool soft = SOFT && cov;
    const float Dw = SOFT ? warp_hide_depth(inside, cov, D) : INFINITY;
    float T = 1.0f, Cr = 0.0f, Cg = 0.0f, Cb = 0.0f, Z = 0.0f;
    int last = 0;
    uint32_t visited = 0, blended = 0;
    bool done = !inside;
    const int2 r = rec.A ? clamp_range(tile_range[tile], rec.cap) : tile_range[tile];
    for (int b = r.x; b < r.y; b += CTA_THREADS) {
        // this barrier also keeps the staging below from overwriting records that
        // another warp of the CTA is still reading from the previous batch
        if (__syncthreads_count(done) == CTA_THREADS) break;
        const int n = min(CTA_THREADS, r.y - b);
        if ((int)threadIdx.x < n) {
            int g = gids[b + threadIdx.x];
            if (g < 0 || g >= N) g = -1;  // an id outside [0, N): an entry that draws nothing
            float4 A, B, C;
            stage_rec(splats, g, A, B, C);
            sA[threadIdx.x] = A;
            sB[threadIdx.x] = B;
            sC[threadIdx.x] = C;
            float4 Dm = make_float4(0.f, 0.f, 0.f, INFINITY);
            if (SOFT && g >= 0) Dm = stage_depth_model(depth_model, g, sp, C.y);
            if (SOFT) sD[threadIdx.x] = Dm;
            if (rec.A) {
                // the staged records of every batch this CTA takes, in list order, for
                // the backward pass (both half-tile CTAs write the batches they take;
                // where they overlap they write the same values)
                const int64_t e = b + threadIdx.x;
                rec.A[e] = A;
                rec.B[e] = B;
                rec.C[e] = C;
                if (SOFT) rec.D[e] = Dm;
            }
        }
        __syncthreads();
        // this warp's hits of the batch (the staged records whose ellipse reaches its
        // block), listed front to back and padded with NO_HIT to whole pairs
        uint8_t* __restrict__ L = sList[threadIdx.x >> 5];
        int cnt = 0;
        for (int m = 0; m * 32 < n; ++m) {
            const int kk = m * 32 + lane;
            const bool hit = kk < n && block_hits(sA[kk], sB[kk], sC[kk].w, pm.x0, pm.y0) && !(SOFT && sD[kk].w > Dw);
            const uint32_t mask = __ballot_sync(0xffffffffu, hit);
            if (hit) L[cnt + __popc(mask & ((1u << lane) - 1u))] = (uint8_t)kk;
            cnt += __popc(mask);
        }
        if (lane < 2) L[cnt + lane] = NO_HIT;
        __syncwarp();
        if (!SOFT && rec.L) {  // the list, for the backward pass (slot of warp w of the tile: w * cap)
            const int wit = (blockIdx.x % CTAS_PER_TILE) * CTA_WARPS + (threadIdx.x >> 5);
            uint8_t* __restrict__ dst = rec.L + (int64_t)wit * rec.cap + b;
#pragma unroll 1
            for (int t = lane; t < n; t += 32) dst[t] = t < cnt ? L[t] : NO_HIT;
        }
        const int pos0 = b - r.x;  // list position of staged record 0
        for (int p = 0; p < cnt; p += 2) {
            if (__all_sync(0xffffffffu, done)) break;
            // two hits at a time, both evaluated before the transmittance chain takes
            // them in list order; every lane evaluates both and keeps what applies to
            // its pixel (a NO_HIT entry reads a staged record and keeps nothing)
            const uint32_t k2 = *reinterpret_cast<const uint16_t*>(L + p);
            const int kq[2] = {(int)(k2 & 0xffu), (int)(k2 >> 8)};
            float4 Cq[2], Bq[2];
            Eval ev[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ks = kq[h] & (CTA_THREADS - 1);
                Cq[h] = sC[ks];
                const float4 A = sA[ks];
                Bq[h] = sB[ks];
                ev[h] = eval_splat(A, Bq[h], px, py);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool live = (h == 0 || kq[h] != NO_HIT) && !done;  // only the second can be padding
                // hard test, sorted by depth: once a Gaussian is not in front of the
                // mesh, none after it is
                const bool occluded = !soft && !(Cq[h].y < D);
                if (STATS) visited += live && !occluded;
                done = done || (live && occluded);
                bool use = live && !occluded && !ev[h].skip;
                float a = ev[h].alpha;
                if (SOFT && soft && use) {  // the Gaussian's part in front of the mesh
                    const float4 Dm = sD[kq[h]];
                    const float zs = fmaf(Dm.x, ev[h].dx, fmaf(Dm.y, ev[h].dy, Cq[h].y));
                    a *= sp.front((D - zs) * Dm.z);
                    use = a >= ALPHA_MIN;
                }
                const float Tn = __fmul_rn(T, __fsub_rn(1.0f, a));
                const bool stop = Tn <= T_STOP;
                done = done || (use && stop);
                const bool blend = use && !stop;
                const float w = a * T;
                Cr = blend ? fmaf(w, Bq[h].z, Cr) : Cr;
                Cg = blend ? fmaf(w, Bq[h].w, Cg) : Cg;
                Cb = blend ? fmaf(w, Cq[h].x, Cb) : Cb;
                Z = blend ? fmaf(w, Cq[h].y, Z) : Z;
                T = blend ? Tn : T;
                last = blend ? pos0 + kq[h] + 1 : last;
                if (STATS) blended += blend;
            }
        }
    }
    if (STATS) {
        block_count(visited, stats);
        block_count(blended, stats + 1);
    }
    if (inside) {
        float tr, tg, tb;
        if (aa_cov) {
            // the layer (coverage a, premultiplied colour) over the background; the
            // colour and depth composited behind it are added by k_composite_back
            const float a = aa_cov[pix], ua = 1.0f - a;
            tr = fmaf(ua, bg.x, mesh_rgb[3 * pix]);
            tg = fmaf(ua, bg.y, mesh_rgb[3 * pix + 1]);
            tb = fmaf(ua, bg.z, mesh_rgb[3 * pix + 2]);
            out_depth[pix] = a > 0.0f ? fmaf(T, a * D, Z) : Z;
            out_alpha[pix] = 1.0f - T * ua;
        } else {
            if (cov) {
                tr = mesh_rgb[3 * pix]; tg = mesh_rgb[3 * pix + 1]; tb = mesh_rgb[3 * pix + 2];
            } else {
                tr = bg.x; tg = bg.y; tb = bg.z;
            }
            out_depth[pix] = cov ? fmaf(T, D, Z) : Z;
            out_alpha[pix] = cov ? 1.0f : 1.0f - T;
        }
        out_rgb[3 * pix] = fmaf(T, tr, Cr);
        out_rgb[3 * pix + 1] = fmaf(T, tg, Cg);
        out_rgb[3 * pix + 2] = fmaf(T, tb, Cb);
        T_final[pix] = T;
        n_contrib[pix] = last;
    }
}

constexpr int NGRAD = 10;
constexpr int GROUP = 4;
constexpr unsigned FULL = 0xffffffffu;

// One level of a reduce-scatter over the lanes xor o: of each pair of values
// (a, b) the lane keeps the one its bit o selects and adds its partner's copy
// of it.
__device__ __forceinline__ float rs_combine(float a, float b, int lane, int o)
{
    const bool hi = lane & o;
    return (hi ? b : a) + __shfl_xor_sync(FULL, hi ? a : b, o);
}

// Accumulator slots of a staged entry: sums over the CTA's pixels of the
// per-pixel terms, ds = dL/d sigma, (dx, dy) = pixel centre - mean, w = alpha
// T_front:
//   0 ds dx, 1 ds dy, 2 ds dx^2 / 2, 3 ds dx dy, 4 ds dy^2 / 2, 5 ds,
//   6 w g_r, 7 w g_g, 8 w g_b, 9 w g_depth;
// with the soft split four more, 10 pz, 11 pz dx, 12 pz dy, 13 psx, where pz =
// dL/dx kappa and psx = dL/dx x for the split's argument x.
//
// The sums become the record's gradient (components 0..9 of the record
// layout) when the entry leaves the stage:
//   sigma = -l / log2e, l = a2 dx^2 + b2 dx dy + c2 dy^2, so d sigma / d mean =
//   -(a dx + b dy, b dx + c dy) with a = -2 a2 / log2e, b = -b2 / log2e,
//   c = -2 c2 / log2e; and dL/d opacity = sum dL/d alpha G = -sum ds / opacity
//   (ds = -dL/d alpha alpha, alpha = opacity G where alpha is not clamped; both
//   terms are zero where it is).
__device__ __forceinline__ void record_grad(const float* acc, const float4& A, const float4& B, float* out)
{
    const float tx = acc[0] * (1.0f / LOG2E), ty = acc[1] * (1.0f / LOG2E);
    out[0] = 2.0f * A.z * tx + A.w * ty;
    out[1] = A.w * tx + 2.0f * B.x * ty;
    out[2] = acc[2];
    out[3] = acc[3];
    out[4] = acc[4];
    out[5] = B.y > 0.0f ? -acc[5] / B.y : 0.0f;
#pragma unroll
    for (int q = 6; q < NGRAD; ++q) out[q] = acc[q];
}

// Adds a gradient row (components 0..9) to its Gaussian's row of v_splats:
// three 16-byte vector atomics, the last of which adds zero to the two padding
// floats.
__device__ __forceinline__ void add_grad_row(float* __restrict__ v_splats, int g, const float* v)
{
    float4* dst = reinterpret_cast<float4*>(v_splats + 12 * (int64_t)g);
    atomicAdd(dst, make_float4(v[0], v[1], v[2], v[3]));
    atomicAdd(dst + 1, make_float4(v[4], v[5], v[6], v[7]));
    atomicAdd(dst + 2, make_float4(v[8], v[9], 0.0f, 0.0f));
}

__device__ __forceinline__ void flush_grad(float* __restrict__ v_splats, int g, const float* acc, const float4& A,
                                           const float4& B)
{
    float v[NGRAD];
    record_grad(acc, A, B, v);
    add_grad_row(v_splats, g, v);
}

// With the soft split the sums 10..13 add their part: the split's argument x =
// (D - z*) kappa, z* = z_c + g . (p - mean2d), so dL/d mean2d += pz g, dL/d z_c
// -= pz, dL/d g -= pz d, dL/d sigma_z = -psx / sigma_z (kappa = 1 / (sigma_z
// softness)).
__device__ __forceinline__ void flush_grad_soft(float* __restrict__ v_splats, float* __restrict__ v_depth_model,
                                                int g, const float* acc, const float4& A, const float4& B,
                                                const float4& Dm, float softness)
{
    float v[NGRAD];
    record_grad(acc, A, B, v);
    v[0] += acc[10] * Dm.x;
    v[1] += acc[10] * Dm.y;
    v[9] -= acc[10];
    add_grad_row(v_splats, g, v);
    atomicAdd(reinterpret_cast<float4*>(v_depth_model) + g,
              make_float4(-acc[11], -acc[12], -acc[13] * Dm.z * softness, 0.0f));
}

// ------------------------------------------- tensor-core reduction ---------
//
// Hard split: the warp's sums over its 32 pixels of the gradient terms of a
// group of eight entries are a small contraction, (8 entries x 32 pixels) x
// (32 pixels x 6 moments) for ds = dL/d sigma and (8 x 32) x (32 x 4 upstream
// gradient channels) for w = alpha T, done with warp-level tf32 MMAs
// (m16n8k8).  With dx = u + i, dy = v + j (u, v the entry's offset at the
// block's first pixel, i, j the pixel's place in the 8 x 4 block) the six
// pixel moments 1, i, j, i^2, i j, j^2 of ds give every ds term.  Each fp32
// value x enters as two tf32 values (rows g and g + 8 of the A operand): hi =
// x with its 13 low mantissa bits cleared, and lo = x - hi (exact in fp32)
// cleared the same way, which keeps about 20 bits (|x - hi - lo| <= 2^-20 |x|);
// a bit mask costs one instruction where a rounding conversion costs several.
// The moments are small integers, exact in tf32, and the upstream gradient is
// split once per CTA with rounding conversions (columns 0..3 hi, 4..7 lo).

constexpr int RGROUP = 8;  // entries per tensor-core group
constexpr int RPAD = 40;   // row stride of the per-warp staging (conflict-free 8-byte fragment loads)

// The staging rows hold a warp's 32 pixels in fragment order: pixel q * 8 + i
// (k-block q, i < 8) at column q * 8 + 2 i for i < 4 and q * 8 + 2 (i - 4) + 1
// otherwise, so that the two pixels c and c + 4 of a lane's A fragment are
// adjacent (one 8-byte load).
__device__ __forceinline__ int frag_col(int pixel)
{
    const int i = pixel & 7;
    return (pixel & ~7) + (i < 4 ? 2 * i : 2 * (i - 4) + 1);
}

struct RedSmem {
    float ds[RGROUP][RPAD];  // [group slot][frag_col(pixel)] dL/d sigma
    float w[RGROUP][RPAD];   // [group slot][frag_col(pixel)] alpha T_front
    float2 gf[4][32];        // B fragments (b0, b1) of the upstream gradient, per 8-pixel k-block
};

__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 8-pixel k-block of the A operand: rows g (hi) and g + 8 (lo) of group
// slot g at pixels kb * 8 + c and kb * 8 + c + 4 (columns p = kb * 8 + 2 c and
// p + 1 of the staging).
__device__ __forceinline__ void a_frag(const float (&m)[RGROUP][RPAD], int g, int p, uint32_t (&a)[4])
{
    const float2 x = *reinterpret_cast<const float2*>(&m[g][p]);
    const float x0 = x.x, x1 = x.y;
    a[0] = __float_as_uint(x0) & 0xffffe000u;
    a[1] = __float_as_uint(x0 - __uint_as_float(a[0])) & 0xffffe000u;
    a[2] = __float_as_uint(x1) & 0xffffe000u;
    a[3] = __float_as_uint(x1 - __uint_as_float(a[2])) & 0xffffe000u;

}

// pixel moment n (1, i, j, i^2, i j, j^2, 0, 0) of the pixel at (i, j)
__device__ __forceinline__ float moment(int n, int i, int j)
{
    return n == 0 ? 1.0f : n == 1 ? (float)i : n == 2 ? (float)j : n == 3 ? (float)(i * i)
         : n == 4 ? (float)(i * j) : n == 5 ? (float)(j * j) : 0.0f;
}

// ---------------------------------------------- bulk-copy staging ---------
//
// The backward pass's shuffle-sum form (the soft split's, and the hard split's
// under GM_BWD_SHUFFLE_REDUCE) takes each batch of a tile's staged
// records (written by the forward pass in list order) with bulk copies
// (cp.async.bulk, the TMA engine's linear mode) into shared memory: one thread
// issues the copies of a batch and an mbarrier counts their bytes; with two
// buffers the next batch's copies are in flight while the CTA works on the
// current one.  The source is always this GPU's own record buffer.

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of the given parity, at most about COPY_WAIT_NS
// nanoseconds (by the global timer); false when it gave up.
constexpr uint64_t COPY_WAIT_NS = 1000000000ull;

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > COPY_WAIT_NS) return false;
    }
}

// n consecutive 16-byte elements from global src to shared dst, counted on bar
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// generic-proxy accesses of shared memory before this point are ordered before
// the bulk copies issued after it
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace

// Set when a bulk copy's wait gave up (gm_get_copy_status).
__device__ uint32_t g_copy_status = 0;

namespace {

// The kernel is bound by instruction issue, and resident warps hide its
// latencies: the gathered hard split runs ten CTAs of 128 threads per SM (48
// registers, 22 KB of shared memory with the tensor-core staging), the shuffle
// sums with two bulk-copied record buffers nine, the soft split eight (64
// registers: four more terms per entry).  BULK: the records come from the
// forward pass's staged records by bulk copies; otherwise each thread gathers
// and stages one record per batch.  MMA: the warp sums of a group of entries
// on the tensor cores (hard split); otherwise by the shuffle reduce-scatter
// into a per-CTA accumulator.  The hard split with staged records (the
// renderers' default) runs k_composite_bwd_lists instead.
template <bool STATS, bool SOFT, bool BULK, bool MMA>
__global__ void __launch_bounds__(CTA_THREADS, SOFT ? 8 : (BULK ? 9 : 10))
k_composite_bwd(Cam c, float3 bg, int N, Split sp, const int2* __restrict__ tile_range,
                const int32_t* __restrict__ gids, const float4* __restrict__ splats,
                const float4* __restrict__ depth_model, const float* __restrict__ mesh_depth,
                const float* __restrict__ mesh_rgb, const int32_t* __restrict__ face_id,
                const float* __restrict__ T_final, const int32_t* __restrict__ n_contrib,
                const float* __restrict__ g_rgb, const float* __restrict__ g_depth, const float* __restrict__ g_alpha,
                float* __restrict__ v_splats, float* __restrict__ v_depth_model, float* __restrict__ v_mesh_depth,
                AaLayer aa, Staged rec, unsigned long long* __restrict__ stats)
{
    constexpr int NACC = SOFT ? NGRAD + 4 : NGRAD;
    static_assert(!(BULK && MMA), "staged records with the tensor-core sums: k_composite_bwd_lists");
    // the bulk-copied records take two buffers: the next batch in flight
    constexpr int NBUF = BULK ? 2 : 1;
    __shared__ __align__(16) float4 sA_buf[NBUF][CTA_THREADS];
    __shared__ __align__(16) float4 sB_buf[NBUF][CTA_THREADS];
    __shared__ __align__(16) float4 sC_buf[NBUF][CTA_THREADS];
    __shared__ __align__(16) float4 sD_buf[SOFT ? NBUF : 1][SOFT ? CTA_THREADS : 1];
    // per-entry sums of the CTA's pixels (the tensor-core form adds each warp's
    // sums to the gradient rows directly and needs none)
    __shared__ float sAcc[MMA ? 1 : CTA_THREADS][NACC + 1];
    __shared__ __align__(8) uint64_t s_bar[NBUF];
    __shared__ int s_max_last;
    // hard split: the tensor-core reduction's staging per warp, and the moments'
    // B fragments (b0, b1) per k-block and lane, shared by the warps
    __shared__ __align__(16) RedSmem sRed[MMA ? CTA_WARPS : 1];
    __shared__ __align__(16) float2 sMf[MMA ? 4 : 1][32];
    // hard split: each warp's hits of the current batch (staged entry indices)
    __shared__ uint8_t sList[MMA ? CTA_WARPS : 1][MMA ? CTA_THREADS + RGROUP : 1];
    int tile;
    const PixelMap pm = pixel_of(c, tile);
    const int lane = threadIdx.x & 31;
    const bool inside = pm.i < c.W && pm.j < c.H;
    const int64_t pix = (int64_t)pm.j * c.W + pm.i;
    const float px = (float)pm.i + 0.5f, py = (float)pm.j + 0.5f;

    float D = -INFINITY, T = 1.0f, gr = 0.f, gg = 0.f, gb = 0.f, gz = 0.f;
    int last = 0;
    // behind = (colour, depth) accumulated behind the current Gaussian, dotted with
    // this pixel's upstream gradient (g_rgb, g_depth); starts with the terminal layer
    float behind = 0.f, aterm = 0.f;
    bool cov = false;
    float vD = 0.0f;  // soft split: dL/d mesh depth at this pixel
    if (inside) {
        D = mesh_depth[pix];
        cov = aa.cov ? D < INFINITY : face_id[pix] >= 0;
        T = T_final[pix];
        last = n_contrib[pix];
        gr = g_rgb[3 * pix]; gg = g_rgb[3 * pix + 1]; gb = g_rgb[3 * pix + 2];
        gz = g_depth[pix];
        if (aa.cov) {
            // behind the front chain: the layer, and through 1 - a what lies behind it
            // (the back chain's colour, depth and transmittance, then the background)
            const float a = aa.cov[pix], ua = 1.0f - a;
            float Tb = 1.0f, Eb = bg.x * gr + bg.y * gg + bg.z * gb;
            if (cov && a < 1.0f) {
                const float4 bk = aa.back[pix];
                Tb = aa.T_back[pix];
                Eb = fmaf(Tb, Eb, bk.x * gr + bk.y * gg + bk.z * gb + bk.w * gz);
            }
            const float own = mesh_rgb[3 * pix] * gr + mesh_rgb[3 * pix + 1] * gg + mesh_rgb[3 * pix + 2] * gb +
                              (a > 0.0f ? a * D * gz : 0.0f);
            behind = T * fmaf(ua, Eb, own);
            aterm = g_alpha[pix] * T * ua * Tb;
        } else if (cov) {
            behind = T * (mesh_rgb[3 * pix] * gr + mesh_rgb[3 * pix + 1] * gg + mesh_rgb[3 * pix + 2] * gb + D * gz);
        } else {
            behind = T * (bg.x * gr + bg.y * gg + bg.z * gb);
            aterm = g_alpha[pix] * T;  // out_alpha = 1 - T_final when uncovered
        }
    }
    int warp_last = last;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) warp_last = max(warp_last, __shfl_xor_sync(0xffffffffu, warp_last, o));
    if constexpr (MMA) {
        // B fragments: moments of pixel (i, j) = (c (+4), kb) for term g; the upstream
        // gradient's channel g & 3 (hi for g < 4, lo for g >= 4) of pixel kb * 8 + c (+4)
        const int g = lane >> 2, c = lane & 3, kb = threadIdx.x >> 5;
        sMf[kb][lane] = make_float2(moment(g, c, kb), moment(g, c + 4, kb));
        RedSmem& R = sRed[threadIdx.x >> 5];
        float* gtmp = &R.ds[0][0];  // 128 floats of scratch before the first group
        gtmp[4 * lane] = gr;
        gtmp[4 * lane + 1] = gg;
        gtmp[4 * lane + 2] = gb;
        gtmp[4 * lane + 3] = gz;
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float b[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float x = gtmp[4 * (q * 8 + c + 4 * h) + (g & 3)];
                const uint32_t hi = to_tf32(x);
                b[h] = g < 4 ? __uint_as_float(hi) : __uint_as_float(to_tf32(x - __uint_as_float(hi)));
            }
            R.gf[q][lane] = make_float2(b[0], b[1]);
        }
        __syncwarp();
    }
    if (threadIdx.x == 0) {
        s_max_last = 0;
        if (BULK) {
#pragma unroll
            for (int q = 0; q < NBUF; ++q) mbar_init(&s_bar[q], 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    __syncthreads();
    if (lane == 0 && warp_last > 0) atomicMax(&s_max_last, warp_last);
    __syncthreads();
    const int2 r = BULK ? clamp_range(tile_range[tile], rec.cap) : tile_range[tile];
    const int end = BULK ? min(r.x + s_max_last, r.y) : r.x + s_max_last;
    const int n_batches = (end - r.x + CTA_THREADS - 1) / CTA_THREADS;
    const bool soft = SOFT && cov;
    const float Dw = SOFT ? warp_hide_depth(inside, cov, D) : INFINITY;
    uint32_t visited = 0, contributed = 0;
    // batch j holds list positions [max(r.x, end - 128 (j + 1)), end - 128 j)
    auto issue = [&](int j) {
        const int hi = end - CTA_THREADS * j, lo = max(r.x, hi - CTA_THREADS);
        const uint32_t bytes = (uint32_t)(hi - lo) * 16u;
        const int q = j % NBUF;
        mbar_arrive_expect_tx(&s_bar[q], bytes * (SOFT ? 4u : 3u));
        bulk_copy(sA_buf[q], rec.A + lo, bytes, &s_bar[q]);
        bulk_copy(sB_buf[q], rec.B + lo, bytes, &s_bar[q]);
        bulk_copy(sC_buf[q], rec.C + lo, bytes, &s_bar[q]);
        if (SOFT) bulk_copy(sD_buf[SOFT ? q : 0], rec.D + lo, bytes, &s_bar[q]);
    };
    if (BULK && threadIdx.x == 0 && n_batches > 0) issue(0);
    int n_prev = 0;
    for (int j = 0;; ++j) {
        const int cur = j % NBUF, prev = (j + NBUF - 1) % NBUF;
        // the previous batch's gradients go out (each thread its own slot) and, for
        // the gathering form, the next batch comes in on the same slot
        if (!MMA && (int)threadIdx.x < n_prev) {
            const int g = rec_id(sC_buf[prev][threadIdx.x]);
            if (g >= 0) {
                if (SOFT)
                    flush_grad_soft(v_splats, v_depth_model, g, sAcc[threadIdx.x], sA_buf[prev][threadIdx.x],
                                    sB_buf[prev][threadIdx.x], sD_buf[SOFT ? prev : 0][threadIdx.x], sp.softness);
                else
                    flush_grad(v_splats, g, sAcc[threadIdx.x], sA_buf[prev][threadIdx.x], sB_buf[prev][threadIdx.x]);
            }
        }
        if (j >= n_batches) break;
        const int b_end = end - CTA_THREADS * j;
        const int b0 = max(r.x, b_end - CTA_THREADS);
        const int n = b_end - b0;
        if ((int)threadIdx.x < n) {
            if (!BULK) {
                int g = gids[b0 + threadIdx.x];
                if (g < 0 || g >= N) g = -1;  // an entry that draws nothing and gets no gradient
                float4 A, B, C;
                stage_rec(splats, g, A, B, C);
                sA_buf[0][threadIdx.x] = A;
                sB_buf[0][threadIdx.x] = B;
                sC_buf[0][threadIdx.x] = C;
                if (SOFT && g >= 0) sD_buf[0][threadIdx.x] = stage_depth_model(depth_model, g, sp, C.y);
            }
            if (!MMA) {
#pragma unroll
                for (int q = 0; q < NACC; ++q) sAcc[threadIdx.x][q] = 0.0f;
            }
        }
        __syncthreads();
        if (BULK) {
            if (threadIdx.x == 0) {
                if (j + 1 < n_batches) {
                    // the other buffer was last read by the flush above: free after the barrier
                    fence_proxy_async_smem();
                    issue(j + 1);
                }
            }
            const bool ok = __syncthreads_and(mbar_wait(&s_bar[cur], (uint32_t)(j / NBUF) & 1u));
            if (!ok) {
                // a copy did not arrive: report, let the copies in flight land, stop
                if (threadIdx.x == 0) atomicOr(&g_copy_status, 1u);
                mbar_wait(&s_bar[cur], (uint32_t)(j / NBUF) & 1u);
                if (j + 1 < n_batches)
                    mbar_wait(&s_bar[(j + 1) % NBUF], (uint32_t)((j + 1) / NBUF) & 1u);
                return;
            }
        }
        const float4* __restrict__ sA = sA_buf[cur];
        const float4* __restrict__ sB = sB_buf[cur];
        const float4* __restrict__ sC = sC_buf[cur];
        const float4* __restrict__ sD = sD_buf[SOFT ? cur : 0];
        // this warp only needs the entries in front of its last composited one, and of
        // those only the ones that can reach its pixels; the tensor-core form takes them
        // from a hit list in groups of eight, the shuffle form from a ballot per 32
        // entries four at a time, both from the back
        const int k_top = min(n, warp_last - (b0 - r.x)) - 1;
        if constexpr (MMA) {
            // the warp's hits of this batch (entries up to k_top whose ellipse reaches
            // its block), listed back to front, padded with NO_HIT to whole groups
            RedSmem& R = sRed[threadIdx.x >> 5];
            uint8_t* __restrict__ L = sList[threadIdx.x >> 5];
            int cnt = 0;
            for (int m = k_top >> 5; m >= 0; --m) {
                const int kk = m * 32 + lane;
                const bool hit = kk <= k_top && block_hits(sA[kk], sB[kk], sC[kk].w, pm.x0, pm.y0);
                const uint32_t mask = __ballot_sync(FULL, hit);
                // hits above this lane in the chunk come first
                if (hit) L[cnt + __popc(mask >> lane) - 1] = (uint8_t)kk;
                cnt += __popc(mask);
            }
            if (lane < RGROUP) L[cnt + lane] = NO_HIT;
            __syncwarp();
            // entries [0, lastk) of the batch lie before the pixel's last composited one
            // (all of them in front of the mesh, which ended the pixel's forward chain);
            // NO_HIT >= CTA_THREADS >= lastk
            const int lastk = min(last - (b0 - r.x), CTA_THREADS);
            const int col = frag_col(lane);
            for (int base = 0; base < cnt; base += RGROUP) {
                // per entry of the group, back to front: w = alpha T_front and ds =
                // dL/d sigma at this lane's pixel, staged for the contraction.  Every
                // lane evaluates every entry (most groups' entries reach some lane of
                // the block) and keeps the result where the entry is composited there.
                bool any = false;
#pragma unroll
                for (int jj = 0; jj < RGROUP; ++jj) {
                    const int k = L[base + jj];
                    const int ks = k & (CTA_THREADS - 1);  // NO_HIT reads a staged record and keeps nothing
                    const float4 C3 = sC[ks], A = sA[ks], B = sB[ks];
                    const Eval e = eval_splat(A, B, px, py);
                    const bool seen = k < lastk;
                    const bool take = seen && !e.skip;
                    if (STATS) {
                        visited += seen;
                        contributed += take;
                    }
                    const float a = e.alpha;
                    const float rom = __fdividef(1.0f, 1.0f - a);
                    const float Tp = T * rom;  // transmittance in front of it
                    const float w = a * Tp;
                    const float front = B.z * gr + B.w * gg + C3.x * gb + C3.y * gz;
                    const float dLda = Tp * front + (aterm - behind) * rom;
                    behind = take ? fmaf(w, front, behind) : behind;
                    T = take ? Tp : T;
                    any |= take;
                    // alpha clamped at 0.99 has no opacity / sigma gradient; elsewhere
                    // d alpha / d sigma = -alpha
                    R.ds[jj][col] = take && !e.clamped ? -dLda * a : 0.0f;
                    R.w[jj][col] = take ? w : 0.0f;
                }
                if (__any_sync(FULL, any)) {
                    __syncwarp();
                    const int g = lane >> 2, c = lane & 3;
                    float dm[4] = {0.f, 0.f, 0.f, 0.f}, dc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t a[4];
                        const float2 bm = sMf[q][lane], bg = R.gf[q][lane];
                        a_frag(R.ds, g, q * 8 + 2 * c, a);
                        mma_tf32(dm, a[0], a[1], a[2], a[3], __float_as_uint(bm.x), __float_as_uint(bm.y));
                        a_frag(R.w, g, q * 8 + 2 * c, a);
                        mma_tf32(dc, a[0], a[1], a[2], a[3], __float_as_uint(bg.x), __float_as_uint(bg.y));
                    }
                    // lane (g, c): group slot g, terms 2c and 2c + 1 (hi rows + lo rows):
                    // S_n = sum ds m_n for c = 0 (S0, Si), 1 (Sj, Sii), 2 (Sij, Sjj); the
                    // colour sums of channels 2c, 2c + 1 (c < 2 hi, c >= 2 lo columns)
                    const float t0 = dm[0] + dm[2], t1 = dm[1] + dm[3];
                    float e0 = dc[0] + dc[2], e1 = dc[1] + dc[3];
                    e0 += __shfl_xor_sync(FULL, e0, 2);
                    e1 += __shfl_xor_sync(FULL, e1, 2);
                    // lane c = 0 collects the entry's six moments and four colour sums
                    const float sj = __shfl_down_sync(FULL, t0, 1), sii = __shfl_down_sync(FULL, t1, 1);
                    const float sij = __shfl_down_sync(FULL, t0, 2), sjj = __shfl_down_sync(FULL, t1, 2);
                    const float eb = __shfl_down_sync(FULL, e0, 1), ez = __shfl_down_sync(FULL, e1, 1);
                    const int k = L[base + g];
                    const int gid = k != NO_HIT ? rec_id(sC[k]) : -1;
                    if (c == 0 && gid >= 0) {
                        // with dx = u + i, dy = v + j (u, v at the block's first pixel):
                        //   sum ds dx = u S0 + Si, sum ds dy = v S0 + Sj,
                        //   sum ds dx^2 / 2 = u (u S0 / 2 + Si) + Sii / 2,
                        //   sum ds dx dy = v (u S0 + Si) + u Sj + Sij,
                        //   sum ds dy^2 / 2 = v (v S0 / 2 + Sj) + Sjj / 2, sum ds = S0
                        const float4 A = sA[k], B = sB[k];
                        const float u = pm.x0 - A.x, v = pm.y0 - A.y;
                        float acc[NGRAD];
                        acc[0] = fmaf(u, t0, t1);
                        acc[1] = fmaf(v, t0, sj);
                        acc[2] = fmaf(u, fmaf(0.5f * u, t0, t1), 0.5f * sii);
                        acc[3] = fmaf(v, acc[0], fmaf(u, sj, sij));
                        acc[4] = fmaf(v, fmaf(0.5f * v, t0, sj), 0.5f * sjj);
                        acc[5] = t0;
                        acc[6] = e0;
                        acc[7] = e1;
                        acc[8] = eb;
                        acc[9] = ez;
                        flush_grad(v_splats, gid, acc, A, B);
                    }
                }
                __syncwarp();  // the staging is rewritten by the next group
            }
        } else
        for (int m = k_top >> 5; m >= 0; --m) {
            const int kk = m * 32 + lane;
            uint32_t mask =
                __ballot_sync(0xffffffffu, kk <= k_top && block_hits(sA[kk], sB[kk], sC[kk].w, pm.x0, pm.y0) &&
                                               !(SOFT && sD[kk].w > Dw));
            while (mask) {
                int kj[GROUP];
#pragma unroll
                for (int jj = 0; jj < GROUP; ++jj) {
                    if (mask) {
                        const int bit = 31 - __clz(mask);
                        kj[jj] = m * 32 + bit;
                        mask &= ~(1u << bit);
                    } else {
                        kj[jj] = -1;
                    }
                }
                // per entry: w = alpha T_front, ds = dL/d sigma (soft split: pz = dL/dx
                // kappa, psx = dL/dx x)
                float pw[GROUP], pds[GROUP], pz[GROUP], psx[GROUP];
                bool any = false;
#pragma unroll
                for (int jj = 0; jj < GROUP; ++jj) {
                    pw[jj] = pds[jj] = pz[jj] = psx[jj] = 0.0f;
                    const int k = kj[jj];
                    if (k < 0 || !inside || b0 - r.x + k >= last) continue;
                    const float4 C3 = sC[k];
                    if (!soft && !(C3.y < D)) continue;
                    if (STATS) ++visited;
                    const float4 A = sA[k], B = sB[k];
                    const Eval e = eval_splat(A, B, px, py);
                    if (e.skip) continue;
                    float a = e.alpha, f = 1.0f, x = 0.0f, kap = 0.0f;
                    if (soft) {  // the composited alpha is alpha f, f = f(x)
                        const float4 Dm = sD[k];
                        const float zs = fmaf(Dm.x, e.dx, fmaf(Dm.y, e.dy, C3.y));
                        kap = Dm.z;
                        x = (D - zs) * kap;
                        f = sp.front(x);
                        a = e.alpha * f;
                        if (a < ALPHA_MIN) continue;
                    }
                    if (STATS) ++contributed;
                    any = true;
                    const float rom = __fdividef(1.0f, 1.0f - a);
                    const float Tp = T * rom;  // transmittance in front of this Gaussian
                    const float w = a * Tp;
                    const float front = B.z * gr + B.w * gg + C3.x * gb + C3.y * gz;
                    const float dLda = Tp * front + (aterm - behind) * rom;  // dL / d(composited alpha)
                    behind = fmaf(w, front, behind);
                    T = Tp;
                    pw[jj] = w;
                    // alpha clamped at 0.99 has no opacity / sigma gradient; elsewhere
                    // d alpha / d sigma = -alpha
                    if (!e.clamped) pds[jj] = -(SOFT ? dLda * f : dLda) * e.alpha;
                    if (soft) {  // dL/dx = dLda alpha f'(x)
                        const float psi = dLda * e.alpha * sp.density(x, f);
                        pz[jj] = psi * kap;
                        psx[jj] = psi * x;
                        vD += psi * kap;
                    }
                }
                if (__any_sync(FULL, any)) {
                    // Warp sums of the four entries' terms by a reduce-scatter over the
                    // lanes.  The terms are products whose factors a lane picks by its
                    // bits 4 and 3 (h4, h3), so the first two levels (lanes xor 16, then
                    // xor 8) need no select: with X = (1, dx), Y = (1, dy) and G =
                    // ((g_r, g_g), (g_b, g_depth)), the lane keeps ds X[h4] Y[h3] and
                    // w G[h4][h3] and sends its partners the other products.  Level 3
                    // (xor 4) then picks the ds- or the w-term, levels 4 and 5 the
                    // entry: lane L ends with term (L >> 2) of entry L & 3.  The
                    // ds dx^2 / 2, ds dy^2 / 2 terms (with the soft split also pz dx, pz
                    // dy) take a second, shorter reduction of the same form; the soft
                    // split's pz and psx a third.
                    const bool h4 = lane & 16, h3 = lane & 8;
                    const float P0 = h4 ? gb : gr, P1 = h4 ? gz : gg, Q0 = h4 ? gr : gb, Q1 = h4 ? gg : gz;
                    const float Gkk = h3 ? P1 : P0, Gks = h3 ? P0 : P1, Gsk = h3 ? Q1 : Q0, Gss = h3 ? Q0 : Q1;
                    float RA[GROUP], RB[GROUP], R2[GROUP];
#pragma unroll
                    for (int jj = 0; jj < GROUP; ++jj) {
                        // pixel offsets recomputed (the same roundings as eval_splat)
                        // rather than kept live through the group: fewer registers; a
                        // missing entry (all terms zero) borrows the first one's mean
                        const float2 mean = *reinterpret_cast<const float2*>(&sA[kj[jj] < 0 ? kj[0] : kj[jj]]);
                        const float dx = __fsub_rn(px, mean.x), dy = __fsub_rn(py, mean.y);
                        const float ds = pds[jj], w = pw[jj];
                        const float dsx = ds * dx;
                        const float Ak = h4 ? dsx : ds, As = h4 ? ds : dsx;  // ds X[h4], ds X[!h4]
                        const float Yk = h3 ? dy : 1.0f, Ys = h3 ? 1.0f : dy;  // Y[h3], Y[!h3]
                        float K = Ak * Yk + __shfl_xor_sync(FULL, As * Yk, 16);
                        float S = Ak * Ys + __shfl_xor_sync(FULL, As * Ys, 16);
                        RA[jj] = K + __shfl_xor_sync(FULL, S, 8);
                        K = w * Gkk + __shfl_xor_sync(FULL, w * Gsk, 16);
                        S = w * Gks + __shfl_xor_sync(FULL, w * Gss, 16);
                        RB[jj] = K + __shfl_xor_sync(FULL, S, 8);
                        // ds dx^2 / 2 kept by h4 = 0, ds dy^2 / 2 by h4 = 1; with the soft
                        // split also pz dx, pz dy: u[b4] F[b3] with u = (dx, dy), F = (u ds / 2,
                        // pz), two select-free levels like the first reduction's
                        const float hds = 0.5f * ds, uk = h4 ? dy : dx, us = h4 ? dx : dy;
                        const float hk = hds * uk, hs = hds * us;
                        if (SOFT) {
                            const float z = pz[jj];
                            K = uk * (h3 ? z : hk) + __shfl_xor_sync(FULL, us * (h3 ? z : hs), 16);
                            S = uk * (h3 ? hk : z) + __shfl_xor_sync(FULL, us * (h3 ? hs : z), 16);
                            R2[jj] = K + __shfl_xor_sync(FULL, S, 8);
                        } else {
                            R2[jj] = hk * uk + __shfl_xor_sync(FULL, hs * us, 16);
                        }
                    }
                    {   // levels 3..5: the term kind, then the entry
                        const float T0 = rs_combine(RA[0], RB[0], lane, 4), T1 = rs_combine(RA[1], RB[1], lane, 4);
                        const float T2 = rs_combine(RA[2], RB[2], lane, 4), T3 = rs_combine(RA[3], RB[3], lane, 4);
                        const float U0 = rs_combine(T0, T2, lane, 2), U1 = rs_combine(T1, T3, lane, 2);
                        const float tot = rs_combine(U0, U1, lane, 1);
                        const int e = lane & 3;
                        const int k = e == 0 ? kj[0] : e == 1 ? kj[1] : e == 2 ? kj[2] : kj[3];
                        // slot of ds X[h4] Y[h3] (lane bit 2 clear) or w G[h4][h3] (set)
                        const int slot = (lane & 4) ? 6 + (h4 ? 2 : 0) + (h3 ? 1 : 0)
                                                    : (h4 ? (h3 ? 3 : 0) : (h3 ? 1 : 5));
                        if (k >= 0 && tot != 0.0f) atomicAdd(&sAcc[k][slot], tot);
                    }
                    if (!SOFT) {  // ds dx^2 / 2, ds dy^2 / 2: the entry by lane bits 3, 2,
                                  // then a butterfly over bits 1, 0
                        const float V0 = rs_combine(R2[0], R2[2], lane, 8), V1 = rs_combine(R2[1], R2[3], lane, 8);
                        float t2 = rs_combine(V0, V1, lane, 4);
                        t2 += __shfl_xor_sync(FULL, t2, 2);
                        t2 += __shfl_xor_sync(FULL, t2, 1);
                        const int e = (lane >> 2) & 3;
                        const int k = e == 0 ? kj[0] : e == 1 ? kj[1] : e == 2 ? kj[2] : kj[3];
                        if ((lane & 3) == 0 && k >= 0 && t2 != 0.0f) atomicAdd(&sAcc[k][h4 ? 4 : 2], t2);
                    } else {
                        {   // ds dx^2 / 2, ds dy^2 / 2, pz dx, pz dy: the entry by lane bits 2,
                            // 1, then a butterfly over bit 0
                            const float W0 = rs_combine(R2[0], R2[2], lane, 4), W1 = rs_combine(R2[1], R2[3], lane, 4);
                            float t2 = rs_combine(W0, W1, lane, 2);
                            t2 += __shfl_xor_sync(FULL, t2, 1);
                            const int e = (lane >> 1) & 3;
                            const int k = e == 0 ? kj[0] : e == 1 ? kj[1] : e == 2 ? kj[2] : kj[3];
                            const int slot = h3 ? (h4 ? 12 : 11) : (h4 ? 4 : 2);
                            if ((lane & 1) == 0 && k >= 0 && t2 != 0.0f) atomicAdd(&sAcc[k][slot], t2);
                        }
                        // pz (kept by h4 = 0), psx (h4 = 1): the entry by lane bits 3, 2, then a
                        // butterfly over bits 1, 0
                        float R3[GROUP];
#pragma unroll
                        for (int jj = 0; jj < GROUP; ++jj)
                            R3[jj] = (h4 ? psx[jj] : pz[jj]) + __shfl_xor_sync(FULL, h4 ? pz[jj] : psx[jj], 16);
                        const float V0 = rs_combine(R3[0], R3[2], lane, 8), V1 = rs_combine(R3[1], R3[3], lane, 8);
                        float t3 = rs_combine(V0, V1, lane, 4);
                        t3 += __shfl_xor_sync(FULL, t3, 2);
                        t3 += __shfl_xor_sync(FULL, t3, 1);
                        const int e = (lane >> 2) & 3;
                        const int k = e == 0 ? kj[0] : e == 1 ? kj[1] : e == 2 ? kj[2] : kj[3];
                        if ((lane & 3) == 0 && k >= 0 && t3 != 0.0f) atomicAdd(&sAcc[k][h4 ? 13 : 10], t3);
                    }
                }
            }
        }
        __syncthreads();
        n_prev = n;
    }
    if (STATS) {
        block_count(visited, stats);
        block_count(contributed, stats + 1);
    }
    if (SOFT && inside && v_mesh_depth) v_mesh_depth[pix] = vD;
}

// Hard split with the forward's staged records and hit lists: every warp works
// through its own lists with no CTA barrier.  It reads the lists of the
// forward's batches back to front, up to the warp's last composited entry, into
// a ring of pending list positions (descending), and takes them eight at a time
// whatever batch they come from, so that only the last group is padded; each
// group's records are loaded from the staged buffer by the warp itself (three
// 16-byte loads a record, one per lane) into a per-warp group buffer, the next
// group's loads in flight while the warp works on the current one.  The
// per-entry chain, the tensor-core sums and the gradient atomics are those of
// k_composite_bwd.
struct GroupRec {
    float4 r[3][RGROUP];  // A, B, C of each group slot
};
constexpr int PEND_RING = 256;         // pending positions a warp holds: < 2 groups + a batch + padding
constexpr int PEND_NONE = 0x7fffffff;  // a padding slot

template <bool STATS>
__global__ void __launch_bounds__(CTA_THREADS, 9)
k_composite_bwd_lists(Cam c, float3 bg, const int2* __restrict__ tile_range, const float* __restrict__ mesh_depth,
                      const float* __restrict__ mesh_rgb, const int32_t* __restrict__ face_id,
                      const float* __restrict__ T_final, const int32_t* __restrict__ n_contrib,
                      const float* __restrict__ g_rgb, const float* __restrict__ g_depth,
                      const float* __restrict__ g_alpha, float* __restrict__ v_splats, AaLayer aa, Staged rec,
                      unsigned long long* __restrict__ stats)
{
    __shared__ __align__(16) RedSmem sRed[CTA_WARPS];
    __shared__ __align__(16) float2 sMf[4][32];
    __shared__ __align__(16) int sPend[CTA_WARPS][PEND_RING];
    __shared__ __align__(16) GroupRec sG[CTA_WARPS];
    int tile;
    const PixelMap pm = pixel_of(c, tile);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool inside = pm.i < c.W && pm.j < c.H;
    const int64_t pix = (int64_t)pm.j * c.W + pm.i;
    const float px = (float)pm.i + 0.5f, py = (float)pm.j + 0.5f;

    float D = -INFINITY, T = 1.0f, gr = 0.f, gg = 0.f, gb = 0.f, gz = 0.f;
    int last = 0;
    // behind = (colour, depth) accumulated behind the current Gaussian, dotted with
    // this pixel's upstream gradient (g_rgb, g_depth); starts with the terminal layer
    float behind = 0.f, aterm = 0.f;
    if (inside) {
        D = mesh_depth[pix];
        const bool cov = aa.cov ? D < INFINITY : face_id[pix] >= 0;
        T = T_final[pix];
        last = n_contrib[pix];
        gr = g_rgb[3 * pix]; gg = g_rgb[3 * pix + 1]; gb = g_rgb[3 * pix + 2];
        gz = g_depth[pix];
        if (aa.cov) {
            // behind the front chain: the layer, and through 1 - a what lies behind it
            // (the back chain's colour, depth and transmittance, then the background)
            const float a = aa.cov[pix], ua = 1.0f - a;
            float Tb = 1.0f, Eb = bg.x * gr + bg.y * gg + bg.z * gb;
            if (cov && a < 1.0f) {
                const float4 bk = aa.back[pix];
                Tb = aa.T_back[pix];
                Eb = fmaf(Tb, Eb, bk.x * gr + bk.y * gg + bk.z * gb + bk.w * gz);
            }
            const float own = mesh_rgb[3 * pix] * gr + mesh_rgb[3 * pix + 1] * gg + mesh_rgb[3 * pix + 2] * gb +
                              (a > 0.0f ? a * D * gz : 0.0f);
            behind = T * fmaf(ua, Eb, own);
            aterm = g_alpha[pix] * T * ua * Tb;
        } else if (cov) {
            behind = T * (mesh_rgb[3 * pix] * gr + mesh_rgb[3 * pix + 1] * gg + mesh_rgb[3 * pix + 2] * gb + D * gz);
        } else {
            behind = T * (bg.x * gr + bg.y * gg + bg.z * gb);
            aterm = g_alpha[pix] * T;  // out_alpha = 1 - T_final when uncovered
        }
    }
    int warp_last = last;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) warp_last = max(warp_last, __shfl_xor_sync(0xffffffffu, warp_last, o));
    RedSmem& R = sRed[w];
    {
        // B fragments: moments of pixel (i, j) = (c (+4), kb) for term g; the upstream
        // gradient's channel g & 3 (hi for g < 4, lo for g >= 4) of pixel kb * 8 + c (+4)
        const int g = lane >> 2, c = lane & 3;
        for (int kb = w; kb < 4; kb += CTA_WARPS) sMf[kb][lane] = make_float2(moment(g, c, kb), moment(g, c + 4, kb));
        float* gtmp = &R.ds[0][0];  // 128 floats of scratch before the first group
        gtmp[4 * lane] = gr;
        gtmp[4 * lane + 1] = gg;
        gtmp[4 * lane + 2] = gb;
        gtmp[4 * lane + 3] = gz;
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float b[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float x = gtmp[4 * (q * 8 + c + 4 * h) + (g & 3)];
                const uint32_t hi = to_tf32(x);
                b[h] = g < 4 ? __uint_as_float(hi) : __uint_as_float(to_tf32(x - __uint_as_float(hi)));
            }
            R.gf[q][lane] = make_float2(b[0], b[1]);
        }
        __syncwarp();
    }
    __syncthreads();  // the moments' fragments, written by every warp
    uint32_t visited = 0, contributed = 0;
    const int2 r = clamp_range(tile_range[tile], rec.cap);
    const int wn = min(warp_last, r.y - r.x);  // this warp's entries: positions [0, wn) after r.x
    int j = (wn + CTA_THREADS - 1) / CTA_THREADS - 1;  // the next of the forward's batches to list
    const int wit = (blockIdx.x % CTAS_PER_TILE) * CTA_WARPS + w;
    const uint8_t* __restrict__ lists = rec.L + (int64_t)wit * rec.cap + r.x;
    int* __restrict__ P = sPend[w];
    GroupRec& G = sG[w];
    const int col = frag_col(lane);
    // the group's records: lane t < 24 loads array t / 8 of slot t % 8
    const int sj = lane & (RGROUP - 1), sa = lane / RGROUP;
    const float4* __restrict__ src = (sa == 0 ? rec.A : sa == 1 ? rec.B : rec.C) + r.x;
    int head = 0, tail = 0;  // pending positions: ring slots [head, tail)
    // Lists the forward's batches, back to front, until two groups are pending:
    // each batch's list (ascending, NO_HIT after its end) contributes its entries
    // below the warp's end, reversed, as positions; after the first batch the
    // pending positions are padded with PEND_NONE to a whole group.
    auto refill = [&]() {
        while (tail - head < 2 * RGROUP && j >= 0) {
            const int b0 = CTA_THREADS * j;
            const int n = min(CTA_THREADS, wn - b0);
            int fl[CTA_THREADS / 32];
            int cnt = 0;
#pragma unroll
            for (int i = 0; i < CTA_THREADS / 32; ++i) {
                const int t = 32 * i + lane;
                fl[i] = t < n ? __ldg(lists + b0 + t) : NO_HIT;
                cnt += __popc(__ballot_sync(FULL, fl[i] < n));
            }
#pragma unroll
            for (int i = 0; i < CTA_THREADS / 32; ++i)
                if (fl[i] < n) P[(tail + cnt - 1 - (32 * i + lane)) & (PEND_RING - 1)] = b0 + fl[i];
            tail += cnt;
            --j;
        }
        if (j < 0) {
            const int end = (tail + RGROUP - 1) & ~(RGROUP - 1);
            if (lane < end - tail) P[(tail + lane) & (PEND_RING - 1)] = PEND_NONE;
            tail = end;
        }
        __syncwarp();
    };
    auto load_slot = [&](int base) {
        const int p = lane < 3 * RGROUP ? P[(base & (PEND_RING - 1)) + sj] : PEND_NONE;
        return p != PEND_NONE ? __ldg(src + p) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    // dL/d alpha of an entry = T_front front + (aterm - behind) / (1 - alpha): the
    // chain carries aterm - behind
    float nbh = aterm - behind;
    refill();
    float4 nxt = head < tail ? load_slot(head) : make_float4(0.f, 0.f, 0.f, 0.f);
    while (head < tail) {
        if (lane < 3 * RGROUP) G.r[sa][sj] = nxt;
        refill();  // the next group pending (its loads in flight while the warp works on this one)
        if (head + RGROUP < tail) nxt = load_slot(head + RGROUP);
        const int* __restrict__ Pg = P + (head & (PEND_RING - 1));
        const int4 pa = *reinterpret_cast<const int4*>(Pg), pb = *reinterpret_cast<const int4*>(Pg + 4);
        const int pos[RGROUP] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
        // per entry of the group, back to front: w = alpha T_front and ds = dL/d
        // sigma at this lane's pixel, staged for the contraction (every lane
        // evaluates every entry and keeps its pixel's part by selects); an entry
        // lies before the pixel's last composited one, and so in front of the mesh,
        // when its position is below the pixel's count (PEND_NONE is not)
        bool any = false;
#pragma unroll
        for (int jj = 0; jj < RGROUP; ++jj) {
            const float4 A = G.r[0][jj], B = G.r[1][jj], C3 = G.r[2][jj];
            const Eval e = eval_splat(A, B, px, py);
            const bool seen = pos[jj] < last;
            const bool take = seen && !e.skip;
            if (STATS) {
                visited += seen;
                contributed += take;
            }
            const float a = e.alpha;
            const float rom = __fdividef(1.0f, 1.0f - a);
            const float Tp = T * rom;  // transmittance in front of it
            const float wv = a * Tp;
            const float front = B.z * gr + B.w * gg + C3.x * gb + C3.y * gz;
            const float wt = take ? wv : 0.0f;  // an entry not taken adds nothing to the chain
            const float dLda = fmaf(Tp, front, nbh * rom);
            nbh = fmaf(-wt, front, nbh);
            T = take ? Tp : T;
            any |= take;
            // alpha clamped at 0.99 has no opacity / sigma gradient; elsewhere
            // d alpha / d sigma = -alpha
            R.ds[jj][col] = take && !e.clamped ? -dLda * a : 0.0f;
            R.w[jj][col] = wt;
        }
        if (__any_sync(FULL, any)) {
            __syncwarp();
            const int g = lane >> 2, c = lane & 3;
            float dm[4] = {0.f, 0.f, 0.f, 0.f}, dc[4] = {0.f, 0.f, 0.f, 0.f};

#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t af[4];
                const float2 bm = sMf[q][lane], bgf = R.gf[q][lane];
                a_frag(R.ds, g, q * 8 + 2 * c, af);
                mma_tf32(dm, af[0], af[1], af[2], af[3], __float_as_uint(bm.x), __float_as_uint(bm.y));
                a_frag(R.w, g, q * 8 + 2 * c, af);
                mma_tf32(dc, af[0], af[1], af[2], af[3], __float_as_uint(bgf.x), __float_as_uint(bgf.y));
            }
            // lane (g, c): group slot g, terms 2c and 2c + 1 (see k_composite_bwd)
            const float t0 = dm[0] + dm[2], t1 = dm[1] + dm[3];
            float e0 = dc[0] + dc[2], e1 = dc[1] + dc[3];
            e0 += __shfl_xor_sync(FULL, e0, 2);
            e1 += __shfl_xor_sync(FULL, e1, 2);
            const float sj = __shfl_down_sync(FULL, t0, 1), sii = __shfl_down_sync(FULL, t1, 1);
            const float sij = __shfl_down_sync(FULL, t0, 2), sjj = __shfl_down_sync(FULL, t1, 2);
            const float eb = __shfl_down_sync(FULL, e0, 1), ez = __shfl_down_sync(FULL, e1, 1);
            const int gid = Pg[g] != PEND_NONE ? rec_id(G.r[2][g]) : -1;
            if (c == 0 && gid >= 0) {
                const float4 A = G.r[0][g], B = G.r[1][g];
                const float u = pm.x0 - A.x, v = pm.y0 - A.y;
                float acc[NGRAD];
                acc[0] = fmaf(u, t0, t1);
                acc[1] = fmaf(v, t0, sj);
                acc[2] = fmaf(u, fmaf(0.5f * u, t0, t1), 0.5f * sii);
                acc[3] = fmaf(v, acc[0], fmaf(u, sj, sij));
                acc[4] = fmaf(v, fmaf(0.5f * v, t0, sj), 0.5f * sjj);
                acc[5] = t0;
                acc[6] = e0;
                acc[7] = e1;
                acc[8] = eb;
                acc[9] = ez;
                flush_grad(v_splats, gid, acc, A, B);
            }
        }
        __syncwarp();  // the group's records and staging are rewritten next
        head += RGROUP;
    }
    if (STATS) {
        block_count(visited, stats);
        block_count(contributed, stats + 1);
    }
}


// ----------------------------------------------------- the back chain -----
//
// Behind a fractional mesh layer (antialiased coverage 0 < a < 1, a split
// depth D) the Gaussians' back parts are composited into a second chain
// (Hybrid rendering, two-layer equation): under the hard split the Gaussians
// at or behind D, under the soft split every Gaussian with alpha (1 - f).
// Such pixels are few (silhouettes), so one warp takes one tile: its lanes take
// the tile's fractional pixels 32 at a time, and the warp stages the tile's
// list 32 entries at a time in shared memory (one coalesced load per entry,
// shared by every lane).  The forward adds T_front (1 - a)(C_b + (T_b - 1) bg)
// to the colour the main pass wrote; the backward adds the Gaussians'
// gradients (global atomics) and writes the layer's gradients (dL/da, dL/dM,
// dL/dD).

constexpr int BACK_WARPS = 4;

// first list position whose Gaussian is not in front of D (the list is sorted
// by centre depth; an invalid id counts as in front)
__device__ __forceinline__ int first_behind(const int32_t* __restrict__ gids, const float4* __restrict__ splats,
                                            int N, int lo, int hi, float D)
{
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int g = gids[mid];
        const float z = (g >= 0 && g < N) ? splats[3 * (int64_t)g + 2].y : -INFINITY;
        if (z < D) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

struct BackStage {
    float4 A[32], B[32], C[32], Dm[32];
    int g[32];
    uint8_t frac[TILE_PIX];
};

// the tile's pixels whose layer has a back chain (0 < a < 1 and a split depth),
// compacted into st.frac; returns their number
__device__ __forceinline__ int gather_frac(const Cam& c, int tile, const float* __restrict__ cov,
                                           const float* __restrict__ mesh_depth, BackStage& st, int lane)
{
    const int tx = tile % c.TW, ty = tile / c.TW;
    int n = 0;
#pragma unroll 1
    for (int k = 0; k < TILE_PIX / 32; ++k) {
        const int tp = k * 32 + lane;
        const int i = tx * TILE + (tp & (TILE - 1)), j = ty * TILE + (tp >> 4);
        bool f = false;
        if (i < c.W && j < c.H) {
            const int64_t pix = (int64_t)j * c.W + i;
            f = mesh_depth[pix] < INFINITY && cov[pix] < 1.0f;
        }
        const uint32_t m = __ballot_sync(0xffffffffu, f);
        if (f) st.frac[n + __popc(m & ((1u << lane) - 1))] = (uint8_t)tp;
        n += __popc(m);
    }
    __syncwarp();
    return n;
}

// stages list entries k0 .. k0 + 31 (those < kend) of the tile: lane l loads entry k0 + l
template <bool SOFT>
__device__ __forceinline__ void stage_back(const int32_t* __restrict__ gids, const float4* __restrict__ splats,
                                           const float4* __restrict__ depth_model, int N, const Split& sp, int k0,
                                           int kend, BackStage& st, int lane)
{
    __syncwarp();
    const int k = k0 + lane;
    int g = k < kend ? gids[k] : -1;
    if (g < 0 || g >= N) g = -1;
    st.g[lane] = g;
    if (g >= 0) {
        stage_rec(splats, g, st.A[lane], st.B[lane], st.C[lane]);
        if (SOFT) st.Dm[lane] = stage_depth_model(depth_model, g, sp, st.C[lane].y);
    }
    __syncwarp();
}

template <bool SOFT>
__global__ void __launch_bounds__(32 * BACK_WARPS)
k_composite_back_fwd(Cam c, float3 bg, int N, Split sp, const int2* __restrict__ tile_range,
                     const int32_t* __restrict__ gids, const float4* __restrict__ splats,
                     const float4* __restrict__ depth_model, const float* __restrict__ mesh_depth,
                     const float* __restrict__ cov, const float* __restrict__ T_final, float* __restrict__ out_rgb,
                     float* __restrict__ out_depth, float* __restrict__ out_alpha, float4* __restrict__ back,
                     float* __restrict__ T_back, int32_t* __restrict__ n_back)
{
    __shared__ BackStage stages[BACK_WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x * BACK_WARPS + warp;
    if (tile >= c.TW * c.TH) return;
    BackStage& st = stages[warp];
    const int nfrac = gather_frac(c, tile, cov, mesh_depth, st, lane);
    const int2 r = tile_range[tile];
    const int tx = tile % c.TW, ty = tile / c.TW;
#pragma unroll 1
    for (int base = 0; base < nfrac; base += 32) {
        const bool act = base + lane < nfrac;
        int64_t pix = 0;
        float px = 0.f, py = 0.f, D = INFINITY;
        if (act) {
            const int tp = st.frac[base + lane];
            const int i = tx * TILE + (tp & (TILE - 1)), j = ty * TILE + (tp >> 4);
            pix = (int64_t)j * c.W + i;
            px = (float)i + 0.5f;
            py = (float)j + 0.5f;
            D = mesh_depth[pix];
        }
        float Dmin = D;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Dmin = fminf(Dmin, __shfl_xor_sync(0xffffffffu, Dmin, o));
        const int start = SOFT ? r.x : first_behind(gids, splats, N, r.x, r.y, Dmin);
        float T = 1.0f, Cr = 0.f, Cg = 0.f, Cb = 0.f, Z = 0.f;
        int last = 0;
        bool done = !act;
#pragma unroll 1
        for (int k0 = start; k0 < r.y; k0 += 32) {
            if (__all_sync(0xffffffffu, done)) break;
            stage_back<SOFT>(gids, splats, depth_model, N, sp, k0, r.y, st, lane);
            const int n = min(32, r.y - k0);
            for (int e = 0; e < n && !done; ++e) {
                if (st.g[e] < 0) continue;
                const float4 C = st.C[e];
                if (!SOFT && C.y < D) continue;
                const float4 B = st.B[e];
                const Eval ev = eval_splat(st.A[e], B, px, py);
                if (ev.skip) continue;
                float part = ev.alpha;
                if (SOFT) {
                    const float4 Dm = st.Dm[e];
                    const float zs = fmaf(Dm.x, ev.dx, fmaf(Dm.y, ev.dy, C.y));
                    part = ev.alpha * (1.0f - sp.front((D - zs) * Dm.z));
                    if (part < ALPHA_MIN) continue;
                }
                const float Tn = __fmul_rn(T, __fsub_rn(1.0f, part));
                if (Tn <= T_STOP) {
                    done = true;
                    break;
                }
                const float w = part * T;
                Cr = fmaf(w, B.z, Cr);
                Cg = fmaf(w, B.w, Cg);
                Cb = fmaf(w, C.x, Cb);
                Z = fmaf(w, C.y, Z);
                T = Tn;
                last = k0 + e - r.x + 1;
            }
        }
        if (act) {
            const float a = cov[pix];
            back[pix] = make_float4(Cr, Cg, Cb, Z);
            T_back[pix] = T;
            n_back[pix] = last;
            const float s = T_final[pix] * (1.0f - a), tm1 = T - 1.0f;
            out_rgb[3 * pix] = fmaf(s, fmaf(tm1, bg.x, Cr), out_rgb[3 * pix]);
            out_rgb[3 * pix + 1] = fmaf(s, fmaf(tm1, bg.y, Cg), out_rgb[3 * pix + 1]);
            out_rgb[3 * pix + 2] = fmaf(s, fmaf(tm1, bg.z, Cb), out_rgb[3 * pix + 2]);
            out_depth[pix] = fmaf(s, Z, out_depth[pix]);
            out_alpha[pix] = 1.0f - s * T;
        }
    }
}

// The layer's gradients at every pixel (the antialiased layer's own terms),
// before the back chains' gradients.
template <bool SOFT>
__global__ void __launch_bounds__(256)
k_layer_grad(int64_t P, float3 bg, const float* __restrict__ mesh_depth, const float* __restrict__ T_final,
             const float* __restrict__ g_rgb, const float* __restrict__ g_depth, const float* __restrict__ g_alpha,
             AaLayer aa, float* __restrict__ v_mesh_depth)
{
    const int64_t pix = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (pix >= P) return;
    const float a = aa.cov[pix], D = mesh_depth[pix], Tf = T_final[pix];
    const bool has_mesh = D < INFINITY, frac = has_mesh && a < 1.0f;
    const float gr = g_rgb[3 * pix], gg = g_rgb[3 * pix + 1], gb = g_rgb[3 * pix + 2], gz = g_depth[pix];
    float Tb = 1.0f, Eb = bg.x * gr + bg.y * gg + bg.z * gb;
    if (frac) {
        const float4 bk = aa.back[pix];
        Tb = aa.T_back[pix];
        Eb = fmaf(Tb, Eb, bk.x * gr + bk.y * gg + bk.z * gb + bk.w * gz);
    }
    // rgb = C + T (M + (1 - a)(C_b + T_b bg)), depth = Z + T (a D + (1 - a) Z_b),
    // alpha = 1 - T (1 - a) T_b
    aa.v_rgb[3 * pix] = Tf * gr;
    aa.v_rgb[3 * pix + 1] = Tf * gg;
    aa.v_rgb[3 * pix + 2] = Tf * gb;
    aa.v_cov[pix] = has_mesh ? Tf * (fmaf(gz, D, -Eb) + g_alpha[pix] * Tb) : 0.0f;
    v_mesh_depth[pix] = (SOFT ? v_mesh_depth[pix] : 0.0f) + (a > 0.0f && has_mesh ? Tf * a * gz : 0.0f);
}

template <bool SOFT>
__global__ void __launch_bounds__(32 * BACK_WARPS)
k_composite_back_bwd(Cam c, float3 bg, int N, Split sp, const int2* __restrict__ tile_range,
                     const int32_t* __restrict__ gids, const float4* __restrict__ splats,
                     const float4* __restrict__ depth_model, const float* __restrict__ mesh_depth,
                     const float* __restrict__ T_final, const float* __restrict__ g_rgb,
                     const float* __restrict__ g_depth, const float* __restrict__ g_alpha, AaLayer aa,
                     float* __restrict__ v_splats, float* __restrict__ v_depth_model, float* __restrict__ v_mesh_depth)
{
    __shared__ BackStage stages[BACK_WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x * BACK_WARPS + warp;
    if (tile >= c.TW * c.TH) return;
    BackStage& st = stages[warp];
    const int nfrac = gather_frac(c, tile, aa.cov, mesh_depth, st, lane);
    const int2 r = tile_range[tile];
    const int tx = tile % c.TW, ty = tile / c.TW;
#pragma unroll 1
    for (int base = 0; base < nfrac; base += 32) {
        const bool act = base + lane < nfrac;
        int64_t pix = 0;
        float px = 0.f, py = 0.f, D = INFINITY;
        int top = -1;  // the last list position of this lane's back chain
        float hr = 0.f, hg = 0.f, hb = 0.f, hz = 0.f, T = 1.0f, behind = 0.f, aterm = 0.f;
        if (act) {
            const int tp = st.frac[base + lane];
            const int i = tx * TILE + (tp & (TILE - 1)), j = ty * TILE + (tp >> 4);
            pix = (int64_t)j * c.W + i;
            px = (float)i + 0.5f;
            py = (float)j + 0.5f;
            D = mesh_depth[pix];
            top = r.x + aa.n_back[pix] - 1;
            // the back chain, back to front, with the upstream gradient scaled by T (1 - a)
            const float s = T_final[pix] * (1.0f - aa.cov[pix]);
            hr = s * g_rgb[3 * pix];
            hg = s * g_rgb[3 * pix + 1];
            hb = s * g_rgb[3 * pix + 2];
            hz = s * g_depth[pix];
            T = aa.T_back[pix];
            behind = T * (bg.x * hr + bg.y * hg + bg.z * hb);
            aterm = s * g_alpha[pix] * T;
        }
        float Dmin = D;
        int tmax = top;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            Dmin = fminf(Dmin, __shfl_xor_sync(0xffffffffu, Dmin, o));
            tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
        }
        const int start = SOFT ? r.x : first_behind(gids, splats, N, r.x, r.y, Dmin);
        float vD = 0.0f;
#pragma unroll 1
        for (int k1 = min(tmax, r.y - 1); k1 >= start; k1 -= 32) {
            const int k0 = max(start, k1 - 31);
            stage_back<SOFT>(gids, splats, depth_model, N, sp, k0, k1 + 1, st, lane);
            for (int e = k1 - k0; e >= 0; --e) {
                const int k = k0 + e;
                if (k > top || st.g[e] < 0) continue;
                const float4 C = st.C[e];
                if (!SOFT && C.y < D) continue;
                const float4 A = st.A[e], B = st.B[e];
                const Eval ev = eval_splat(A, B, px, py);
                if (ev.skip) continue;
                float part = ev.alpha, f = 0.0f, x = 0.0f;
                float4 Dm = make_float4(0.f, 0.f, 0.f, 0.f);
                if (SOFT) {
                    Dm = st.Dm[e];
                    const float zs = fmaf(Dm.x, ev.dx, fmaf(Dm.y, ev.dy, C.y));
                    x = (D - zs) * Dm.z;
                    f = sp.front(x);
                    part = ev.alpha * (1.0f - f);
                    if (part < ALPHA_MIN) continue;
                }
                const float rom = __fdividef(1.0f, 1.0f - part);
                const float Tp = T * rom;
                const float w = part * Tp;
                const float front = B.z * hr + B.w * hg + C.x * hb + C.y * hz;
                const float dLdp = Tp * front + (aterm - behind) * rom;  // dL / d(the back part)
                behind = fmaf(w, front, behind);
                T = Tp;
                // record gradient: sigma = (a dx^2 + c dy^2) / 2 + b dx dy of the record's conic
                const int g = st.g[e];
                const float4* rec = splats + 3 * (int64_t)g;
                const float4 s0 = rec[0], s1 = rec[1];
                float vg[10] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, w * hr, w * hg, w * hb, w * hz};
                const float dLdal = SOFT ? dLdp * (1.0f - f) : dLdp;
                if (!ev.clamped) {
                    const float ds = -dLdal * ev.alpha;  // d alpha / d sigma = -alpha
                    vg[0] = -ds * (s0.z * ev.dx + s0.w * ev.dy);
                    vg[1] = -ds * (s0.w * ev.dx + s1.x * ev.dy);
                    vg[2] = 0.5f * ds * ev.dx * ev.dx;
                    vg[3] = ds * ev.dx * ev.dy;
                    vg[4] = 0.5f * ds * ev.dy * ev.dy;
                    vg[5] = dLdal * ev.G;
                }
                if (SOFT) {  // the back part alpha (1 - f(x)): dL/dx = -dLdp alpha f'(x)
                    const float psi = -dLdp * ev.alpha * sp.density(x, f);
                    const float pz = psi * Dm.z;
                    vg[0] += pz * Dm.x;
                    vg[1] += pz * Dm.y;
                    vg[9] -= pz;
                    vD += pz;
                    atomicAdd(reinterpret_cast<float4*>(v_depth_model) + g,
                              make_float4(-pz * ev.dx, -pz * ev.dy, -psi * x * Dm.z * sp.softness, 0.0f));
                }
                float4* dst = reinterpret_cast<float4*>(v_splats + 12 * (int64_t)g);
                atomicAdd(dst, make_float4(vg[0], vg[1], vg[2], vg[3]));
                atomicAdd(dst + 1, make_float4(vg[4], vg[5], vg[6], vg[7]));
                atomicAdd(dst + 2, make_float4(vg[8], vg[9], 0.0f, 0.0f));
            }
        }
        if (act && SOFT) v_mesh_depth[pix] += vD;
    }
}

}  // namespace

static Staged staged_of(float* staged, int cap)
{
    Staged r{nullptr, nullptr, nullptr, nullptr, nullptr, 0};
    if (!staged || cap <= 0) return r;
    float4* b = reinterpret_cast<float4*>(staged);
    r.A = b;
    r.B = b + cap;
    r.C = b + 2 * (int64_t)cap;
    r.D = b + 3 * (int64_t)cap;                  // soft split: depth models
    r.L = reinterpret_cast<uint8_t*>(r.D);       // hard split: 8 hit-list bytes a position
    r.cap = cap;
    return r;
}

size_t staged_bytes(int cap, bool soft) { return (size_t)(cap > 0 ? cap : 0) * (soft ? 64 : 56); }

cudaError_t copy_status(uint32_t* flags, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_copy_status, sizeof(uint32_t));
    if (e == cudaSuccess && clear) {
        const uint32_t z = 0;
        e = cudaMemcpyToSymbol(g_copy_status, &z, sizeof(z));
    }
    return e;
}

cudaError_t composite_fwd(const Cam& c, const float bg[3], int N, float softness, int split, const int32_t* tile_range,
                          const int32_t* gids, const float* splats, const float* depth_model, const float* mesh_depth,
                          const float* mesh_rgb, const int32_t* face_id, float* out_rgb, float* out_depth,
                          float* out_alpha, float* T_final, int32_t* n_contrib, const AaLayer& aa, float* staged,
                          int staged_cap, uint64_t* stats, cudaStream_t s)
{
    const bool soft = softness > 0.0f;
    const Staged rec = staged_of(staged, staged_cap);
    auto kern = soft ? (stats ? k_composite_fwd<true, true> : k_composite_fwd<false, true>)
                     : (stats ? k_composite_fwd<true, false> : k_composite_fwd<false, false>);
    kern<<<c.TW * c.TH * CTAS_PER_TILE, CTA_THREADS, 0, s>>>(
        c, make_float3(bg[0], bg[1], bg[2]), N, Split{softness, split == 1}, reinterpret_cast<const int2*>(tile_range),
        gids,
        reinterpret_cast<const float4*>(splats), reinterpret_cast<const float4*>(depth_model), mesh_depth, mesh_rgb,
        face_id, out_rgb, out_depth, out_alpha, T_final, n_contrib, aa.cov, rec,
        reinterpret_cast<unsigned long long*>(stats));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !aa.cov) return e;
    const int64_t P = (int64_t)c.W * c.H;
    const unsigned grid = (unsigned)((P + 255) / 256);
    auto back = soft ? k_composite_back_fwd<true> : k_composite_back_fwd<false>;
    const unsigned tgrid = (unsigned)((c.TW * c.TH + BACK_WARPS - 1) / BACK_WARPS);
    (void)grid;
    back<<<tgrid, 32 * BACK_WARPS, 0, s>>>(c, make_float3(bg[0], bg[1], bg[2]), N, Split{softness, split == 1},
                              reinterpret_cast<const int2*>(tile_range), gids, reinterpret_cast<const float4*>(splats),
                              reinterpret_cast<const float4*>(depth_model), mesh_depth, aa.cov, T_final, out_rgb,
                              out_depth, out_alpha, aa.back, aa.T_back, aa.n_back);
    return cudaGetLastError();
}

cudaError_t composite_bwd(const Cam& c, const float bg[3], int N, float softness, int split, const int32_t* tile_range,
                          const int32_t* gids, const float* splats, const float* depth_model, const float* mesh_depth,
                          const float* mesh_rgb, const int32_t* face_id, const float* T_final,
                          const int32_t* n_contrib, const float* g_rgb, const float* g_depth, const float* g_alpha,
                          float* v_splats, float* v_depth_model, float* v_mesh_depth, const AaLayer& aa,
                          const float* staged, int staged_cap, uint64_t* stats, cudaStream_t s)
{
    const bool soft = softness > 0.0f;
    const Staged rec = staged_of(const_cast<float*>(staged), staged_cap);
    const bool bulk = rec.A != nullptr && !getenv("GM_BWD_GATHER");
    const bool mma = !soft && !getenv("GM_BWD_SHUFFLE_REDUCE");
    if (bulk && mma) {
        // the forward's hit lists: every warp through its own lists
        auto lk = stats ? k_composite_bwd_lists<true> : k_composite_bwd_lists<false>;
        lk<<<c.TW * c.TH * CTAS_PER_TILE, CTA_THREADS, 0, s>>>(
            c, make_float3(bg[0], bg[1], bg[2]), reinterpret_cast<const int2*>(tile_range), mesh_depth, mesh_rgb,
            face_id, T_final, n_contrib, g_rgb, g_depth, g_alpha, v_splats, aa, rec,
            reinterpret_cast<unsigned long long*>(stats));
    } else {
        using K = decltype(&k_composite_bwd<false, false, false, false>);
        K kern;
        if (soft)
            kern = stats ? (bulk ? k_composite_bwd<true, true, true, false> : k_composite_bwd<true, true, false, false>)
                         : (bulk ? k_composite_bwd<false, true, true, false> : k_composite_bwd<false, true, false, false>);
        else if (mma)  // gathered records (the staged ones go to k_composite_bwd_lists)
            kern = stats ? k_composite_bwd<true, false, false, true> : k_composite_bwd<false, false, false, true>;
        else
            kern = stats ? (bulk ? k_composite_bwd<true, false, true, false> : k_composite_bwd<true, false, false, false>)
                         : (bulk ? k_composite_bwd<false, false, true, false> : k_composite_bwd<false, false, false, false>);
        kern<<<c.TW * c.TH * CTAS_PER_TILE, CTA_THREADS, 0, s>>>(
            c, make_float3(bg[0], bg[1], bg[2]), N, Split{softness, split == 1}, reinterpret_cast<const int2*>(tile_range),
            gids,
            reinterpret_cast<const float4*>(splats), reinterpret_cast<const float4*>(depth_model), mesh_depth, mesh_rgb,
            face_id, T_final, n_contrib, g_rgb, g_depth, g_alpha, v_splats, v_depth_model, v_mesh_depth, aa,
            bulk ? rec : Staged{nullptr, nullptr, nullptr, nullptr, nullptr, 0}, reinterpret_cast<unsigned long long*>(stats));
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !aa.cov) return e;
    const int64_t P = (int64_t)c.W * c.H;
    const unsigned grid = (unsigned)((P + 255) / 256);
    auto lg = soft ? k_layer_grad<true> : k_layer_grad<false>;
    lg<<<grid, 256, 0, s>>>(P, make_float3(bg[0], bg[1], bg[2]), mesh_depth, T_final, g_rgb, g_depth, g_alpha, aa,
                            v_mesh_depth);
    auto back = soft ? k_composite_back_bwd<true> : k_composite_back_bwd<false>;
    const unsigned tgrid = (unsigned)((c.TW * c.TH + BACK_WARPS - 1) / BACK_WARPS);
    back<<<tgrid, 32 * BACK_WARPS, 0, s>>>(c, make_float3(bg[0], bg[1], bg[2]), N, Split{softness, split == 1},
                                           reinterpret_cast<const int2*>(tile_range), gids,
                                           reinterpret_cast<const float4*>(splats),
                                           reinterpret_cast<const float4*>(depth_model), mesh_depth, T_final, g_rgb,
                                           g_depth, g_alpha, aa, v_splats, v_depth_model, v_mesh_depth);
    return cudaGetLastError();
}

}  // namespace gm

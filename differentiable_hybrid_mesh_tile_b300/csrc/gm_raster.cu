// Direct z-buffer ("A Lightweight and Differentiable Renderer for Joint Mesh
// and 3D Gaussian Splat Scenes", Mesh rasterizer, item 1): the per-pixel
// coverage and depth test of the tile z-buffer (gm_mesh.cu), taken over
// (triangle, pixel) pairs instead of per-tile triangle lists, so that no
// binning or sort is needed.  Each covered pixel keeps its winner by a 64-bit
// atomicMin of (complemented reciprocal-depth bits << 32 | face id): the
// largest reciprocal depth (nearest surface) and, on an equal depth, the
// smaller face id -- the tile z-buffer's rule, whatever order the pairs are
// taken in.  The coverage and depth arithmetic is the tile z-buffer's, rounding
// for rounding, so both give the same face ids bit for bit.
//
// Triangles whose pixel-centre box holds at most SMALL_TRI pixels: a warp sets
// up 32 consecutive faces in shared memory and takes their box rows in runs of
// RUN consecutive pixels, one run per lane per round (the owner lookup and the
// record loads once per run; each edge function's row term once per run).  Larger triangles
// go to a queue that persistent blocks work through in chunks of CHUNK pixels;
// a block that finds no new triangle helps with the chunks of unfinished ones,
// so one full-screen triangle still spreads over several blocks.
#include "gm_internal.cuh"

namespace gm {
namespace {

constexpr int SMALL_TRI = 2048;
constexpr int RUN = 4;
constexpr int CHUNK = 1024;
constexpr int ZB_THREADS = 256;
constexpr int HELP_PASSES = 8;  // each queued triangle is offered to up to this many blocks
constexpr int ZB_NLARGE = 0, ZB_CURSOR = 1;

// A set-up triangle.  Edge k runs from vertex a to vertex b with (du, dv) =
// (u_b - u_a, v_b - v_a) rounded once, as the tile z-buffer's edge function
// rounds them; w_k = 1 / (area z_k), so that the reciprocal depth at a pixel is
// sum_k e_k w_k.
struct ZTri {
    float4 a;  // u0, v0, u1, v1
    float4 b;  // u2, v2, area (twice the signed area), w0
    float4 c;  // edge 0 (v1 -> v2): du, dv; edge 1 (v2 -> v0): du, dv
    float4 d;  // edge 2 (v0 -> v1): du, dv; w1, w2
    int4 e;    // box x0, y0, box width, face id
    int4 g;    // 1 / width (float bits), box pixels, runs per box row, 1 / runs per row (float bits)
};

__device__ __forceinline__ ZTri make_ztri(const Tri& t, int f)
{
    ZTri z;
    z.a = make_float4(t.u[0], t.v[0], t.u[1], t.v[1]);
    z.b = make_float4(t.u[2], t.v[2], t.area, 1.0f / (t.area * t.z[0]));
    z.c = make_float4(__fsub_rn(t.u[2], t.u[1]), __fsub_rn(t.v[2], t.v[1]), __fsub_rn(t.u[0], t.u[2]),
                      __fsub_rn(t.v[0], t.v[2]));
    z.d = make_float4(__fsub_rn(t.u[1], t.u[0]), __fsub_rn(t.v[1], t.v[0]), 1.0f / (t.area * t.z[1]),
                      1.0f / (t.area * t.z[2]));
    const int w = t.x1 - t.x0 + 1, h = t.y1 - t.y0 + 1;
    z.e = make_int4(t.x0, t.y0, w, f);
    const int rw = (w + RUN - 1) / RUN;
    z.g = make_int4(__float_as_int(__frcp_rn((float)w)), w * h, rw, __float_as_int(__frcp_rn((float)rw)));
    return z;
}

// the edge function of an edge with precomputed (du, dv) from (ua, va)
__device__ __forceinline__ float edge_pre(float du, float dv, float ua, float va, float px, float py)
{
    return __fsub_rn(__fmul_rn(du, __fsub_rn(py, va)), __fmul_rn(dv, __fsub_rn(px, ua)));
}

// Coverage and depth of pixel (i, j) of the triangle; a covered pixel offers
// the triangle to the pixel's key.
__device__ __forceinline__ void zb_pixel(const ZTri& z, int i, int j, int W, unsigned long long* __restrict__ key)
{
    const float px = (float)i + 0.5f, py = (float)j + 0.5f;
    const float e0 = edge_pre(z.c.x, z.c.y, z.a.z, z.a.w, px, py);
    const float e1 = edge_pre(z.c.z, z.c.w, z.b.x, z.b.y, px, py);
    const float e2 = edge_pre(z.d.x, z.d.y, z.a.x, z.a.y, px, py);
    const bool in = z.b.z > 0.0f ? (e0 >= 0.0f && e1 >= 0.0f && e2 >= 0.0f) : (e0 <= 0.0f && e1 <= 0.0f && e2 <= 0.0f);
    if (!in) return;
    const float inv_d = fmaf(e0, z.b.w, fmaf(e1, z.d.z, e2 * z.d.w));
    if (!(inv_d > 0.0f)) return;  // the tile z-buffer's winner starts at reciprocal depth 0
    const unsigned long long k = ((unsigned long long)(~__float_as_uint(inv_d)) << 32) | (uint32_t)z.e.w;
    atomicMin(key + (int64_t)j * W + i, k);
}

// Up to RUN pixels (i0 .. i0 + n - 1, row j) of the triangle: the edge
// functions as edge_pre computes them, with the row term du (py - va) of each
// edge formed once.
__device__ __forceinline__ void zb_run(const ZTri& z, int i0, int j, int n, int W,
                                       unsigned long long* __restrict__ key)
{
    const float py = (float)j + 0.5f;
    const float r0 = __fmul_rn(z.c.x, __fsub_rn(py, z.a.w));
    const float r1 = __fmul_rn(z.c.z, __fsub_rn(py, z.b.y));
    const float r2 = __fmul_rn(z.d.x, __fsub_rn(py, z.a.y));
    const bool pos = z.b.z > 0.0f;
    unsigned long long* row = key + (int64_t)j * W;
#pragma unroll
    for (int k = 0; k < RUN; ++k) {
        if (k >= n) break;
        const int i = i0 + k;
        const float px = (float)i + 0.5f;
        const float e0 = __fsub_rn(r0, __fmul_rn(z.c.y, __fsub_rn(px, z.a.z)));
        const float e1 = __fsub_rn(r1, __fmul_rn(z.c.w, __fsub_rn(px, z.b.x)));
        const float e2 = __fsub_rn(r2, __fmul_rn(z.d.y, __fsub_rn(px, z.a.x)));
        const bool in = pos ? (e0 >= 0.0f && e1 >= 0.0f && e2 >= 0.0f) : (e0 <= 0.0f && e1 <= 0.0f && e2 <= 0.0f);
        if (!in) continue;
        const float inv_d = fmaf(e0, z.b.w, fmaf(e1, z.d.z, e2 * z.d.w));
        if (!(inv_d > 0.0f)) continue;
        atomicMin(row + i, ((unsigned long long)(~__float_as_uint(inv_d)) << 32) | (uint32_t)z.e.w);
    }
}

// Pixel r (row-major) of the triangle's box.
__device__ __forceinline__ void box_pixel(const ZTri& z, int r, int& i, int& j)
{
    int row, col;
    divmod_small(r, z.e.z, __int_as_float(z.g.x), row, col);
    i = z.e.x + col;
    j = z.e.y + row;
}

__global__ void __launch_bounds__(ZB_THREADS)
k_zb_small(Cam c, const float* __restrict__ V, int nV, const int32_t* __restrict__ F, int nF,
           ZTri* __restrict__ large, int32_t* __restrict__ taken, int32_t* ctl, unsigned long long* __restrict__ key)
{
    __shared__ ZTri s[ZB_THREADS];
    const int f = blockIdx.x * ZB_THREADS + threadIdx.x;
    const int lane = threadIdx.x & 31, wbase = threadIdx.x & ~31;
    int area = 0;
    if (f < nF) {
        Tri t;
        if (tri_setup(c, V, nV, F, f, t)) {
            const ZTri z = make_ztri(t, f);
            if (z.g.y <= SMALL_TRI) {
                s[threadIdx.x] = z;
                area = z.g.z * (t.y1 - t.y0 + 1);  // runs of the box
            } else {  // queued for the chunked pass (at most nF of them)
                const int q = atomicAdd(ctl + ZB_NLARGE, 1);
                large[q] = z;
                taken[q] = 0;
            }
        }
    }
    // the (triangle, run) pairs of the warp's small triangles, flattened
    int o = area;  // inclusive prefix sum over the lanes
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, o, d);
        if (lane >= d) o += y;
    }
    const int total = __shfl_sync(0xffffffffu, o, 31);
    o -= area;
    __syncwarp();
    for (int base = 0; base < total; base += 32) {
        const int p = base + lane;
        // owner of pair p: the last lane whose first pair is at or before p
        int j = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
            const int oj = __shfl_sync(0xffffffffu, o, j + step);
            if (oj <= p) j += step;
        }
        const int oj = __shfl_sync(0xffffffffu, o, j);
        if (p < total) {
            const ZTri& z = s[wbase + j];
            int row, seg;
            divmod_small(p - oj, z.g.z, __int_as_float(z.g.w), row, seg);
            const int c0 = seg * RUN;
            zb_run(z, z.e.x + c0, z.e.y + row, min(RUN, z.e.z - c0), c.W, key);
        }
    }
}

// Persistent blocks over the queue of large triangles: a block takes a
// triangle from the cursor, claims its chunks one by one (taken[q] counts the
// claims) and, when the cursor has passed every triangle HELP_PASSES times,
// stops.  A triangle is thus worked on by the block that took it first and by
// up to HELP_PASSES - 1 helpers.
__global__ void __launch_bounds__(ZB_THREADS)
k_zb_large(Cam c, const ZTri* __restrict__ large, int32_t* __restrict__ taken, int32_t* ctl,
           unsigned long long* __restrict__ key)
{
    __shared__ int s_q, s_chunk;
    const int L = ctl[ZB_NLARGE];
    if (L <= 0) return;
    for (;;) {
        if (threadIdx.x == 0) {
            s_q = -1;
            for (;;) {
                const int i = atomicAdd(ctl + ZB_CURSOR, 1);
                if (i >= HELP_PASSES * L) break;
                const int q = i % L;
                const int nch = (large[q].g.y + CHUNK - 1) / CHUNK;
                const int ch = atomicAdd(taken + q, 1);
                if (ch < nch) {
                    s_q = q;
                    s_chunk = ch;
                    break;
                }
            }
        }
        __syncthreads();
        const int q = s_q;
        if (q < 0) break;
        const ZTri z = large[q];
        const int n = z.g.y, nch = (n + CHUNK - 1) / CHUNK;
        int ch = s_chunk;
        while (ch < nch) {
            for (int k = threadIdx.x; k < CHUNK; k += ZB_THREADS) {
                const int r = ch * CHUNK + k;
                if (r >= n) break;
                int pi, pj;
                box_pixel(z, r, pi, pj);
                zb_pixel(z, pi, pj, c.W, key);
            }
            __syncthreads();  // every thread has read s_chunk
            if (threadIdx.x == 0) s_chunk = atomicAdd(taken + q, 1);
            __syncthreads();
            ch = s_chunk;
        }
        __syncthreads();  // every thread has read s_q before it is rewritten
    }
}

__global__ void __launch_bounds__(256)
k_zb_resolve(int64_t n, const unsigned long long* __restrict__ key, int32_t* __restrict__ face_id)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const unsigned long long k = key[i];
    face_id[i] = k == ~0ull ? -1 : (int32_t)(uint32_t)k;
}

size_t a256(size_t b) { return (b + 255) & ~(size_t)255; }

struct ZbWs {
    unsigned long long* key;
    ZTri* large;
    int32_t *taken, *ctl;
};

ZbWs carve_zb_ws(void* ws, int nF, int W, int H)
{
    const size_t n = nF > 0 ? (size_t)nF : 1;
    ZbWs w;
    uint8_t* b = (uint8_t*)ws;
    w.key = (unsigned long long*)b;
    b += a256(sizeof(unsigned long long) * (size_t)W * (size_t)H);
    w.large = (ZTri*)b;
    b += a256(sizeof(ZTri) * n);
    w.taken = (int32_t*)b;
    b += a256(sizeof(int32_t) * n);
    w.ctl = (int32_t*)b;
    return w;
}

}  // namespace

size_t zbuffer_direct_ws_bytes(int nF, int W, int H)
{
    const size_t n = nF > 0 ? (size_t)nF : 1;
    return a256(sizeof(unsigned long long) * (size_t)W * (size_t)H) + a256(sizeof(ZTri) * n) +
           a256(sizeof(int32_t) * n) + 256;
}

cudaError_t zbuffer_direct(const Cam& c, const float* V, int nV, const int32_t* F, int nF, int32_t* face_id,
                           void* ws, cudaStream_t s)
{
    ZbWs w = carve_zb_ws(ws, nF, c.W, c.H);
    const int64_t npix = (int64_t)c.W * c.H;
    cudaError_t e = cudaMemsetAsync(w.key, 0xff, sizeof(unsigned long long) * (size_t)npix, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(w.ctl, 0, 2 * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    if (nF > 0) {
        k_zb_small<<<(nF + ZB_THREADS - 1) / ZB_THREADS, ZB_THREADS, 0, s>>>(c, V, nV, F, nF, w.large, w.taken,
                                                                           w.ctl, w.key);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_zb_large<<<num_sms() * 4, ZB_THREADS, 0, s>>>(c, w.large, w.taken, w.ctl, w.key);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (npix > 0) k_zb_resolve<<<(unsigned)((npix + 255) / 256), 256, 0, s>>>(npix, w.key, face_id);
    return cudaGetLastError();
}

}  // namespace gm

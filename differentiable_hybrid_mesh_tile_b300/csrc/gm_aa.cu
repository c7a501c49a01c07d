// Analytic edge antialiasing of the mesh layer ("A Lightweight and
// Differentiable Renderer for Joint Mesh and 3D Gaussian Splat Scenes",
// Design Details > Mesh rasterizer, item 3; Limitations: a per-axis 1D
// approximation): neighbouring pixels that see a silhouette share coverage by
// where the nearer surface's silhouette edge crosses between their centres,
// giving each pixel a mesh layer (coverage a, premultiplied colour M, split
// depth D) for the two-layer compositing of Hybrid rendering; and its
// backward pass to the interpolated colours and depths and to the silhouette
// vertices.  Edge adjacency (which face lies across each edge) comes from a
// radix sort of the faces' edge keys.
//
// Every decision (occluder, the faces crossed, the exit edge, silhouette or
// internal edge, the axis of the edge, the side of the crossing) is taken in
// fp32 with the rasterizer's own correctly rounded operations, so it is the
// one any IEEE evaluation of the same formulas takes; the crossing t itself is
// evaluated in fp64 (few pixel pairs reach it), free of the cancellation that
// fp32 screen coordinates of the order of a thousand pixels would bring.
#include "gm_internal.cuh"

namespace gm {
namespace {

constexpr int AA_WALK = 8;  // faces a crossing may pass through before it gives up

// ----------------------------------------------------------- adjacency ----

__global__ void __launch_bounds__(256)
k_edge_keys(const int32_t* __restrict__ F, int nF, int bits, uint64_t* __restrict__ keys, int32_t* __restrict__ vals,
            int32_t* __restrict__ n_dev)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) *n_dev = 3 * nF;
    if (i >= 3 * (int64_t)nF) return;
    const int64_t f = i / 3;
    const int k = (int)(i - 3 * f);
    const uint32_t a = (uint32_t)__ldg(F + 3 * f + (k + 1) % 3), b = (uint32_t)__ldg(F + 3 * f + (k + 2) % 3);
    const uint64_t lo = a < b ? a : b, hi = a < b ? b : a;
    keys[i] = (lo << bits) | hi;
    vals[i] = (int32_t)i;
}

// after the sort: a key shared by exactly two face edges pairs them; one alone
// has no neighbour (-1); three or more mark every one of them (-2)
__global__ void __launch_bounds__(256)
k_edge_pairs(const uint64_t* __restrict__ keys, const int32_t* __restrict__ vals, int64_t n, int nF,
             int32_t* __restrict__ adj)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint64_t k = keys[i];
    const bool prev = i > 0 && keys[i - 1] == k, next = i + 1 < n && keys[i + 1] == k;
    const bool prev2 = prev && i > 1 && keys[i - 2] == k, next2 = next && i + 2 < n && keys[i + 2] == k;
    int32_t r;
    if (!prev && !next) r = -1;
    else if (prev2 || next2 || (prev && next)) r = -2;
    else r = vals[prev ? i - 1 : i + 1] / 3;
    const int32_t v = vals[i];
    if (v >= 0 && v < 3 * nF) adj[v] = r;
}

// ------------------------------------------------------------ one pair -----

// screen position of vertex vid in fp32, the rasterizer's operations
__device__ __forceinline__ bool vtx_f32(const Cam& c, const float* __restrict__ V, int nV, int vid, float& u,
                                        float& v)
{
    if (vid < 0 || vid >= nV) return false;
    const float X = __ldg(V + 3 * (int64_t)vid), Y = __ldg(V + 3 * (int64_t)vid + 1), Z = __ldg(V + 3 * (int64_t)vid + 2);
    const float x = cam_row_rn(c, 0, X, Y, Z), y = cam_row_rn(c, 1, X, Y, Z), z = cam_row_rn(c, 2, X, Y, Z);
    if (!(z > c.znear)) return false;
    u = __fadd_rn(__fdiv_rn(__fmul_rn(c.fx, x), z), c.cx);
    v = __fadd_rn(__fdiv_rn(__fmul_rn(c.fy, y), z), c.cy);
    return true;
}

// camera-space position and screen position of vertex vid in fp64
__device__ __forceinline__ void vtx_f64(const Cam& c, const float* __restrict__ V, int vid, double xc[3], double& u,
                                        double& v)
{
    const double X = __ldg(V + 3 * (int64_t)vid), Y = __ldg(V + 3 * (int64_t)vid + 1), Z = __ldg(V + 3 * (int64_t)vid + 2);
#pragma unroll
    for (int r = 0; r < 3; ++r)
        xc[r] = __dadd_rn(__dadd_rn(__dadd_rn(__dmul_rn((double)c.R[3 * r], X), __dmul_rn((double)c.R[3 * r + 1], Y)),
                                    __dmul_rn((double)c.R[3 * r + 2], Z)),
                          (double)c.t[r]);
    u = __dadd_rn(__ddiv_rn(__dmul_rn((double)c.fx, xc[0]), xc[2]), (double)c.cx);
    v = __dadd_rn(__ddiv_rn(__dmul_rn((double)c.fy, xc[1]), xc[2]), (double)c.cy);
}

__device__ __forceinline__ double edge64(double ua, double va, double ub, double vb, double px, double py)
{
    return __dsub_rn(__dmul_rn(__dsub_rn(ub, ua), __dsub_rn(py, va)), __dmul_rn(__dsub_rn(vb, va), __dsub_rn(px, ua)));
}

struct Mesh {
    const float* V;
    const int32_t* F;
    const int32_t* adj;
    const int32_t* face_id;
    const float* depth;
    const float* rgb;
    int nV, nF;
};

struct PairHit {
    int64_t occ, other;  // the occluder's pixel and the other one
    double t;            // crossing, from the occluder's centre (0) to the other's (1)
    int face, k;         // the silhouette edge: edge k (corners k+1, k+2) of this face
    bool far_side;       // t >= 0.5 (fp32 decision): the weight falls on the other pixel
};

// The pair of neighbouring pixels pp, pq: where they see different faces, the
// nearer surface (smaller mesh depth) is followed from the occluder's centre
// towards the other centre through its faces, across internal edges (one face
// across, on the other side of the edge in the image), to the first
// silhouette edge it leaves by; a pair along x only takes an edge more
// vertical than horizontal, a pair along y the others.
__device__ bool aa_pair(const Cam& c, const Mesh& m, int64_t pp, int64_t pq, PairHit& h)
{
    const int fp = m.face_id[pp], fq = m.face_id[pq];
    if (fp == fq) return false;
    const float Dp = fp >= 0 ? m.depth[pp] : INFINITY, Dq = fq >= 0 ? m.depth[pq] : INFINITY;
    int64_t o, nb;
    if (Dp < Dq) { o = pp; nb = pq; }
    else if (Dq < Dp) { o = pq; nb = pp; }
    else return false;
    const int oi = (int)(o % c.W), oj = (int)(o / c.W), ni = (int)(nb % c.W), nj = (int)(nb / c.W);
    const float ox = (float)oi + 0.5f, oy = (float)oj + 0.5f, nx = (float)ni + 0.5f, ny = (float)nj + 0.5f;
    int X = m.face_id[o], entry = -1, exit_k = -1;
    float u[3], v[3], best = INFINITY;
    bool found = false;
    for (int step = 0; step < AA_WALK; ++step) {
        if (X < 0 || X >= m.nF) return false;
        int vid[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            vid[k] = __ldg(m.F + 3 * (int64_t)X + k);
            if (!vtx_f32(c, m.V, m.nV, vid[k], u[k], v[k])) return false;
        }
        const bool pos = edge_rn(u[0], v[0], u[1], v[1], u[2], v[2]) > 0.0f;
        exit_k = -1;
        best = INFINITY;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            if (k == entry) continue;
            const int a = (k + 1) % 3, b = (k + 2) % 3;
            const float eo = edge_rn(u[a], v[a], u[b], v[b], ox, oy);
            const float en = edge_rn(u[a], v[a], u[b], v[b], nx, ny);
            const float so = pos ? eo : -eo, sn = pos ? en : -en;
            if (step == 0 && so < 0.0f) return false;  // the face no longer covers the occluder's centre
            if (!(sn < 0.0f)) continue;
            if (so < 0.0f) return false;  // the segment misses this face
            const float tk = __fdiv_rn(eo, __fsub_rn(eo, en));
            if (tk < best) {
                best = tk;
                exit_k = k;
            }
        }
        if (exit_k < 0) return false;  // the other centre lies on the surface
        const int a = (exit_k + 1) % 3, b = (exit_k + 2) % 3;
        const int nf = __ldg(m.adj + 3 * (int64_t)X + exit_k);
        if (nf < 0 || nf >= m.nF) { found = true; break; }
        int third = -1, back = -1;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int vk = __ldg(m.F + 3 * (int64_t)nf + k);
            if (vk != vid[a] && vk != vid[b]) { third = vk; back = k; }
        }
        float u3, v3;
        if (third < 0 || !vtx_f32(c, m.V, m.nV, third, u3, v3)) { found = true; break; }
        const float sX = edge_rn(u[a], v[a], u[b], v[b], u[exit_k], v[exit_k]);
        const float sN = edge_rn(u[a], v[a], u[b], v[b], u3, v3);
        if (!((sX < 0.0f && sN > 0.0f) || (sX > 0.0f && sN < 0.0f))) { found = true; break; }  // folded
        X = nf;  // the surface goes on across the edge
        entry = back;
    }
    if (!found) return false;
    const int a = (exit_k + 1) % 3, b = (exit_k + 2) % 3;
    const float du = __fsub_rn(u[b], u[a]), dv = __fsub_rn(v[b], v[a]);
    if ((oj == nj) != (fabsf(dv) > fabsf(du))) return false;
    double xc[3], ua, va, ub, vb;
    vtx_f64(c, m.V, __ldg(m.F + 3 * (int64_t)X + a), xc, ua, va);
    vtx_f64(c, m.V, __ldg(m.F + 3 * (int64_t)X + b), xc, ub, vb);
    const double eo = edge64(ua, va, ub, vb, (double)ox, (double)oy);
    const double en = edge64(ua, va, ub, vb, (double)nx, (double)ny);
    double t = __ddiv_rn(eo, __dsub_rn(eo, en));
    t = t < 0.0 ? 0.0 : (t > 1.0 ? 1.0 : t);
    h.occ = o;
    h.other = nb;
    h.t = t;
    h.face = X;
    h.k = exit_k;
    h.far_side = best >= 0.5f;
    return true;
}

__device__ __forceinline__ void load_rgb(const float* __restrict__ rgb, int64_t p, float c[3])
{
    c[0] = rgb[3 * p];
    c[1] = rgb[3 * p + 1];
    c[2] = rgb[3 * p + 2];
}

// The pixel's layer before clamping: the four pairs (left, right, up, down)
// whose weight falls on it move (a, M) towards the other pixel's layer.
// Returns the unclamped coverage; src (optional) = the occluder pixel whose
// depth an uncovered pixel takes (-1: none).
__device__ float aa_layer(const Cam& c, const Mesh& m, int i, int j, float M[3], float& Dout, int64_t* src)
{
    const int64_t pp = (int64_t)j * c.W + i;
    const bool cov = m.face_id[pp] >= 0;
    float cp[3];
    load_rgb(m.rgb, pp, cp);
    float a = cov ? 1.0f : 0.0f;
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) M[ch] = cov ? cp[ch] : 0.0f;
    float Dnear = INFINITY;
    int64_t from = -1;
    const int di[4] = {-1, 1, 0, 0}, dj[4] = {0, 0, -1, 1};
#pragma unroll 1
    for (int s = 0; s < 4; ++s) {
        const int qi = i + di[s], qj = j + dj[s];
        if (qi < 0 || qj < 0 || qi >= c.W || qj >= c.H) continue;
        const int64_t pq = (int64_t)qj * c.W + qi;
        if (m.face_id[pq] == m.face_id[pp]) continue;
        PairHit h;
        if (!aa_pair(c, m, pp, pq, h)) continue;
        const bool onto_me = h.far_side ? h.other == pp : h.occ == pp;
        if (!onto_me) continue;
        const float w = (float)fabs(h.t - 0.5);
        float co[3], cn[3];
        load_rgb(m.rgb, h.occ, co);
        if (h.occ == pp) {  // the surface leaves part of this pixel
            const bool cov_n = m.face_id[h.other] >= 0;
            load_rgb(m.rgb, h.other, cn);
            a = fmaf(w, (cov_n ? 1.0f : 0.0f) - 1.0f, a);
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) M[ch] = fmaf(w, (cov_n ? cn[ch] : 0.0f) - co[ch], M[ch]);
        } else {  // the surface reaches into this pixel
            a = fmaf(w, 1.0f - (cov ? 1.0f : 0.0f), a);
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) M[ch] = fmaf(w, co[ch] - (cov ? cp[ch] : 0.0f), M[ch]);
            if (!cov && w > 0.0f) {
                const float Do = m.depth[h.occ];
                if (Do < Dnear) {
                    Dnear = Do;
                    from = h.occ;
                }
            }
        }
    }
    Dout = cov ? m.depth[pp] : Dnear;
    if (src) *src = cov ? -1 : from;
    return a;
}

__global__ void __launch_bounds__(TILE_PIX)
k_antialias(Cam c, Mesh m, float* __restrict__ cov, float* __restrict__ rgb_aa, float* __restrict__ depth_aa,
            float* __restrict__ tile_far, uint8_t* __restrict__ tile_full)
{
    __shared__ float s_max[TILE_PIX / 32];
    const int tile = blockIdx.x;
    const int tx = tile % c.TW, ty = tile / c.TW;
    const int i = tx * TILE + (threadIdx.x & (TILE - 1));
    const int j = ty * TILE + (threadIdx.x >> 4);
    const bool inside = i < c.W && j < c.H;
    float a = 0.0f, D = INFINITY;
    if (inside) {
        const int64_t pix = (int64_t)j * c.W + i;
        float M[3];
        a = aa_layer(c, m, i, j, M, D, nullptr);
        a = fminf(fmaxf(a, 0.0f), 1.0f);
        cov[pix] = a;
        rgb_aa[3 * pix] = M[0];
        rgb_aa[3 * pix + 1] = M[1];
        rgb_aa[3 * pix + 2] = M[2];
        depth_aa[pix] = D;
    }
    // a tile is full when every pixel is fully covered; far = its largest split depth
    const int all = __syncthreads_and(!inside || a >= 1.0f);
    float mx = inside ? D : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float far = s_max[0];
        for (int w = 1; w < TILE_PIX / 32; ++w) far = fmaxf(far, s_max[w]);
        tile_far[tile] = all ? far : INFINITY;
        tile_full[tile] = (uint8_t)(all ? 1 : 0);
    }
}

// ------------------------------------------------------------ backward ----

// dL/d(screen positions of the edge's ends) -> dL/d world positions, added
__device__ void scatter_vertex_grad(const Cam& c, const float* __restrict__ V, int vid, double gu, double gv,
                                    float* __restrict__ v_verts)
{
    double xc[3], u, v;
    vtx_f64(c, V, vid, xc, u, v);
    const double iz = 1.0 / xc[2];
    const double gx = gu * (double)c.fx * iz, gy = gv * (double)c.fy * iz;
    const double gz = -(gu * (u - (double)c.cx) + gv * (v - (double)c.cy)) * iz;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        const double g = (double)c.R[d] * gx + (double)c.R[3 + d] * gy + (double)c.R[6 + d] * gz;
        atomicAdd(v_verts + 3 * (int64_t)vid + d, (float)g);
    }
}

// Per pixel: dL/d its interpolated colour and depth (through its own layer and
// the layers of the neighbours its pairs move), and, for the pairs it owns
// (right and down neighbour), dL/d the silhouette vertices through the
// crossing t.  Weights that fall on a pixel whose coverage left [0, 1] carry
// no coverage gradient (the clamp).
__global__ void __launch_bounds__(TILE_PIX)
k_antialias_bwd(Cam c, Mesh m, const float* __restrict__ v_cov, const float* __restrict__ v_rgb_aa,
                const float* __restrict__ v_depth_aa, float* __restrict__ v_mesh_rgb, float* __restrict__ v_mesh_depth,
                float* __restrict__ v_verts)
{
    const int tile = blockIdx.x;
    const int tx = tile % c.TW, ty = tile / c.TW;
    const int i = tx * TILE + (threadIdx.x & (TILE - 1));
    const int j = ty * TILE + (threadIdx.x >> 4);
    if (i >= c.W || j >= c.H) return;
    const int64_t pp = (int64_t)j * c.W + i;
    const bool cov = m.face_id[pp] >= 0;
    const float a0 = cov ? 1.0f : 0.0f;
    float vc[3], vM[3];
    load_rgb(v_rgb_aa, pp, vM);
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) vc[ch] = a0 * vM[ch];
    float vD = cov ? v_depth_aa[pp] : 0.0f;
    const int di[4] = {-1, 1, 0, 0}, dj[4] = {0, 0, -1, 1};
#pragma unroll 1
    for (int s = 0; s < 4; ++s) {
        const int qi = i + di[s], qj = j + dj[s];
        if (qi < 0 || qj < 0 || qi >= c.W || qj >= c.H) continue;
        const int64_t pq = (int64_t)qj * c.W + qi;
        if (m.face_id[pq] == m.face_id[pp]) continue;
        PairHit h;
        if (!aa_pair(c, m, pp, pq, h)) continue;
        const int64_t tgt = h.far_side ? h.other : h.occ;
        const float w = (float)fabs(h.t - 0.5);
        float vMt[3];
        load_rgb(v_rgb_aa, tgt, vMt);
        const bool cov_o = true, cov_n = m.face_id[h.other] >= 0;
        (void)cov_o;
        // this pixel's colour in the moved layer
        if (tgt == pp) {
            const float k = h.occ == pp ? -w : -w * a0;
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) vc[ch] = fmaf(k, vM[ch], vc[ch]);
        } else {
            const float k = h.occ == pp ? w : w * a0;
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) vc[ch] = fmaf(k, vMt[ch], vc[ch]);
        }
        // an uncovered neighbour that took this pixel's depth
        if (tgt == pq && h.occ == pp && m.face_id[pq] < 0 && w > 0.0f) {
            float Mq[3], Dq;
            int64_t src;
            aa_layer(c, m, qi, qj, Mq, Dq, &src);
            if (src == pp) vD += v_depth_aa[pq];
        }
        // the crossing, for the pairs this pixel owns
        if (s == 1 || s == 3) {
            float Mt[3], Dt;
            const float at = aa_layer(c, m, (int)(tgt % c.W), (int)(tgt / c.W), Mt, Dt, nullptr);
            const float va = (at >= 0.0f && at <= 1.0f) ? v_cov[tgt] : 0.0f;
            float co[3], cn[3];
            load_rgb(m.rgb, h.occ, co);
            load_rgb(m.rgb, h.other, cn);
            const float an = cov_n ? 1.0f : 0.0f;
            float dLdw;
            if (tgt == h.occ) {  // (a, M) += w ((a0, M0)(other) - (1, c_o))
                dLdw = va * (an - 1.0f);
#pragma unroll
                for (int ch = 0; ch < 3; ++ch) dLdw = fmaf(vMt[ch], an * cn[ch] - co[ch], dLdw);
            } else {  // (a, M) += w ((1, c_o) - (a0, M0)(other))
                dLdw = va * (1.0f - an);
#pragma unroll
                for (int ch = 0; ch < 3; ++ch) dLdw = fmaf(vMt[ch], co[ch] - an * cn[ch], dLdw);
            }
            const double dLdt = h.t >= 0.5 ? (double)dLdw : -(double)dLdw;
            if (dLdt != 0.0 && h.t > 0.0 && h.t < 1.0) {
                const int ka = (h.k + 1) % 3, kb = (h.k + 2) % 3;
                const int vida = __ldg(m.F + 3 * (int64_t)h.face + ka), vidb = __ldg(m.F + 3 * (int64_t)h.face + kb);
                double xc[3], ua, va_, ub, vb;
                vtx_f64(c, m.V, vida, xc, ua, va_);
                vtx_f64(c, m.V, vidb, xc, ub, vb);
                const double ox = (double)(h.occ % c.W) + 0.5, oy = (double)(h.occ / c.W) + 0.5;
                const double nx = (double)(h.other % c.W) + 0.5, ny = (double)(h.other / c.W) + 0.5;
                const double eo = edge64(ua, va_, ub, vb, ox, oy), en = edge64(ua, va_, ub, vb, nx, ny);
                const double den = (eo - en) * (eo - en);
                const double geo = dLdt * (-en / den), gen = dLdt * (eo / den);
                // e(p) = (ub - ua)(py - va) - (vb - va)(px - ua)
                const double gua = geo * (vb - oy) + gen * (vb - ny);
                const double gub = geo * (oy - va_) + gen * (ny - va_);
                const double gva = geo * (ox - ub) + gen * (nx - ub);
                const double gvb = geo * (ua - ox) + gen * (ua - nx);
                scatter_vertex_grad(c, m.V, vida, gua, gva, v_verts);
                scatter_vertex_grad(c, m.V, vidb, gub, gvb, v_verts);
            }
        }
    }
    v_mesh_rgb[3 * pp] = vc[0];
    v_mesh_rgb[3 * pp + 1] = vc[1];
    v_mesh_rgb[3 * pp + 2] = vc[2];
    v_mesh_depth[pp] = vD;
}

}  // namespace

// ------------------------------------------------------------ host side ---

static int bits_for(int n)
{
    return n > 1 ? 32 - __builtin_clz((unsigned)(n - 1)) : 1;
}

size_t mesh_edges_ws_bytes(int nF)
{
    const int64_t n = 3 * (int64_t)(nF > 0 ? nF : 1);
    return ((sizeof(uint64_t) * n + 255) & ~(size_t)255) + ((sizeof(int32_t) * n + 255) & ~(size_t)255) + 256 +
           sort_ws_bytes(n);
}

cudaError_t mesh_edges(const int32_t* F, int nF, int nV, int32_t* adj, int32_t* counters, void* ws, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(counters, 0, 4 * sizeof(int32_t), s);
    if (e != cudaSuccess || nF <= 0) return e;
    const int64_t n = 3 * (int64_t)nF;
    uint8_t* b = (uint8_t*)ws;
    uint64_t* keys = (uint64_t*)b;
    b += (sizeof(uint64_t) * n + 255) & ~(size_t)255;
    int32_t* vals = (int32_t*)b;
    b += (sizeof(int32_t) * n + 255) & ~(size_t)255;
    int32_t* n_dev = (int32_t*)b;
    b += 256;
    SortWs so;
    carve_sort_ws(b, n, so);
    const int bits = bits_for(nV);
    k_edge_keys<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(F, nF, bits, keys, vals, n_dev);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = radix_sort(keys, vals, so.keys_alt, so.vals_alt, (int)n, 0, 2 * bits, n_dev, counters, so, s);
    if (e != cudaSuccess) return e;
    const bool alt = sort_passes(0, 2 * bits) % 2 != 0;
    k_edge_pairs<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(alt ? so.keys_alt : keys, alt ? so.vals_alt : vals, n,
                                                              nF, adj);
    return cudaGetLastError();
}

cudaError_t antialias(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const int32_t* adj,
                      const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb, float* cov,
                      float* rgb_aa, float* depth_aa, float* tile_far, uint8_t* tile_full, cudaStream_t s)
{
    const Mesh m{V, F, adj, face_id, mesh_depth, mesh_rgb, nV, nF};
    k_antialias<<<c.TW * c.TH, TILE_PIX, 0, s>>>(c, m, cov, rgb_aa, depth_aa, tile_far, tile_full);
    return cudaGetLastError();
}

cudaError_t antialias_bwd(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const int32_t* adj,
                          const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb, const float* v_cov,
                          const float* v_rgb_aa, const float* v_depth_aa, float* v_mesh_rgb, float* v_mesh_depth,
                          float* v_verts, cudaStream_t s)
{
    const Mesh m{V, F, adj, face_id, mesh_depth, mesh_rgb, nV, nF};
    k_antialias_bwd<<<c.TW * c.TH, TILE_PIX, 0, s>>>(c, m, v_cov, v_rgb_aa, v_depth_aa, v_mesh_rgb, v_mesh_depth,
                                                      v_verts);
    return cudaGetLastError();
}

}  // namespace gm

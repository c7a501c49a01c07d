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
// evaluated in double-float arithmetic (about 48 significant bits from pairs of
// fp32 values; fp64 runs at a small fraction of the fp32 rate on this GPU),
// free of the cancellation that fp32 screen coordinates of the order of a
// thousand pixels would bring.
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

// Double-float arithmetic: a value is hi + lo with |lo| <= ulp(hi) / 2, built on
// the error-free transformations two-sum (Knuth: a + b = s + e exactly) and
// two-product (Dekker's, here with a fused multiply-add: a b = p + e exactly).
struct DF {
    float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

__device__ __forceinline__ DF fast_two_sum(float a, float b)  // |a| >= |b|
{
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ DF two_prod(float a, float b)
{
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ DF df_add(DF a, DF b)
{
    DF s = two_sum(a.hi, b.hi);
    const DF t = two_sum(a.lo, b.lo);
    s = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
    return fast_two_sum(s.hi, __fadd_rn(s.lo, t.lo));
}

__device__ __forceinline__ DF df_neg(DF a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ DF df_sub(DF a, DF b) { return df_add(a, df_neg(b)); }

__device__ __forceinline__ DF df_mul(DF a, DF b)
{
    DF p = two_prod(a.hi, b.hi);
    return fast_two_sum(p.hi, __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo)));
}

// a / b: a correctly rounded fp32 quotient refined twice by the exact remainder
__device__ __forceinline__ DF df_div(DF a, DF b)
{
    const float q1 = __fdiv_rn(a.hi, b.hi);
    DF r = df_sub(a, df_mul(b, DF{q1, 0.0f}));
    const float q2 = __fdiv_rn(r.hi, b.hi);
    r = df_sub(r, df_mul(b, DF{q2, 0.0f}));
    const float q3 = __fdiv_rn(r.hi, b.hi);
    return df_add(fast_two_sum(q1, q2), DF{q3, 0.0f});
}

// screen position of vertex vid in double-float (the vertex and camera are fp32)
__device__ __forceinline__ void vtx_df(const Cam& c, const float* __restrict__ V, int vid, DF& u, DF& v)
{
    const float X = __ldg(V + 3 * (int64_t)vid), Y = __ldg(V + 3 * (int64_t)vid + 1), Z = __ldg(V + 3 * (int64_t)vid + 2);
    DF xc[3];
#pragma unroll
    for (int r = 0; r < 3; ++r)
        xc[r] = df_add(df_add(df_add(two_prod(c.R[3 * r], X), two_prod(c.R[3 * r + 1], Y)), two_prod(c.R[3 * r + 2], Z)),
                       DF{c.t[r], 0.0f});
    u = df_add(df_div(df_mul(DF{c.fx, 0.0f}, xc[0]), xc[2]), DF{c.cx, 0.0f});
    v = df_add(df_div(df_mul(DF{c.fy, 0.0f}, xc[1]), xc[2]), DF{c.cy, 0.0f});
}

// e(a -> b, p) = (ub - ua)(py - va) - (vb - va)(px - ua)
__device__ __forceinline__ DF edge_df(DF ua, DF va, DF ub, DF vb, float px, float py)
{
    return df_sub(df_mul(df_sub(ub, ua), df_sub(DF{py, 0.0f}, va)), df_mul(df_sub(vb, va), df_sub(DF{px, 0.0f}, ua)));
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
    float t;             // crossing, from the occluder's centre (0) to the other's (1)
    float eo, en;        // the silhouette edge's function at the two centres (t = eo / (eo - en))
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
    DF ua, va, ub, vb;
    vtx_df(c, m.V, __ldg(m.F + 3 * (int64_t)X + a), ua, va);
    vtx_df(c, m.V, __ldg(m.F + 3 * (int64_t)X + b), ub, vb);
    const DF eo = edge_df(ua, va, ub, vb, ox, oy);
    const DF en = edge_df(ua, va, ub, vb, nx, ny);
    const float t = df_div(eo, df_sub(eo, en)).hi;
    h.occ = o;
    h.other = nb;
    h.t = t < 0.0f ? 0.0f : (t > 1.0f ? 1.0f : t);
    h.eo = eo.hi;
    h.en = en.hi;
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
        const float w = fabsf(h.t - 0.5f);
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

// dL/d(screen position of a vertex) -> dL/d its world position, added
__device__ void scatter_vertex_grad(const Cam& c, const float* __restrict__ V, int vid, float gu, float gv,
                                    float* __restrict__ v_verts)
{
    const float X = __ldg(V + 3 * (int64_t)vid), Y = __ldg(V + 3 * (int64_t)vid + 1), Z = __ldg(V + 3 * (int64_t)vid + 2);
    const float x = fmaf(c.R[0], X, fmaf(c.R[1], Y, fmaf(c.R[2], Z, c.t[0])));
    const float y = fmaf(c.R[3], X, fmaf(c.R[4], Y, fmaf(c.R[5], Z, c.t[1])));
    const float z = fmaf(c.R[6], X, fmaf(c.R[7], Y, fmaf(c.R[8], Z, c.t[2])));
    const float iz = 1.0f / z;
    // u = fx x / z + cx, v = fy y / z + cy
    const float gx = gu * c.fx * iz, gy = gv * c.fy * iz;
    const float gz = -(gu * c.fx * x + gv * c.fy * y) * iz * iz;
#pragma unroll
    for (int d = 0; d < 3; ++d)
        atomicAdd(v_verts + 3 * (int64_t)vid + d, c.R[d] * gx + c.R[3 + d] * gy + c.R[6 + d] * gz);
}

// Per pixel, the terms of its own layer: M0 = a0 c (dL/dc += a0 dL/dM) and, where
// the mesh covers the pixel, D_aa = D.  Written; the pair kernel then adds.
__global__ void __launch_bounds__(256)
k_aa_bwd_own(int64_t P, const int32_t* __restrict__ face_id, const float* __restrict__ v_rgb_aa,
             const float* __restrict__ v_depth_aa, float* __restrict__ v_mesh_rgb, float* __restrict__ v_mesh_depth)
{
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const bool cov = face_id[p] >= 0;
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) v_mesh_rgb[3 * p + ch] = cov ? v_rgb_aa[3 * p + ch] : 0.0f;
    v_mesh_depth[p] = cov ? v_depth_aa[p] : 0.0f;
}

// Each pair once, by the pixel on its left / top: the weight w moved the target's
// layer, (a, M)(tgt) += w ((a, M)(from) - (a0, M0)(tgt)) with the surface pixel's
// layer (1, c_o) on one side and the other pixel's (a0, a0 c) on the other.  Adds
// dL/d the two colours (and the depth an uncovered target took from the surface
// pixel) to the pixels' gradients, and dL/dt of the crossing to the silhouette
// edge's vertices.  A target whose coverage sits at 0 or 1 after the clamp
// passes no coverage gradient.
__global__ void __launch_bounds__(256)
k_aa_bwd_pairs(Cam c, Mesh m, const float* __restrict__ cov, const float* __restrict__ depth_aa,
               const float* __restrict__ v_cov, const float* __restrict__ v_rgb_aa,
               const float* __restrict__ v_depth_aa, float* __restrict__ v_mesh_rgb,
               float* __restrict__ v_mesh_depth, float* __restrict__ v_verts)
{
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= (int64_t)c.W * c.H) return;
    const int i = (int)(p % c.W), j = (int)(p / c.W);
#pragma unroll 1
    for (int s = 0; s < 2; ++s) {
        const int qi = i + (s == 0), qj = j + (s == 1);
        if (qi >= c.W || qj >= c.H) continue;
        const int64_t q = (int64_t)qj * c.W + qi;
        if (m.face_id[q] == m.face_id[p]) continue;
        PairHit h;
        if (!aa_pair(c, m, p, q, h)) continue;
        const int64_t tgt = h.far_side ? h.other : h.occ;
        const float w = fabsf(h.t - 0.5f);
        const bool cov_n = m.face_id[h.other] >= 0;
        const float an = cov_n ? 1.0f : 0.0f;
        float vM[3], co[3], cn[3];
        load_rgb(v_rgb_aa, tgt, vM);
        load_rgb(m.rgb, h.occ, co);
        load_rgb(m.rgb, h.other, cn);
        float dLdw;
        const float at = cov[tgt];
        const float va = (at > 0.0f && at < 1.0f) ? v_cov[tgt] : 0.0f;
        if (tgt == h.occ) {  // (a, M)(o) += w ((a0, a0 c)(n) - (1, c_o))
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) {
                atomicAdd(v_mesh_rgb + 3 * h.occ + ch, -w * vM[ch]);
                if (cov_n) atomicAdd(v_mesh_rgb + 3 * h.other + ch, w * vM[ch]);
            }
            dLdw = va * (an - 1.0f);
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) dLdw = fmaf(vM[ch], an * cn[ch] - co[ch], dLdw);
        } else {  // (a, M)(n) += w ((1, c_o) - (a0, a0 c)(n))
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) {
                atomicAdd(v_mesh_rgb + 3 * h.occ + ch, w * vM[ch]);
                if (cov_n) atomicAdd(v_mesh_rgb + 3 * h.other + ch, -w * vM[ch]);
            }
            dLdw = va * (1.0f - an);
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) dLdw = fmaf(vM[ch], co[ch] - an * cn[ch], dLdw);
            // an uncovered pixel takes the depth of the first (left, right, up, down)
            // of its nearest reaching surface pixels
            const float Do = m.depth[h.occ];
            if (!cov_n && w > 0.0f && __float_as_uint(depth_aa[tgt]) == __float_as_uint(Do)) {
                const int ti = (int)(tgt % c.W), tj = (int)(tgt / c.W);
                const int di[4] = {-1, 1, 0, 0}, dj[4] = {0, 0, -1, 1};
                bool first = true;
                for (int r = 0; r < 4; ++r) {
                    const int ri = ti + di[r], rj = tj + dj[r];
                    if (ri < 0 || rj < 0 || ri >= c.W || rj >= c.H) continue;
                    const int64_t pr = (int64_t)rj * c.W + ri;
                    if (pr == h.occ) break;
                    if (m.face_id[pr] < 0 || __float_as_uint(m.depth[pr]) != __float_as_uint(Do)) continue;
                    PairHit h2;  // an earlier neighbour at the same depth: does it reach the pixel?
                    if (aa_pair(c, m, tgt, pr, h2) && h2.occ == pr && h2.far_side && fabsf(h2.t - 0.5f) > 0.0f) {
                        first = false;
                        break;
                    }
                }
                if (first) atomicAdd(v_mesh_depth + h.occ, v_depth_aa[tgt]);
            }
        }
        // through the crossing: t = eo / (eo - en), w = |t - 0.5|
        const float dLdt = h.t >= 0.5f ? dLdw : -dLdw;
        if (dLdt != 0.0f && h.t > 0.0f && h.t < 1.0f) {
            const int ka = (h.k + 1) % 3, kb = (h.k + 2) % 3;
            const int vida = __ldg(m.F + 3 * (int64_t)h.face + ka), vidb = __ldg(m.F + 3 * (int64_t)h.face + kb);
            float ua, va_, ub, vb;
            vtx_f32(c, m.V, m.nV, vida, ua, va_);
            vtx_f32(c, m.V, m.nV, vidb, ub, vb);
            const float ox = (float)(h.occ % c.W) + 0.5f, oy = (float)(h.occ / c.W) + 0.5f;
            const float nx = (float)(h.other % c.W) + 0.5f, ny = (float)(h.other / c.W) + 0.5f;
            const float d = h.eo - h.en;
            const float geo = dLdt * (-h.en / (d * d)), gen = dLdt * (h.eo / (d * d));
            // e(p) = (ub - ua)(py - va) - (vb - va)(px - ua)
            scatter_vertex_grad(c, m.V, vida, geo * (vb - oy) + gen * (vb - ny), geo * (ox - ub) + gen * (nx - ub),
                                v_verts);
            scatter_vertex_grad(c, m.V, vidb, geo * (oy - va_) + gen * (ny - va_),
                                geo * (ua - ox) + gen * (ua - nx), v_verts);
        }
    }
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
                          const int32_t* face_id, const float* mesh_depth, const float* mesh_rgb, const float* cov,
                          const float* depth_aa, const float* v_cov, const float* v_rgb_aa, const float* v_depth_aa,
                          float* v_mesh_rgb, float* v_mesh_depth, float* v_verts, cudaStream_t s)
{
    const Mesh m{V, F, adj, face_id, mesh_depth, mesh_rgb, nV, nF};
    const int64_t P = (int64_t)c.W * c.H;
    const unsigned grid = (unsigned)((P + 255) / 256);
    k_aa_bwd_own<<<grid, 256, 0, s>>>(P, face_id, v_rgb_aa, v_depth_aa, v_mesh_rgb, v_mesh_depth);
    k_aa_bwd_pairs<<<grid, 256, 0, s>>>(c, m, cov, depth_aa, v_cov, v_rgb_aa, v_depth_aa, v_mesh_rgb, v_mesh_depth,
                                         v_verts);
    return cudaGetLastError();
}

}  // namespace gm

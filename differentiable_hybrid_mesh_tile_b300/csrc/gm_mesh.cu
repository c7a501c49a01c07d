// Mesh layer of the hybrid renderer ("A Lightweight and Differentiable
// Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Design Details >
// Mesh rasterizer, items 1 and 2): triangle tile bins, the z-buffer, the
// perspective-correct interpolation of depth and vertex colour, and its
// backward pass to vertex positions and colours.
#include "gm_internal.cuh"

namespace gm {
namespace {

// ------------------------------------------------------------- bins ------

__global__ void __launch_bounds__(256)
k_tri_count(Cam c, const float* __restrict__ V, int nV, const int32_t* __restrict__ F, int nF,
            int32_t* __restrict__ counts)
{
    int f = blockIdx.x * blockDim.x + threadIdx.x;
    if (f >= nF) return;
    Tri t;
    int n = 0;
    if (tri_setup(c, V, nV, F, f, t))
        n = (t.x1 / TILE - t.x0 / TILE + 1) * (t.y1 / TILE - t.y0 / TILE + 1);
    counts[f] = n;
}

__global__ void __launch_bounds__(256)
k_tri_emit(Cam c, const float* __restrict__ V, int nV, const int32_t* __restrict__ F, int nF,
           const int32_t* __restrict__ offsets, int cap, int32_t* counters, uint64_t* __restrict__ keys,
           int32_t* __restrict__ vals)
{
    int f = blockIdx.x * blockDim.x + threadIdx.x;
    if (f == 0 && counters[GM_CNT_K] > cap) atomicOr(counters + GM_CNT_FLAGS, GM_FLAG_OVERFLOW);
    if (f >= nF) return;
    Tri t;
    if (!tri_setup(c, V, nV, F, f, t)) return;
    int64_t o = offsets[f];
    for (int ty = t.y0 / TILE; ty <= t.y1 / TILE; ++ty)
        for (int tx = t.x0 / TILE; tx <= t.x1 / TILE; ++tx, ++o) {
            if (o < 0 || o >= cap) return;
            keys[o] = (uint64_t)(uint32_t)(ty * c.TW + tx) << 32;
            vals[o] = f;
        }
}

// ---------------------------------------------------------- z-buffer ------

// A staged triangle, four 16-byte vectors (one shared-memory load each):
// (u0, v0, u1, v1), (u2, v2, area, w0), (w1, w2, face id, -), pixel-centre box
// (x0, x1, y0, y1); w_k = 1 / (area z_k): depth reciprocal = sum_k e_k w_k.
struct TriRec {
    float4 p, q, w;
    int4 box;
};

__global__ void __launch_bounds__(TILE_PIX)
k_zbuffer(Cam c, const float* __restrict__ V, int nV, const int32_t* __restrict__ F, int nF,
          const int2* __restrict__ tile_range, const int32_t* __restrict__ tri_ids, int32_t* __restrict__ face_id)
{
    __shared__ TriRec sm[TILE_PIX];
    const int tile = blockIdx.x;
    const int tx = tile % c.TW, ty = tile / c.TW;
    // warp w covers the 8 x 4 pixel block at (8 (w % 2), 4 (w / 2)) of the tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = tx * TILE + (warp & 1) * 8, by = ty * TILE + (warp >> 1) * 4;
    const int i = bx + (lane & 7);
    const int j = by + (lane >> 3);
    const bool inside = i < c.W && j < c.H;
    const float px = (float)i + 0.5f, py = (float)j + 0.5f;
    const int2 r = tile_range[tile];
    float best = 0.0f;  // reciprocal depth of the winner (0 = none)
    int best_f = -1;
    for (int b = r.x; b < r.y; b += TILE_PIX) {
        const int n = min(TILE_PIX, r.y - b);
        if ((int)threadIdx.x < n) {
            int f = tri_ids[b + threadIdx.x];
            Tri t;
            TriRec& q = sm[threadIdx.x];
            // an id outside [0, nF) (possible only when the sort that built the
            // lists gave up a bounded wait) is skipped
            if (f >= 0 && f < nF && tri_setup(c, V, nV, F, f, t)) {
                q.p = make_float4(t.u[0], t.v[0], t.u[1], t.v[1]);
                q.q = make_float4(t.u[2], t.v[2], t.area, 1.0f / (t.area * t.z[0]));
                q.w = make_float4(1.0f / (t.area * t.z[1]), 1.0f / (t.area * t.z[2]), __int_as_float(f), 0.0f);
                q.box = make_int4(t.x0, t.x1, t.y0, t.y1);
            } else {
                q.w = make_float4(0.0f, 0.0f, __int_as_float(-1), 0.0f);
                q.box = make_int4(1, 0, 1, 0);
            }
        }
        __syncthreads();
        // per 32 staged triangles, a ballot of those whose pixel-centre box meets
        // this warp's block; the warp visits only those, in ascending face order
        for (int m = 0; m * 32 < n; ++m) {
            const int kk = m * 32 + lane;
            bool h = false;
            if (kk < n) {
                const int4 bb = sm[kk].box;
                h = bb.y >= bx && bb.x <= bx + 7 && bb.w >= by && bb.z <= by + 3;
            }
            uint32_t mask = __ballot_sync(0xffffffffu, h);
            while (mask) {
                const int k = m * 32 + __ffs(mask) - 1;
                mask &= mask - 1;
                const int4 bb = sm[k].box;
                if (!inside || i < bb.x || i > bb.y || j < bb.z || j > bb.w) continue;
                const float4 a = sm[k].p, b = sm[k].q;
                // vertices (a.x, a.y), (a.z, a.w), (b.x, b.y); area b.z
                float e0 = edge_rn(a.z, a.w, b.x, b.y, px, py);
                float e1 = edge_rn(b.x, b.y, a.x, a.y, px, py);
                float e2 = edge_rn(a.x, a.y, a.z, a.w, px, py);
                bool in = b.z > 0.0f ? (e0 >= 0.0f && e1 >= 0.0f && e2 >= 0.0f)
                                     : (e0 <= 0.0f && e1 <= 0.0f && e2 <= 0.0f);
                if (!in) continue;
                const float4 w = sm[k].w;
                float inv_d = fmaf(e0, b.w, fmaf(e1, w.x, e2 * w.y));
                if (inv_d > best) {  // lists ascend in face id: an equal depth keeps the smaller id
                    best = inv_d;
                    best_f = __float_as_int(w.z);
                }
            }
        }
        __syncthreads();
    }
    if (inside) face_id[(int64_t)j * c.W + i] = best_f;
}

// ------------------------------------------------------------- interp -----

struct Persp {
    float u[3], v[3], z[3], x[3], y[3];
    float e[3], area, lam[3], q[3], s, D, w[3];
};

// false when a vertex index is out of range (the face is then treated as absent)
__device__ __forceinline__ bool load_face(const float* __restrict__ V, int nV, const int32_t* __restrict__ F,
                                          int f, int vid[3], float X[3][3])
{
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        vid[k] = __ldg(F + 3 * (int64_t)f + k);
        if (vid[k] < 0 || vid[k] >= nV) return false;
    }
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int d = 0; d < 3; ++d) X[k][d] = __ldg(V + 3 * (int64_t)vid[k] + d);
    return true;
}

// perspective-correct weights at pixel centre (px, py)
__device__ __forceinline__ void persp(const Cam& c, const float X[3][3], float px, float py, Persp& P)
{
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        float x = fmaf(c.R[0], X[k][0], fmaf(c.R[1], X[k][1], fmaf(c.R[2], X[k][2], c.t[0])));
        float y = fmaf(c.R[3], X[k][0], fmaf(c.R[4], X[k][1], fmaf(c.R[5], X[k][2], c.t[1])));
        float z = fmaf(c.R[6], X[k][0], fmaf(c.R[7], X[k][1], fmaf(c.R[8], X[k][2], c.t[2])));
        P.x[k] = x; P.y[k] = y; P.z[k] = z;
        float iz = 1.0f / z;
        P.u[k] = fmaf(c.fx * x, iz, c.cx);
        P.v[k] = fmaf(c.fy * y, iz, c.cy);
    }
    P.area = (P.u[1] - P.u[0]) * (P.v[2] - P.v[0]) - (P.u[2] - P.u[0]) * (P.v[1] - P.v[0]);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int a = (k + 1) % 3, b = (k + 2) % 3;
        P.e[k] = (P.u[b] - P.u[a]) * (py - P.v[a]) - (P.v[b] - P.v[a]) * (px - P.u[a]);
    }
    float ia = 1.0f / P.area;
    P.s = 0.0f;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        P.lam[k] = P.e[k] * ia;
        P.q[k] = P.lam[k] / P.z[k];
        P.s += P.q[k];
    }
    P.D = 1.0f / P.s;
#pragma unroll
    for (int k = 0; k < 3; ++k) P.w[k] = P.q[k] * P.D;
}

__global__ void __launch_bounds__(TILE_PIX)
k_interp(Cam c, const float* __restrict__ V, int nV, const int32_t* __restrict__ F, int nF,
         const float* __restrict__ vcol, const int32_t* __restrict__ face_id, float* __restrict__ mesh_depth,
         float* __restrict__ mesh_rgb, float* __restrict__ tile_far, uint8_t* __restrict__ tile_full)
{
    __shared__ float s_max[TILE_PIX / 32];
    const int tile = blockIdx.x;
    const int tx = tile % c.TW, ty = tile / c.TW;
    const int i = tx * TILE + (threadIdx.x & (TILE - 1));
    const int j = ty * TILE + (threadIdx.x >> 4);
    const bool inside = i < c.W && j < c.H;
    float D = INFINITY;
    bool covered = false;
    if (inside) {
        const int64_t pix = (int64_t)j * c.W + i;
        int f = face_id[pix];
        float rgb[3] = {0.0f, 0.0f, 0.0f};
        int vid[3];
        float X[3][3];
        if (f >= 0 && f < nF && load_face(V, nV, F, f, vid, X)) {
            Persp P;
            persp(c, X, (float)i + 0.5f, (float)j + 0.5f, P);
            D = P.D;
            covered = true;
#pragma unroll
            for (int k = 0; k < 3; ++k)
#pragma unroll
                for (int ch = 0; ch < 3; ++ch) rgb[ch] = fmaf(P.w[k], __ldg(vcol + 3 * (int64_t)vid[k] + ch), rgb[ch]);
        }
        mesh_depth[pix] = D;
        mesh_rgb[3 * pix + 0] = rgb[0];
        mesh_rgb[3 * pix + 1] = rgb[1];
        mesh_rgb[3 * pix + 2] = rgb[2];
    }
    const int all = __syncthreads_and(!inside || covered);
    float m = inside ? D : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float far = s_max[0];
        for (int w = 1; w < TILE_PIX / 32; ++w) far = fmaxf(far, s_max[w]);
        tile_far[tile] = all ? far : INFINITY;
        tile_full[tile] = (uint8_t)(all ? 1 : 0);
    }
}

// ------------------------------------------------------------ backward ----

// dL/d(world vertex positions, vertex colours) of one covered pixel, given
// dL/dD (gD) and dL/d(mesh colour) (gc), for the interpolation of k_interp.
__device__ __forceinline__ void interp_grad(const Cam& c, const float X[3][3], const float C[3][3], float px,
                                            float py, float gD, const float gc[3], float gX[3][3], float gC[3][3])
{
    Persp P;
    persp(c, X, px, py, P);
    float gw[3];
    float cm[3] = {0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        gw[k] = gc[0] * C[k][0] + gc[1] * C[k][1] + gc[2] * C[k][2];
#pragma unroll
        for (int ch = 0; ch < 3; ++ch) {
            gC[k][ch] = P.w[k] * gc[ch];
            cm[ch] = fmaf(P.w[k], C[k][ch], cm[ch]);
        }
    }
    const float gwbar = gc[0] * cm[0] + gc[1] * cm[1] + gc[2] * cm[2];
    // q_k = l_k / z_k, s = sum q, D = 1/s, w_k = q_k D
    float gl[3], gz[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        float gq = -gD * P.D * P.D + P.D * (gw[k] - gwbar);
        gl[k] = gq / P.z[k];
        gz[k] = -gq * P.q[k] / P.z[k];
    }
    // l_k = e_k / area
    const float ia = 1.0f / P.area;
    float garea = 0.0f;
    float ge[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        ge[k] = gl[k] * ia;
        garea -= gl[k] * P.lam[k] * ia;
    }
    float gu[3] = {0.0f, 0.0f, 0.0f}, gv[3] = {0.0f, 0.0f, 0.0f};
    // e_k = (ub - ua)(py - va) - (vb - va)(px - ua), a = k+1, b = k+2
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int a = (k + 1) % 3, b = (k + 2) % 3;
        gu[b] += ge[k] * (py - P.v[a]);
        gu[a] += ge[k] * (P.v[b] - py);
        gv[b] -= ge[k] * (px - P.u[a]);
        gv[a] += ge[k] * (px - P.u[b]);
    }
    // area = (u1 - u0)(v2 - v0) - (u2 - u0)(v1 - v0)
    gu[0] += garea * (P.v[1] - P.v[2]);
    gu[1] += garea * (P.v[2] - P.v[0]);
    gu[2] += garea * (P.v[0] - P.v[1]);
    gv[0] += garea * (P.u[2] - P.u[1]);
    gv[1] += garea * (P.u[0] - P.u[2]);
    gv[2] += garea * (P.u[1] - P.u[0]);
    // u = fx x / z + cx, v = fy y / z + cy; then world = R^T camera
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const float iz = 1.0f / P.z[k];
        const float gx = gu[k] * c.fx * iz;
        const float gy = gv[k] * c.fy * iz;
        const float gzz = gz[k] - (gu[k] * (P.u[k] - c.cx) + gv[k] * (P.v[k] - c.cy)) * iz;
        gX[k][0] = c.R[0] * gx + c.R[3] * gy + c.R[6] * gzz;
        gX[k][1] = c.R[1] * gx + c.R[4] * gy + c.R[7] * gzz;
        gX[k][2] = c.R[2] * gx + c.R[5] * gy + c.R[8] * gzz;
    }
}

// Per-face sums of a warp's pixel gradients.  Each pixel has 18 values (the
// position and the colour gradient of the face's three vertices); the lanes
// park them in shared memory, then take the (face, component) sums of the
// warp's distinct faces 32 at a time: each adds its component over the face's
// pixels and issues one global atomic.  A warp with K faces thus costs
// ceil(18 K / 32) rounds instead of 18 K warp-wide sums.
constexpr int MB_WARPS = TILE_PIX / 32;
constexpr int MB_VALS = 18;

struct MeshBwdStage {
    float val[MB_WARPS][MB_VALS][33];  // [warp][component][lane], padded: conflict-free reads across components
    int vid[MB_WARPS][3][32];
    uint32_t peers[MB_WARPS][32];
    uint8_t lead[MB_WARPS][32];
};

// DIRECT: g_rgb / g_depth are already dL/d(interpolated colour, depth) per pixel
// (from the antialiasing's backward); otherwise they are the image's upstream
// gradient, weighted here by the transmittance in front of the mesh.
//
// At most 64 registers (4 CTAs of 256 threads per SM): the kernel waits on the
// gathers of the faces' vertices and colours, and more resident warps hide them.
template <bool DIRECT>
__global__ void __launch_bounds__(TILE_PIX, 4)
k_mesh_bwd(Cam c, const float* __restrict__ V, int nV, const int32_t* __restrict__ F, int nF,
           const float* __restrict__ vcol, const int32_t* __restrict__ face_id, const float* __restrict__ T_final,
           const float* __restrict__ g_rgb, const float* __restrict__ g_depth,
           const float* __restrict__ v_mesh_depth, float* __restrict__ v_verts, float* __restrict__ v_vcol)
{
    __shared__ MeshBwdStage st;
    const int tile = blockIdx.x;
    const int tx = tile % c.TW, ty = tile / c.TW;
    const int i = tx * TILE + (threadIdx.x & (TILE - 1));
    const int j = ty * TILE + (threadIdx.x >> 4);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int f = -1;
    if (i < c.W && j < c.H) f = face_id[(int64_t)j * c.W + i];
    float gX[3][3], gC[3][3];
    int vid[3] = {0, 0, 0};
    float X[3][3], C[3][3];
    const bool act = f >= 0 && f < nF && load_face(V, nV, F, f, vid, X);
    if (act) {
        const int64_t pix = (int64_t)j * c.W + i;
#pragma unroll
        for (int k = 0; k < 3; ++k)
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) C[k][ch] = __ldg(vcol + 3 * (int64_t)vid[k] + ch);
        const float T = DIRECT ? 1.0f : T_final[pix];
        const float gc[3] = {T * g_rgb[3 * pix], T * g_rgb[3 * pix + 1], T * g_rgb[3 * pix + 2]};
        // dL/dD: through the depth output (T D), and through the soft split when given
        const float gD = T * g_depth[pix] + (!DIRECT && v_mesh_depth ? v_mesh_depth[pix] : 0.0f);
        interp_grad(c, X, C, (float)i + 0.5f, (float)j + 0.5f, gD, gc, gX, gC);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            st.vid[w][k][lane] = vid[k];
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                st.val[w][3 * k + d][lane] = gX[k][d];
                st.val[w][9 + 3 * k + d][lane] = gC[k][d];
            }
        }
    }
    // the lanes of each face; a face's lowest lane leads it
    const uint32_t peers = __match_any_sync(0xffffffffu, act ? f : -1);
    const bool leader = act && lane == __ffs(peers) - 1;
    const uint32_t leaders = __ballot_sync(0xffffffffu, leader);
    if (leader) {
        st.peers[w][lane] = peers;
        st.lead[w][__popc(leaders & ((1u << lane) - 1u))] = (uint8_t)lane;
    }
    __syncwarp();
    const int items = MB_VALS * __popc(leaders);
    for (int t = lane; t < items; t += 32) {
        const int fi = t / MB_VALS, q = t - fi * MB_VALS;
        const int ld = st.lead[w][fi];
        uint32_t m = st.peers[w][ld];
        float sum = 0.0f;
        while (m) {
            sum += st.val[w][q][__ffs(m) - 1];
            m &= m - 1;
        }
        const int k = (q % 9) / 3, d = q % 3;
        float* dst = q < 9 ? v_verts : v_vcol;
        if (sum != 0.0f) atomicAdd(dst + 3 * (int64_t)st.vid[w][k][ld] + d, sum);
    }
}

}  // namespace

// ------------------------------------------------------------ host side ---

static int tile_bits(int n_tiles)
{
    return n_tiles > 1 ? 32 - __builtin_clz((unsigned)(n_tiles - 1)) : 0;
}

size_t tri_bin_ws_bytes(int nF, int cap)
{
    int64_t n = nF > 0 ? nF : 1, k = cap > 0 ? cap : 1;
    return scan_ws_bytes(n) + 2 * ((sizeof(int32_t) * n + 255) & ~(size_t)255) +
           ((sizeof(uint64_t) * k + 255) & ~(size_t)255) + sort_ws_bytes(k);
}

cudaError_t tri_bin(const Cam& c, const float* V, int nV, const int32_t* F, int nF, int32_t* tile_range,
                    int32_t* tri_ids, int cap, int32_t* counters, void* ws, cudaStream_t s)
{
    int64_t n = nF > 0 ? nF : 1, k = cap > 0 ? cap : 1;
    uint8_t* b = (uint8_t*)ws;
    ScanWs sw;
    b += carve_scan_ws(b, n, sw);
    int32_t* counts = (int32_t*)b;
    b += (sizeof(int32_t) * n + 255) & ~(size_t)255;
    int32_t* offsets = (int32_t*)b;
    b += (sizeof(int32_t) * n + 255) & ~(size_t)255;
    uint64_t* keysA = (uint64_t*)b;
    b += (sizeof(uint64_t) * k + 255) & ~(size_t)255;
    SortWs so;
    carve_sort_ws(b, k, so);

    cudaError_t e = cudaMemsetAsync(counters, 0, 4 * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    const int T = c.TW * c.TH;
    const int passes = sort_passes(32, 32 + tile_bits(T));
    uint64_t* ek = passes % 2 ? so.keys_alt : keysA;
    int32_t* ev = passes % 2 ? so.vals_alt : tri_ids;
    if (nF > 0) {
        k_tri_count<<<(nF + 255) / 256, 256, 0, s>>>(c, V, nV, F, nF, counts);
        if ((e = exclusive_scan(counts, nullptr, offsets, nF, counters, sw, s)) != cudaSuccess) return e;
        k_tri_emit<<<(nF + 255) / 256, 256, 0, s>>>(c, V, nV, F, nF, offsets, cap, counters, ek, ev);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (passes % 2)
            e = radix_sort(so.keys_alt, so.vals_alt, keysA, tri_ids, cap, 32, 32 + tile_bits(T), counters + GM_CNT_K,
                           counters, so, s);
        else
            e = radix_sort(keysA, tri_ids, so.keys_alt, so.vals_alt, cap, 32, 32 + tile_bits(T), counters + GM_CNT_K,
                           counters, so, s);
        if (e != cudaSuccess) return e;
    }
    return tile_ranges(keysA, nF > 0 ? cap : 0, counters, tile_range, T, s);
}

cudaError_t zbuffer(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const int32_t* tile_range,
                    const int32_t* tri_ids, int32_t* face_id, cudaStream_t s)
{
    k_zbuffer<<<c.TW * c.TH, TILE_PIX, 0, s>>>(c, V, nV, F, nF, reinterpret_cast<const int2*>(tile_range), tri_ids,
                                                face_id);
    return cudaGetLastError();
}

cudaError_t interp(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const float* vcol,
                   const int32_t* face_id, float* mesh_depth, float* mesh_rgb, float* tile_far, uint8_t* tile_full,
                   cudaStream_t s)
{
    k_interp<<<c.TW * c.TH, TILE_PIX, 0, s>>>(c, V, nV, F, nF, vcol, face_id, mesh_depth, mesh_rgb, tile_far,
                                               tile_full);
    return cudaGetLastError();
}

cudaError_t mesh_bwd(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const float* vcol,
                     const int32_t* face_id, const float* T_final, const float* g_rgb, const float* g_depth,
                     const float* v_mesh_depth, float* v_verts, float* v_vcol, cudaStream_t s)
{
    k_mesh_bwd<false><<<c.TW * c.TH, TILE_PIX, 0, s>>>(c, V, nV, F, nF, vcol, face_id, T_final, g_rgb, g_depth,
                                                        v_mesh_depth, v_verts, v_vcol);
    return cudaGetLastError();
}

cudaError_t interp_bwd(const Cam& c, const float* V, int nV, const int32_t* F, int nF, const float* vcol,
                       const int32_t* face_id, const float* v_mesh_rgb, const float* v_mesh_depth, float* v_verts,
                       float* v_vcol, cudaStream_t s)
{
    k_mesh_bwd<true><<<c.TW * c.TH, TILE_PIX, 0, s>>>(c, V, nV, F, nF, vcol, face_id, nullptr, v_mesh_rgb,
                                                       v_mesh_depth, nullptr, v_verts, v_vcol);
    return cudaGetLastError();
}

}  // namespace gm

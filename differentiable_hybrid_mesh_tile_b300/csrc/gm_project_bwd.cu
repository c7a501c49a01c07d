// Backward of the Gaussian projection ("A Lightweight and Differentiable
// Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Hybrid rendering:
// everything is differentiable; projection and SH colour adapted from gsplat).
// Given dL/d of each projected record (mean2d, conic, opacity, rgb, depth --
// what the composite backward produces), the chain rule through the EWA
// projection and the SH colour gives dL/d of the Gaussian's 3D mean,
// log-scales, quaternion, opacity logit and colour coefficients.
//
// One thread per Gaussian: the forward intermediates are recomputed in fp32
// from the inputs (nothing is stored between the passes), and each thread
// writes only its own Gaussian's rows, so no atomics are needed.  Gaussians
// the forward culled (radius 0) get zero gradients.
#include <algorithm>

#include "gm_internal.cuh"
#include "gm_proj.cuh"

namespace gm {
namespace {

// dL/d(x, y, z) of sum_k vY[k] Y_k(x, y, z), each Y_k the polynomial of
// sh_basis in the components of the unit direction (treated as independent;
// the normalisation is applied by the caller).
template <int DEG>
__device__ __forceinline__ void sh_basis_vjp(float x, float y, float z, const float* vY, float& gx, float& gy,
                                             float& gz)
{
    gx = gy = gz = 0.0f;
    if (DEG >= 1) {
        gy += SH_C1 * vY[1];
        gz += SH_C1 * vY[2];
        gx += SH_C1 * vY[3];
    }
    if (DEG >= 2) {
        gx += SH_C2a * (y * vY[4] + z * vY[7]) + 2.0f * SH_C2e * x * vY[8];
        gy += SH_C2a * (x * vY[4] + z * vY[5]) - 2.0f * SH_C2e * y * vY[8];
        gz += SH_C2a * (y * vY[5] + x * vY[7]) + 6.0f * SH_C2c * z * vY[6];
        if (DEG >= 3) {
            const float xx = x * x, yy = y * y, zz = z * z;
            // Y9 = C3a y (3x^2 - y^2), Y10 = C3b x y z, Y11 = C3c y (5z^2 - 1),
            // Y12 = C3d z (5z^2 - 3), Y13 = C3c x (5z^2 - 1), Y14 = C3f z (x^2 - y^2),
            // Y15 = C3a x (x^2 - 3y^2)
            gx += SH_C3a * 6.0f * x * y * vY[9] + SH_C3b * y * z * vY[10] + SH_C3c * (5.0f * zz - 1.0f) * vY[13] +
                  SH_C3f * 2.0f * x * z * vY[14] + SH_C3a * 3.0f * (xx - yy) * vY[15];
            gy += SH_C3a * 3.0f * (xx - yy) * vY[9] + SH_C3b * x * z * vY[10] + SH_C3c * (5.0f * zz - 1.0f) * vY[11] -
                  SH_C3f * 2.0f * y * z * vY[14] - SH_C3a * 6.0f * x * y * vY[15];
            gz += SH_C3b * x * y * vY[10] + SH_C3c * 10.0f * y * z * vY[11] + SH_C3d * (15.0f * zz - 3.0f) * vY[12] +
                  SH_C3c * 10.0f * x * z * vY[13] + SH_C3f * (xx - yy) * vY[14];
        }
    }
}

// The additions of gradients over calls or views are separately rounded
// (__fadd_rn is never contracted into a multiply-add), so a batched sum over
// views and a sequence of accumulating per-view calls agree bit for bit.
__device__ __forceinline__ void put(float* dst, float v, bool acc)
{
    *dst = acc ? __fadd_rn(*dst, v) : v;
}

__device__ __forceinline__ void add_or_set(float& x, float v, bool first)
{
    x = first ? v : __fadd_rn(x, v);
}

// The gradient of one Gaussian's parameters from one view's record gradient.
template <int DEG>
struct ProjGrad {
    static constexpr int K = DEG < 0 ? 1 : (DEG + 1) * (DEG + 1);
    float vmu[3], vls[3], vq[4], vlogit;
    float vcol[3 * K];
};

// DEG < 0: colours are RGB [N][3]; else SH coefficients [N][(DEG+1)^2][3].
// radius: of this Gaussian in this view (0 = culled: zero gradient);
// vsp: its record gradient (3 float4); sh_row: its SH row staged in shared
// memory (ShStage), or null.
template <int DEG>
__device__ __forceinline__ void project_bwd_gaussian(const Cam& c, const ProjConsts& pc, int g,
                                                     const float* __restrict__ means,
                                                     const float* __restrict__ log_scales,
                                                     const float4* __restrict__ quats,
                                                     const float* __restrict__ logits,
                                                     const float* __restrict__ colors, int radius,
                                                     const float4* __restrict__ vsp,
                                                     const float4* __restrict__ vdm, bool first,
                                                     ProjGrad<DEG>& out, const float4* sh_row = nullptr)
{
    constexpr int K = ProjGrad<DEG>::K;
    // this view's gradient: written into out (first view) or added to it, one
    // finished value per parameter, so the sum over views is taken in view order
    float vmu[3] = {0.f, 0.f, 0.f}, vls[3] = {0.f, 0.f, 0.f}, vq[4] = {0.f, 0.f, 0.f, 0.f}, vlogit = 0.f;
    float* vcol = out.vcol;
    if (first) {
#pragma unroll
        for (int i = 0; i < 3 * K; ++i) vcol[i] = 0.0f;
    }

    if (radius > 0) {
        const float mx = __ldg(means + 3 * (int64_t)g), my = __ldg(means + 3 * (int64_t)g + 1),
                    mz = __ldg(means + 3 * (int64_t)g + 2);
        const float tx = fmaf(c.R[0], mx, fmaf(c.R[1], my, fmaf(c.R[2], mz, c.t[0])));
        const float ty = fmaf(c.R[3], mx, fmaf(c.R[4], my, fmaf(c.R[5], mz, c.t[1])));
        const float tz = fmaf(c.R[6], mx, fmaf(c.R[7], my, fmaf(c.R[8], mz, c.t[2])));
        const float4 q = __ldg(quats + g);
        const float qi = 1.0f / sqrtf(q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
        const float w = q.x * qi, x = q.y * qi, y = q.z * qi, z = q.w * qi;
        const float Rq[3][3] = {{1.f - 2.f * (y * y + z * z), 2.f * (x * y - w * z), 2.f * (x * z + w * y)},
                                {2.f * (x * y + w * z), 1.f - 2.f * (x * x + z * z), 2.f * (y * z - w * x)},
                                {2.f * (x * z - w * y), 2.f * (y * z + w * x), 1.f - 2.f * (x * x + y * y)}};
        float s[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) s[k] = expf(__ldg(log_scales + 3 * (int64_t)g + k));
        // RR = R_cw R(q); the camera-frame factor is WM = RR diag(s)
        float RR[3][3], WM[3][3];
#pragma unroll
        for (int r = 0; r < 3; ++r)
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                RR[r][k] = c.R[3 * r] * Rq[0][k] + c.R[3 * r + 1] * Rq[1][k] + c.R[3 * r + 2] * Rq[2][k];
                WM[r][k] = RR[r][k] * s[k];
            }
        const float iz = 1.0f / tz;
        const float rx = tx * iz, ry = ty * iz;
        const bool clx = rx > pc.limx_pos || rx < -pc.limx_neg;
        const bool cly = ry > pc.limy_pos || ry < -pc.limy_neg;
        const float lx = fminf(pc.limx_pos, fmaxf(-pc.limx_neg, rx));
        const float ly = fminf(pc.limy_pos, fmaxf(-pc.limy_neg, ry));
        const float j00 = c.fx * iz, j02 = -c.fx * lx * iz;
        const float j11 = c.fy * iz, j12 = -c.fy * ly * iz;
        float G0[3], G1[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            G0[k] = fmaf(j00, WM[0][k], j02 * WM[2][k]);
            G1[k] = fmaf(j11, WM[1][k], j12 * WM[2][k]);
        }
        const float a = G0[0] * G0[0] + G0[1] * G0[1] + G0[2] * G0[2] + 0.3f;
        const float b = G0[0] * G1[0] + G0[1] * G1[1] + G0[2] * G1[2];
        const float cc = G1[0] * G1[0] + G1[1] * G1[1] + G1[2] * G1[2] + 0.3f;
        const float idet = 1.0f / (a * cc - b * b);

        // upstream: record = (u, v, A, B, C | o, r, g | b, depth)
        const float4 v0 = __ldg(vsp), v1 = __ldg(vsp + 1), v2 = __ldg(vsp + 2);
        const float gu = v0.x, gv = v0.y, go = v1.y, gz = v2.y;
        float gA = v0.z, gB = v0.w, gC = v1.x;
        const float grgb[3] = {v1.z, v1.w, v2.x};

        // depth model of the soft split, when its gradient is given: g = conic b,
        // sigma_z^2 = szz - b . g, with b = G WM_2^T and szz = |WM_2|^2
        float vbu = 0.f, vbv = 0.f, vszz = 0.f;
        if (vdm) {
            const float4 vd = __ldg(vdm);
            const float bu = G0[0] * WM[2][0] + G0[1] * WM[2][1] + G0[2] * WM[2][2];
            const float bv = G1[0] * WM[2][0] + G1[1] * WM[2][1] + G1[2] * WM[2][2];
            const float szz = WM[2][0] * WM[2][0] + WM[2][1] * WM[2][1] + WM[2][2] * WM[2][2];
            const float cA = cc * idet, cB = -b * idet, cC = a * idet;
            const float dgu = cA * bu + cB * bv, dgv = cB * bu + cC * bv;
            const float var = szz - (bu * dgu + bv * dgv);
            const float vvar = var > 1e-12f ? 0.5f * vd.z / sqrtf(var) : 0.0f;  // sigma_z = sqrt(var)
            vszz = vvar;
            const float wgu = vd.x - vvar * bu, wgv = vd.y - vvar * bv;  // dL/dg, the variance path included
            vbu = cA * wgu + cB * wgv - vvar * dgu;
            vbv = cB * wgu + cC * wgv - vvar * dgv;
            gA += wgu * bu;  // dL/d conic = dL/dg b^T (the off-diagonal B appears twice)
            gB += wgu * bv + wgv * bu;
            gC += wgv * bv;
        }

        // conic (A, B, C) = (cc, -b, a) / det, det = a cc - b^2
        const float Qd = (gA * cc - gB * b + gC * a) * idet;  // L_conic = Q / det, Qd = Q / det
        const float ga = (gC - Qd * cc) * idet;
        const float gcc = (gA - Qd * a) * idet;
        const float gb = (2.0f * Qd * b - gB) * idet;
        // a = |G0|^2 + 0.3, b = G0 . G1, cc = |G1|^2 + 0.3
        float vG0[3], vG1[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            vG0[k] = 2.0f * ga * G0[k] + gb * G1[k] + vbu * WM[2][k];
            vG1[k] = 2.0f * gcc * G1[k] + gb * G0[k] + vbv * WM[2][k];
        }
        // G0 = j00 WM0 + j02 WM2, G1 = j11 WM1 + j12 WM2
        float vWM[3][3];
        float vj00 = 0.f, vj02 = 0.f, vj11 = 0.f, vj12 = 0.f;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            vWM[0][k] = j00 * vG0[k];
            vWM[1][k] = j11 * vG1[k];
            vWM[2][k] = j02 * vG0[k] + j12 * vG1[k] + vbu * G0[k] + vbv * G1[k] + 2.0f * vszz * WM[2][k];
            vj00 = fmaf(vG0[k], WM[0][k], vj00);
            vj02 = fmaf(vG0[k], WM[2][k], vj02);
            vj11 = fmaf(vG1[k], WM[1][k], vj11);
            vj12 = fmaf(vG1[k], WM[2][k], vj12);
        }
        // camera-frame mean: u = fx tx / tz + cx, v = fy ty / tz + cy, depth = tz;
        // j00 = fx / tz, j02 = -fx lx / tz with lx = tx / tz unless clamped (then constant)
        const float iz2 = iz * iz;
        float vtx = gu * c.fx * iz, vty = gv * c.fy * iz;
        float vtz = gz - (gu * c.fx * tx + gv * c.fy * ty) * iz2 - (vj00 * c.fx + vj11 * c.fy) * iz2;
        if (clx) {
            vtz += vj02 * c.fx * lx * iz2;
        } else {
            vtx -= vj02 * c.fx * iz2;
            vtz += vj02 * 2.0f * c.fx * lx * iz2;
        }
        if (cly) {
            vtz += vj12 * c.fy * ly * iz2;
        } else {
            vty -= vj12 * c.fy * iz2;
            vtz += vj12 * 2.0f * c.fy * ly * iz2;
        }
        // t = R_cw mu + t_cw
#pragma unroll
        for (int m = 0; m < 3; ++m) vmu[m] = c.R[m] * vtx + c.R[3 + m] * vty + c.R[6 + m] * vtz;
        // WM[r][k] = RR[r][k] s[k], s = exp(log_s)
        float vRq[3][3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            float vs = 0.0f;
#pragma unroll
            for (int r = 0; r < 3; ++r) vs = fmaf(vWM[r][k], RR[r][k], vs);
            vls[k] = vs * s[k];
#pragma unroll
            for (int m = 0; m < 3; ++m)
                vRq[m][k] = (c.R[m] * vWM[0][k] + c.R[3 + m] * vWM[1][k] + c.R[6 + m] * vWM[2][k]) * s[k];
        }
        // R(q) of the unit quaternion (w, x, y, z)
        const float vw = 2.f * (-z * vRq[0][1] + y * vRq[0][2] + z * vRq[1][0] - x * vRq[1][2] - y * vRq[2][0] +
                                x * vRq[2][1]);
        const float vx = 2.f * (y * vRq[0][1] + z * vRq[0][2] + y * vRq[1][0] - 2.f * x * vRq[1][1] - w * vRq[1][2] +
                                z * vRq[2][0] + w * vRq[2][1] - 2.f * x * vRq[2][2]);
        const float vy = 2.f * (-2.f * y * vRq[0][0] + x * vRq[0][1] + w * vRq[0][2] + x * vRq[1][0] +
                                z * vRq[1][2] - w * vRq[2][0] + z * vRq[2][1] - 2.f * y * vRq[2][2]);
        const float vz = 2.f * (-2.f * z * vRq[0][0] - w * vRq[0][1] + x * vRq[0][2] + w * vRq[1][0] -
                                2.f * z * vRq[1][1] + y * vRq[1][2] + x * vRq[2][0] + y * vRq[2][1]);
        // unit quaternion = q / |q|: project out the radial part
        const float dot = vw * w + vx * x + vy * y + vz * z;
        vq[0] = (vw - dot * w) * qi;
        vq[1] = (vx - dot * x) * qi;
        vq[2] = (vy - dot * y) * qi;
        vq[3] = (vz - dot * z) * qi;
        // opacity = sigmoid(logit)
        const float op = 1.0f / (1.0f + expf(-__ldg(logits + g)));
        vlogit = go * op * (1.0f - op);
        // colour
        if (DEG < 0) {
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) add_or_set(vcol[ch], grgb[ch], first);
        } else {
            float dx = mx - pc.cpx, dy = my - pc.cpy, dz = mz - pc.cpz;
            const float dn = 1.0f / sqrtf(dx * dx + dy * dy + dz * dz);
            dx *= dn; dy *= dn; dz *= dn;
            float Y[16];
            sh_basis<DEG>(dx, dy, dz, Y);
            float cf[3 * K];
            const float* src = colors + (int64_t)g * (3 * K);
            if ((3 * K) % 4 == 0) {
                const float4* src4 = reinterpret_cast<const float4*>(src);
#pragma unroll
                for (int v4 = 0; v4 < 3 * K / 4; ++v4) {
                    const float4 e = sh_row ? sh_row[v4] : __ldg(src4 + v4);
                    cf[4 * v4] = e.x; cf[4 * v4 + 1] = e.y; cf[4 * v4 + 2] = e.z; cf[4 * v4 + 3] = e.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 3 * K; ++i) cf[i] = __ldg(src + i);
            }
            // rgb = max(0, sum_k Y_k c_k + 0.5): no gradient where the clamp holds
            float gch[3];
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) {
                float accum = 0.5f;
#pragma unroll
                for (int k = 0; k < K; ++k) accum = fmaf(Y[k], cf[3 * k + ch], accum);
                gch[ch] = accum > 0.0f ? grgb[ch] : 0.0f;
            }
            float vY[16];
#pragma unroll
            for (int k = 0; k < K; ++k) {
                vY[k] = gch[0] * cf[3 * k] + gch[1] * cf[3 * k + 1] + gch[2] * cf[3 * k + 2];
#pragma unroll
                for (int ch = 0; ch < 3; ++ch) add_or_set(vcol[3 * k + ch], gch[ch] * Y[k], first);
            }
            // direction d = n / |n|, n = mu - camera centre
            float gx, gy, gzd;
            sh_basis_vjp<DEG>(dx, dy, dz, vY, gx, gy, gzd);
            const float dd = gx * dx + gy * dy + gzd * dz;
            vmu[0] += (gx - dd * dx) * dn;
            vmu[1] += (gy - dd * dy) * dn;
            vmu[2] += (gzd - dd * dz) * dn;
        }
    }

#pragma unroll
    for (int k = 0; k < 3; ++k) {
        add_or_set(out.vmu[k], vmu[k], first);
        add_or_set(out.vls[k], vls[k], first);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) add_or_set(out.vq[k], vq[k], first);
    add_or_set(out.vlogit, vlogit, first);
}

template <int DEG>
__device__ __forceinline__ void store_grad(int g, const ProjGrad<DEG>& G, bool acc, float* __restrict__ v_means,
                                           float* __restrict__ v_log_scales, float4* __restrict__ v_quats,
                                           float* __restrict__ v_logits, float* __restrict__ v_colors)
{
    constexpr int K = ProjGrad<DEG>::K;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        put(v_means + 3 * (int64_t)g + k, G.vmu[k], acc);
        put(v_log_scales + 3 * (int64_t)g + k, G.vls[k], acc);
    }
    {
        float4 o = make_float4(G.vq[0], G.vq[1], G.vq[2], G.vq[3]);
        if (acc) {
            const float4 p = v_quats[g];
            o = make_float4(__fadd_rn(p.x, o.x), __fadd_rn(p.y, o.y), __fadd_rn(p.z, o.z), __fadd_rn(p.w, o.w));
        }
        v_quats[g] = o;
    }
    put(v_logits + g, G.vlogit, acc);
    float* dst = v_colors + (int64_t)g * (3 * K);
    if ((3 * K) % 4 == 0) {
        float4* dst4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int v4 = 0; v4 < 3 * K / 4; ++v4) {
            float4 o = make_float4(G.vcol[4 * v4], G.vcol[4 * v4 + 1], G.vcol[4 * v4 + 2], G.vcol[4 * v4 + 3]);
            if (acc) {
                const float4 p = dst4[v4];
                o = make_float4(__fadd_rn(p.x, o.x), __fadd_rn(p.y, o.y), __fadd_rn(p.z, o.z), __fadd_rn(p.w, o.w));
            }
            dst4[v4] = o;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 3 * K; ++i) put(dst + i, G.vcol[i], acc);
    }
}

template <int DEG>
__global__ void __launch_bounds__(256)
k_project_bwd(Cam c, ProjConsts pc, int N, const float* __restrict__ means, const float* __restrict__ log_scales,
              const float4* __restrict__ quats, const float* __restrict__ logits, const float* __restrict__ colors,
              const int32_t* __restrict__ radii, const float4* __restrict__ v_splats,
              const float4* __restrict__ v_depth_model, bool acc, float* __restrict__ v_means,
              float* __restrict__ v_log_scales, float4* __restrict__ v_quats, float* __restrict__ v_logits,
              float* __restrict__ v_colors)
{
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= N) return;
    ProjGrad<DEG> G;
    project_bwd_gaussian<DEG>(c, pc, g, means, log_scales, quats, logits, colors, __ldg(radii + g),
                              v_splats + 3 * (int64_t)g, v_depth_model ? v_depth_model + g : nullptr, true, G);
    store_grad<DEG>(g, G, acc, v_means, v_log_scales, v_quats, v_logits, v_colors);
}

// The views of a batch summed in registers (in view order, the order in which
// per-view calls with accumulation would add them), written once.
template <int DEG>
__global__ void __launch_bounds__(PROJ_THREADS)
k_project_bwd_views(ViewBatch vb, int N, const float* __restrict__ means, const float* __restrict__ log_scales,
                    const float4* __restrict__ quats, const float* __restrict__ logits,
                    const float* __restrict__ colors, const int32_t* __restrict__ radii,
                    const float4* __restrict__ v_splats, const float4* __restrict__ v_depth_model, bool acc,
                    float* __restrict__ v_means,
                    float* __restrict__ v_log_scales, float4* __restrict__ v_quats, float* __restrict__ v_logits,
                    float* __restrict__ v_colors)
{
    // the SH rows of the CTA's Gaussians, staged once for every view
    constexpr int ROW4 = ShStage<DEG>::ROW4;
    __shared__ float4 s_sh[ROW4 ? PROJ_THREADS * ShStage<DEG>::STRIDE : 1];
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    if constexpr (ROW4 > 0) {
        stage_sh_rows<DEG>(colors, blockIdx.x * blockDim.x, N, s_sh);
        __syncthreads();
    }
    if (g >= N) return;
    ProjGrad<DEG> total;
    for (int v = 0; v < vb.n; ++v) {
        const int64_t i = (int64_t)v * N + g;
        project_bwd_gaussian<DEG>(vb.cam[v], vb.pc[v], g, means, log_scales, quats, logits, colors,
                                  __ldg(radii + i), v_splats + 3 * i, v_depth_model ? v_depth_model + i : nullptr,
                                  v == 0, total, ROW4 ? s_sh + threadIdx.x * ShStage<DEG>::STRIDE : nullptr);
    }
    store_grad<DEG>(g, total, acc, v_means, v_log_scales, v_quats, v_logits, v_colors);
}

}  // namespace

cudaError_t project_bwd(const Cam& c, int sh_degree, int N, const float* means, const float* log_scales,
                        const float* quats, const float* logits, const float* colors, const int32_t* radii,
                        const float* v_splats, const float* v_depth_model, bool accumulate, float* v_means,
                        float* v_log_scales, float* v_quats, float* v_logits, float* v_colors, cudaStream_t s)
{
    if (N <= 0) return cudaSuccess;
    const ProjConsts pc = make_proj_consts(c);
    const int grid = (N + 255) / 256;
    auto* q4 = reinterpret_cast<const float4*>(quats);
    auto* vs4 = reinterpret_cast<const float4*>(v_splats);
    auto* vd4 = reinterpret_cast<const float4*>(v_depth_model);
    auto* vq4 = reinterpret_cast<float4*>(v_quats);
#define GM_PROJ_BWD(D)                                                                                      \
    k_project_bwd<D><<<grid, 256, 0, s>>>(c, pc, N, means, log_scales, q4, logits, colors, radii, vs4, vd4,        \
                                          accumulate, v_means, v_log_scales, vq4, v_logits, v_colors)
    switch (sh_degree) {
        case -1: GM_PROJ_BWD(-1); break;
        case 0: GM_PROJ_BWD(0); break;
        case 1: GM_PROJ_BWD(1); break;
        case 2: GM_PROJ_BWD(2); break;
        case 3: GM_PROJ_BWD(3); break;
        default: return cudaErrorInvalidValue;
    }
#undef GM_PROJ_BWD
    return cudaGetLastError();
}

cudaError_t project_bwd_views(const Cam* cams, int V, int sh_degree, int N, const float* means,
                              const float* log_scales, const float* quats, const float* logits, const float* colors,
                              const int32_t* radii, const float* v_splats, const float* v_depth_model,
                              bool accumulate, float* v_means, float* v_log_scales, float* v_quats, float* v_logits,
                              float* v_colors, cudaStream_t s)
{
    if (N <= 0) return cudaSuccess;
    const int grid = (N + PROJ_THREADS - 1) / PROJ_THREADS;  // 128-thread CTAs: the SH-3 body is register heavy
    auto* q4 = reinterpret_cast<const float4*>(quats);
    auto* vq4 = reinterpret_cast<float4*>(v_quats);
    for (int v0 = 0; v0 < V; v0 += MAX_VIEWS) {
        ViewBatch vb;
        vb.n = std::min(MAX_VIEWS, V - v0);
        for (int v = 0; v < vb.n; ++v) {
            vb.cam[v] = cams[v0 + v];
            vb.pc[v] = make_proj_consts(cams[v0 + v]);
        }
        const int64_t off = (int64_t)v0 * N;
        auto* vs4 = reinterpret_cast<const float4*>(v_splats + 12 * off);
        auto* vd4 = v_depth_model ? reinterpret_cast<const float4*>(v_depth_model + 4 * off) : nullptr;
        const bool acc = accumulate || v0 > 0;  // later batches add to the earlier ones
#define GM_PROJ_BWD_V(D)                                                                                          \
    k_project_bwd_views<D><<<grid, PROJ_THREADS, 0, s>>>(vb, N, means, log_scales, q4, logits, colors, radii + off, vs4,   \
                                                vd4, acc, v_means, v_log_scales, vq4, v_logits, v_colors)
        switch (sh_degree) {
            case -1: GM_PROJ_BWD_V(-1); break;
            case 0: GM_PROJ_BWD_V(0); break;
            case 1: GM_PROJ_BWD_V(1); break;
            case 2: GM_PROJ_BWD_V(2); break;
            case 3: GM_PROJ_BWD_V(3); break;
            default: return cudaErrorInvalidValue;
        }
#undef GM_PROJ_BWD_V
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gm

// Projection constants and the real SH basis, shared by the projection
// (gm_gauss.cu) and its backward (gm_project_bwd.cu).
#pragma once

#include "gm_internal.cuh"

namespace gm {

// Real spherical harmonics, index l*l + l + m (m = -l..l), orthonormal on the
// sphere, without the Condon-Shortley phase: e.g. Y_1,-1 = sqrt(3/4pi) y.
constexpr float SH_C0 = 0.28209479177387814f;   // 1/(2 sqrt(pi))
constexpr float SH_C1 = 0.4886025119029199f;    // sqrt(3/(4 pi))
constexpr float SH_C2a = 1.0925484305920792f;   // sqrt(15/pi)/2
constexpr float SH_C2c = 0.31539156525252005f;  // sqrt(5/pi)/4
constexpr float SH_C2e = 0.5462742152960396f;   // sqrt(15/pi)/4
constexpr float SH_C3a = 0.5900435899266435f;   // sqrt(35/(2 pi))/4
constexpr float SH_C3b = 2.890611442640554f;    // sqrt(105/pi)/2
constexpr float SH_C3c = 0.4570457994644658f;   // sqrt(21/(2 pi))/4
constexpr float SH_C3d = 0.3731763325901154f;   // sqrt(7/pi)/4
constexpr float SH_C3f = 1.445305721320277f;    // sqrt(105/pi)/4

template <int DEG>
__device__ __forceinline__ void sh_basis(float x, float y, float z, float* Y)
{
    Y[0] = SH_C0;
    if (DEG >= 1) {
        Y[1] = SH_C1 * y;
        Y[2] = SH_C1 * z;
        Y[3] = SH_C1 * x;
    }
    if (DEG >= 2) {
        const float xx = x * x, yy = y * y, zz = z * z;
        Y[4] = SH_C2a * x * y;
        Y[5] = SH_C2a * y * z;
        Y[6] = SH_C2c * (3.0f * zz - 1.0f);
        Y[7] = SH_C2a * x * z;
        Y[8] = SH_C2e * (xx - yy);
        if (DEG >= 3) {
            Y[9] = SH_C3a * y * (3.0f * xx - yy);
            Y[10] = SH_C3b * x * y * z;
            Y[11] = SH_C3c * y * (5.0f * zz - 1.0f);
            Y[12] = SH_C3d * z * (5.0f * zz - 3.0f);
            Y[13] = SH_C3c * x * (5.0f * zz - 1.0f);
            Y[14] = SH_C3f * z * (xx - yy);
            Y[15] = SH_C3a * x * (xx - 3.0f * yy);
        }
    }
}

struct ProjConsts {
    float limx_pos, limx_neg, limy_pos, limy_neg;  // clamp of tx/tz, ty/tz
    float cpx, cpy, cpz;                           // camera centre in world space
};

// The direction t / t_z used in the Jacobian is clamped to 1.3 x the tangent
// of the half field of view on each side of the principal point.
inline ProjConsts make_proj_consts(const Cam& c)
{
    ProjConsts pc;
    pc.limx_pos = 1.3f * ((float)c.W - c.cx) / c.fx;
    pc.limx_neg = 1.3f * c.cx / c.fx;
    pc.limy_pos = 1.3f * ((float)c.H - c.cy) / c.fy;
    pc.limy_neg = 1.3f * c.cy / c.fy;
    // camera centre = -R^T t
    pc.cpx = -(c.R[0] * c.t[0] + c.R[3] * c.t[1] + c.R[6] * c.t[2]);
    pc.cpy = -(c.R[1] * c.t[0] + c.R[4] * c.t[1] + c.R[7] * c.t[2]);
    pc.cpz = -(c.R[2] * c.t[0] + c.R[5] * c.t[1] + c.R[8] * c.t[2]);
    return pc;
}

// Cameras of one batched launch (passed by value as a kernel parameter).
// SH rows of 3 (DEG + 1)^2 floats that are whole float4s (degrees 1 and 3) are
// staged per CTA in shared memory: read from DRAM by coalesced 16-byte loads
// of the CTA's contiguous rows, issued before any other work, and kept at an
// odd stride of float4s so that each lane's reads of its own row are free of
// bank conflicts.
template <int DEG>
struct ShStage {
    static constexpr int K = DEG < 0 ? 1 : (DEG + 1) * (DEG + 1);
    static constexpr int ROW4 = (DEG >= 1 && (3 * K) % 4 == 0) ? 3 * K / 4 : 0;  // float4s a row; 0: not staged
    static constexpr int STRIDE = ROW4 % 2 ? ROW4 : ROW4 + 1;                     // float4s between staged rows
};

constexpr int PROJ_THREADS = 128;

// Stages the SH rows of Gaussians [g0, g0 + PROJ_THREADS) (those below N) in
// sh; every thread of the CTA calls it, then waits at a barrier.
template <int DEG>
__device__ __forceinline__ void stage_sh_rows(const float* __restrict__ colors, int g0, int N, float4* sh)
{
    constexpr int ROW4 = ShStage<DEG>::ROW4, STRIDE = ShStage<DEG>::STRIDE;
    const int rows = min(PROJ_THREADS, N - g0);
    const float4* __restrict__ src = reinterpret_cast<const float4*>(colors) + (int64_t)g0 * ROW4;
    float4 v[ROW4 ? ROW4 : 1];
#pragma unroll
    for (int m = 0; m < ROW4; ++m) {
        const int i = m * PROJ_THREADS + threadIdx.x;
        if (i < rows * ROW4) v[m] = __ldg(src + i);
    }
#pragma unroll
    for (int m = 0; m < ROW4; ++m) {
        const int i = m * PROJ_THREADS + threadIdx.x;
        if (i < rows * ROW4) sh[(i / ROW4) * STRIDE + i % ROW4] = v[m];
    }
}

constexpr int MAX_VIEWS = 8;
struct ViewBatch {
    Cam cam[MAX_VIEWS];
    ProjConsts pc[MAX_VIEWS];
    int n;
};

}  // namespace gm

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
constexpr int MAX_VIEWS = 8;
struct ViewBatch {
    Cam cam[MAX_VIEWS];
    ProjConsts pc[MAX_VIEWS];
    int n;
};

}  // namespace gm

"""Pins of the oracle's projection gradient (the projection / SH backward that
completes the Gaussian training gradients; page "A Lightweight and
Differentiable Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Hybrid
rendering: everything is differentiable; projection and SH adapted from
gsplat).  The oracle differentiates its own double-precision projection by
central differences; these tests fix its scale, sign and chain structure with
closed forms and invariants of the projection map."""

import math

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes

MEAN, LOGS, QUAT, LOGIT, COLOR = 0, 3, 6, 10, 11
F_MX, F_MY, F_CA, F_CB, F_CC, F_OP, F_R, F_G, F_B, F_Z = range(10)
SH_C0 = 0.5 / math.sqrt(math.pi)
SH_C1 = math.sqrt(3.0 / (4.0 * math.pi))


def cam_identity(w=128, h=128, f=100.0, cx=64.0, cy=64.0):
    return scenes.Camera(w, h, f, f, cx, cy, scenes.NEAR, scenes.FAR,
                         np.eye(3, dtype=np.float32), np.zeros(3, np.float32))


def one(mean, log_s=(-2.0, -2.0, -2.0), quat=(1.0, 0.0, 0.0, 0.0), logit=0.3, colors=None, deg=-1):
    if colors is None:
        colors = np.full((1, 3), 0.4) if deg < 0 else np.zeros((1, (deg + 1) ** 2, 3))
    return scenes.Gaussians(np.asarray([mean], np.float32), np.asarray([log_s], np.float32),
                            np.asarray([quat], np.float32), np.asarray([logit], np.float32),
                            np.asarray(colors, np.float32).reshape(1, -1), deg)


def grad(orc, cam, g, field, params, h=1e-3, v=None):
    if v is None:
        v = np.zeros((1, 12), np.float32)
        v[0, field] = 1.0
    params = np.asarray(params, np.int32)
    gr, st = orc.project_fd(cam, g, v, np.zeros(len(params), np.int32), params, np.full(len(params), h))
    return gr, st


def test_conic_wrt_log_scale_closed_form(orc):
    # identity rotation on the optical axis: Sigma2 = diag((f s_k / z)^2 + 0.3), b = 0, so
    # conic a = 1 / ((f s0 / z)^2 + 0.3) and d a / d log s0 = -2 k^2 / (k^2 + 0.3)^2
    cam = cam_identity()
    z, ls = 5.0, (-2.0, -1.5, -1.0)
    g = one((0.0, 0.0, z), log_s=ls)
    k0, k1 = (100.0 * math.exp(ls[0]) / z) ** 2, (100.0 * math.exp(ls[1]) / z) ** 2
    gr, st = grad(orc, cam, g, F_CA, [LOGS, LOGS + 1, LOGS + 2])
    assert (st == 0).all()
    np.testing.assert_allclose(gr[0], -2.0 * k0 / (k0 + 0.3) ** 2, rtol=1e-7)
    np.testing.assert_allclose(gr[1:], 0.0, atol=1e-9)
    gr, st = grad(orc, cam, g, F_CC, [LOGS, LOGS + 1, LOGS + 2])
    np.testing.assert_allclose(gr[1], -2.0 * k1 / (k1 + 0.3) ** 2, rtol=1e-7)
    np.testing.assert_allclose(gr[[0, 2]], 0.0, atol=1e-9)


def test_mean2d_and_depth_wrt_mean(orc):
    # u = fx x / z + cx, v = fy y / z + cy, depth = z (world = camera frame)
    cam = cam_identity()
    x, y, z = 0.5, -0.3, 5.0
    g = one((x, y, z))
    gu, st = grad(orc, cam, g, F_MX, [MEAN, MEAN + 1, MEAN + 2])
    assert (st == 0).all()
    np.testing.assert_allclose(gu, [100.0 / z, 0.0, -100.0 * x / z ** 2], rtol=1e-7, atol=1e-9)
    gv, _ = grad(orc, cam, g, F_MY, [MEAN, MEAN + 1, MEAN + 2])
    np.testing.assert_allclose(gv, [0.0, 100.0 / z, -100.0 * y / z ** 2], rtol=1e-7, atol=1e-9)
    gz, _ = grad(orc, cam, g, F_Z, [MEAN, MEAN + 1, MEAN + 2])
    np.testing.assert_allclose(gz, [0.0, 0.0, 1.0], rtol=1e-9, atol=1e-9)


def test_opacity_wrt_logit(orc):
    cam = cam_identity()
    for logit in (-2.0, 0.0, 1.7):
        g = one((0.1, 0.2, 4.0), logit=logit)
        o = 1.0 / (1.0 + math.exp(-float(np.float32(logit))))
        gr, st = grad(orc, cam, g, F_OP, [LOGIT])
        assert st[0] == 0
        np.testing.assert_allclose(gr[0], o * (1.0 - o), rtol=1e-8)


def test_colour_coefficients_are_linear(orc):
    # degree 0: r = C0 c_00 + 0.5; degree 1 with only c_{1,0} (index 2, Y = C1 d_z) set:
    # r = 0.5 + C1 d_z c, so d r / d c = C1 d_z and d r / d mean = C1 c (e_z - d_z d) / |mean|
    cam = cam_identity()
    g = one((0.2, 0.1, 4.0), deg=0, colors=[[0.3, 0.1, -0.2]])
    gr, st = grad(orc, cam, g, F_R, [COLOR, COLOR + 1, COLOR + 2])
    assert (st == 0).all()
    np.testing.assert_allclose(gr, [SH_C0, 0.0, 0.0], rtol=1e-8, atol=1e-10)
    mu = np.array([0.6, -0.4, 3.0])
    col = np.zeros((4, 3))
    col[2, 0] = 0.7
    g = one(tuple(mu), deg=1, colors=col)
    d = mu.astype(np.float32).astype(np.float64)
    n = np.linalg.norm(d)
    d /= n
    gr, st = grad(orc, cam, g, F_R, [COLOR + 3 * 2, MEAN, MEAN + 1, MEAN + 2])
    assert (st == 0).all()
    c = float(np.float32(0.7))
    np.testing.assert_allclose(gr[0], SH_C1 * d[2], rtol=1e-8)
    np.testing.assert_allclose(gr[1:], SH_C1 * c * (np.array([0.0, 0.0, 1.0]) - d[2] * d) / n, rtol=1e-6,
                               atol=1e-9)


def test_quaternion_gradient_invariants(orc):
    # the record depends on q only through q / |q|: sum_j q_j dL/dq_j = 0; an isotropic
    # Gaussian does not depend on q at all
    cam = cam_identity()
    rng = np.random.default_rng(7)
    v = rng.normal(size=(1, 12)).astype(np.float32)
    v[0, 10:] = 0.0
    for _ in range(4):
        q = rng.normal(size=4)
        g = one(tuple(rng.uniform(-0.5, 0.5, 2)) + (4.0,), log_s=tuple(rng.normal(-2.5, 0.4, 3)), quat=tuple(q))
        gq, st = grad(orc, cam, g, None, [QUAT, QUAT + 1, QUAT + 2, QUAT + 3], v=v)
        assert (st == 0).all()
        assert abs(float(np.dot(gq, q.astype(np.float32)))) <= 1e-6 * np.abs(gq).max() * np.linalg.norm(q)
        assert np.abs(gq).max() > 1e-3  # anisotropic: q matters
        g = one((0.1, 0.0, 4.0), log_s=(-2.2, -2.2, -2.2), quat=tuple(q))
        gq, st = grad(orc, cam, g, None, [QUAT, QUAT + 1, QUAT + 2, QUAT + 3], v=v)
        np.testing.assert_allclose(gq, 0.0, atol=1e-6)


def test_clamped_jacobian_direction_freezes_conic(orc):
    # beyond 1.3 x the half field of view the Jacobian is evaluated at the clamped
    # direction, so the conic no longer depends on the mean's x, while u still does
    cam = cam_identity()
    x = 0.64 * 1.3 * 4.0 * 1.6  # tx/tz = 1.3 * 0.64 * 1.6: well past the clamp
    g = one((x, 0.0, 4.0), log_s=(0.6, 0.6, 0.6))  # large enough to reach the image
    ga, st = grad(orc, cam, g, F_CA, [MEAN])
    assert st[0] == 0
    np.testing.assert_allclose(ga[0], 0.0, atol=1e-12)
    gu, st = grad(orc, cam, g, F_MX, [MEAN])
    np.testing.assert_allclose(gu[0], 100.0 / 4.0, rtol=1e-7)
    # inside the clamp the same conic gradient is not zero
    g = one((0.3, 0.0, 4.0), log_s=(0.6, -1.0, -2.0), quat=(0.9, 0.2, 0.3, 0.1))
    ga, st = grad(orc, cam, g, F_CA, [MEAN])
    assert st[0] == 0 and abs(ga[0]) > 1e-6


def test_decision_boundaries_are_reported(orc):
    cam = cam_identity()
    # behind the camera: culled throughout, zero gradient
    g = one((0.0, 0.0, -3.0))
    gr, st = grad(orc, cam, g, F_MX, [MEAN, LOGS, QUAT, LOGIT])
    assert (st == 0).all() and (gr == 0).all()
    # on the near plane: culled on one side only
    g = one((0.0, 0.0, scenes.NEAR))
    gr, st = grad(orc, cam, g, F_Z, [MEAN + 2], h=1e-3)
    assert st[0] == 1
    # exactly at the clamp of the Jacobian direction
    lim = 1.3 * 64.0 / 100.0
    g = one((lim * 4.0, 0.0, 4.0), log_s=(0.6, 0.6, 0.6))
    gr, st = grad(orc, cam, g, F_CA, [MEAN], h=1e-3)
    assert st[0] == 1
    # a colour clamped at zero in one direction of the step
    g = one((0.0, 0.0, 4.0), deg=0, colors=[[-0.5 / SH_C0, 0.2, 0.2]])
    gr, st = grad(orc, cam, g, F_R, [COLOR], h=1e-3)
    assert st[0] == 1


def test_unknown_parameter_is_unused(orc):
    cam = cam_identity()
    g = one((0.0, 0.0, 4.0))
    gr, st = grad(orc, cam, g, F_MX, [orc.proj_nparams(-1), -1])
    assert (st == 5).all()


def test_depth_model_gradient_closed_form(orc):
    # identity rotation on the optical axis: Sigma_c = diag(s^2), J e_z = 0, so g = 0 and
    # sigma_z = s_2: d sigma_z / d log s = (0, 0, s_2); d g_u / d log s_0 = 0
    cam = cam_identity()
    ls = (-2.0, -1.5, -1.0)
    g = one((0.0, 0.0, 5.0), log_s=ls)
    v = np.zeros((1, 12), np.float32)
    vd = np.zeros((1, 4), np.float32)
    vd[0, 2] = 1.0
    gr, st = orc.project_fd(cam, g, v, np.zeros(3, np.int32), np.array([LOGS, LOGS + 1, LOGS + 2], np.int32),
                            np.full(3, 1e-3), v_depth_model=vd)
    assert (st == 0).all()
    np.testing.assert_allclose(gr, [0.0, 0.0, float(np.exp(np.float32(ls[2])))], rtol=1e-7, atol=1e-9)
    # off axis the slope g_u = Sigma_uv,z / (Sigma_uv + 0.3) grows with x: d g_u / d mean_x < 0
    # for an isotropic Gaussian (j02 = -f x / z^2 turns negative)
    g = one((0.2, 0.0, 5.0), log_s=(-1.0, -1.0, -1.0))
    vd[0] = [1.0, 0.0, 0.0, 0.0]
    gr, st = orc.project_fd(cam, g, v, np.zeros(1, np.int32), np.array([MEAN], np.int32), np.full(1, 1e-4),
                            v_depth_model=vd)
    assert st[0] == 0 and gr[0] < 0

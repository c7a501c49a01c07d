"""Pins of the oracle's Gaussian steps: EWA projection, SH colour, tile bins and
the sort (page "A Lightweight and Differentiable Renderer for Joint Mesh and 3D
Gaussian Splat Scenes", Hybrid rendering; the projection, SH and tile sorting
kernels it says are adapted from gsplat; Limitations: centre-depth order; the
stored parameterisation of the "Gaussian splatting reference" page, Output
writing)."""

import json
import math
import os

import numpy as np
import pytest
from scipy.spatial.transform import Rotation
from scipy.special import expit, sph_harm_y

from differentiable_hybrid_mesh_tile_b300 import scenes

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


def cam_identity(w, h, f, cx, cy):
    return scenes.Camera(w, h, f, f, cx, cy, scenes.NEAR, scenes.FAR,
                         np.eye(3, dtype=np.float32), np.zeros(3, np.float32))


def gaussians(means, log_scales, quats, logits, colors, deg=-1):
    return scenes.Gaussians(np.asarray(means, np.float32), np.asarray(log_scales, np.float32),
                            np.asarray(quats, np.float32), np.asarray(logits, np.float32),
                            np.asarray(colors, np.float32), deg)


def test_isotropic_on_axis_closed_form(orc):
    cam = cam_identity(64, 48, 50.0, 32.0, 24.0)
    rng = np.random.default_rng(3)
    n = 6
    z = np.array([1.0, 2.0, 3.5, 5.0, 0.5, 8.0])
    s = np.array([0.01, 0.05, 0.2, 0.03, 0.004, 0.5])
    means = np.stack([np.zeros(n), np.zeros(n), z], 1)
    q = rng.normal(size=(n, 4))
    g = gaussians(means, np.log(s)[:, None].repeat(3, 1), q, rng.normal(size=n), rng.uniform(size=(n, 3)))
    splats, radii, _, _ = orc.project(cam, g)
    var = (50.0 * s / z) ** 2 + 0.3
    np.testing.assert_allclose(splats[:, 0], 32.0, atol=1e-6)
    np.testing.assert_allclose(splats[:, 1], 24.0, atol=1e-6)
    np.testing.assert_allclose(splats[:, 2], 1.0 / var, rtol=1e-6)
    np.testing.assert_allclose(splats[:, 3], 0.0, atol=1e-6 / var.min())
    np.testing.assert_allclose(splats[:, 4], 1.0 / var, rtol=1e-6)
    np.testing.assert_allclose(splats[:, 9], z, rtol=1e-7)
    np.testing.assert_array_equal(radii, np.ceil(3.0 * np.sqrt(var)).astype(np.int32))
    np.testing.assert_allclose(splats[:, 5], expit(g.logits.astype(np.float64)), rtol=1e-6)


def _sigma2_reference(cam, mean, log_s, q_wxyz):
    """2D covariance from an independent route: scipy's rotation of the
    quaternion and the Jacobian of the pinhole map by central differences."""
    R = cam.R.astype(np.float64)
    t = cam.t.astype(np.float64)
    rot = Rotation.from_quat([q_wxyz[1], q_wxyz[2], q_wxyz[3], q_wxyz[0]]).as_matrix()
    S = np.diag(np.exp(np.asarray(log_s, np.float64)))
    cov = rot @ S @ S @ rot.T
    X = R @ np.asarray(mean, np.float64) + t

    def proj(Y):
        return np.array([cam.fx * Y[0] / Y[2] + cam.cx, cam.fy * Y[1] / Y[2] + cam.cy])

    J = np.zeros((2, 3))
    for k in range(3):
        e = np.zeros(3)
        e[k] = 1e-6 * max(1.0, abs(X[k]))
        J[:, k] = (proj(X + e) - proj(X - e)) / (2 * e[k])
    S2 = J @ (R @ cov @ R.T) @ J.T + 0.3 * np.eye(2)
    return S2, proj(X), X[2]


def test_anisotropic_matches_fd_jacobian_and_scipy_rotation(orc):
    cam = scenes.look_at((0.7, -0.4, 3.2), (0.1, 0, 0), 160, 120, 140.0, 130.0, 77.0, 61.0)
    rng = np.random.default_rng(11)
    n = 200
    means = rng.uniform(-0.8, 0.8, size=(n, 3))
    ls = rng.normal(-3.0, 0.7, size=(n, 3))
    q = rng.normal(size=(n, 4))
    g = gaussians(means, ls, q, rng.normal(size=n), rng.uniform(size=(n, 3)))
    splats, radii, touched, _ = orc.project(cam, g)
    checked = 0
    for k in range(n):
        S2, m2, z = _sigma2_reference(cam, g.means[k], g.log_scales[k], g.quats[k].astype(np.float64))
        if radii[k] == 0:
            continue
        checked += 1
        conic = np.linalg.inv(S2)
        np.testing.assert_allclose(splats[k, 0:2], m2, rtol=1e-6, atol=1e-4)
        scale = math.sqrt(conic[0, 0] * conic[1, 1])
        np.testing.assert_allclose(splats[k, [2, 3, 4]], [conic[0, 0], conic[0, 1], conic[1, 1]],
                                   atol=2e-6 * scale)
        np.testing.assert_allclose(splats[k, 9], z, rtol=1e-7)
        lam = np.linalg.eigvalsh(S2).max()
        ext = 3.0 * math.sqrt(lam)
        if abs(ext - round(ext)) > 1e-4:
            assert radii[k] == math.ceil(ext)
    assert checked > 150


def test_jacobian_clamp_beyond_field_of_view(orc):
    """Past 1.3x the tangent of the half field of view the Jacobian is taken at
    the clamp: a Gaussian beyond it gets the conic of the same Gaussian placed
    on the clamp direction at the same depth; one inside the clamp does not."""
    cam = cam_identity(100, 80, 50.0, 50.0, 40.0)
    z = 2.0
    lim = 1.3 * (cam.width - cam.cx) / cam.fx
    xs = [1.5 * lim * z, lim * z, 0.8 * lim * z]
    means = [[x, 0.1, z] for x in xs]
    q = [0.9, 0.2, -0.3, 0.1]
    ls = [-0.4, -0.9, -0.6]
    g = gaussians(means, [ls] * 3, [q] * 3, [0.0] * 3, [[0.5] * 3] * 3)
    splats, radii, _, _ = orc.project(cam, g)
    assert np.all(radii > 0)
    conics = splats[:, [2, 3, 4]].astype(np.float64)
    np.testing.assert_allclose(conics[0], conics[1], rtol=1e-6)
    assert np.abs(conics[2] - conics[1]).max() > 1e-3 * np.abs(conics[1]).max()
    # the one on the clamp direction is unclamped: it matches the independent route
    S2, _, _ = _sigma2_reference(cam, g.means[1], g.log_scales[1], g.quats[1].astype(np.float64))
    inv = np.linalg.inv(S2)
    np.testing.assert_allclose(conics[1], [inv[0, 0], inv[0, 1], inv[1, 1]], rtol=1e-5, atol=1e-9)


def test_projection_culls(orc):
    cam = cam_identity(64, 64, 64.0, 32.0, 32.0)
    means = [[0, 0, 0.005], [0, 0, -1.0], [50.0, 0, 1.0], [0, 0, 2.0]]
    g = gaussians(means, [[-3.0] * 3] * 4, [[1, 0, 0, 0]] * 4, [0.0] * 4, [[0.5] * 3] * 4)
    splats, radii, touched, _ = orc.project(cam, g)
    assert radii.tolist()[:3] == [0, 0, 0] and radii[3] > 0
    assert touched[3] > 0 and np.all(splats[:3] == 0)


def _real_sh_scipy(deg, d):
    theta = math.acos(max(-1.0, min(1.0, d[2])))
    phi = math.atan2(d[1], d[0])
    out = []
    for l in range(deg + 1):
        for m in range(-l, l + 1):
            am = abs(m)
            Y = sph_harm_y(l, am, theta, phi)
            if m == 0:
                out.append(Y.real)
            elif m > 0:
                out.append(math.sqrt(2) * (-1) ** m * Y.real)
            else:
                out.append(math.sqrt(2) * (-1) ** m * Y.imag)
    return np.array(out)


def test_sh_basis_matches_scipy_and_cartesian_table(orc):
    rng = np.random.default_rng(5)
    for _ in range(50):
        d = rng.normal(size=3)
        d /= np.linalg.norm(d)
        Y = orc.sh_basis(3, d)
        np.testing.assert_allclose(Y, _real_sh_scipy(3, d), atol=1e-12)
        x, y, z = d
        c1 = math.sqrt(3 / (4 * math.pi))
        np.testing.assert_allclose(Y[1:4], [c1 * y, c1 * z, c1 * x], atol=1e-12)
        np.testing.assert_allclose(Y[4], 0.5 * math.sqrt(15 / math.pi) * x * y, atol=1e-12)
        np.testing.assert_allclose(Y[6], 0.25 * math.sqrt(5 / math.pi) * (3 * z * z - 1), atol=1e-12)
        np.testing.assert_allclose(Y[15], 0.25 * math.sqrt(35 / (2 * math.pi)) * x * (x * x - 3 * y * y), atol=1e-12)
    assert abs(orc.sh_basis(0, [0, 0, 1])[0] - 0.5 / math.sqrt(math.pi)) < 1e-15


def test_sh_orthonormal_by_quadrature(orc):
    nt, nphi = 24, 48
    xs, ws = np.polynomial.legendre.leggauss(nt)
    G = np.zeros((16, 16))
    for ct, w in zip(xs, ws):
        st = math.sqrt(1 - ct * ct)
        for k in range(nphi):
            ph = 2 * math.pi * k / nphi
            Y = orc.sh_basis(3, [st * math.cos(ph), st * math.sin(ph), ct])
            G += w * (2 * math.pi / nphi) * np.outer(Y, Y)
    np.testing.assert_allclose(G, np.eye(16), atol=1e-12)


def test_sh_colour(orc):
    cam = scenes.look_at((0.5, 1.0, 3.0), (0, 0, 0), 64, 64, 60, 60)
    rng = np.random.default_rng(9)
    n = 40
    means = rng.uniform(-0.5, 0.5, size=(n, 3))
    sh = rng.normal(0, 0.2, size=(n, 16, 3))
    sh[:, 0] = rng.normal(0.5, 0.2, size=(n, 3))
    g = gaussians(means, np.full((n, 3), -3.0), np.tile([1, 0, 0, 0], (n, 1)), np.zeros(n), sh, deg=3)
    splats, radii, _, _ = orc.project(cam, g)
    cpos = -cam.R.astype(np.float64).T @ cam.t.astype(np.float64)
    for k in range(n):
        if radii[k] == 0:
            continue
        d = g.means[k].astype(np.float64) - cpos
        d /= np.linalg.norm(d)
        Y = _real_sh_scipy(3, d)
        rgb = np.maximum(0.0, Y @ g.colors[k].astype(np.float64) + 0.5)
        np.testing.assert_allclose(splats[k, 6:9], rgb, atol=1e-6)
    # degree 0 is C0 * dc + 0.5
    g0 = gaussians(means, np.full((n, 3), -3.0), np.tile([1, 0, 0, 0], (n, 1)), np.zeros(n), sh[:, :1], deg=0)
    s0, r0, _, _ = orc.project(cam, g0)
    ok = r0 > 0
    np.testing.assert_allclose(s0[ok, 6:9], np.maximum(0, 0.5 / math.sqrt(math.pi) * sh[ok, 0] + 0.5), atol=1e-6)


def test_rect_hand_cases(orc):
    for case in GOLDEN["gauss_rect"]:
        cam = cam_identity(case["width"], case["height"], 10.0, 0.0, 0.0)
        splats = np.zeros((1, 12), np.float32)
        splats[0, 0:2] = case["mean"]
        splats[0, 9] = 1.0
        keys, gids, pre = orc.bin_gaussians(cam, splats, np.array([case["radius"]], np.int32))
        tiles = sorted((keys >> np.uint64(32)).astype(np.int64).tolist())
        TW = (case["width"] + 15) // 16
        if case["rect"] is None:
            assert tiles == []
        else:
            x0, y0, x1, y1 = case["rect"]
            assert tiles == sorted(ty * TW + tx for ty in range(y0, y1) for tx in range(x0, x1))


def test_bins_sorted_like_lexsort_and_cull(orc):
    s = scenes.tiny()
    cam = s.camera
    splats, radii, touched, _ = orc.project(cam, s.gaussians)
    keys, gids, pre = orc.bin_gaussians(cam, splats, radii)
    assert pre == len(keys) == touched.sum()
    tile = (keys >> np.uint64(32)).astype(np.int64)
    depth = splats[gids, 9]
    order = np.lexsort((gids, depth, tile))
    np.testing.assert_array_equal(order, np.arange(len(keys)))
    # depth bits are monotone in depth for positive depths
    assert np.all((keys & np.uint64(0xFFFFFFFF)).astype(np.uint32) == depth.view(np.uint32))
    # cull: fully covered tiles drop exactly the entries at or beyond their far depth
    T = orc.n_tiles(cam)
    rng = np.random.default_rng(1)
    full = (rng.uniform(size=T) < 0.5).astype(np.uint8)
    far = np.where(full == 1, rng.uniform(3.0, 5.0, size=T), np.inf).astype(np.float32)
    kc, gc, prec = orc.bin_gaussians(cam, splats, radii, far, full, cull=True)
    assert prec == len(keys)
    keep = ~((full[tile] == 1) & (depth >= far[tile]))
    np.testing.assert_array_equal(kc, keys[keep])
    np.testing.assert_array_equal(gc, gids[keep])
    assert keep.sum() < len(keys)


def test_tile_lists_match_bins(orc):
    s = scenes.tiny()
    splats, radii, _, _ = orc.project(s.camera, s.gaussians)
    keys, gids, _ = orc.bin_gaussians(s.camera, splats, radii)
    start, entries = orc.tile_lists(s.camera, splats, radii)
    np.testing.assert_array_equal(entries, gids)
    counts = np.bincount((keys >> np.uint64(32)).astype(np.int64), minlength=orc.n_tiles(s.camera))
    np.testing.assert_array_equal(np.diff(start), counts)

"""Pins of the oracle's soft split (page "A Lightweight and Differentiable
Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Hybrid rendering: each
Gaussian is split at the mesh surface; its depth given the pixel is Gaussian
with mean z*(p) = z_c + g . (p - mean2d) and standard deviation sigma from the
projected 3D covariance; the part in front is f = Phi((D - z*)/(sigma
softness)); a flat Gaussian lying on a tilted surface tilts with it).

The depth model is pinned by closed forms and by the page's own property of
flat Gaussians; the compositing by a single-Gaussian closed form with an
independent normal CDF (scipy.special.ndtr), by the hard-split limit and by
the unchanged uncovered pixels; the finite differences through the depth
model by closed-form derivatives.  The same pins cover the optional logistic
form of the front fraction, sigmoid(1.702 x) (scipy.special.expit), which
stays within 0.0095 of Phi."""

import math

import numpy as np
import pytest
from scipy.special import expit, ndtr
from scipy.spatial.transform import Rotation

from differentiable_hybrid_mesh_tile_b300 import scenes

S_MX, S_MY, S_CA, S_CB, S_CC, S_OP, S_R, S_G, S_B, S_Z = range(10)
F_GU, F_GV, F_SZ = 12, 13, 14


def cam_identity(w=64, h=64, f=100.0, cx=32.0, cy=32.0):
    return scenes.Camera(w, h, f, f, cx, cy, scenes.NEAR, scenes.FAR,
                         np.eye(3, dtype=np.float32), np.zeros(3, np.float32))


def gaussians(means, log_scales, quats, logits, colors):
    return scenes.Gaussians(np.asarray(means, np.float32), np.asarray(log_scales, np.float32),
                            np.asarray(quats, np.float32), np.asarray(logits, np.float32),
                            np.asarray(colors, np.float32), -1)


def test_depth_model_isotropic_on_axis(orc):
    # Sigma_c = s^2 I on the optical axis: J e_z = 0, so g = 0 and sigma_z = s
    cam = cam_identity()
    s = np.array([0.02, 0.1, 0.3])
    n = len(s)
    g = gaussians(np.stack([np.zeros(n), np.zeros(n), [2.0, 4.0, 6.0]], 1), np.log(s)[:, None].repeat(3, 1),
                  np.random.default_rng(1).normal(size=(n, 4)), np.zeros(n), np.full((n, 3), 0.5))
    dm = orc.project_depth_model(cam, g)
    np.testing.assert_allclose(dm[:, :2], 0.0, atol=1e-9)
    np.testing.assert_allclose(dm[:, 2], s.astype(np.float32), rtol=1e-6)


def test_depth_model_isotropic_off_axis_closed_form(orc):
    # isotropic Sigma_c = s^2 I at (x, 0, z): Sigma_uv,z = s^2 (j02, 0) with j02 = -f x / z^2,
    # Sigma_uv = s^2 diag(j00^2 + j02^2, j11^2); g_u = s^2 j02 / (s^2 (j00^2 + j02^2) + 0.3),
    # sigma_z^2 = s^2 - s^2 j02 g_u
    cam = cam_identity()
    x, z, s = 0.4, 4.0, 0.05
    g = gaussians([[x, 0.0, z]], [[math.log(s)] * 3], [[1, 0, 0, 0]], [0.0], [[0.5, 0.5, 0.5]])
    dm = orc.project_depth_model(cam, g)
    xf, zf, sf = (float(np.float32(v)) for v in (x, z, s))
    sf = float(np.exp(np.float32(math.log(s))))
    j00, j02 = 100.0 / zf, -100.0 * xf / zf ** 2
    gu = sf ** 2 * j02 / (sf ** 2 * (j00 ** 2 + j02 ** 2) + 0.3)
    var = sf ** 2 - sf ** 2 * j02 * gu
    np.testing.assert_allclose(dm[0, 0], gu, rtol=1e-6)
    np.testing.assert_allclose(dm[0, 1], 0.0, atol=1e-9)
    np.testing.assert_allclose(dm[0, 2], math.sqrt(var), rtol=1e-6)


def test_flat_gaussian_depth_follows_its_plane(orc):
    # a flat Gaussian (scales 0.6, 0.6, 1e-5) lying in a tilted plane: z*(p) is the depth of
    # that plane seen through pixel p, to first order in p - mean2d (the eps = 0.3 px^2 of the
    # splat shrinks g by ~0.3 / Sigma_uv ~ 1e-4 here)
    cam = cam_identity(w=256, h=256, f=200.0, cx=128.0, cy=128.0)
    normal = np.array([0.3, -0.5, -1.0])
    normal /= np.linalg.norm(normal)
    # rotation taking e_z to the plane normal
    rot, _ = Rotation.align_vectors([normal], [[0.0, 0.0, 1.0]])
    qx, qy, qz, qw = rot.as_quat()
    c0 = np.array([0.2, -0.1, 5.0])
    g = gaussians([c0], [[math.log(0.6), math.log(0.6), math.log(1e-5)]], [[qw, qx, qy, qz]], [0.0],
                  [[0.5, 0.5, 0.5]])
    dm = orc.project_depth_model(cam, g)
    sp, rad, _, _ = orc.project(cam, g)
    c0 = c0.astype(np.float32).astype(np.float64)
    mx, my, zc = float(sp[0, S_MX]), float(sp[0, S_MY]), float(sp[0, S_Z])
    def z_plane(u, v):  # depth of the plane n . X = n . c0 seen through pixel (u, v)
        ray = np.array([(u - 128.0) / 200.0, (v - 128.0) / 200.0, 1.0])
        return normal.dot(c0) / normal.dot(ray) * ray[2]

    # g is the pixel gradient of that depth at the splat's centre (the affine map of the
    # splat is the projection's derivative there)
    e = 1e-3
    grad = np.array([(z_plane(mx + e, my) - z_plane(mx - e, my)) / (2 * e),
                     (z_plane(mx, my + e) - z_plane(mx, my - e)) / (2 * e)])
    np.testing.assert_allclose(z_plane(mx, my), zc, rtol=1e-6)
    np.testing.assert_allclose(dm[0, :2], grad, rtol=2e-3, atol=1e-7)
    assert np.abs(grad).max() > 1e-3
    # a flat Gaussian has no depth spread of its own; what remains is the splat's 0.3 px^2
    # blur times the depth slope: sigma_z^2 = 0.3 g^T Sigma_uv (Sigma_uv + 0.3 I)^-1 g_exact
    # ~ 0.3 |g|^2 (Sigma_uv ~ 600 px^2 here)
    np.testing.assert_allclose(dm[0, 2], math.sqrt(0.3) * np.linalg.norm(grad), rtol=2e-2)


def _one(D, softness, alpha_logit=0.5, z=4.0, gu=0.01, gv=-0.02, sz=0.05, px=10.5, py=9.5, f32=False):
    splats = np.zeros((1, 12), np.float32)
    splats[0, :10] = [10.0, 10.0, 0.02, 0.003, 0.03, expit(alpha_logit), 0.9, 0.2, 0.4, z]
    dm = np.array([[gu, gv, sz, 0.0]], np.float32)
    return splats, dm


def _front(x, split):
    # the two forms of the front fraction: scipy's normal CDF, or the logistic
    # approximation sigmoid(1.702 x) through scipy's expit
    return float(ndtr(x)) if split == 0 else float(expit(1.702 * x))


def _front_density(x, split):
    if split == 0:
        return math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    f = float(expit(1.702 * x))
    return 1.702 * f * (1.0 - f)


@pytest.mark.parametrize("split", [0, 1], ids=["phi", "logistic"])
def test_single_gaussian_soft_split_closed_form(orc, split):
    cm, bg = (0.1, 0.7, 0.3), (1.0, 1.0, 1.0)
    for D in (3.9, 4.0, 4.05, 4.2):
        for softness in (0.5, 1.0, 2.0):
            splats, dm = _one(D, softness)
            s = splats[0].astype(np.float64)
            d = np.array([10.5 - s[S_MX], 9.5 - s[S_MY]])
            sigma = 0.5 * (s[S_CA] * d[0] ** 2 + s[S_CC] * d[1] ** 2) + s[S_CB] * d[0] * d[1]
            alpha = min(0.99, s[S_OP] * math.exp(-sigma))
            zs = s[S_Z] + float(dm[0, 0]) * d[0] + float(dm[0, 1]) * d[1]
            f = _front((D - zs) / (float(dm[0, 2]) * softness), split)
            o = orc.composite_one(10.5, 9.5, splats, [0], D=D, covered=True, cm=cm, bg=bg, f32=False,
                                  depth_model=dm, softness=softness, split=split)
            a = alpha * f
            if a < 1.0 / 255.0:  # the skip applies to the composited alpha
                a = 0.0
            np.testing.assert_allclose(o["rgb"], a * s[S_R:S_B + 1] + (1 - a) * np.array(cm), rtol=1e-12,
                                       atol=1e-14)
            np.testing.assert_allclose(o["T"], 1 - a, rtol=1e-12)
            np.testing.assert_allclose(o["depth"], a * s[S_Z] + (1 - a) * D, rtol=1e-12)


def test_soft_split_limits(orc):
    cm, bg = (0.1, 0.7, 0.3), (1.0, 1.0, 1.0)
    rng = np.random.default_rng(3)
    n = 6
    splats = np.zeros((n, 12), np.float32)
    splats[:, 0] = rng.uniform(8, 12, n)
    splats[:, 1] = rng.uniform(8, 12, n)
    splats[:, 2] = 0.05
    splats[:, 4] = 0.05
    splats[:, 5] = rng.uniform(0.3, 0.9, n)
    splats[:, 6:9] = rng.uniform(size=(n, 3))
    splats[:, 9] = np.sort(rng.uniform(3.0, 5.0, n))
    dm = np.zeros((n, 4), np.float32)
    dm[:, 0:2] = rng.normal(0, 0.01, (n, 2))
    dm[:, 2] = 0.02
    D = 4.0
    hard = orc.composite_one(10.5, 10.5, splats, np.arange(n), D=D, covered=True, cm=cm, bg=bg, f32=False)
    # a vanishing softness turns the split into the hard depth test (no Gaussian is within a
    # few sigma_z softness of the mesh here)
    zs = splats[:, 9] + dm[:, 0] * (10.5 - splats[:, 0]) + dm[:, 1] * (10.5 - splats[:, 1])
    assert np.abs(zs - D).min() > 1e-3
    sharp = orc.composite_one(10.5, 10.5, splats, np.arange(n), D=D, covered=True, cm=cm, bg=bg, f32=False,
                              depth_model=dm, softness=1e-3)
    np.testing.assert_allclose(sharp["rgb"], hard["rgb"], atol=1e-12)
    # an uncovered pixel (no mesh, D = inf) is not changed by the split
    for soft in (0.5, 3.0):
        a = orc.composite_one(10.5, 10.5, splats, np.arange(n), covered=False, cm=cm, bg=bg, f32=True)
        b = orc.composite_one(10.5, 10.5, splats, np.arange(n), covered=False, cm=cm, bg=bg, f32=True,
                              depth_model=dm, softness=soft)
        assert all(np.array_equal(np.asarray(a[k]), np.asarray(b[k])) for k in a)
    # a Gaussian well behind the mesh still shows a little through the soft split
    far = splats.copy()
    far[:, 9] = 4.05
    s1 = orc.composite_one(10.5, 10.5, far, np.arange(n), D=D, covered=True, cm=cm, bg=bg, f32=False,
                           depth_model=dm, softness=1.0)
    assert 0.0 < 1.0 - s1["T"] < 0.2


def test_logistic_split_is_close_to_phi(orc):
    """The logistic form differs from Phi by at most 0.0095 in f (the known bound of
    the 1.702 approximation), so a single Gaussian's composited alpha by at most
    0.0095 alpha; both reach the hard split as the softness vanishes."""
    cm = (0.1, 0.7, 0.3)
    xs = np.linspace(-6, 6, 2001)
    assert np.abs(ndtr(xs) - expit(1.702 * xs)).max() < 0.0095
    for D in (3.95, 4.0, 4.03, 4.1):
        splats, dm = _one(D, 1.0)
        a = [1.0 - orc.composite_one(10.5, 9.5, splats, [0], D=D, covered=True, cm=cm, f32=False,
                                     depth_model=dm, softness=1.0, split=k)["T"] for k in (0, 1)]
        assert abs(a[0] - a[1]) <= 0.0095 * 0.99 + 1e-12
    rng = np.random.default_rng(3)
    n = 5
    splats = np.zeros((n, 12), np.float32)
    splats[:, 0:2] = rng.uniform(8, 12, (n, 2))
    splats[:, 2] = splats[:, 4] = 0.05
    splats[:, 5] = rng.uniform(0.3, 0.9, n)
    splats[:, 6:9] = rng.uniform(size=(n, 3))
    splats[:, 9] = np.sort(rng.uniform(3.0, 5.0, n))
    dm = np.zeros((n, 4), np.float32)
    dm[:, 2] = 0.02
    hard = orc.composite_one(10.5, 10.5, splats, np.arange(n), D=4.0, covered=True, cm=cm, f32=False)
    sharp = orc.composite_one(10.5, 10.5, splats, np.arange(n), D=4.0, covered=True, cm=cm, f32=False,
                              depth_model=dm, softness=1e-3, split=1)
    np.testing.assert_allclose(sharp["rgb"], hard["rgb"], atol=1e-12)


def _flat_scene():
    """A 16 x 16 image fully covered by a mesh at depth D = 4 (mesh colour cm),
    one Gaussian near the surface."""
    cam = cam_identity(w=16, h=16, f=16.0, cx=8.0, cy=8.0)
    splats = np.zeros((1, 12), np.float32)
    splats[0, :10] = [7.6, 8.3, 0.08, 0.01, 0.06, 0.7, 0.9, 0.2, 0.4, 3.98]
    dm = np.array([[0.004, -0.003, 0.03, 0.0]], np.float32)
    radii = np.array([12], np.int32)
    lists = (np.array([0, 1], np.int64), np.array([0], np.int32))
    D = np.full(256, 4.0, np.float32)
    cm = np.tile(np.array([0.1, 0.7, 0.3], np.float32), (256, 1))
    face = np.zeros(256, np.int32)
    return cam, splats, dm, radii, lists, D, cm, face


@pytest.mark.parametrize("split", [0, 1], ids=["phi", "logistic"])
def test_finite_differences_through_the_depth_model(orc, split):
    """d/d(sigma_z, g_u, z_c) of L = sum_p g_rgb . rgb against the closed forms
    sum_p alpha (c - cm) . g_rgb f'(x) dx/d(.), x = (D - z_c - g . d) / (sigma_z s),
    f' the normal density or, for the logistic form, 1.702 f (1 - f)."""
    cam, splats, dm, radii, lists, D, cm, face = _flat_scene()
    rng = np.random.default_rng(5)
    g_rgb = rng.uniform(-1, 1, (16, 16, 3)).astype(np.float32)
    zero = np.zeros((16, 16), np.float32)
    softness = 1.5
    s = splats[0].astype(np.float64)
    gu, gv, sz = (float(v) for v in dm[0, :3])
    want = {F_SZ: 0.0, F_GU: 0.0, S_Z: 0.0}
    for j in range(16):
        for i in range(16):
            d = np.array([i + 0.5 - s[S_MX], j + 0.5 - s[S_MY]])
            sig = 0.5 * (s[S_CA] * d[0] ** 2 + s[S_CC] * d[1] ** 2) + s[S_CB] * d[0] * d[1]
            alpha = min(0.99, s[S_OP] * math.exp(-sig))
            x = (4.0 - s[S_Z] - gu * d[0] - gv * d[1]) / (sz * softness)
            f = _front(x, split)
            if sig < 0 or alpha * f < 1 / 255:
                continue
            phi = _front_density(x, split)
            k = alpha * float(np.dot(s[S_R:S_B + 1] - cm[0].astype(np.float64), g_rgb[j, i])) * phi
            want[F_SZ] += k * (-x / sz)
            want[F_GU] += k * (-d[0] / (sz * softness))
            want[S_Z] += k * (-1.0 / (sz * softness))
    fields = np.array([F_SZ, F_GU, S_Z], np.int32)
    hs = np.array([1e-5, 1e-6, 1e-6])
    got, st = orc.composite_fd(cam, (1, 1, 1), splats, radii, lists, D.reshape(16, 16), cm.reshape(16, 16, 3),
                               face.reshape(16, 16), (g_rgb, zero, zero), np.zeros(3, np.int32), fields, hs,
                               depth_model=dm, softness=softness, split=split)
    assert (st == 0).all(), st
    for k, fld in enumerate(fields):
        np.testing.assert_allclose(got[k], want[int(fld)], rtol=2e-5, atol=1e-9)


@pytest.mark.parametrize("split", [0, 1], ids=["phi", "logistic"])
def test_skip_margin_carries_the_split_rounding(orc, split):
    """The reported alpha-skip margin of a covered pixel covers the rounding bound
    of x = (D - z*) / (sigma_z softness): a thin depth extent makes the decision
    ill-conditioned where the surface z* meets the mesh, and the margin says so
    there (negative) and only there."""
    cam, splats, dm, radii, lists, D, cm, face = _flat_scene()
    out = {}
    for sz in (0.5, 1e-6):
        d = dm.copy()
        d[0, 2] = sz
        o = orc.composite_fwd(cam, (1, 1, 1), splats, lists, D.reshape(16, 16), cm.reshape(16, 16, 3),
                              face.reshape(16, 16), depth_model=d, softness=1.0, split=split)
        out[sz] = o["margins"][..., 1]
    wide, thin = out[0.5], out[1e-6]
    assert np.isfinite(wide).all() and (wide > 1e-3).mean() > 0.9
    # with sigma_z = 1e-6 the decision is ill-conditioned exactly where the surface
    # z*(p) passes within a few hundred sigma_z of the mesh depth, and nowhere else
    s = splats[0].astype(np.float64)
    j, i = np.mgrid[0:16, 0:16]
    zs = s[S_Z] + float(dm[0, 0]) * (i + 0.5 - s[S_MX]) + float(dm[0, 1]) * (j + 0.5 - s[S_MY])
    near = np.abs(4.0 - zs) < 1e-4
    assert near.any() and (thin[near] < 0).all()
    assert (thin[np.abs(4.0 - zs) > 1e-3] > 0).all()

"""Pins of the oracle's analytic edge antialiasing (page "A Lightweight and
Differentiable Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Mesh
rasterizer item 3: neighbouring pixels that see a silhouette share coverage by
where the front triangle's edge crosses between their centres, and blend over a
farther surface; internal edges of a connected surface are left alone;
Limitations: a per-axis 1D approximation, exact for straight edges away from
corners; Hybrid rendering: the coverage a_m enters the two-layer compositing).

Pinned by: the edge adjacency of closed meshes; exact coverage of axis-aligned
edges; the per-line coverage sums of slanted straight edges against the exact
clipped pixel areas; colour blending over a farther surface; the interior of a
closed surface left untouched; the two-layer compositing equation on one pixel;
and the silhouette gradient against its closed form."""

import math

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes

NO_GAUSS = scenes.Gaussians(np.zeros((0, 3), np.float32), np.zeros((0, 3), np.float32),
                            np.zeros((0, 4), np.float32), np.zeros(0, np.float32), np.zeros((0, 3), np.float32), -1)


def cam_id(w=48, h=48, f=48.0):
    return scenes.Camera(w, h, f, f, w / 2, h / 2, scenes.NEAR, scenes.FAR, np.eye(3, dtype=np.float32),
                         np.zeros(3, np.float32))


def unproject(cam, pts, z):
    return np.array([((u - cam.cx) * z / cam.fx, (v - cam.cy) * z / cam.fy, z) for u, v in pts], np.float32)


def quad(cam, u0, u1, v0, v1, z, col):
    V = unproject(cam, [(u0, v0), (u1, v0), (u1, v1), (u0, v1)], z)
    F = np.array([[0, 1, 2], [0, 2, 3]], np.int32)
    return V, F, np.tile(np.asarray(col, np.float32), (4, 1))


def render(orc, cam, V, F, vcol, bg=(1.0, 1.0, 1.0)):
    sc = scenes.Scene("t", [cam], scenes.Mesh(V, F, vcol), NO_GAUSS, bg)
    return orc.render(sc, antialias_edges=True)


def test_edge_adjacency(orc):
    v, f = scenes.icosphere(2)
    adj = orc.mesh_edges(f)
    assert (adj >= 0).all()
    for face in range(len(f)):
        for k in range(3):
            other = adj[face, k]
            e = {f[face, (k + 1) % 3], f[face, (k + 2) % 3]}
            back = [kk for kk in range(3) if {f[other, (kk + 1) % 3], f[other, (kk + 2) % 3]} == e]
            assert len(back) == 1 and adj[other, back[0]] == face
    assert (orc.mesh_edges(np.array([[0, 1, 2]], np.int32)) == -1).all()
    fan = np.array([[0, 1, 2], [1, 0, 3], [0, 1, 4]], np.int32)  # edge {0, 1} shared three times
    a = orc.mesh_edges(fan)
    assert a[0, 2] == -2 and a[1, 2] == -2 and a[2, 2] == -2
    assert (a[:, :2] == -1).all()


def test_axis_aligned_edges_exact(orc):
    """A quad with edges at x = 10.0 / 30.3 and y = 8.0 / 39.6: a pixel [i, i+1] x [j, j+1]
    gets exactly the covered fraction away from the corners; the quad's internal diagonal
    changes nothing; the colour is premultiplied by the coverage."""
    cam = cam_id()
    V, F, vc = quad(cam, 10.0, 30.3, 8.0, 39.6, 5.0, (0.9, 0.2, 0.4))
    r = render(orc, cam, V, F, vc)
    cov, rgb = r["cov"].astype(np.float64), r["rgb_aa"].astype(np.float64)
    for j in range(12, 36):
        np.testing.assert_allclose(cov[j, 30], 0.3, atol=2e-6)
        np.testing.assert_allclose(cov[j, 31], 0.0, atol=0)
        # the edge at x = 10 sits on a pixel boundary: weight 0 up to the fp32 vertex
        np.testing.assert_allclose(cov[j, 9:11], [0.0, 1.0], atol=2e-6)
        np.testing.assert_allclose(cov[j, 11:30], 1.0, atol=0)
        np.testing.assert_allclose(rgb[j, 30], 0.3 * np.array([0.9, 0.2, 0.4]), atol=2e-6)
    for i in range(14, 28):
        np.testing.assert_allclose(cov[39, i], 0.6, atol=2e-6)
        np.testing.assert_allclose(cov[9:39, i], 1.0, atol=0)
        np.testing.assert_allclose(cov[7:9, i], [0.0, 1.0], atol=2e-6)
    # no Gaussians: the image is the layer over the background
    np.testing.assert_allclose(r["rgb"].astype(np.float64), rgb + (1 - cov)[..., None] * 1.0, atol=1e-6)
    np.testing.assert_allclose(r["alpha"], cov, atol=1e-6)


def _clip_area(nrm, c, i, j):
    """Area of the pixel square [i, i+1] x [j, j+1] on the side (p - c) . nrm <= 0."""
    poly = [(i, j), (i + 1, j), (i + 1, j + 1), (i, j + 1)]
    side = [(p[0] - c[0]) * nrm[0] + (p[1] - c[1]) * nrm[1] for p in poly]
    out = []
    for k in range(4):
        a, b, fa, fb = poly[k], poly[(k + 1) % 4], side[k], side[(k + 1) % 4]
        if fa <= 0:
            out.append(a)
        if (fa < 0) != (fb < 0) and fa != fb:
            t = fa / (fa - fb)
            out.append((a[0] + t * (b[0] - a[0]), a[1] + t * (b[1] - a[1])))
    if len(out) < 3:
        return 0.0
    x, y = np.array([p[0] for p in out]), np.array([p[1] for p in out])
    return 0.5 * abs(np.dot(x, np.roll(y, -1)) - np.dot(y, np.roll(x, -1)))


@pytest.mark.parametrize("deg", [7, 20, 33, 44, 50, 70])
def test_slanted_edge_line_sums_exact(orc, deg):
    """A straight edge at deg degrees: each line of pixels across it (columns for a
    shallow edge, rows for a steep one) holds exactly the covered area in total; a
    single pixel is within 0.13 of its own area."""
    cam = cam_id()
    t = math.radians(deg)
    d, nrm, c0 = np.array([-math.sin(t), math.cos(t)]), np.array([math.cos(t), math.sin(t)]), np.array([24.3, 23.8])
    V = unproject(cam, [c0 + 100 * d, c0 - 100 * d, c0 - 100 * nrm], 5.0)
    r = render(orc, cam, V, np.array([[0, 1, 2]], np.int32), np.ones((3, 3), np.float32))
    # the edge as the fp32 vertices place it
    P = V[:2].astype(np.float64)
    uv = np.stack([cam.fx * P[:, 0] / P[:, 2] + cam.cx, cam.fy * P[:, 1] / P[:, 2] + cam.cy], 1)
    dd = uv[1] - uv[0]
    n2 = np.array([dd[1], -dd[0]])
    if np.dot(n2, (c0 - 100 * nrm) - uv[0]) > 0:
        n2 = -n2
    ex = np.array([[_clip_area(n2, uv[0], i, j) for i in range(48)] for j in range(48)])
    cov = r["cov"].astype(np.float64)
    inner = slice(8, 40)
    shallow = abs(dd[1]) < abs(dd[0])
    s_aa = cov[:, inner].sum(0) if shallow else cov[inner, :].sum(1)
    s_ex = ex[:, inner].sum(0) if shallow else ex[inner, :].sum(1)
    np.testing.assert_allclose(s_aa, s_ex, atol=2e-5)
    assert np.abs(cov - ex)[inner, inner].max() < 0.13


def test_colour_over_farther_surface_and_depth(orc):
    """A front quad over a farther one: at the front quad's right edge the pixel behind
    it stays fully covered and blends towards the front colour by the crossing; where
    the front quad reaches into an uncovered pixel, that pixel takes its depth."""
    cam = cam_id()
    Vf, Ff, cf = quad(cam, 10.0, 30.3, 8.0, 20.0, 4.0, (1.0, 0.0, 0.0))
    Vb, Fb, cb = quad(cam, 4.0, 44.0, 14.0, 44.0, 8.0, (0.0, 0.0, 1.0))
    V = np.concatenate([Vf, Vb])
    F = np.concatenate([Ff, Fb + 4])
    r = render(orc, cam, V, F, np.concatenate([cf, cb]))
    j = 17  # a row where the front quad lies over the back one
    np.testing.assert_allclose(r["cov"][j, 31], 1.0, atol=0)
    np.testing.assert_allclose(r["rgb_aa"][j, 31], [0.0, 0.0, 1.0], atol=0)
    np.testing.assert_allclose(r["cov"][j, 30], 1.0, atol=0)
    np.testing.assert_allclose(r["rgb_aa"][j, 30], [0.3, 0.0, 0.7], atol=2e-6)  # 0.3 front + 0.7 back
    np.testing.assert_allclose(r["depth_aa"][j, 30], r["mesh_depth"][j, 30], atol=0)
    j = 10  # the front quad alone: pixel 30 is not covered and takes 0.3 and pixel 29's depth
    assert r["face_id"][j, 30] < 0
    np.testing.assert_allclose(r["cov"][j, 30], 0.3, atol=2e-6)
    np.testing.assert_allclose(r["depth_aa"][j, 30], r["mesh_depth"][j, 29], atol=0)
    Vq, Fq, cq = quad(cam, 10.0, 30.7, 8.0, 20.0, 4.0, (1.0, 0.0, 0.0))
    r2 = render(orc, cam, Vq, Fq, cq)
    np.testing.assert_allclose(r2["cov"][10, 30:32], [0.7, 0.0], atol=2e-6)  # the edge leaves pixel 30
    np.testing.assert_allclose(r2["depth_aa"][10, 30], r2["mesh_depth"][10, 30], atol=0)
    assert np.isinf(r2["depth_aa"][10, 31])


def test_closed_surface_interior_untouched(orc):
    """On an icosphere the internal edges between front faces do nothing: away from the
    outline every pixel keeps coverage 1 and its own colour; only the outline is soft."""
    v, f = scenes.icosphere(3)
    cam = scenes.look_at((0, 0, 3.2), (0, 0, 0), 64, 64, 64, 64)
    rng = np.random.default_rng(1)
    r = render(orc, cam, v.astype(np.float32), f, rng.uniform(0, 1, (len(v), 3)).astype(np.float32))
    covered = r["face_id"] >= 0
    far_in = covered.copy()
    for _ in range(2):  # two pixels inside the outline
        far_in[1:-1, 1:-1] &= covered[:-2, 1:-1] & covered[2:, 1:-1] & covered[1:-1, :-2] & covered[1:-1, 2:]
        covered = far_in.copy()
    assert far_in.sum() > 1000
    assert (r["cov"][far_in] == 1.0).all()
    np.testing.assert_array_equal(r["rgb_aa"][far_in], r["mesh_rgb"][far_in])
    soft = (r["cov"] > 0) & (r["cov"] < 1)
    assert soft.sum() > 50 and not (soft & far_in).any()


def test_two_layer_compositing_one_pixel(orc):
    """rgb = C_f + T_f (M + (1 - a)(C_b + T_b bg)) with a Gaussian in front of the mesh
    layer (z < D) and one behind it, over a layer of coverage 0.3."""
    splats = np.zeros((2, 12), np.float32)
    splats[:, 0:2] = 10.0
    splats[:, 2] = splats[:, 4] = 0.1
    splats[:, 5] = [0.6, 0.5]
    splats[0, 6:9] = [1.0, 0.0, 0.0]
    splats[1, 6:9] = [0.0, 1.0, 0.0]
    splats[:, 9] = [3.0, 6.0]
    a, c, bg, D = 0.3, np.array([0.2, 0.3, 0.9]), np.array([1.0, 1.0, 1.0]), 4.0
    o = orc.composite_one(10.5, 10.5, splats, [0, 1], D=D, cov=a, cm=a * c, bg=bg, f32=False)
    sp = splats.astype(np.float64)
    s = 0.5 * sp[0, 2] * 0.25 * 2
    a1, a2 = sp[0, 5] * math.exp(-s), sp[1, 5] * math.exp(-s)
    want = a1 * splats[0, 6:9] + (1 - a1) * (a * c + (1 - a) * (a2 * splats[1, 6:9] + (1 - a2) * bg))
    np.testing.assert_allclose(o["rgb"], want, rtol=1e-12)
    np.testing.assert_allclose(o["depth"], a1 * 3.0 + (1 - a1) * (a * D + (1 - a) * a2 * 6.0), rtol=1e-12)
    np.testing.assert_allclose(o["alpha"], 1 - (1 - a1) * (1 - a) * (1 - a2), rtol=1e-12)
    np.testing.assert_allclose(o["T"], 1 - a1, rtol=1e-12)
    # coverage 1 hides the back Gaussian; coverage 0 with no mesh depth is one chain
    o1 = orc.composite_one(10.5, 10.5, splats, [0, 1], D=D, cov=1.0, cm=c, bg=bg, f32=False)
    np.testing.assert_allclose(o1["rgb"], a1 * splats[0, 6:9] + (1 - a1) * c, rtol=1e-12)
    o0 = orc.composite_one(10.5, 10.5, splats, [0, 1], D=np.inf, cov=0.0, cm=(0, 0, 0), bg=bg, f32=False)
    h = orc.composite_one(10.5, 10.5, splats, [0, 1], covered=False, bg=bg, f32=False)
    np.testing.assert_allclose(o0["rgb"], h["rgb"], rtol=0, atol=0)


def test_silhouette_gradient_closed_form(orc):
    """Moving a vertex of the quad's vertical right edge along world x shifts the edge
    crossing in row j by fx / z times (1 - s_j) for the top vertex (s_j the row's
    position along the edge): dL/dX = sum_j g_j . (c - bg) fx / z (1 - s_j) over the rows
    away from the corners (upstream gradient zero elsewhere; one colour, no Gaussians)."""
    cam = cam_id()
    z, col, bg = 5.0, np.array([0.9, 0.2, 0.4]), np.array([1.0, 1.0, 1.0])
    # no edge on a pixel boundary (there the side of a crossing at t = 0.5 is a tie)
    V, F, vc = quad(cam, 10.2, 30.3, 8.3, 39.6, z, col)
    r = render(orc, cam, V, F, vc)
    rng = np.random.default_rng(2)
    g_rgb = np.zeros((48, 48, 3), np.float32)
    rows = np.arange(12, 36)
    g_rgb[rows, 30] = rng.uniform(-1, 1, (len(rows), 3))
    zero = np.zeros((48, 48), np.float32)
    grads = (g_rgb, zero, zero)
    vids = np.array([1, 2], np.int32)  # top-right, bottom-right
    got, st = orc.mesh_fd(cam, bg, V, F, vc, r["face_id"], np.zeros((1, 12), np.float32), r["lists"],
                          r["mesh_depth"], r["mesh_rgb"], grads, vids, np.zeros(2, np.int32), np.full(2, 1e-4),
                          adj=r["adj"])
    assert (st == 0).all(), st
    uv = V[:, 1].astype(np.float64) * cam.fy / z + cam.cy
    s = (rows + 0.5 - uv[1]) / (uv[2] - uv[1])
    k = (g_rgb[rows, 30].astype(np.float64) @ (col - bg)) * cam.fx / z
    np.testing.assert_allclose(got, [np.sum(k * (1 - s)), np.sum(k * s)], rtol=1e-5)

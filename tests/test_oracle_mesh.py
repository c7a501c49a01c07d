"""Pins of the oracle's mesh steps against closed forms, exact arithmetic and
invariants (page "A Lightweight and Differentiable Renderer for Joint Mesh and
3D Gaussian Splat Scenes", Design Details > Mesh rasterizer, items 1 and 2)."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


def cam_identity(w, h, f, cx, cy):
    return scenes.Camera(w, h, f, f, cx, cy, scenes.NEAR, scenes.FAR,
                         np.eye(3, dtype=np.float32), np.zeros(3, np.float32))


def test_single_triangle_coverage_exact(orc):
    # camera at the origin looking down +z, fx = fy = 8, principal point (8, 8);
    # vertices at depth 2 project to (5, 5), (13, 5), (5, 13): a right triangle,
    # every coordinate a small dyadic rational (exact in fp32).
    cam = cam_identity(16, 16, 8.0, 8.0, 8.0)
    V = np.array([[-0.75, -0.75, 2.0], [1.25, -0.75, 2.0], [-0.75, 1.25, 2.0]], np.float32)
    F = np.array([[0, 1, 2]], np.int32)
    fid, best, _ = orc.zbuffer(cam, V, F)
    fid = fid.reshape(16, 16)
    # exact inside set from the projected vertices (rational arithmetic on the
    # float32 inputs): u - 5 >= 0, v - 5 >= 0, (u - 5) + (v - 5) <= 8
    u = [Fraction(float(x)) * 8 / 2 + 8 for x in V[:, 0]]
    assert u[0] == 5 and u[1] == 13
    for j in range(16):
        for i in range(16):
            px, py = Fraction(2 * i + 1, 2), Fraction(2 * j + 1, 2)
            inside = px >= 5 and py >= 5 and (px - 5) + (py - 5) <= 8
            assert (fid[j, i] == 0) == inside, (i, j)
    assert np.all(best.reshape(16, 16)[fid == 0] == 2.0)


def test_fronto_parallel_barycentrics(orc):
    cam = cam_identity(16, 16, 8.0, 8.0, 8.0)
    V = np.array([[-0.75, -0.75, 2.0], [1.25, -0.75, 2.0], [-0.75, 1.25, 2.0]], np.float32)
    F = np.array([[0, 1, 2]], np.int32)
    vcol = np.eye(3, dtype=np.float32)
    fid, _, _ = orc.zbuffer(cam, V, F)
    depth, rgb = orc.interp_mesh(cam, V, F, vcol, fid)
    for p in np.nonzero(fid >= 0)[0]:
        i, j = p % 16, p // 16
        l1 = (i + 0.5 - 5.0) / 8.0
        l2 = (j + 0.5 - 5.0) / 8.0
        np.testing.assert_allclose(rgb[p], [1 - l1 - l2, l1, l2], atol=1e-6)
        assert abs(depth[p] - 2.0) < 1e-6


def _tilted_scene():
    rng = np.random.default_rng(7)
    cam = scenes.look_at((0.3, -0.2, 3.0), (0, 0, 0), 48, 40, 60.0, 55.0, 23.0, 21.5)
    V = np.array([[-0.9, -0.7, 0.4], [0.8, -0.5, -0.6], [0.1, 0.9, 0.2]], np.float32)
    F = np.array([[0, 1, 2]], np.int32)
    vcol = rng.uniform(0, 1, size=(3, 3)).astype(np.float32)
    return cam, V, F, vcol


def test_perspective_depth_matches_ray_plane(orc):
    """D at a pixel centre equals the camera-z of the ray's hit on the triangle's
    plane, and the colour equals the 3D barycentric blend at the hit point."""
    cam, V, F, vcol = _tilted_scene()
    fid, _, _ = orc.zbuffer(cam, V, F)
    depth, rgb = orc.interp_mesh(cam, V, F, vcol, fid)
    R, t = cam.R.astype(np.float64), cam.t.astype(np.float64)
    Xc = (R @ V.astype(np.float64).T).T + t
    n = np.cross(Xc[1] - Xc[0], Xc[2] - Xc[0])
    covered = np.nonzero(fid >= 0)[0]
    assert len(covered) > 100
    for p in covered:
        i, j = p % cam.width, p // cam.width
        d = np.array([(i + 0.5 - cam.cx) / cam.fx, (j + 0.5 - cam.cy) / cam.fy, 1.0])
        s = (n @ Xc[0]) / (n @ d)
        hit = s * d
        assert abs(depth[p] - hit[2]) <= 2e-7 * hit[2]
        # 3D barycentrics of the hit point by sub-triangle areas
        A = np.linalg.norm(n)
        b0 = np.linalg.norm(np.cross(Xc[1] - hit, Xc[2] - hit)) / A
        b1 = np.linalg.norm(np.cross(Xc[2] - hit, Xc[0] - hit)) / A
        b2 = 1.0 - b0 - b1
        np.testing.assert_allclose(rgb[p], b0 * vcol[0] + b1 * vcol[1] + b2 * vcol[2], atol=2e-6)


def test_screen_space_blend_would_differ(orc):
    """Guards the test above: on this tilted triangle the affine (screen-space)
    blend differs from the perspective-correct one by far more than the tolerance."""
    cam, V, F, vcol = _tilted_scene()
    fid, _, _ = orc.zbuffer(cam, V, F)
    _, rgb = orc.interp_mesh(cam, V, F, vcol, fid)
    R, t = cam.R.astype(np.float64), cam.t.astype(np.float64)
    Xc = (R @ V.astype(np.float64).T).T + t
    uv = np.stack([cam.fx * Xc[:, 0] / Xc[:, 2] + cam.cx, cam.fy * Xc[:, 1] / Xc[:, 2] + cam.cy], 1)
    worst = 0.0
    for p in np.nonzero(fid >= 0)[0]:
        q = np.array([p % cam.width + 0.5, p // cam.width + 0.5])
        M = np.array([[uv[0, 0], uv[1, 0], uv[2, 0]], [uv[0, 1], uv[1, 1], uv[2, 1]], [1, 1, 1]])
        lam = np.linalg.solve(M, [q[0], q[1], 1.0])
        worst = max(worst, np.abs(lam @ vcol - rgb[p]).max())
    assert worst > 1e-2


def test_diagonal_tie_smaller_id_wins(orc):
    case = GOLDEN["diagonal_tie"]
    cam = cam_identity(16, 16, 8.0, 0.0, 0.0)
    V = np.array(case["verts"], np.float32)
    F = np.array(case["faces"], np.int32)
    for order in ([0, 1], [1, 0]):
        Fo = F[order]
        fid, best, second = orc.zbuffer(cam, V, Fo)
        fid = fid.reshape(16, 16)
        for i, j in case["diagonal_pixels"]:
            assert fid[j, i] == 0
            assert best[j * 16 + i] == 2.0 and second[j * 16 + i] == 2.0
        # off the diagonal each side belongs to its own face
        assert fid[4, 8] == order.index(0)   # (u, v) = (8.5, 4.5): below the diagonal, face 0 of the file
        assert fid[8, 4] == order.index(1)


def test_nearest_wins_and_near_plane_skip(orc):
    cam = cam_identity(16, 16, 8.0, 8.0, 8.0)
    far_tri = [[-2, -2, 4.0], [2, -2, 4.0], [0, 2, 4.0]]
    near_tri = [[-1, -1, 2.0], [1, -1, 2.0], [0, 1, 2.0]]
    V = np.array(far_tri + near_tri, np.float32)
    F = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    fid, _, _ = orc.zbuffer(cam, V, F)
    assert fid.reshape(16, 16)[8, 8] == 1  # the nearer triangle, though its id is larger
    # a vertex in front of the near plane drops the whole triangle
    V2 = V.copy()
    V2[3, 2] = 0.005
    fid2, _, _ = orc.zbuffer(cam, V2, F)
    assert fid2.reshape(16, 16)[8, 8] == 0
    assert np.all(fid2 != 1)
    # a zero-area triangle covers nothing
    V3 = np.array([[0, 0, 2], [1, 1, 2], [2, 2, 2]], np.float32)
    fid3, _, _ = orc.zbuffer(cam, V3, np.array([[0, 1, 2]], np.int32))
    assert np.all(fid3 == -1)


def test_triangle_bins_cover_exactly_the_boxes(orc):
    """Bins hold a triangle in every tile where the brute-force z-buffer sees it
    (ignoring occlusion: one triangle at a time), face ids ascend per tile, and
    each binned tile meets the triangle's pixel-centre box."""
    s = scenes.tiny()
    cam = scenes.look_at((0.4, 0.3, 2.2), (0, 0, 0), 96, 80, 90, 90)
    V, F = s.mesh.verts, s.mesh.faces
    counts, ids = orc.bin_triangles(cam, V, F)
    TW = (cam.width + 15) // 16
    start = np.concatenate([[0], np.cumsum(counts)])
    per_tile = [ids[start[t]:start[t + 1]] for t in range(len(counts))]
    for lst in per_tile:
        assert np.all(np.diff(lst) > 0)
    for f in range(len(F)):
        fid, _, _ = orc.zbuffer(cam, V, F[f:f + 1])
        pix = np.nonzero(fid >= 0)[0]
        tiles = set(((pix // cam.width) // 16 * TW + (pix % cam.width) // 16).tolist())
        binned = {t for t in range(len(counts)) if f in per_tile[t]}
        assert tiles <= binned
        if binned:
            # the binned tiles form the rectangle spanned by the covered tiles or more,
            # never a tile outside the projected vertex box
            R, tt = cam.R.astype(np.float64), cam.t.astype(np.float64)
            Xc = (R @ V[F[f]].astype(np.float64).T).T + tt
            u = cam.fx * Xc[:, 0] / Xc[:, 2] + cam.cx
            v = cam.fy * Xc[:, 1] / Xc[:, 2] + cam.cy
            for t in binned:
                tx, ty = t % TW, t // TW
                assert u.max() >= tx * 16 + 0.5 - 1e-3 and u.min() <= tx * 16 + 15.5 + 1e-3
                assert v.max() >= ty * 16 + 0.5 - 1e-3 and v.min() <= ty * 16 + 15.5 + 1e-3


def test_tile_depth_bounds(orc):
    cam = cam_identity(40, 24, 8.0, 20.0, 12.0)
    md = np.full((24, 40), np.inf, np.float32)
    md[:16, :16] = np.arange(256, dtype=np.float32).reshape(16, 16) + 1.0
    md[:16, 16:32] = 3.0
    md[5, 20] = np.inf
    md[16:, 32:] = 7.0   # ragged corner tile: 8x8 in-image pixels, all covered
    far, full = orc.tile_depth_bounds(cam, md)
    assert full.tolist() == [1, 0, 0, 0, 0, 1]
    assert far[0] == 256.0 and far[5] == 7.0
    assert np.isinf(far[1]) and np.isinf(far[2])

"""GPU parity of the mesh layer (gm_bin_triangles, gm_zbuffer, gm_interp_mesh)
against the CPU oracle ("A Lightweight and Differentiable Renderer for Joint
Mesh and 3D Gaussian Splat Scenes", Design Details > Mesh rasterizer)."""

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu

TIE = 1e-6  # near-tie band of the z-buffer: two nearest depths within 1e-6 relative


def _mesh_cases():
    tiny = scenes.tiny()
    sph = scenes.sphere512()
    ragged = scenes.look_at((0.3, 0.5, 2.6), (0, 0, 0), 101, 77, 90, 95, 47.3, 40.1)
    close = scenes.look_at((0.1, 0.2, 1.6), (0, 0, 0), 130, 96, 120, 120)
    return [("tiny", tiny.camera, tiny.mesh), ("sphere512", sph.camera, sph.mesh),
            ("ragged", ragged, tiny.mesh), ("close", close, scenes.sphere512().mesh)]


@pytest.fixture(scope="module", params=_mesh_cases(), ids=lambda c: c[0])
def case(request):
    H.need_gpu()
    return request.param


def test_triangle_bins_exact(case, orc):
    name, cam, mesh = case
    g = H.run_mesh(cam, mesh)
    counts, ids = orc.bin_triangles(cam, mesh.verts, mesh.faces)
    assert g["K"] == len(ids)
    tr = g["tile_range"]
    np.testing.assert_array_equal(tr[:, 1] - tr[:, 0], counts)
    start = np.concatenate([[0], np.cumsum(counts)])
    np.testing.assert_array_equal(tr[counts > 0, 0], start[:-1][counts > 0])
    np.testing.assert_array_equal(g["tri_ids"], ids)  # tile-major, ascending face id within a tile


def test_zbuffer_matches_brute_force(case, orc):
    name, cam, mesh = case
    g = H.run_mesh(cam, mesh)
    fid, best, second = orc.zbuffer(cam, mesh.verts, mesh.faces)
    fid = fid.reshape(cam.height, cam.width)
    gpu = g["face_id"]
    assert np.all(gpu >= -1)
    tie = (second <= best * (1 + TIE)).reshape(fid.shape) & (fid >= 0)
    diff = gpu != fid
    bad = diff & ~tie
    print("%s: %d covered px, %d near-tie px, %d differ at ties" % (name, (fid >= 0).sum(), tie.sum(),
                                                                    (diff & tie).sum()))
    assert not bad.any(), np.argwhere(bad)[:10]
    # where they differ at a near tie the GPU's face covers the pixel at the tied depth
    for j, i in np.argwhere(diff):
        f = gpu[j, i]
        one, d1, _ = orc.zbuffer(cam, mesh.verts, mesh.faces[f:f + 1], pixels=np.array([j * cam.width + i]))
        assert one[0] == 0 and abs(d1[0] - best[j * cam.width + i]) <= TIE * best[j * cam.width + i]


def test_interp_teacher_forced(case, orc):
    """Depth and colour from the GPU's own face ids, against the oracle's
    double-precision interpolation of the same ids.  Bound per pixel: 4 x the
    change of the oracle's result when the vertices move by one fp32 rounding
    of their camera-space coordinates (large only on edge-on triangles), plus
    4 eps relative on depth and 2e-6 on colour."""
    name, cam, mesh = case
    g = H.run_mesh(cam, mesh)
    fid = g["face_id"]
    depth, rgb = orc.interp_mesh(cam, mesh.verts, mesh.faces, mesh.vcol, fid.reshape(-1))
    depth = depth.reshape(fid.shape)
    rgb = rgb.reshape(fid.shape + (3,))
    cov = fid >= 0
    assert np.all(np.isinf(g["mesh_depth"][~cov])) and np.all(g["mesh_rgb"][~cov] == 0)
    sd = np.zeros(fid.shape)
    sc = np.zeros(fid.shape)
    for V2 in H.input_ulp_perturbations(cam, mesh.verts):
        d2, c2 = orc.interp_mesh(cam, V2, mesh.faces, mesh.vcol, fid.reshape(-1))
        d2 = d2.reshape(fid.shape).astype(np.float64)
        # uncovered pixels hold +inf depth on both sides: compare covered ones only
        sd[cov] = np.maximum(sd[cov], np.abs(d2[cov] - depth[cov]))
        sc = np.maximum(sc, np.abs(c2.reshape(fid.shape + (3,)).astype(np.float64) - rgb).max(-1))
    d_err = np.zeros(fid.shape)
    d_err[cov] = np.abs(g["mesh_depth"][cov].astype(np.float64) - depth[cov])
    d_tol = 4 * sd + 4 * H.EPS32 * np.abs(depth)
    assert np.all(d_err[cov] <= d_tol[cov]), (d_err[cov] / d_tol[cov]).max()
    c_err = np.abs(g["mesh_rgb"].astype(np.float64) - rgb).max(-1)
    c_tol = 4 * sc + 2e-6
    assert np.all(c_err[cov] <= c_tol[cov]), (c_err[cov] / c_tol[cov]).max()
    far, full = orc.tile_depth_bounds(cam, g["mesh_depth"])
    np.testing.assert_array_equal(g["tile_full"], full)
    np.testing.assert_array_equal(g["tile_far"], far)  # max over the same fp32 depths: exact
    ill = (sc > 2.5e-5) & cov
    print("%s: colour err max %.2e, %d px ill-conditioned (one-ulp input change moves the colour > 2.5e-5), "
          "%d full tiles" % (name, c_err[cov].max(), ill.sum(), full.sum()))


def test_empty_and_degenerate_meshes(orc):
    H.need_gpu()
    cam = scenes.look_at((0, 0, 3), (0, 0, 0), 40, 24, 30, 30)
    empty = scenes.empty_mesh()
    g = H.run_mesh(cam, empty)
    assert g["K"] == 0 and np.all(g["face_id"] == -1) and np.all(g["tile_full"] == 0)
    assert np.all(np.isinf(g["tile_far"])) and np.all(g["tile_range"] == 0)
    # behind the camera, straddling the near plane, zero area, off-image, bad index
    V = np.array([[0, 0, 4.0], [1, 0, 4], [0, 1, 4],       # behind the camera (z_c < 0)
                  [-1, -1, 2.995], [1, -1, 1.0], [0, 1, 1.0],  # one vertex in front of near
                  [0, 0, 1.0], [0.5, 0.5, 1.0], [1, 1, 1.0],   # collinear
                  [50, 50, 0], [51, 50, 0], [50, 51, 0],       # off image
                  [-0.5, -0.5, 0], [0.5, -0.5, 0], [0, 0.5, 0]], np.float32)
    F = np.array([[0, 1, 2], [3, 4, 5], [6, 7, 8], [9, 10, 11], [12, 13, 99], [12, 13, 14]], np.int32)
    mesh = scenes.Mesh(V, F, np.ones_like(V))
    g = H.run_mesh(cam, mesh)
    fid, _, _ = orc.zbuffer(cam, V, F[5:6])
    assert set(np.unique(g["face_id"])) <= {-1, 5}
    np.testing.assert_array_equal(g["face_id"].reshape(-1) == 5, fid == 0)
    assert g["K"] == (g["tile_range"][:, 1] - g["tile_range"][:, 0]).sum()

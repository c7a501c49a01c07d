"""GPU parity of gm_zbuffer_direct (the z-buffer over (triangle, pixel) pairs,
no triangle lists): the same face ids as the tile z-buffer bit for bit, and
the CPU oracle's brute-force z-buffer up to near ties ("A Lightweight and
Differentiable Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Design
Details > Mesh rasterizer, item 1)."""

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu

TIE = 1e-6


def _quad(z, half, col=0.5):
    """Two triangles of a square at depth z (world z = -z seen from the origin
    camera below), half-width half."""
    V = np.array([[-half, -half, z], [half, -half, z], [half, half, z], [-half, half, z]], np.float32)
    return V, np.array([[0, 1, 2], [0, 2, 3]], np.int32)


def _big_scene(seed, W, H):
    """A quad that fills the image, 40 triangles of several thousand pixels at
    random depths in front of it, and a small-triangle soup: small, queued and
    huge triangles in one mesh."""
    rng = np.random.default_rng(seed)
    cam = scenes.look_at((0, 0, 0.0), (0, 0, 1.0), W, H, 0.9 * W, 0.9 * W)
    Vq, Fq = _quad(3.0, 4.0)
    Vs, Fs = [Vq], [Fq]
    n = 4
    for _ in range(40):
        c = np.array([rng.uniform(-1.2, 1.2), rng.uniform(-0.8, 0.8), rng.uniform(1.5, 2.9)])
        tri = c + rng.normal(0, 0.35, (3, 3)) * np.array([1, 1, 0.2])
        Vs.append(tri.astype(np.float32))
        Fs.append(np.array([[n, n + 1, n + 2]], np.int32))
        n += 3
    sv, sf = scenes.triangle_soup(rng, 3000, (-1.5, -1.0, 1.2), (1.5, 1.0, 2.8), 0.03)
    Vs.append(sv.astype(np.float32))
    Fs.append(sf.astype(np.int32) + n)
    V = np.concatenate(Vs).astype(np.float32)
    F = np.concatenate(Fs).astype(np.int32)
    return cam, scenes.Mesh(V, F, np.ones_like(V))


def _cases():
    tiny = scenes.tiny()
    sph = scenes.sphere512()
    soup = scenes.soup1080(n_gauss=10, n_tri=40_000)
    ragged = scenes.look_at((0.3, 0.5, 2.6), (0, 0, 0), 101, 77, 90, 95, 47.3, 40.1)
    close = scenes.look_at((0.1, 0.2, 1.6), (0, 0, 0), 130, 96, 120, 120)
    return [("tiny", tiny.camera, tiny.mesh), ("sphere512", sph.camera, sph.mesh),
            ("ragged", ragged, tiny.mesh), ("close", close, sph.mesh),
            ("soup_40k", soup.camera, soup.mesh), ("big", *_big_scene(5, 256, 192))]


@pytest.fixture(scope="module", params=_cases(), ids=lambda c: c[0])
def case(request):
    H.need_gpu()
    return request.param


def test_direct_equals_tile_zbuffer(case):
    name, cam, mesh = case
    direct = H.run_zbuffer_direct(cam, mesh)
    tile = H.run_mesh(cam, mesh)["face_id"]
    print("%s: %d covered px" % (name, (tile >= 0).sum()))
    assert (tile >= 0).any()
    np.testing.assert_array_equal(direct, tile)


def test_direct_matches_brute_force(case, orc):
    name, cam, mesh = case
    if cam.width * cam.height > 600_000:
        pytest.skip("brute force too slow at this size; covered by the tile comparison")
    gpu = H.run_zbuffer_direct(cam, mesh)
    fid, best, second = orc.zbuffer(cam, mesh.verts, mesh.faces)
    fid = fid.reshape(cam.height, cam.width)
    tie = (second <= best * (1 + TIE)).reshape(fid.shape) & (fid >= 0)
    bad = (gpu != fid) & ~tie
    assert not bad.any(), np.argwhere(bad)[:10]


def test_big_scene_takes_the_queue():
    """The big scene's quad and large triangles exceed the small-triangle
    limit (2048 box pixels), so the chunked pass draws them."""
    cam, mesh = _big_scene(5, 256, 192)
    V, F = mesh.verts.astype(np.float64), mesh.faces
    u = 0.9 * 256 * V[:, 0] / V[:, 2] + 128
    v = 0.9 * 256 * V[:, 1] / V[:, 2] + 96
    w = np.ptp(u[F], axis=1).clip(0, 256) * np.ptp(v[F], axis=1).clip(0, 192)
    assert (w > 4096).sum() >= 10


def test_giant_triangles_past_two_to_the_21():
    """A quad filling a 2100 x 1100 image: box pixel indices beyond 2^21 take the
    integer-division branch of the box walk; every pixel is covered by the quad
    and ties on its diagonal go to the smaller face id."""
    H.need_gpu()
    cam = scenes.look_at((0, 0, 0.0), (0, 0, 1.0), 2100, 1100, 1000, 1000)
    V, F = _quad(2.0, 4.0)
    mesh = scenes.Mesh(V, F, np.ones_like(V))
    direct = H.run_zbuffer_direct(cam, mesh)
    tile = H.run_mesh(cam, mesh)["face_id"]
    np.testing.assert_array_equal(direct, tile)
    assert np.all(direct >= 0)


def test_empty_and_degenerate_meshes():
    H.need_gpu()
    cam = scenes.look_at((0, 0, 3), (0, 0, 0), 40, 24, 30, 30)
    assert np.all(H.run_zbuffer_direct(cam, scenes.empty_mesh()) == -1)
    V = np.array([[0, 0, 4.0], [1, 0, 4], [0, 1, 4],
                  [-1, -1, 2.995], [1, -1, 1.0], [0, 1, 1.0],
                  [0, 0, 1.0], [0.5, 0.5, 1.0], [1, 1, 1.0],
                  [50, 50, 0], [51, 50, 0], [50, 51, 0],
                  [-0.5, -0.5, 0], [0.5, -0.5, 0], [0, 0.5, 0]], np.float32)
    F = np.array([[0, 1, 2], [3, 4, 5], [6, 7, 8], [9, 10, 11], [12, 13, 99], [12, 13, 14]], np.int32)
    mesh = scenes.Mesh(V, F, np.ones_like(V))
    direct = H.run_zbuffer_direct(cam, mesh)
    np.testing.assert_array_equal(direct, H.run_mesh(cam, mesh)["face_id"])
    assert set(np.unique(direct)) == {-1, 5}

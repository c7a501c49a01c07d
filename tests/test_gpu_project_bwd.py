"""GPU parity of gm_project_gaussians_bwd -- the projection / SH backward that
completes the Gaussian training gradients ("A Lightweight and Differentiable
Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Hybrid rendering:
everything is differentiable; projection and SH adapted from gsplat) --
against the oracle's central differences of its double-precision projection."""

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu

# Per parameter: |gpu - fd| <= RTOL |fd| + ATOL + COND_K * cond, where cond is how far
# the oracle's own gradient moves when every fp32 input moves by one ulp (the kernel
# reads the same fp32 inputs and computes in fp32, so its error is of that order).
RTOL, ATOL, COND_K = 1e-3, 1e-5, 8.0
H_STEP = 1e-3


def _cases():
    tiny = scenes.tiny()
    sph = scenes.sphere512()
    soup = scenes.soup1080(n_gauss=50_000, n_tri=10)
    out = [("tiny_rgb", tiny.camera, tiny.gaussians), ("sphere_rgb", sph.camera, sph.gaussians),
           ("soup_sh3", soup.camera, soup.gaussians)]
    for d in (0, 1, 2):
        g = soup.gaussians
        k = (d + 1) ** 2
        out.append(("soup_sh%d" % d, soup.camera,
                    scenes.Gaussians(g.means[:20000], g.log_scales[:20000], g.quats[:20000], g.logits[:20000],
                                     np.ascontiguousarray(g.colors[:20000, :k]), d)))
    orbit = scenes.orbit1080(n_gauss=50_000, levels=1)
    out.append(("orbit_view3_sh3", orbit.cameras[3], orbit.gaussians))
    return out


def _one_ulp(g, rng):
    def nudge(a):
        a = np.asarray(a, np.float32)
        up = rng.random(a.shape) < 0.5
        return np.where(up, np.nextafter(a, np.float32(np.inf)), np.nextafter(a, np.float32(-np.inf))).astype(
            np.float32)
    return scenes.Gaussians(nudge(g.means), nudge(g.log_scales), nudge(g.quats), nudge(g.logits), nudge(g.colors),
                            g.sh_degree)


def _compare(orc, name, cam, g, v, pick, gpu, rng, vd=None):
    P = orc.proj_nparams(g.sh_degree)
    gids = np.repeat(pick, P).astype(np.int32)
    params = np.tile(np.arange(P), len(pick)).astype(np.int32)
    hs = np.full(len(gids), H_STEP)
    fd, st = orc.project_fd(cam, g, v, gids, params, hs, v_depth_model=vd)
    fd2, st2 = orc.project_fd(cam, _one_ulp(g, rng), v, gids, params, hs, v_depth_model=vd)
    cond = np.abs(fd2 - fd)
    ok = (st == 0) & (st2 == 0)
    got = gpu[gids, params]
    err = np.abs(got - fd)
    tol = RTOL * np.abs(fd) + ATOL + COND_K * cond
    bad = ok & (err > tol)
    print("%s: %d parameters, %d checked, %d at a decision boundary, max err/tol %.3g" % (
        name, len(gids), ok.sum(), (~ok).sum(), float(np.max(err[ok] / tol[ok]))))
    if bad.any():
        i = np.flatnonzero(bad)[:10]
        raise AssertionError("projection gradient mismatch (g, param, gpu, fd, tol):\n" + "\n".join(
            "%d %d %.9g %.9g %.3g" % (gids[j], params[j], got[j], fd[j], tol[j]) for j in i))
    assert (~ok).mean() < 0.02


@pytest.fixture(scope="module", params=_cases(), ids=lambda c: c[0])
def case(request):
    H.need_gpu()
    return request.param


def test_projection_backward_matches_fd(case, orc):
    name, cam, g = case
    N = len(g.means)
    rng = np.random.default_rng(31)
    v = rng.normal(size=(N, 12)).astype(np.float32)
    v[:, 10:] = 0.0
    v[:, 0:2] *= 0.1          # pixel-scale fields
    v[:, 2:5] *= 1e-3 * 10.0  # conic entries ~ 1 / px^2
    radii, (vm, vls, vq, vlo, vc) = H.run_project_bwd(cam, g, v)
    gpu = np.concatenate([vm, vls, vq, vlo[:, None], vc.reshape(N, -1)], 1)
    P = orc.proj_nparams(g.sh_degree)
    assert gpu.shape[1] == P
    vis = np.flatnonzero(radii > 0)
    culled = np.flatnonzero(radii == 0)
    assert len(vis) > 0
    np.testing.assert_array_equal(gpu[culled], 0.0)  # culled: zero gradients, every row written
    pick = rng.choice(vis, size=min(96, len(vis)), replace=False)
    _compare(orc, name, cam, g, v, pick, gpu, rng)


def test_depth_model_gradient_matches_fd(case, orc):
    """dL/d(g_u, g_v, sigma_z) of the soft split's depth model chained into the
    3D parameters (record gradient zero, so only that chain is exercised)."""
    name, cam, g = case
    N = len(g.means)
    rng = np.random.default_rng(37)
    v = np.zeros((N, 12), np.float32)
    vd = rng.normal(size=(N, 4)).astype(np.float32)
    vd[:, 3] = 0.0
    radii, (vm, vls, vq, vlo, vc) = H.run_project_bwd(cam, g, v, v_depth_model=vd)
    gpu = np.concatenate([vm, vls, vq, vlo[:, None], vc.reshape(N, -1)], 1)
    vis = np.flatnonzero(radii > 0)
    np.testing.assert_array_equal(gpu[np.flatnonzero(radii == 0)], 0.0)
    np.testing.assert_array_equal(vlo, 0.0)  # opacity and colour do not enter the depth model
    np.testing.assert_array_equal(vc, 0.0)
    pick = rng.choice(vis, size=min(96, len(vis)), replace=False)
    _compare(orc, name + "_depth_model", cam, g, v, pick, gpu, rng, vd=vd)


def test_accumulate_adds(case, orc):
    name, cam, g = case
    N = len(g.means)
    rng = np.random.default_rng(5)
    v = rng.normal(size=(N, 12)).astype(np.float32)
    _, first = H.run_project_bwd(cam, g, v)
    _, twice = H.run_project_bwd(cam, g, v, accumulate_into=first)
    for a, b in zip(first, twice):
        np.testing.assert_allclose(b, 2.0 * a, rtol=1e-6, atol=0)


def test_chain_from_composite_backward(orc):
    """The whole Gaussian gradient chain on the 64 x 64 scene: composite backward
    into v_splats, projection backward into the 3D parameters, against the
    oracle's central differences of the projection for the same v_splats."""
    H.need_gpu()
    sc = scenes.tiny()
    cam, g = sc.camera, sc.gaussians
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    r = gm.HybridRenderer(cam, bg=sc.bg)
    r.upload(sc.mesh, g)
    r.forward()
    gr = [torch.as_tensor(x).cuda() for x in scenes.upstream_grads(3, cam.width, cam.height)]
    v_splats, _, _ = r.backward(*gr, mesh_grads=False)
    v = v_splats.cpu().numpy()
    radii, (vm, vls, vq, vlo, vc) = H.run_project_bwd(cam, g, v)
    N = len(g.means)
    gpu = np.concatenate([vm, vls, vq, vlo[:, None], vc.reshape(N, -1)], 1)
    used = np.flatnonzero(np.abs(v).sum(1) > 0)
    assert len(used) > 50
    _compare(orc, "tiny_chain", cam, g, v, used, gpu, np.random.default_rng(8))

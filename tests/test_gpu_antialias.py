"""GPU parity of the analytic edge antialiasing ("A Lightweight and
Differentiable Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Mesh
rasterizer item 3; Hybrid rendering: the two-layer equation over a fractional
coverage) against the CPU oracle.

- gm_mesh_edges: bit-exact adjacency;
- gm_antialias over the GPU's own mesh images (the oracle reads the same face
  ids, depths and colours): coverage and premultiplied colour within 2e-6 (the
  decisions are the same fp32 operations on both sides, the crossing is fp64
  on both; what remains is the fp32 sum of the weights), split depth and tile
  bounds exact;
- the composite over that layer (front and back chains, hard and soft split)
  within 1e-4, with the occlusion cull on the antialiased tile bounds changing
  nothing;
- the backward (Gaussians of both chains, the layer, the silhouette vertices
  and the interpolation) against the oracle's central differences;
- the renderer classes with antialias=True against the per-call path."""

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu

ATOL_IMG = 1e-4
G_ATOL, G_RTOL = 1e-5, 1e-3
SOFTNESS = 1.0


def _scene(name):
    if name == "tiny":
        return scenes.tiny()
    if name == "sphere512":
        return scenes.sphere512()
    if name == "soup_small":
        s = scenes.soup1080(n_gauss=150_000, n_tri=30_000)
        cam = scenes.look_at((0, 0, 6), (0, 0, 0), 480, 272, 300, 300)
        return scenes.Scene(s.name, [cam], s.mesh, s.gaussians, s.bg)
    if name == "orbit_small":
        s = scenes.orbit1080(n_gauss=100_000, levels=5)
        cam = scenes.look_at((5.0, 0.0, 0.0), (0, 0, 0), 640, 360, 400, 400)
        return scenes.Scene(s.name, [cam], s.mesh, s.gaussians, s.bg)
    raise KeyError(name)


def aa_pipeline(scene, softness=0.0, cull=True):
    cam = scene.camera
    m = H.run_mesh(cam, scene.mesh)
    aa = H.run_antialias(cam, scene.mesh, m)
    sp, rad, tt, dm = H.run_project(cam, scene.gaussians, scene.bg, depth_model=True)
    b = H.run_bin(cam, sp, rad, aa["tile_far"], aa["tile_full"], cull=cull and softness == 0.0)
    f = H.run_composite_aa(cam, scene.bg, b["tile_range"], b["gids"], sp, aa, softness=softness,
                           depth_model=dm if softness > 0 else None)
    return dict(cam=cam, mesh=m, aa=aa, splats=sp, radii=rad, dm=dm, bins=b, fwd=f)


@pytest.fixture(scope="module", params=["tiny", "sphere512", "soup_small", "orbit_small"])
def run(request):
    H.need_gpu()
    s = _scene(request.param)
    return request.param, s, aa_pipeline(s)


def test_mesh_edges_match_oracle(orc):
    H.need_gpu()
    for F, nV in [(scenes.icosphere(3)[1], len(scenes.icosphere(3)[0])),
                  (scenes.soup1080(n_gauss=10, n_tri=5000).mesh.faces, 15000),
                  (np.array([[0, 1, 2], [1, 0, 3], [0, 1, 4], [2, 1, 5]], np.int32), 6)]:
        np.testing.assert_array_equal(H.run_mesh_edges(F, nV), orc.mesh_edges(F))
    v, f = scenes.icosphere(7)
    np.testing.assert_array_equal(H.run_mesh_edges(f, len(v)), orc.mesh_edges(f))


def test_layer_matches_oracle(run, orc):
    name, s, r = run
    cam, m, aa = r["cam"], r["mesh"], r["aa"]
    cov, rgb, depth, codes = orc.antialias(cam, s.mesh.verts, s.mesh.faces, aa["adj"], m["face_id"],
                                           m["mesh_depth"], m["mesh_rgb"])
    np.testing.assert_allclose(aa["cov"], cov, rtol=0, atol=2e-6)
    np.testing.assert_allclose(aa["rgb_aa"], rgb, rtol=0, atol=2e-6)
    np.testing.assert_array_equal(aa["depth_aa"], depth)
    far, full = orc.tile_bounds_cov(cam, aa["cov"], aa["depth_aa"])
    np.testing.assert_array_equal(aa["tile_full"], full)
    np.testing.assert_array_equal(aa["tile_far"], far)
    frac = (cov > 0) & (cov < 1)
    reached = (m["face_id"] < 0) & (cov > 0)
    print("%s: %d px with fractional coverage, %d uncovered px reached, %d full tiles" % (
        name, frac.sum(), reached.sum(), full.sum()))
    if name != "soup_small":
        assert frac.sum() > 20


def test_forward_matches_oracle(run, orc):
    name, s, r = run
    cam, aa, f = r["cam"], r["aa"], r["fwd"]
    lists = orc.tile_lists(cam, r["splats"], r["radii"])
    o = orc.composite_fwd(cam, s.bg, r["splats"], lists, aa["depth_aa"], aa["rgb_aa"], r["mesh"]["face_id"],
                          mesh_cov=aa["cov"])
    tie = H.tie_pixels(o["margins"])
    ok = ~tie
    for k in ("rgb", "depth", "alpha"):
        err = np.abs(f[k] - o[k])
        if err.ndim == 3:
            err = err.max(-1)
        assert np.all(err[ok] <= ATOL_IMG), (k, err[ok].max(), np.argwhere((err > ATOL_IMG) & ok)[:5])
    np.testing.assert_array_equal(f["n_contrib"][ok], o["n_contrib"][ok])
    np.testing.assert_allclose(f["T"][ok], o["T"][ok], rtol=1e-4, atol=1e-7)
    assert tie.sum() <= max(2, tie.size // 1000)
    frac = (aa["cov"] > 0) & (aa["cov"] < 1) & np.isfinite(aa["depth_aa"])
    print("%s: %d ties, %d px with a back chain (mean length %.1f), max |rgb err| %.2e" % (
        name, tie.sum(), frac.sum(), f["n_back"][frac].mean() if frac.any() else 0.0,
        np.abs(f["rgb"] - o["rgb"])[ok].max()))


def test_cull_changes_nothing(run):
    """Bins culled on the antialiased tile bounds give a bit-identical image."""
    name, s, r = run
    cam, aa = r["cam"], r["aa"]
    b0 = H.run_bin(cam, r["splats"], r["radii"], aa["tile_far"], aa["tile_full"], cull=False)
    f0 = H.run_composite_aa(cam, s.bg, b0["tile_range"], b0["gids"], r["splats"], aa)
    for k in ("rgb", "depth", "alpha", "T"):
        np.testing.assert_array_equal(f0[k], r["fwd"][k])
    print("%s: K %d -> %d with the cull" % (name, b0["K"], r["bins"]["K"]))


def test_soft_forward_matches_oracle(orc):
    H.need_gpu()
    s = _scene("sphere512")
    r = aa_pipeline(s, softness=SOFTNESS)
    cam, aa, f = r["cam"], r["aa"], r["fwd"]
    lists = orc.tile_lists(cam, r["splats"], r["radii"])
    o = orc.composite_fwd(cam, s.bg, r["splats"], lists, aa["depth_aa"], aa["rgb_aa"], r["mesh"]["face_id"],
                          mesh_cov=aa["cov"], depth_model=r["dm"], softness=SOFTNESS)
    ok = ~H.tie_pixels(o["margins"])
    for k in ("rgb", "depth", "alpha"):
        err = np.abs(f[k] - o[k])
        if err.ndim == 3:
            err = err.max(-1)
        assert np.all(err[ok] <= ATOL_IMG), (k, err[ok].max())
    assert (~ok).sum() <= max(2, ok.size // 1000)


def _fd_gauss(rng, r, n):
    """Half of the sample among Gaussians near a pixel with fractional coverage."""
    aa, sp, rad = r["aa"], r["splats"], r["radii"]
    frac = (aa["cov"] > 0) & (aa["cov"] < 1)
    Hh, W = frac.shape
    ix = np.clip(np.floor(sp[:, 0]).astype(np.int64), 0, W - 1)
    iy = np.clip(np.floor(sp[:, 1]).astype(np.int64), 0, Hh - 1)
    pad = np.zeros_like(frac)
    for dj in range(-3, 4):
        for di in range(-3, 4):
            pad |= np.roll(np.roll(frac, dj, 0), di, 1)
    near = (rad > 0) & pad[iy, ix]
    pick = []
    for pool, k in ((np.flatnonzero(near), n // 2), (np.flatnonzero((rad > 0) & ~near), n)):
        k = min(k, len(pool), n - len(pick))
        pick.extend(rng.choice(pool, k, replace=False).tolist())
    return np.sort(np.asarray(pick, np.int64))


def _steps(splats, gid, fld):
    s = splats[gid]
    h = np.empty(len(gid))
    h[fld <= 1] = 1e-3
    sc = np.maximum(np.abs(s[:, 2]), np.abs(s[:, 4]))
    mid = (fld >= 2) & (fld <= 4)
    h[mid] = 1e-4 * sc[mid]
    h[fld == 5] = 1e-4
    h[(fld >= 6) & (fld <= 8)] = 1e-2
    h[fld == 9] = 1e-5 * s[fld == 9, 9]
    return h


@pytest.mark.parametrize("name,n_gauss,n_vert,softness", [("tiny", 400, 42, 0.0), ("sphere512", 200, 150, 0.0),
                                                          ("sphere512", 150, 100, SOFTNESS)])
def test_backward_matches_finite_differences(name, n_gauss, n_vert, softness, orc):
    H.need_gpu()
    s = _scene(name)
    r = aa_pipeline(s, softness=softness)
    cam, m, aa, f = r["cam"], r["mesh"], r["aa"], r["fwd"]
    grads = scenes.upstream_grads(29, cam.width, cam.height)
    b = H.run_backward_aa(cam, s.bg, f, grads, len(r["radii"]), s.mesh, m, aa["adj"])
    lists = orc.tile_lists(cam, r["splats"], r["radii"])
    rng = np.random.default_rng(12)
    pick = _fd_gauss(rng, r, n_gauss)
    gid, fld = np.repeat(pick, 10), np.tile(np.arange(10), len(pick))
    soft = dict(depth_model=r["dm"], softness=softness) if softness > 0 else {}
    fd, st = orc.composite_fd(cam, np.float64(s.bg), r["splats"], r["radii"], lists, aa["depth_aa"], aa["rgb_aa"],
                              m["face_id"], grads, gid, fld, _steps(r["splats"], gid, fld), mesh_cov=aa["cov"],
                              **soft)
    got = b["v_splats"][gid, fld].astype(np.float64)
    ok = st == 0
    bad = ok & (np.abs(got - fd) > G_ATOL + G_RTOL * np.abs(fd))
    for k in np.nonzero(bad)[0][:10]:
        print("  gaussian %d field %d: gpu %.7g fd %.7g" % (gid[k], fld[k], got[k], fd[k]))
    print("%s: %d splat parameters checked, %d excluded" % (name, ok.sum(), (~ok).sum()))
    assert not bad.any()
    assert ok.sum() >= 0.75 * len(st)
    # mesh vertices through the layer: half of them on silhouette edges
    frac = (aa["cov"] > 0) & (aa["cov"] < 1)
    covered = m["face_id"] >= 0
    sil_faces = np.unique(m["face_id"][frac & covered])
    all_faces = np.unique(m["face_id"][covered])
    vs = np.unique(s.mesh.faces[sil_faces].reshape(-1))
    va = np.unique(s.mesh.faces[all_faces].reshape(-1))
    verts = np.unique(np.concatenate([rng.choice(vs, min(len(vs), n_vert // 2), replace=False),
                                      rng.choice(va, min(len(va), n_vert // 2), replace=False)]))
    vid, vf = np.repeat(verts, 6), np.tile(np.arange(6), len(verts))
    vh = np.where(vf < 3, 1e-6, 1e-2)
    args = (cam, np.float64(s.bg))
    rest = (s.mesh.faces, s.mesh.vcol, m["face_id"].reshape(-1), r["splats"], lists, m["mesh_depth"].reshape(-1),
            m["mesh_rgb"].reshape(-1, 3), grads, vid, vf, vh)
    vfd, vst = orc.mesh_fd(*args, s.mesh.verts, *rest, adj=aa["adj"], **soft)
    vgot = np.where(vf < 3, b["v_verts"][vid, np.minimum(vf, 2)], b["v_vcol"][vid, np.maximum(vf - 3, 0)])
    vok = vst == 0
    sens = np.zeros(len(vid))
    for V2 in H.input_ulp_perturbations(cam, s.mesh.verts, draws=2):
        v2, st2 = orc.mesh_fd(*args, V2, *rest, adj=aa["adj"], **soft)
        sens = np.maximum(sens, np.where(st2 == 0, np.abs(v2 - vfd), np.inf))
    vok &= np.isfinite(sens)
    vbad = vok & (np.abs(vgot - vfd) > G_ATOL + G_RTOL * np.abs(vfd) + 4 * sens)
    for k in np.nonzero(vbad)[0][:10]:
        print("  vertex %d field %d: gpu %.7g fd %.7g" % (vid[k], vf[k], vgot[k], vfd[k]))
    on_sil = np.isin(vid, vs)
    print("%s: %d mesh parameters checked (%d on silhouettes), %d excluded (%s)" % (
        name, vok.sum(), (vok & on_sil).sum(), (~vok).sum(),
        {orc.FD_STATUS.get(v, "ulp-sensitivity"): int((vst[~vok] == v).sum()) for v in np.unique(vst[~vok])}))
    assert not vbad.any()
    # a vertex moves the depth of every pixel of its faces and the silhouettes near
    # them: on the 512 px sphere, where the Gaussians lie on the surface, some of
    # those pixels flip a depth test or a crossing decision within the step and are
    # reported, not compared (with a position step of 1e-6, 83 % of these requests
    # are smooth for the oracle on its own inputs; measured on the GPU's layer,
    # 60 to 64 % pass every exclusion, against 40 % with a step of 2e-5)
    assert vok.sum() >= 0.55 * len(vst) and (vok & on_sil & (vf < 3)).sum() > 20


def test_renderer_antialias_matches_calls():
    """HybridRenderer(antialias=True) reproduces the per-call path bit for bit in the
    forward pass; its backward gives the same gradients up to the order of atomic sums;
    a captured graph replays it."""
    H.need_gpu()
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    s = _scene("sphere512")
    r = aa_pipeline(s)
    cam = r["cam"]
    rr = gm.HybridRenderer(cam, bg=s.bg, antialias=True)
    rr.upload(s.mesh, s.gaussians)
    rgb, depth, alpha = (H.host(t) for t in rr.forward())
    np.testing.assert_array_equal(H.host(rr.cov), r["aa"]["cov"])
    np.testing.assert_array_equal(rgb, r["fwd"]["rgb"])
    np.testing.assert_array_equal(depth, r["fwd"]["depth"])
    np.testing.assert_array_equal(alpha, r["fwd"]["alpha"])
    grads = scenes.upstream_grads(31, cam.width, cam.height)
    b = H.run_backward_aa(cam, s.bg, r["fwd"], grads, len(r["radii"]), s.mesh, r["mesh"], r["aa"]["adj"])
    vs, vv, vc = rr.backward(*(torch.as_tensor(x).cuda() for x in grads))
    for got, want in ((H.host(vs), b["v_splats"]), (H.host(vv), b["v_verts"]), (H.host(vc), b["v_vcol"])):
        scale = np.abs(want).max(0, keepdims=True) + 1e-12
        assert np.all(np.abs(got - want) <= 1e-4 * np.abs(want) + 1e-5 * scale)
    graph = rr.capture_step(*(torch.as_tensor(x).cuda() for x in grads))
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(H.host(rr.out_rgb), rgb)
    assert not rr.overflowed()


def test_multiview_antialias_matches_single_views():
    H.need_gpu()
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    sc = scenes.orbit1080(n_gauss=40_000, levels=4)
    cams = sc.cameras[:3]
    mv = gm.MultiViewRenderer(cams, bg=sc.bg, streams=2, antialias=True)
    mv.upload(sc.mesh, sc.gaussians)
    outs = [[t.clone() for t in o] for o in mv.forward()]
    grads = [[torch.as_tensor(x).cuda() for x in scenes.upstream_grads(50 + k, c.width, c.height)]
             for k, c in enumerate(cams)]
    res = [x.clone() for x in mv.backward(grads)]
    torch.cuda.synchronize()
    assert not mv.overflowed()
    sum_v = torch.zeros_like(res[5])
    for k, c in enumerate(cams):
        r = gm.HybridRenderer(c, bg=sc.bg, antialias=True)
        r.upload(sc.mesh, sc.gaussians)
        rgb, depth, alpha = r.forward()
        assert torch.equal(rgb, outs[k][0]) and torch.equal(depth, outs[k][1]) and torch.equal(alpha, outs[k][2])
        _, v_verts, _ = r.backward(*grads[k])
        sum_v += v_verts
    torch.testing.assert_close(res[5], sum_v, rtol=1e-4, atol=1e-4 * float(sum_v.abs().max()))

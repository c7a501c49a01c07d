"""GPU parity of the soft split at the mesh surface ("A Lightweight and
Differentiable Renderer for Joint Mesh and 3D Gaussian Splat Scenes", Hybrid
rendering: a Gaussian that straddles the mesh is only partly in front of it)
against the CPU oracle.

- the projection's depth model (g, sigma_z) against the oracle's fp64 one,
  within a bound derived from the fp32 arithmetic and the conditioning of
  (Sigma_uv + 0.3 I);
- the soft forward composite against the oracle's (same inputs, same fp32
  decisions; tie pixels left out as for the hard split), and bit-identical to
  the hard split at pixels the mesh does not cover;
- the soft backward (record fields, depth-model fields, and the mesh vertices
  through dL/dD at the split) against the oracle's central differences;
- the renderer classes with softness > 0 against the per-call path;
- the logistic form of the front fraction on the same checks (forward, skip,
  finite differences)."""

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu

SOFTNESS = 1.0
ATOL_IMG = 1e-4
G_ATOL, G_RTOL = 1e-5, 1e-3
F_GU, F_GV, F_SZ = 12, 13, 14
FIELDS = {0: "mx", 1: "my", 2: "ca", 3: "cb", 4: "cc", 5: "op", 6: "r", 7: "g", 8: "b", 9: "z",
          F_GU: "g_u", F_GV: "g_v", F_SZ: "sigma_z"}


def _scene(name):
    if name == "tiny":
        return scenes.tiny()
    if name == "sphere512":
        return scenes.sphere512()
    if name == "soup_small":
        s = scenes.soup1080(n_gauss=150_000, n_tri=30_000)
        cam = scenes.look_at((0, 0, 6), (0, 0, 0), 480, 272, 300, 300)
        return scenes.Scene(s.name, [cam], s.mesh, s.gaussians, s.bg)
    raise KeyError(name)


def soft_pipeline(scene, softness=SOFTNESS, split=0):
    """Mesh, projection with the depth model, bins without the occlusion cull
    (the soft split turns it off), soft composite."""
    cam = scene.camera
    m = H.run_mesh(cam, scene.mesh)
    sp, rad, tt, dm = H.run_project(cam, scene.gaussians, scene.bg, depth_model=True)
    b = H.run_bin(cam, sp, rad, m["tile_far"], m["tile_full"], cull=False)
    f = H.run_composite(cam, scene.bg, b["tile_range"], b["gids"], sp, m["mesh_depth"], m["mesh_rgb"],
                        m["face_id"], softness=softness, depth_model=dm, soft_split=split)
    return dict(cam=cam, mesh=m, splats=sp, radii=rad, dm=dm, bins=b, fwd=f, split=split)


# scene, front fraction (0: Phi, 1: logistic)
@pytest.fixture(scope="module", params=[("tiny", 0), ("sphere512", 0), ("soup_small", 0), ("tiny", 1),
                                        ("sphere512", 1)], ids=lambda p: p[0] + ("_logistic" if p[1] else ""))
def run(request):
    H.need_gpu()
    name, split = request.param
    s = _scene(name)
    return name + ("_logistic" if split else ""), s, soft_pipeline(s, split=split)


def _quat_rot(q):
    q = q.astype(np.float64)
    q = q / np.linalg.norm(q, axis=1, keepdims=True)
    w, x, y, z = q.T
    return np.stack([
        np.stack([1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)], -1),
        np.stack([2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)], -1),
        np.stack([2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)], -1)], 1)


def test_depth_model_matches_oracle(run, orc):
    """g = (Sigma_uv + 0.3 I)^-1 Sigma_uv,z and sigma_z^2 = Sigma_zz - Sigma_uv,z . g.
    Bound: the kernel forms g from the fp32 conic, so |dg| <= 128 eps (cond |g| +
    sqrt(lam_max Sigma_zz) / lam_min) (|Sigma_uv,z|^2 <= lam_max Sigma_zz); the
    variance loses 64 eps (Sigma_zz + sqrt(lam_max Sigma_zz) |g|) to cancellation plus
    |Sigma_uv,z| |dg|."""
    name, s, r = run
    cam, g = r["cam"], s.gaussians
    want = orc.project_depth_model(cam, g)
    vis = np.flatnonzero(r["radii"] > 0)
    got = r["dm"][vis].astype(np.float64)
    ref = want[vis].astype(np.float64)
    # eigenvalues of Sigma_uv + 0.3 I from the conic (its inverse) of the projected record
    a, b, c = (r["splats"][vis, k].astype(np.float64) for k in (2, 3, 4))
    tr, det = a + c, a * c - b * b
    disc = np.sqrt(np.maximum(0.25 * tr * tr - det, 0.0))
    lam_min, lam_max = 1.0 / (0.5 * tr + disc), 1.0 / (0.5 * tr - disc)
    cond = lam_max / lam_min
    # Sigma_zz = |row 2 of R_cam R(q) S|^2
    Rq = _quat_rot(g.quats[vis])
    S = np.exp(g.log_scales[vis].astype(np.float64))
    WM2 = np.einsum("k,nkj->nj", cam.R[2].astype(np.float64), Rq) * S
    szz = (WM2 ** 2).sum(1)
    gn = np.linalg.norm(ref[:, :2], axis=1)
    eps = H.EPS32
    cross = np.sqrt(lam_max * szz)
    tol_g = 128 * eps * (cond * gn + cross / lam_min)
    err_g = np.linalg.norm(got[:, :2] - ref[:, :2], axis=1)
    assert np.all(err_g <= tol_g), (err_g / tol_g).max()
    tol_var = 64 * eps * (szz + cross * gn) + cross * tol_g + 1e-12
    err_var = np.abs(got[:, 2] ** 2 - ref[:, 2] ** 2)
    assert np.all(err_var <= tol_var), (err_var / tol_var).max()
    print("%s: %d Gaussians, max err/tol g %.3g, var %.3g; sigma_z median %.3g" % (
        name, len(vis), (err_g / tol_g).max(), (err_var / tol_var).max(), np.median(ref[:, 2])))


def test_reach_bounds_the_depth_slope(run):
    """The reach R (4th float of the depth model) bounds g . (p - mean2d) at
    every pixel centre where alpha can reach 1/255, checked by brute force over
    the Gaussian's pixel rectangle (fp64 from the record), and is not loose."""
    name, s, r = run
    sp, dm, rad = r["splats"], r["dm"], r["radii"]
    vis = np.flatnonzero(rad > 0)
    rng = np.random.default_rng(3)
    pick = rng.choice(vis, size=min(300, len(vis)), replace=False)
    worst = 0.0
    for i in pick:
        mx, my, a, b, c, o = (float(sp[i, k]) for k in range(6))
        R = float(dm[i, 3])
        assert np.isfinite(R) and R >= 0.0
        L = np.log(255.0 * o)
        if L <= 0:
            continue
        rr = int(rad[i])
        xs = np.floor(mx) + np.arange(-rr, rr + 1) + 0.5
        ys = np.floor(my) + np.arange(-rr, rr + 1) + 0.5
        dx, dy = np.meshgrid(xs - mx, ys - my)
        sig = 0.5 * (a * dx * dx + c * dy * dy) + b * dx * dy
        inside = sig <= L
        if not inside.any():
            continue
        slope = dm[i, 0].astype(np.float64) * dx + dm[i, 1].astype(np.float64) * dy
        top = float(np.abs(slope[inside]).max())
        assert top <= R, (i, top, R)
        worst = max(worst, top / R if R > 0 else 0.0)
    print("%s: reach checked on %d Gaussians, largest |g . d| / R %.3f" % (name, len(pick), worst))
    assert worst > 0.5


def test_soft_cull_changes_nothing(run):
    """The soft split's occlusion cull (records carrying their hide depth, full
    tiles) only removes list entries every pixel of the tile would skip: the
    image is bit-identical to the unculled bins', with fewer entries."""
    name, s, r = run
    cam, m = r["cam"], r["mesh"]
    split = r["split"]
    sp, rad, tt, dm = H.run_project(cam, s.gaussians, s.bg, depth_model=True, softness=SOFTNESS, soft_split=split)
    np.testing.assert_array_equal(sp[:, :10], r["splats"][:, :10])  # only field 10 differs
    vis = rad > 0
    assert np.all(sp[vis, 10] < sp[vis, 9]) and np.all(sp[~vis, 10] == 0.0)
    b1 = H.run_bin(cam, sp, rad, m["tile_far"], m["tile_full"], cull=True, softness=SOFTNESS)
    f1 = H.run_composite(cam, s.bg, b1["tile_range"], b1["gids"], sp, m["mesh_depth"], m["mesh_rgb"],
                         m["face_id"], softness=SOFTNESS, depth_model=dm, soft_split=split)
    f0 = r["fwd"]
    for k in ("rgb", "depth", "alpha", "T"):
        np.testing.assert_array_equal(f0[k], f1[k])
    print("%s: K %d -> %d with the soft cull" % (name, r["bins"]["K"], b1["K"]))
    if m["tile_full"].any():
        assert b1["K"] < r["bins"]["K"]


def test_hidden_gaussian_skip_changes_nothing(run):
    """The per-block skip of Gaussians hidden behind the mesh only removes work:
    with every reach set to +inf (nothing skipped) the forward pass is bit-identical
    and the backward equal up to the order of the atomic sums."""
    name, s, r = run
    cam, m, b = r["cam"], r["mesh"], r["bins"]
    dm = r["dm"].copy()
    dm[:, 3] = np.inf
    f0 = H.run_composite(cam, s.bg, b["tile_range"], b["gids"], r["splats"], m["mesh_depth"], m["mesh_rgb"],
                         m["face_id"], softness=SOFTNESS, depth_model=dm, soft_split=r["split"])
    f1 = r["fwd"]
    for k in ("rgb", "depth", "alpha", "T", "n_contrib"):
        np.testing.assert_array_equal(f0[k], f1[k])
    grads = scenes.upstream_grads(13, cam.width, cam.height)
    N = len(r["radii"])
    g0 = H.run_composite_bwd(cam, s.bg, f0, grads, N)
    g1 = H.run_composite_bwd(cam, s.bg, f1, grads, N)
    for k in ("v_splats", "v_depth_model"):
        scale = np.abs(g0[k]).max(0, keepdims=True) + 1e-12
        assert np.all(np.abs(g1[k] - g0[k]) <= 1e-5 * np.abs(g0[k]) + 1e-6 * scale), k
    np.testing.assert_array_equal(g0["v_mesh_depth"], g1["v_mesh_depth"])


def test_soft_forward_matches_oracle(run, orc):
    name, s, r = run
    cam, f, m = r["cam"], r["fwd"], r["mesh"]
    lists = orc.tile_lists(cam, r["splats"], r["radii"])
    o = orc.composite_fwd(cam, s.bg, r["splats"], lists, m["mesh_depth"], m["mesh_rgb"], m["face_id"],
                          depth_model=r["dm"], softness=SOFTNESS, split=r["split"])
    tie = H.tie_pixels(o["margins"])
    ok = ~tie
    for k in ("rgb", "depth", "alpha"):
        err = np.abs(f[k] - o[k])
        if err.ndim == 3:
            err = err.max(-1)
        assert np.all(err[ok] <= ATOL_IMG), (k, err[ok].max(), np.argwhere((err > ATOL_IMG) & ok)[:5])
    np.testing.assert_array_equal(f["n_contrib"][ok], o["n_contrib"][ok])
    np.testing.assert_allclose(f["T"][ok], o["T"][ok], rtol=1e-4, atol=1e-7)
    n_tie = int(tie.sum())
    # the split matters on this scene: the soft image differs from the hard one at covered pixels
    hard = orc.composite_fwd(cam, s.bg, r["splats"], lists, m["mesh_depth"], m["mesh_rgb"], m["face_id"])
    cov = m["face_id"] >= 0
    moved = (np.abs(hard["rgb"] - o["rgb"]).max(-1) > 1e-3) & cov
    print("%s: %d px, %d ties, %d covered px changed by the split, max |rgb err| %.2e" % (
        name, tie.size, n_tie, moved.sum(), np.abs(f["rgb"] - o["rgb"])[ok].max()))
    assert n_tie <= max(2, tie.size // 1000)
    if cov.any():
        assert moved.any()


def test_uncovered_pixels_as_hard_split(run):
    """Where the mesh does not cover the pixel the soft split is the hard one: the
    same lists give bit-identical outputs there."""
    name, s, r = run
    cam, m, b = r["cam"], r["mesh"], r["bins"]
    hard = H.run_composite(cam, s.bg, b["tile_range"], b["gids"], r["splats"], m["mesh_depth"], m["mesh_rgb"],
                           m["face_id"])
    unc = m["face_id"] < 0
    for k in ("rgb", "depth", "alpha", "T", "n_contrib"):
        np.testing.assert_array_equal(hard[k][unc], r["fwd"][k][unc])


def _fd_requests(rng, r, n_gauss, fields):
    """Half of the sample among the Gaussians whose centre lies within 3 sigma_z of
    the mesh surface at its own pixel (where the split acts), half among the rest."""
    radii, sp, dm, m = r["radii"], r["splats"], r["dm"], r["mesh"]
    H_, W_ = m["face_id"].shape
    ix = np.clip(np.floor(sp[:, 0]).astype(np.int64), 0, W_ - 1)
    iy = np.clip(np.floor(sp[:, 1]).astype(np.int64), 0, H_ - 1)
    D = m["mesh_depth"][iy, ix]
    near = (radii > 0) & (m["face_id"][iy, ix] >= 0) & (np.abs(sp[:, 9] - D) < 3 * SOFTNESS * dm[:, 2])
    pick = []
    for pool, k in ((np.flatnonzero(near), n_gauss // 2), (np.flatnonzero((radii > 0) & ~near), n_gauss)):
        k = min(k, len(pool), n_gauss - len(pick))
        pick.extend(rng.choice(pool, k, replace=False).tolist())
    pick = np.sort(np.asarray(pick, np.int64))
    return np.repeat(pick, len(fields)), np.tile(np.array(list(fields)), len(pick))


def _steps(splats, dm, gid, fld):
    s, d = splats[gid], dm[gid]
    h = np.empty(len(gid))
    h[fld <= 1] = 1e-3
    sc = np.maximum(np.abs(s[:, 2]), np.abs(s[:, 4]))
    mid = (fld >= 2) & (fld <= 4)
    h[mid] = 1e-4 * sc[mid]
    h[fld == 5] = 1e-4
    h[(fld >= 6) & (fld <= 8)] = 1e-2
    # z, g and sigma_z enter through x = (D - z - g . d) / (sigma_z s): steps a small
    # fraction of sigma_z (per pixel of offset for g)
    h[fld == 9] = 1e-3 * d[fld == 9, 2]
    gsel = (fld == F_GU) | (fld == F_GV)
    h[gsel] = 1e-4 * d[gsel, 2]
    h[fld == F_SZ] = 1e-4 * d[fld == F_SZ, 2]
    return h


@pytest.mark.parametrize("name,n_gauss,n_vert,split", [("tiny", 600, 42, 0), ("sphere512", 250, 120, 0),
                                                       ("tiny", 600, 42, 1)])
def test_soft_backward_matches_finite_differences(name, n_gauss, n_vert, split, orc):
    H.need_gpu()
    s = _scene(name)
    r = soft_pipeline(s, split=split)
    cam, m, f, dm = r["cam"], r["mesh"], r["fwd"], r["dm"]
    grads = scenes.upstream_grads(17, cam.width, cam.height)
    b = H.run_composite_bwd(cam, s.bg, f, grads, len(r["radii"]), s.mesh, mesh_grads=True)
    # every pixel's dL/dD is written; zero where the mesh does not cover it
    cov = m["face_id"] >= 0
    np.testing.assert_array_equal(b["v_mesh_depth"][~cov], 0.0)
    lists = orc.tile_lists(cam, r["splats"], r["radii"])
    rng = np.random.default_rng(9)
    fields = list(range(10)) + [F_GU, F_GV, F_SZ]
    gid, fld = _fd_requests(rng, r, n_gauss, fields)
    hs = _steps(r["splats"], dm, gid, fld)
    fd, st = orc.composite_fd(cam, np.float64(s.bg), r["splats"], r["radii"], lists, m["mesh_depth"],
                              m["mesh_rgb"], m["face_id"], grads, gid, fld, hs, depth_model=dm, softness=SOFTNESS,
                              split=split)
    got = np.where(fld < 12, b["v_splats"][gid, np.minimum(fld, 11)],
                   b["v_depth_model"][gid, np.clip(fld - 12, 0, 3)]).astype(np.float64)
    ok = st == 0
    err = np.abs(got - fd)
    tol = G_ATOL + G_RTOL * np.abs(fd)
    bad = ok & (err > tol)
    for k in np.nonzero(bad)[0][:10]:
        print("  gaussian %d %s: gpu %.7g fd %.7g" % (gid[k], FIELDS[int(fld[k])], got[k], fd[k]))
    print("%s: %d parameters checked, %d excluded (%s), %d depth-model ones non-zero" % (
        name, ok.sum(), (~ok).sum(), {orc.FD_STATUS[v]: int((st == v).sum()) for v in np.unique(st[~ok])},
        int((ok & (fld >= 12) & (np.abs(fd) > 1e-6)).sum())))
    assert not bad.any()
    assert ok.sum() >= 0.8 * len(st)
    assert (ok & (fld >= 12) & (np.abs(fd) > 1e-6)).sum() > 20  # the split is exercised
    # mesh vertices: the interpolated depth now also moves each Gaussian's front part
    covered_faces = np.unique(m["face_id"][cov])
    verts = np.unique(s.mesh.faces[covered_faces].reshape(-1))
    if len(verts) > n_vert:
        verts = np.sort(rng.choice(verts, n_vert, replace=False))
    vid = np.repeat(verts, 6)
    vf = np.tile(np.arange(6), len(verts))
    vh = np.where(vf < 3, 1e-6, 1e-2)
    args = (cam, np.float64(s.bg))
    rest = (s.mesh.faces, s.mesh.vcol, m["face_id"].reshape(-1), r["splats"], lists, m["mesh_depth"].reshape(-1),
            m["mesh_rgb"].reshape(-1, 3), grads, vid, vf, vh)
    vfd, vst = orc.mesh_fd(*args, s.mesh.verts, *rest, depth_model=dm, softness=SOFTNESS, split=split)
    vgot = np.where(vf < 3, b["v_verts"][vid, np.minimum(vf, 2)], b["v_vcol"][vid, np.maximum(vf - 3, 0)])
    vok = vst == 0
    sens = np.zeros(len(vid))
    for V2 in H.input_ulp_perturbations(cam, s.mesh.verts, draws=2):
        v2, st2 = orc.mesh_fd(*args, V2, *rest, depth_model=dm, softness=SOFTNESS, split=split)
        sens = np.maximum(sens, np.where(st2 == 0, np.abs(v2 - vfd), np.inf))
    vok &= np.isfinite(sens)
    verr = np.abs(vgot - vfd)
    vbad = vok & (verr > G_ATOL + G_RTOL * np.abs(vfd) + 4 * sens)
    for k in np.nonzero(vbad)[0][:10]:
        print("  vertex %d field %d: gpu %.7g fd %.7g" % (vid[k], vf[k], vgot[k], vfd[k]))
    print("%s: %d mesh parameters checked, %d excluded" % (name, vok.sum(), (~vok).sum()))
    assert not vbad.any()
    assert vok.sum() >= 0.75 * len(vst)


def test_renderer_soft_matches_calls():
    """HybridRenderer(softness) reproduces the per-call soft path bit for bit in
    the forward pass, and its backward (one call, Gaussian part then mesh part)
    gives the same gradients up to the order of the atomic sums."""
    H.need_gpu()
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    s = scenes.sphere512()
    r = soft_pipeline(s)
    cam = r["cam"]
    rr = gm.HybridRenderer(cam, bg=s.bg, softness=SOFTNESS)
    rr.upload(s.mesh, s.gaussians)
    rgb, depth, alpha = (H.host(t) for t in rr.forward())
    np.testing.assert_array_equal(H.host(rr.depth_model)[r["radii"] > 0], r["dm"][r["radii"] > 0])
    np.testing.assert_array_equal(rgb, r["fwd"]["rgb"])
    np.testing.assert_array_equal(depth, r["fwd"]["depth"])
    np.testing.assert_array_equal(alpha, r["fwd"]["alpha"])
    grads = scenes.upstream_grads(23, cam.width, cam.height)
    b = H.run_composite_bwd(cam, s.bg, r["fwd"], grads, len(r["radii"]), s.mesh, mesh_grads=True)
    vs, vv, vc = rr.backward(*(torch.as_tensor(x).cuda() for x in grads))
    for got, want in ((H.host(vs), b["v_splats"]), (H.host(rr.v_depth_model), b["v_depth_model"]),
                      (H.host(vv), b["v_verts"]), (H.host(vc), b["v_vcol"])):
        scale = np.abs(want).max(0, keepdims=True) + 1e-12
        assert np.all(np.abs(got - want) <= 1e-4 * np.abs(want) + 1e-5 * scale)
    np.testing.assert_array_equal(H.host(rr.v_mesh_depth), b["v_mesh_depth"])
    # captured as one graph
    graph = rr.capture_step(*(torch.as_tensor(x).cuda() for x in grads))
    graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(H.host(rr.out_rgb), rgb)
    assert not rr.overflowed()


def test_multiview_soft_matches_single_views():
    """MultiViewRenderer(softness): per view the single-view soft renderer's
    images bit for bit; summed parameter gradients equal per-view projection
    backward calls (record and depth-model gradients) accumulated in view order."""
    H.need_gpu()
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    sc = scenes.orbit1080(n_gauss=40_000, levels=3)
    cams = sc.cameras[:3]
    mv = gm.MultiViewRenderer(cams, bg=sc.bg, streams=2, softness=SOFTNESS)
    mv.upload(sc.mesh, sc.gaussians)
    outs = [[t.clone() for t in o] for o in mv.forward()]
    grads = [[torch.as_tensor(x).cuda() for x in scenes.upstream_grads(40 + k, c.width, c.height)]
             for k, c in enumerate(cams)]
    res = [x.clone() for x in mv.backward(grads)]
    torch.cuda.synchronize()
    assert not mv.overflowed()
    for k, c in enumerate(cams):
        r = gm.HybridRenderer(c, bg=sc.bg, softness=SOFTNESS)
        r.upload(sc.mesh, sc.gaussians)
        rgb, depth, alpha = r.forward()
        assert torch.equal(rgb, outs[k][0]) and torch.equal(depth, outs[k][1]) and torch.equal(alpha, outs[k][2])
    o = mv.opts
    v0 = mv.views[0]
    args = [v0.means, v0.log_scales, v0.quats, v0.logits, v0.colors]
    seq = [torch.zeros_like(a) for a in args]
    for k in range(len(cams)):
        gm.gm_project_gaussians_bwd(mv.cams[k], o, *args, mv.radii[k], mv.v_splats[k], *seq, accumulate=k > 0,
                                    v_depth_model=mv.v_depth_model[k])
    for a, b in zip(res[:5], seq):
        assert torch.equal(a, b)
    assert float(mv.v_depth_model.abs().max()) > 0.0

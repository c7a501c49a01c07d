"""GPU parity of the Gaussian steps (gm_project_gaussians, gm_bin_sort_gaussians)
against the CPU oracle ("A Lightweight and Differentiable Renderer for Joint
Mesh and 3D Gaussian Splat Scenes", Hybrid rendering: the projection, SH and
tile sorting kernels; the cull_occluded bullet; Limitations: centre-depth
order)."""

import math

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu

# radius ties: 3 sqrt(lambda_max) within this relative distance of an integer.
# lambda_max comes from the stable form m + sqrt(h^2 + b^2) of fp32 entries
# whose relative error stays below ~1e-6, so 3 sqrt(.) errs by < 1e-6.
RADIUS_TIE = 4e-6


def _proj_cases():
    tiny = scenes.tiny()
    sph = scenes.sphere512()
    soup = scenes.soup1080(n_gauss=60_000, n_tri=10)
    out = [("tiny_rgb", tiny.camera, tiny.gaussians), ("sphere_rgb", sph.camera, sph.gaussians),
           ("soup_sh3", soup.camera, soup.gaussians)]
    rng = np.random.default_rng(12)
    for d in (0, 1, 2):
        g = soup.gaussians
        k = (d + 1) ** 2
        sub = scenes.Gaussians(g.means[:20000], g.log_scales[:20000], g.quats[:20000], g.logits[:20000],
                               np.ascontiguousarray(g.colors[:20000, :k]), d)
        out.append(("soup_sh%d" % d, soup.camera, sub))
    # unnormalised quaternions, a Gaussian behind the camera, one past far
    g = tiny.gaussians
    q = g.quats * rng.uniform(0.2, 5.0, size=(len(g.quats), 1)).astype(np.float32)
    m = g.means.copy()
    m[0] = [0, 0, 10.0]
    m[1] = [0, 0, 3.995]
    out.append(("tiny_edge", tiny.camera, scenes.Gaussians(m, g.log_scales, q, g.logits, g.colors, -1)))
    return out


@pytest.fixture(scope="module", params=_proj_cases(), ids=lambda c: c[0])
def pcase(request):
    H.need_gpu()
    return request.param


def test_projection_matches_oracle(pcase, orc):
    name, cam, g = pcase
    sp, rad, tt = H.run_project(cam, g)
    osp, orad, ott, margin = orc.project(cam, g)
    tie = margin < RADIUS_TIE
    both = (rad > 0) & (orad > 0)
    mism = rad != orad
    print("%s: %d projected, %d radius ties, %d radius mismatches" % (name, (orad > 0).sum(), tie.sum(), mism.sum()))
    # a mismatch is a culled/visible flip only at a tie, or a one-unit radius step at a tie
    assert np.all(tie[mism]), np.nonzero(mism & ~tie)[0][:10]
    assert np.all(np.abs(rad[mism] - orad[mism]) <= 1)
    # culled Gaussians write zero records
    assert np.all(sp[rad == 0] == 0) and np.all(tt[rad == 0] == 0)
    ok = both & ~mism
    # mean2d = f t / z + c: ~8 fp32 operations on values up to |m| + |c| px
    m_err = np.abs(sp[ok, :2] - osp[ok, :2])
    scale = np.abs(osp[ok, :2]) + np.array([abs(cam.cx), abs(cam.cy)])
    assert np.all(m_err <= 16 * H.EPS32 * scale + 1e-5), (m_err / scale).max()
    # conic: Sigma2 entries carry an absolute fp32 error ~ eps * lambda_max; the inverse
    # amplifies it by 1 / lambda_min^2 (both eigenvalues from the oracle's fp64 values)
    a, b, c = (osp[ok, k].astype(np.float64) for k in (2, 3, 4))
    det = a * c - b * b
    tr = a + c
    lam_min_inv = 0.5 * (tr + np.sqrt(np.maximum((a - c) ** 2 + 4 * b * b, 0)))  # largest conic eigenvalue
    lam_max_inv = det / lam_min_inv                                              # smallest conic eigenvalue
    bound = 64 * H.EPS32 * lam_min_inv ** 2 / lam_max_inv
    c_err = np.abs(sp[ok, 2:5] - osp[ok, 2:5]).max(1)
    assert np.all(c_err <= bound), (c_err / bound).max()
    np.testing.assert_allclose(sp[ok, 5], osp[ok, 5], rtol=4 * H.EPS32, atol=1e-7)      # opacity
    np.testing.assert_allclose(sp[ok, 6:9], osp[ok, 6:9], rtol=0, atol=2e-6)           # colour
    np.testing.assert_allclose(sp[ok, 9], osp[ok, 9], rtol=4 * H.EPS32)               # depth
    assert np.all(sp[:, 10:] == 0)
    # tile rectangles agree except where a rectangle edge (m +- r)/16 lies within the
    # mean's error of an integer
    same_rect = tt[ok] == ott[ok]
    if not same_rect.all():
        idx = np.nonzero(ok)[0][~same_rect]
        for k in idx:
            edges = np.array([osp[k, 0] - orad[k], osp[k, 0] + orad[k], osp[k, 1] - orad[k], osp[k, 1] + orad[k]]) / 16
            assert np.min(np.abs(edges - np.round(edges))) * 16 < 1e-3, k


def test_sh_colour_clamp_and_view_dependence(orc):
    H.need_gpu()
    cam = scenes.look_at((0, 0, 3), (0, 0, 0), 64, 64, 60, 60)
    n = 256
    rng = np.random.default_rng(0)
    sh = rng.normal(0, 1.0, size=(n, 16, 3)).astype(np.float32)  # large: many colours clamp at 0
    g = scenes.Gaussians(rng.uniform(-0.5, 0.5, (n, 3)).astype(np.float32), np.full((n, 3), -3, np.float32),
                         np.tile(np.float32([1, 0, 0, 0]), (n, 1)), np.zeros(n, np.float32), sh, 3)
    sp, rad, _ = H.run_project(cam, g)
    osp, orad, _, _ = orc.project(cam, g)
    ok = (rad > 0) & (orad > 0)
    assert (sp[ok, 6:9] == 0).sum() > 50
    np.testing.assert_allclose(sp[ok, 6:9], osp[ok, 6:9], atol=2e-5)


def _bin_inputs(name):
    if name == "tiny":
        s = scenes.tiny()
    elif name == "sphere512":
        s = scenes.sphere512()
    else:
        s = scenes.soup1080(n_gauss=200_000, n_tri=40_000)
    m = H.run_mesh(s.camera, s.mesh)
    sp, rad, _ = H.run_project(s.camera, s.gaussians)
    return s.camera, sp, rad, m


@pytest.fixture(scope="module", params=["tiny", "sphere512", "soup_200k"])
def bcase(request):
    H.need_gpu()
    return (request.param,) + _bin_inputs(request.param)


@pytest.mark.parametrize("cull", [False, True])
def test_bin_sort_teacher_forced_exact(bcase, cull, orc):
    """Keys, ids and tile ranges from the GPU's own projected splats equal the
    oracle's (stable sort on (tile, depth bits), then id) bit for bit, with
    and without the occlusion cull; the pre-cull count too."""
    name, cam, sp, rad, m = bcase
    g = H.run_bin(cam, sp, rad, m["tile_far"], m["tile_full"], cull)
    keys, gids, pre = orc.bin_gaussians(cam, sp, rad, m["tile_far"], m["tile_full"], cull)
    assert g["K"] == len(keys) and g["counters"][1] == pre and g["counters"][2] == 0
    np.testing.assert_array_equal(g["keys"], keys)
    np.testing.assert_array_equal(g["gids"], gids)
    start, _ = H.lists_from_bins(cam, keys, gids)
    tr = g["tile_range"]
    cnt = np.diff(start)
    np.testing.assert_array_equal(tr[:, 1] - tr[:, 0], cnt)
    np.testing.assert_array_equal(tr[cnt > 0, 0], start[:-1][cnt > 0])
    if name == "sphere512":  # rectangles of more than 16 tiles take the warp-wide path
        assert (np.bincount(gids) > 16).any()
    print("%s cull=%d: K=%d (pre-cull %d), %d sort partitions" % (name, cull, len(keys), pre, -(-len(keys) // 3840)))


def test_sort_stability_and_ragged_sizes(orc):
    """Many Gaussians at one depth in the same tiles (ids must stay ascending),
    K not a multiple of the partition size, several thousand partitions."""
    H.need_gpu()
    cam = scenes.look_at((0, 0, 3), (0, 0, 0), 480, 272, 300, 300)
    rng = np.random.default_rng(3)
    for n in (1, 7, 3839, 3841, 50_001):
        sp = np.zeros((n, 12), np.float32)
        sp[:, 0] = rng.uniform(0, 480, n)
        sp[:, 1] = rng.uniform(0, 272, n)
        sp[:, 9] = rng.choice(np.float32([0.5, 1.0, 1.0, 2.0]), n)  # heavy duplicates
        rad = rng.integers(1, 40, n).astype(np.int32)
        g = H.run_bin(cam, sp, rad)
        keys, gids, _ = orc.bin_gaussians(cam, sp, rad)
        np.testing.assert_array_equal(g["keys"], keys)
        np.testing.assert_array_equal(g["gids"], gids)


def test_capacity_overflow_is_reported_and_contained(orc):
    H.need_gpu()
    s = scenes.tiny()
    sp, rad, tt = H.run_project(s.camera, s.gaussians)
    need = int(tt.sum())
    # synchronous mode: GM_ERR_CAPACITY with the needed count, then a retry that fits
    g = H.run_bin(s.camera, sp, rad, cap=need // 3)
    assert g["cap"] == need + 1 and g["K"] == need
    # asynchronous mode: no error at the call, the overflow flag is set, no write past cap
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    cap = need // 2
    keys = torch.zeros(cap + 64, dtype=torch.int64, device="cuda")
    gids = torch.full((cap + 64,), -1, dtype=torch.int32, device="cuda")
    tr = torch.zeros(H.n_tiles(s.camera), 2, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(4, dtype=torch.int32, device="cuda")
    ws = torch.empty(gm.gm_bin_sort_gaussians_workspace_size(len(rad), cap, 64, 64), dtype=torch.uint8, device="cuda")
    gm.gm_bin_sort_gaussians(gm.make_camera(s.camera), gm.make_opts(cull_occluded=False, tile_test=False), H.dev(sp), H.dev(rad),
                             None, None, keys, gids, tr, cap, cnt, ws, sync=False)
    c = H.host(cnt)
    assert c[0] == need and c[2] & gm.GM_FLAG_OVERFLOW
    assert np.all(H.host(gids)[cap:] == -1) and np.all(H.host(keys)[cap:] == 0)


def _largest_dropped_alpha(cam, osp, dg, dt, n_max=20000, seed=2):
    """Largest o exp(-sigma) in double, over the in-image pixel centres of tile
    dt[k], of Gaussian dg[k] (the oracle's projection osp), on a seeded sample
    of at most n_max pairs."""
    TW = (cam.width + 15) // 16
    rng = np.random.default_rng(seed)
    if len(dg) > n_max:
        sel = rng.choice(len(dg), n_max, replace=False)
        dg, dt = dg[sel], dt[sel]
    off = np.arange(16) + 0.5
    worst = 0.0
    for lo in range(0, len(dg), 4096):
        g, t = dg[lo:lo + 4096], dt[lo:lo + 4096]
        rec = osp[g].astype(np.float64)
        tx, ty = (t % TW) * 16, (t // TW) * 16
        xs = tx[:, None] + off[None, :]
        ys = ty[:, None] + off[None, :]
        dx = xs[:, None, :] - rec[:, 0, None, None]
        dy = ys[:, :, None] - rec[:, 1, None, None]
        sig = 0.5 * (rec[:, 2, None, None] * dx * dx + rec[:, 4, None, None] * dy * dy) + rec[:, 3, None, None] * dx * dy
        inside = (xs[:, None, :] < cam.width) & (ys[:, :, None] < cam.height)
        a = rec[:, 5, None, None] * np.exp(-np.maximum(sig, 0.0))
        a = np.where(inside & (sig >= 0), a, 0.0)
        worst = max(worst, float(a.max()) if a.size else 0.0)
    return worst


def _tile_test_cases():
    soup = scenes.soup1080(n_gauss=150_000, n_tri=30_000)
    cam = scenes.look_at((0, 0, 6), (0, 0, 0), 480, 272, 300, 300)
    return [("tiny", scenes.tiny()), ("sphere512", scenes.sphere512()),
            ("soup_small", scenes.Scene(soup.name, [cam], soup.mesh, soup.gaussians, soup.bg))]


@pytest.mark.parametrize("case", _tile_test_cases(), ids=lambda c: c[0])
def test_tile_test_drops_only_unreachable_pairs(case, orc):
    """With opts.tile_test each tile's list is the exact rectangle list with some
    entries removed, in the same order, and every removed (Gaussian, tile) pair
    is one whose alpha stays below 1/255 at every pixel centre of the tile
    (checked in double from the oracle's projection), so compositing cannot
    change."""
    H.need_gpu()
    name, s = case
    cam = s.camera
    sp, rad, _ = H.run_project(cam, s.gaussians)
    m = H.run_mesh(cam, s.mesh)
    ex = H.run_bin(cam, sp, rad, m["tile_far"], m["tile_full"], cull=True)
    ti = H.run_bin(cam, sp, rad, m["tile_far"], m["tile_full"], cull=True, tile_test=True)
    assert ti["K"] <= ex["K"]
    T = H.n_tiles(cam)
    TW = (cam.width + 15) // 16
    dropped_g, dropped_t = [], []
    for t in range(T):
        a0, a1 = ex["tile_range"][t]
        b0, b1 = ti["tile_range"][t]
        le = ex["gids"][a0:a1] if a1 > a0 else np.zeros(0, np.int32)
        lt = ti["gids"][b0:b1] if b1 > b0 else np.zeros(0, np.int32)
        keep = np.isin(le, lt)
        np.testing.assert_array_equal(le[keep], lt)  # same order, nothing new
        dropped_g.append(le[~keep])
        dropped_t.append(np.full((~keep).sum(), t))
    dg = np.concatenate(dropped_g)
    dt = np.concatenate(dropped_t)
    osp, _, _, _ = orc.project(cam, s.gaussians)
    worst = _largest_dropped_alpha(cam, osp, dg, dt)
    print("%s: K %d -> %d (%.1f %% dropped); largest alpha of a dropped pair %.3g" % (
        name, ex["K"], ti["K"], 100.0 * (1 - ti["K"] / max(ex["K"], 1)), worst))
    assert worst < 1.0 / 255.0
    if name == "soup_small":
        assert ti["K"] < 0.9 * ex["K"]


def test_split_binning_equals_one_call():
    """gm_sort_gaussians_by_depth + gm_bin_gaussians (the two halves the renderer
    overlaps with the mesh layer) give bit-identical keys, ids, ranges and counts
    to gm_bin_sort_gaussians, with and without the cull."""
    H.need_gpu()
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    s = scenes.sphere512()
    cam = s.camera
    m = H.run_mesh(cam, s.mesh)
    sp, rad, _ = H.run_project(cam, s.gaussians, s.bg)
    c = gm.make_camera(cam)
    T = H.n_tiles(cam)
    for cull in (False, True):
        o = gm.make_opts(s.bg, cull, -1, True)
        ref = H.run_bin(cam, sp, rad, m["tile_far"], m["tile_full"], cull=cull, tile_test=True)
        cap = ref["cap"]
        keys = torch.zeros(cap, dtype=torch.int64, device="cuda")
        gids = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
        tr = torch.full((T, 2), -5, dtype=torch.int32, device="cuda")
        cnt = torch.full((4,), -9, dtype=torch.int32, device="cuda")
        ws = torch.empty(gm.gm_bin_sort_gaussians_workspace_size(len(rad), cap, cam.width, cam.height),
                         dtype=torch.uint8, device="cuda")
        spd, radd = H.dev(sp, torch.float32), H.dev(rad, torch.int32)
        gm.gm_sort_gaussians_by_depth(c, spd, radd, cap, cnt, ws)
        K = gm.gm_bin_gaussians(c, o, spd, radd, H.dev(m["tile_far"], torch.float32),
                                H.dev(m["tile_full"], torch.uint8), keys, gids, tr, cap, cnt, ws)
        assert K == ref["K"]
        np.testing.assert_array_equal(H.host(keys)[:K].view(np.uint64), ref["keys"])
        np.testing.assert_array_equal(H.host(gids)[:K], ref["gids"])
        np.testing.assert_array_equal(H.host(tr), ref["tile_range"])
        np.testing.assert_array_equal(H.host(cnt), ref["counters"])


@pytest.fixture(scope="module")
def bench_bins():
    """The 1080p workload (1,000,000 Gaussians with degree-3 SH, 200,000-triangle
    soup) as the renderer the benchmark times bins it: its projected records,
    mesh tile bounds and its own bins (tile test and occlusion cull on)."""
    H.need_gpu()
    import differentiable_hybrid_mesh_tile_b300 as gm
    s = scenes.soup1080()
    r = gm.HybridRenderer(s.camera, bg=s.bg)
    r.upload(s.mesh, s.gaussians)
    r.forward(sync=True)
    K = int(r.K_gauss)
    out = dict(scene=s, sp=H.host(r.splats), rad=H.host(r.radii), tile_far=H.host(r.tile_far),
               tile_full=H.host(r.tile_full), keys=H.host(r.keys)[:K].view(np.uint64), gids=H.host(r.gids)[:K],
               tile_range=H.host(r.g_range), K=K, counters=H.host(r.g_counters))
    del r
    torch_sync()
    return out


def torch_sync():
    import torch
    torch.cuda.synchronize()


@pytest.mark.parametrize("cull", [False, True])
def test_bin_sort_exact_at_bench_size(bench_bins, cull, orc):
    """Rectangle bins of the full 1080p workload (6.5 M entries before the cull,
    four depth passes over 1 M keys and two tile passes) equal the oracle's
    bit for bit: keys, ids, tile ranges and counts, with and without the cull."""
    b = bench_bins
    cam = b["scene"].camera
    g = H.run_bin(cam, b["sp"], b["rad"], b["tile_far"], b["tile_full"], cull)
    keys, gids, pre = orc.bin_gaussians(cam, b["sp"], b["rad"], b["tile_far"], b["tile_full"], cull)
    assert g["K"] == len(keys) and g["counters"][1] == pre and g["counters"][2] == 0
    np.testing.assert_array_equal(g["keys"], keys)
    np.testing.assert_array_equal(g["gids"], gids)
    start, _ = H.lists_from_bins(cam, keys, gids)
    tr = g["tile_range"]
    cnt = np.diff(start)
    np.testing.assert_array_equal(tr[:, 1] - tr[:, 0], cnt)
    np.testing.assert_array_equal(tr[cnt > 0, 0], start[:-1][cnt > 0])
    print("1080p cull=%d: K=%d (pre-cull %d)" % (cull, len(keys), pre))


def test_renderer_bins_at_bench_size_thin_the_exact_bins(bench_bins, orc):
    """The renderer's own bins in the benchmark's configuration (tile test and
    cull on) are the oracle's exact culled bins with entries removed: the same
    keys in the same order for what is kept, consistent tile ranges, and every
    removed (Gaussian, tile) pair below alpha 1/255 at every pixel centre of
    its tile (a seeded sample of 20,000, in double)."""
    b = bench_bins
    s = b["scene"]
    cam = s.camera
    keys, gids, pre = orc.bin_gaussians(cam, b["sp"], b["rad"], b["tile_far"], b["tile_full"], True)
    assert b["counters"][1] == pre and b["counters"][2] == 0 and b["counters"][0] == b["K"]
    ce = ((keys >> np.uint64(32)).astype(np.int64) << 32) | gids.astype(np.int64)
    cr = ((b["keys"] >> np.uint64(32)).astype(np.int64) << 32) | b["gids"].astype(np.int64)
    keep = np.isin(ce, cr)
    assert keep.sum() == len(cr)
    np.testing.assert_array_equal(ce[keep], cr)          # same entries in the same order
    np.testing.assert_array_equal(keys[keep], b["keys"])  # with the same depth bits
    start, _ = H.lists_from_bins(cam, b["keys"], b["gids"])
    cnt = np.diff(start)
    tr = b["tile_range"]
    np.testing.assert_array_equal(tr[:, 1] - tr[:, 0], cnt)
    np.testing.assert_array_equal(tr[cnt > 0, 0], start[:-1][cnt > 0])
    osp, _, _, _ = orc.project(cam, s.gaussians)
    dg = gids[~keep]
    dt = (keys[~keep] >> np.uint64(32)).astype(np.int64)
    worst = _largest_dropped_alpha(cam, osp, dg, dt)
    print("1080p renderer bins: %d exact culled entries, %d kept (%.1f %% dropped by the tile test); largest alpha "
          "of a dropped pair %.3g" % (len(keys), len(cr), 100.0 * (1 - len(cr) / len(keys)), worst))
    assert worst < 1.0 / 255.0


def test_long_tile_lists(orc):
    """6,000 Gaussians centred in one tile (heavy depth duplicates, so the id
    order decides), plus a spread of others, binned bit-exact against the
    oracle: one tile list of more than 6,000 entries spans several sort
    partitions."""
    H.need_gpu()
    cam = scenes.look_at((0, 0, 3), (0, 0, 0), 480, 272, 300, 300)
    rng = np.random.default_rng(21)
    n_hot, n_rest = 6000, 20000
    sp = np.zeros((n_hot + n_rest, 12), np.float32)
    sp[:n_hot, 0] = rng.uniform(100.5, 110.5, n_hot)  # all inside tile (6, 6)
    sp[:n_hot, 1] = rng.uniform(100.5, 110.5, n_hot)
    sp[n_hot:, 0] = rng.uniform(0, 480, n_rest)
    sp[n_hot:, 1] = rng.uniform(0, 272, n_rest)
    sp[:, 9] = rng.choice(np.float32([0.5, 1.0, 1.0, 2.0, 3.0]), n_hot + n_rest)
    rad = np.concatenate([np.full(n_hot, 3, np.int32), rng.integers(1, 30, n_rest).astype(np.int32)])
    perm = rng.permutation(n_hot + n_rest)  # hot Gaussians spread over the ids
    sp, rad = sp[perm], rad[perm]
    g = H.run_bin(cam, sp, rad)
    keys, gids, _ = orc.bin_gaussians(cam, sp, rad)
    np.testing.assert_array_equal(g["keys"], keys)
    np.testing.assert_array_equal(g["gids"], gids)
    counts = np.bincount((keys >> np.uint64(32)).astype(np.int64))
    assert counts.max() > 2 * 2048, counts.max()

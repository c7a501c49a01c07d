"""Pins of the oracle's hybrid compositing and of its finite-difference
gradients (page "A Lightweight and Differentiable Renderer for Joint Mesh and
3D Gaussian Splat Scenes", Design Details > Hybrid rendering: front-to-back
compositing of depth-tested Gaussians over one opaque mesh layer; culling of
hidden Gaussians does not change the result)."""

import json
import math
import os

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))
A_MIN = np.float32(1.0 / 255.0)


def splat(mx, my, a, b, c, o, rgb, z):
    s = np.zeros(12, np.float32)
    s[:10] = [mx, my, a, b, c, o, rgb[0], rgb[1], rgb[2], z]
    return s


def test_single_gaussian_at_pixel_centre(orc):
    for o in [0.3, 0.9, 0.995]:
        S = np.stack([splat(3.5, 2.5, 0.7, 0.1, 0.4, o, (0.2, 0.6, 0.9), 2.0)])
        r = orc.composite_one(3.5, 2.5, S, [0], bg=(1, 1, 1))
        a = min(0.99, o)
        np.testing.assert_allclose(r["rgb"], a * np.array([0.2, 0.6, 0.9]) + (1 - a), atol=1e-7)
        assert abs(r["alpha"] - a) < 1e-7 and abs(r["depth"] - a * 2.0) < 1e-6
        assert r["n_contrib"] == 1


def test_offset_gaussian_closed_form(orc):
    a, b, c, o = 0.8, -0.25, 0.5, 0.7
    S = np.stack([splat(10.0, 20.0, a, b, c, o, (1, 0, 0), 1.0)])
    a, b, c, o = (float(v) for v in S[0, 2:6])  # the record holds fp32 values
    px, py = 11.5, 19.5
    dx, dy = px - 10.0, py - 20.0
    alpha = o * math.exp(-(0.5 * (a * dx * dx + c * dy * dy) + b * dx * dy))
    r = orc.composite_one(px, py, S, [0], bg=(0, 0, 0), f32=False)
    assert abs(r["rgb"][0] - alpha) < 1e-12 and abs(r["T"] - (1 - alpha)) < 1e-12


def test_two_layer_golden(orc):
    case = GOLDEN["two_layer_pixel"]
    S = np.stack([splat(0.5, 0.5, 1, 0, 1, 0.5, (1, 0, 0), 1.0),
                  splat(0.5, 0.5, 1, 0, 1, 0.25, (0, 1, 0), 2.0)])
    for f32 in (True, False):
        r = orc.composite_one(0.5, 0.5, S, [0, 1], D=3.0, covered=True, cm=(0, 0, 1), f32=f32)
        np.testing.assert_allclose(r["rgb"], case["rgb"], atol=1e-7)
        assert abs(r["depth"] - case["depth"]) < 1e-6
        assert r["alpha"] == case["alpha"] and abs(r["T"] - case["T"]) < 1e-7


def test_weights_and_transmittance_sum_to_one(orc):
    rng = np.random.default_rng(2)
    n = 60
    S = np.stack([splat(5 + rng.normal(), 5 + rng.normal(), rng.uniform(0.2, 2), rng.uniform(-0.1, 0.1),
                        rng.uniform(0.2, 2), rng.uniform(0.01, 0.6), (1, 1, 1), 1.0 + k) for k in range(n)])
    for f32 in (True, False):
        r = orc.composite_one(5.5, 5.5, S, list(range(n)), bg=(0, 0, 0), f32=f32)
        assert abs(r["rgb"][0] + r["T"] - 1.0) < 1e-6
        assert abs(r["alpha"] - (1 - r["T"])) < 1e-12


def test_hidden_gaussians_change_nothing(orc):
    rng = np.random.default_rng(4)
    S = np.stack([splat(2.5, 2.5, 1, 0, 1, 0.8, rng.uniform(size=3), 3.0 + k) for k in range(5)])
    r = orc.composite_one(2.5, 2.5, S, list(range(5)), D=3.0, covered=True, cm=(0.1, 0.2, 0.3))
    np.testing.assert_array_equal(r["rgb"], [0.1, 0.2, 0.3])
    assert r["depth"] == 3.0 and r["alpha"] == 1.0 and r["n_contrib"] == 0


def test_alpha_skip_threshold(orc):
    below = np.stack([splat(0.5, 0.5, 1, 0, 1, 1.0 / 256.0, (0, 0, 0), 1.0)])
    r = orc.composite_one(0.5, 0.5, below, [0], bg=(1, 1, 1))
    assert r["n_contrib"] == 0 and np.all(r["rgb"] == 1.0)
    above = np.stack([splat(0.5, 0.5, 1, 0, 1, 1.0 / 254.0, (0, 0, 0), 1.0)])
    r = orc.composite_one(0.5, 0.5, above, [0], bg=(1, 1, 1))
    assert r["n_contrib"] == 1 and r["rgb"][0] < 1.0


def test_transmittance_stop_excludes_the_gaussian(orc):
    # 0.99 then 0.99: T would fall to 1e-4 -> the second is not composited
    S = np.stack([splat(0.5, 0.5, 1, 0, 1, 0.999, (1, 0, 0), 1.0),
                  splat(0.5, 0.5, 1, 0, 1, 0.999, (0, 1, 0), 2.0),
                  splat(0.5, 0.5, 1, 0, 1, 0.5, (0, 0, 1), 3.0)])
    r = orc.composite_one(0.5, 0.5, S, [0, 1, 2], bg=(0, 0, 0))
    assert r["n_contrib"] == 1
    assert abs(r["T"] - (1 - np.float32(0.99))) < 1e-9 and r["rgb"][1] == 0.0 and r["rgb"][2] == 0.0
    # slightly more transparent second Gaussian: T' just above 1e-4 -> composited
    S[1, 5] = 0.9895
    r = orc.composite_one(0.5, 0.5, S, [0, 1, 2], bg=(0, 0, 0))
    assert r["n_contrib"] == 2 and r["rgb"][1] > 0
    # three opacities (found by a search over fp32 values) whose fp32 transmittance
    # product lands exactly on float32(1e-4): equality stops, the third is excluded
    ops = np.float32([0.98863285779953, 0.9863587021827698, 0.35509905219078064])
    one = np.float32(1.0)
    T2 = np.float32(np.float32(one - ops[0]) * np.float32(one - ops[1]))
    assert np.float32(T2 * np.float32(one - ops[2])) == np.float32(1e-4)
    S3 = np.stack([splat(0.5, 0.5, 1, 0, 1, float(o), (1, 0, 0), 1.0 + k) for k, o in enumerate(ops)])
    r = orc.composite_one(0.5, 0.5, S3, [0, 1, 2], bg=(0, 0, 0))
    assert r["n_contrib"] == 2 and abs(r["T"] - float(T2)) == 0.0


def test_depth_test_tie_goes_to_the_mesh(orc):
    S = np.stack([splat(0.5, 0.5, 1, 0, 1, 0.8, (1, 0, 0), 2.0)])
    r = orc.composite_one(0.5, 0.5, S, [0], D=2.0, covered=True, cm=(0, 0, 1))
    assert r["n_contrib"] == 0
    r = orc.composite_one(0.5, 0.5, S, [0], D=float(np.nextafter(np.float32(2.0), np.float32(3.0))),
                          covered=True, cm=(0, 0, 1))
    assert r["n_contrib"] == 1


def test_f32_and_f64_modes_agree(orc):
    rng = np.random.default_rng(8)
    n = 200
    S = np.stack([splat(8 + 3 * rng.normal(), 8 + 3 * rng.normal(), rng.uniform(0.05, 1), rng.uniform(-0.02, 0.02),
                        rng.uniform(0.05, 1), rng.uniform(0.01, 0.5), rng.uniform(size=3), 1 + 0.01 * k)
                  for k in range(n)])
    for p in range(20):
        px, py = 8.5 + rng.integers(-4, 4), 8.5 + rng.integers(-4, 4)
        r32 = orc.composite_one(px, py, S, list(range(n)), D=1.5, covered=True, cm=(0.3, 0.3, 0.3))
        r64 = orc.composite_one(px, py, S, list(range(n)), D=1.5, covered=True, cm=(0.3, 0.3, 0.3), f32=False)
        np.testing.assert_allclose(r32["rgb"], r64["rgb"], atol=1e-5)
        assert r32["n_contrib"] == r64["n_contrib"]


# ------------------------------------------------------------------ 4x4 ----

def _cam4():
    return scenes.Camera(4, 4, 4.0, 4.0, 0.0, 0.0, scenes.NEAR, scenes.FAR,
                         np.eye(3, dtype=np.float32), np.zeros(3, np.float32))


def test_brute_force_4x4_scene(orc):
    """4x4 image, one fronto-parallel triangle at depth 2 covering the pixels
    with i + j <= 3 (screen barycentrics = perspective-correct ones on a plane
    of constant depth), one Gaussian in front of it and one behind its plane:
    each pixel against the over operator applied by hand in depth order."""
    cam = _cam4()
    # (u, v) = (0, 0), (4, 0), (0, 4) at z = 2: pixel centres with i + j + 1 <= 4 are covered
    V = np.array([[0, 0, 2], [2, 0, 2], [0, 2, 2]], np.float32)
    F = np.array([[0, 1, 2]], np.int32)
    vcol = np.array([[1, 0, 0], [0, 1, 0], [0, 0, 1]], np.float32)
    g = scenes.Gaussians(
        # centres project to the pixel centres (1.5, 0.5) at depth 1 (in front of
        # the mesh) and (2.5, 2.5) at depth 3 (behind the mesh plane)
        means=np.array([[0.375, 0.125, 1.0], [1.875, 1.875, 3.0]], np.float32),
        log_scales=np.full((2, 3), math.log(0.02), np.float32),
        quats=np.tile(np.float32([1, 0, 0, 0]), (2, 1)),
        logits=np.float32([0.0, 1.0]),
        colors=np.float32([[0, 0, 0], [1, 1, 0]]), sh_degree=-1)
    scene = scenes.Scene("4x4", [cam], scenes.Mesh(V, F, vcol), g, bg=(1.0, 1.0, 1.0))
    out = orc.render(scene)
    fid = out["face_id"]
    for j in range(4):
        for i in range(4):
            assert (fid[j, i] == 0) == (i + j + 1 <= 4)
    sp = out["splats"]
    np.testing.assert_allclose(sp[0, :2], [1.5, 0.5], atol=1e-6)
    np.testing.assert_allclose(sp[1, :2], [2.5, 2.5], atol=1e-6)
    for j in range(4):
        for i in range(4):
            px, py = i + 0.5, j + 0.5
            cov = i + j + 1 <= 4
            lam = np.array([1 - px / 4 - py / 4, px / 4, py / 4])
            base = lam @ vcol if cov else np.ones(3)
            expect = base.copy()
            for k in range(2):
                mx, my = sp[k, 0], sp[k, 1]
                a_, b_, c_ = sp[k, 2], sp[k, 3], sp[k, 4]
                dx, dy = px - mx, py - my
                al = min(0.99, sp[k, 5] * math.exp(-(0.5 * (a_ * dx * dx + c_ * dy * dy) + b_ * dx * dy)))
                in_front = (not cov) or sp[k, 9] < 2.0
                if al >= 1 / 255 and in_front:
                    expect = al * sp[k, 6:9] + (1 - al) * expect
            np.testing.assert_allclose(out["rgb"][j, i], expect, atol=1e-6)
    assert out["alpha"][0, 1] == 1.0 and abs(out["alpha"][2, 2] - 1 / (1 + math.exp(-1.0))) < 1e-6


def test_culled_lists_give_identical_images(orc):
    s = scenes.tiny()
    # closer than the workload's own camera, so that some tiles are fully covered
    cam = scenes.look_at((0.2, 0.1, 2.0), (0, 0, 0), 80, 64, 64, 64)
    s = scenes.Scene(s.name, [cam], s.mesh, s.gaussians, s.bg)
    out = orc.render(s)
    far, full = orc.tile_depth_bounds(cam, out["mesh_depth"])
    assert full.sum() > 0
    keys, gids, pre = orc.bin_gaussians(cam, out["splats"], out["radii"], far, full, cull=True)
    assert len(keys) < pre
    T = orc.n_tiles(cam)
    start = np.zeros(T + 1, np.int64)
    np.add.at(start, (keys >> np.uint64(32)).astype(np.int64) + 1, 1)
    start = np.cumsum(start)
    culled = orc.composite_fwd(cam, s.bg, out["splats"], (start, gids), out["mesh_depth"],
                               out["mesh_rgb"], out["face_id"])
    for k in ("rgb", "depth", "alpha", "T", "n_contrib"):
        np.testing.assert_array_equal(culled[k], out[k])


# ------------------------------------------------------ finite differences ----

def _one_gaussian_frame(o=0.6, b=0.05):
    cam = scenes.Camera(16, 16, 16.0, 16.0, 8.0, 8.0, scenes.NEAR, scenes.FAR,
                        np.eye(3, dtype=np.float32), np.zeros(3, np.float32))
    S = np.stack([splat(7.3, 8.6, 0.35, b, 0.5, o, (0.9, 0.2, 0.4), 2.0)])
    radii = np.array([6], np.int32)
    return cam, S, radii


def test_fd_matches_closed_form_single_gaussian(orc):
    cam, S, radii = _one_gaussian_frame()
    lists = orc.tile_lists(cam, S, radii)
    H = W = 16
    g_rgb, g_depth, g_alpha = scenes.upstream_grads(0, W, H)
    face = np.full(H * W, -1, np.int32)
    md = np.full(H * W, np.inf, np.float32)
    mrgb = np.zeros((H * W, 3), np.float32)
    bg = np.float64([1.0, 1.0, 1.0])
    fields = [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]
    hs = [1e-4, 1e-4, 1e-5, 1e-5, 1e-5, 1e-6, 1e-3, 1e-3, 1e-3, 1e-4]
    grad, status = orc.composite_fd(cam, bg, S, radii, lists, md, mrgb, face, (g_rgb, g_depth, g_alpha),
                                    [0] * 10, fields, hs)
    assert np.all(status == 0)
    mx, my, a, b, c, o = (float(v) for v in S[0, :6])
    col, z = S[0, 6:9].astype(np.float64), float(S[0, 9])
    ref = np.zeros(10)
    for j in range(H):
        for i in range(W):
            dx, dy = i + 0.5 - mx, j + 0.5 - my
            sig = 0.5 * (a * dx * dx + c * dy * dy) + b * dx * dy
            G = math.exp(-sig)
            al = o * G
            if al < 1 / 255:
                continue
            # out = al*col + (1-al)*bg ; depth = al*z ; alpha = al
            dL_dal = g_rgb[j, i] @ (col - bg) + g_depth[j, i] * z + g_alpha[j, i]
            dal_dsig = -al
            ref[0] += dL_dal * dal_dsig * -(a * dx + b * dy)
            ref[1] += dL_dal * dal_dsig * -(b * dx + c * dy)
            ref[2] += dL_dal * dal_dsig * 0.5 * dx * dx
            ref[3] += dL_dal * dal_dsig * dx * dy
            ref[4] += dL_dal * dal_dsig * 0.5 * dy * dy
            ref[5] += dL_dal * G
            ref[6:9] += al * g_rgb[j, i]
            ref[9] += al * g_depth[j, i]
    np.testing.assert_allclose(grad, ref, rtol=1e-6, atol=1e-8)


def test_fd_reports_flips(orc):
    # an opacity right at the 0.99 clamp flips under +-h at the centre pixel
    cam, S, radii = _one_gaussian_frame(o=0.99)
    S[0, 0:2] = [7.5, 8.5]
    lists = orc.tile_lists(cam, S, radii)
    g = scenes.upstream_grads(0, 16, 16)
    face = np.full(256, -1, np.int32)
    grad, status = orc.composite_fd(cam, np.float64([1, 1, 1]), S, radii, lists, np.full(256, np.inf, np.float32),
                                    np.zeros((256, 3), np.float32), face, g, [0], [5], [1e-4], tie_band=0.0)
    assert status[0] in (1, 2)


def test_mesh_fd_closed_forms(orc):
    """Fronto-parallel triangle, no Gaussians: a joint z shift of the three
    vertices moves every covered depth by the same amount, and the colour
    gradient of vertex k is the sum of its screen barycentric over the pixels."""
    cam = scenes.Camera(16, 16, 8.0, 8.0, 8.0, 8.0, scenes.NEAR, scenes.FAR,
                        np.eye(3, dtype=np.float32), np.zeros(3, np.float32))
    V = np.array([[-0.75, -0.75, 2.0], [1.25, -0.75, 2.0], [-0.75, 1.25, 2.0]], np.float32)
    F = np.array([[0, 1, 2]], np.int32)
    vcol = np.float32([[0.2, 0.4, 0.6], [0.9, 0.1, 0.3], [0.5, 0.5, 0.1]])
    fid, _, _ = orc.zbuffer(cam, V, F)
    md, mrgb = orc.interp_mesh(cam, V, F, vcol, fid)
    S = np.zeros((0, 12), np.float32)
    lists = orc.tile_lists(cam, S, np.zeros(0, np.int32))
    g = scenes.upstream_grads(3, 16, 16)
    vids = [0, 1, 2] * 2 + [0, 0, 0, 1, 1, 1, 2, 2, 2]
    fields = [2, 2, 2, 0, 1, 0] + [3, 4, 5] * 3
    hs = [1e-5] * 6 + [1e-3] * 9
    grad, status = orc.mesh_fd(cam, np.float64([1, 1, 1]), V, F, vcol, fid, S, lists, md, mrgb, g,
                               vids, fields, hs)
    assert np.all(status == 0)
    cov = np.nonzero(fid >= 0)[0]
    # with one uniform vertex colour the colour term is constant (weights sum to
    # one), so a joint z shift of the plane only moves the depth: sum_k dL/dz_k
    # = sum of g_depth over the covered pixels
    flat = np.full((3, 3), 0.25, np.float32)
    md_f, mrgb_f = orc.interp_mesh(cam, V, F, flat, fid)
    gz, st = orc.mesh_fd(cam, np.float64([1, 1, 1]), V, F, flat, fid, S, lists, md_f, mrgb_f, g,
                         [0, 1, 2], [2, 2, 2], [1e-5] * 3)
    assert np.all(st == 0)
    assert abs(gz.sum() - g[1].reshape(-1)[cov].astype(np.float64).sum()) < 1e-6
    for k in range(3):
        acc = np.zeros(3)
        for p in cov:
            px, py = p % 16 + 0.5, p // 16 + 0.5
            lam = [1 - (px - 5) / 8 - (py - 5) / 8, (px - 5) / 8, (py - 5) / 8][k]
            acc += lam * g[0].reshape(-1, 3)[p]
        np.testing.assert_allclose(grad[6 + 3 * k: 9 + 3 * k], acc, atol=1e-6)

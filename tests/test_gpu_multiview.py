"""Batched views (page "A Lightweight and Differentiable Renderer
for Joint Mesh and 3D Gaussian Splat Scenes", Hybrid rendering: the renderer
is run per camera; a training batch holds several cameras of one scene).

The batched projection must equal the per-view projection bit for bit (it is
the same arithmetic on the same inputs), the batched projection backward must
equal per-view calls that accumulate in view order, and the multi-view
renderer must reproduce the single-view renderer's images exactly and its
gradients up to the order of atomic sums.  The single-view path is the one
the other parity tests check against the oracle."""

import numpy as np
import pytest

from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _orbit(n_gauss=40_000, views=8):
    sc = scenes.orbit1080(n_gauss=n_gauss, levels=3)
    return sc, sc.cameras[:views]


def _tiny_views(n):
    sc = scenes.tiny()
    cams = []
    for k in range(n):
        a = 2.0 * np.pi * k / n
        cams.append(scenes.look_at((4.0 * np.cos(a), 0.5, 4.0 * np.sin(a)), (0, 0, 0), 64, 64, 64, 64))
    return sc, cams


@pytest.mark.parametrize("case", ["orbit_sh3_8", "tiny_rgb_10"])
def test_views_projection_and_backward_match_per_view(case):
    H.need_gpu()
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    sc, cams = _orbit() if case == "orbit_sh3_8" else _tiny_views(10)
    g = sc.gaussians
    V, N = len(cams), len(g.means)
    o = gm.make_opts((1, 1, 1), True, g.sh_degree)
    cc = [gm.make_camera(c) for c in cams]
    args = [H.dev(g.means, torch.float32), H.dev(g.log_scales, torch.float32), H.dev(g.quats, torch.float32),
            H.dev(g.logits, torch.float32), H.dev(g.colors, torch.float32)]
    sp = torch.full((V, N, 12), 5.0, dtype=torch.float32, device="cuda")
    rad = torch.full((V, N), -1, dtype=torch.int32, device="cuda")
    tt = torch.full((V, N), -1, dtype=torch.int32, device="cuda")
    gm.gm_project_gaussians_views(cc, o, *args, sp, rad, tt)
    for v in range(V):
        s1 = torch.empty(N, 12, dtype=torch.float32, device="cuda")
        r1 = torch.empty(N, dtype=torch.int32, device="cuda")
        t1 = torch.empty(N, dtype=torch.int32, device="cuda")
        gm.gm_project_gaussians(cc[v], o, *args, s1, r1, t1)
        assert torch.equal(sp[v], s1) and torch.equal(rad[v], r1) and torch.equal(tt[v], t1), v
    rng = np.random.default_rng(4)
    vs = H.dev(rng.normal(size=(V, N, 12)).astype(np.float32), torch.float32)
    batched = [torch.full(a.shape, 9.0, dtype=torch.float32, device="cuda") for a in args]
    gm.gm_project_gaussians_bwd_views(cc, o, *args, rad, vs, *batched)
    seq = [torch.full(a.shape, 9.0, dtype=torch.float32, device="cuda") for a in args]
    for v in range(V):
        gm.gm_project_gaussians_bwd(cc[v], o, *args, rad[v], vs[v], *seq, accumulate=v > 0)
    for a, b in zip(batched, seq):
        if V <= 8:
            assert torch.equal(a, b)
        else:  # groups of eight views are summed first
            torch.testing.assert_close(a, b, rtol=1e-5, atol=1e-6 * float(b.abs().max()))


def test_multiview_renderer_matches_single_views():
    H.need_gpu()
    import torch
    import differentiable_hybrid_mesh_tile_b300 as gm
    sc, cams = _orbit(views=4)
    mv = gm.MultiViewRenderer(cams, bg=sc.bg, streams=3)
    mv.upload(sc.mesh, sc.gaussians)
    outs = [[t.clone() for t in o] for o in mv.forward()]
    grads = [[torch.as_tensor(x).cuda() for x in scenes.upstream_grads(20 + k, c.width, c.height)]
             for k, c in enumerate(cams)]
    res = [x.clone() for x in mv.backward(grads)]
    torch.cuda.synchronize()
    assert not mv.overflowed()
    sum_mesh = [torch.zeros_like(res[5]), torch.zeros_like(res[6])]
    for k, c in enumerate(cams):
        r = gm.HybridRenderer(c, bg=sc.bg)
        r.upload(sc.mesh, sc.gaussians)
        rgb, depth, alpha = r.forward()
        assert torch.equal(rgb, outs[k][0]) and torch.equal(depth, outs[k][1]) and torch.equal(alpha, outs[k][2])
        v_splats, v_verts, v_vcol = r.backward(*grads[k])
        # atomic sums in another order: a tolerance on the scale of each record field
        scale = v_splats.abs().amax(0, keepdim=True).clamp_min(1e-12)
        assert bool(((mv.v_splats[k] - v_splats).abs() <= 1e-4 * v_splats.abs() + 1e-5 * scale).all())
        sum_mesh[0] += v_verts
        sum_mesh[1] += v_vcol
    torch.testing.assert_close(res[5], sum_mesh[0], rtol=1e-4, atol=1e-4 * float(sum_mesh[0].abs().max()))
    torch.testing.assert_close(res[6], sum_mesh[1], rtol=1e-4, atol=1e-4 * float(sum_mesh[1].abs().max()))
    # the summed parameter gradients against per-view projection backward calls on the
    # renderer's own record gradients
    o = mv.opts
    v0 = mv.views[0]
    args = [v0.means, v0.log_scales, v0.quats, v0.logits, v0.colors]
    seq = [torch.zeros_like(a) for a in args]
    for k in range(len(cams)):
        gm.gm_project_gaussians_bwd(mv.cams[k], o, *args, mv.radii[k], mv.v_splats[k], *seq, accumulate=k > 0)
    for a, b in zip(res[:5], seq):
        assert torch.equal(a, b)
    # one CUDA graph for the batch reproduces the eager pass
    graph = mv.capture_step(grads)
    graph.replay()
    torch.cuda.synchronize()
    for k in range(len(cams)):
        assert torch.equal(mv.views[k].out_rgb, outs[k][0])
    torch.testing.assert_close(mv.v_means, res[0], rtol=1e-4, atol=1e-4 * float(res[0].abs().max()))

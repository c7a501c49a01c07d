"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and bring results back as numpy; tolerances derived from fp32 error
bounds (each stated where it is used)."""

import numpy as np
import pytest
import torch

import differentiable_hybrid_mesh_tile_b300 as gm
from differentiable_hybrid_mesh_tile_b300 import build as gm_build
from differentiable_hybrid_mesh_tile_b300 import scenes

EPS32 = float(np.finfo(np.float32).eps)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gm_build.build()
    gm.lib()


def dev(x, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda().contiguous()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def n_tiles(cam):
    return ((cam.width + 15) // 16) * ((cam.height + 15) // 16)


def run_mesh(cam, mesh):
    """GPU gm_bin_triangles -> gm_zbuffer -> gm_interp_mesh."""
    c = gm.make_camera(cam)
    V, F, vcol = dev(mesh.verts, torch.float32), dev(mesh.faces, torch.int32), dev(mesh.vcol, torch.float32)
    T = n_tiles(cam)
    tr = torch.zeros(T, 2, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(4, dtype=torch.int32, device="cuda")
    cap = 16
    for _ in range(2):
        ids = torch.zeros(cap, dtype=torch.int32, device="cuda")
        ws = torch.empty(gm.gm_bin_triangles_workspace_size(len(F), cap, cam.width, cam.height), dtype=torch.uint8,
                         device="cuda")
        try:
            K = gm.gm_bin_triangles(c, V, F, tr, ids, cap, cnt, ws)
            break
        except gm.GmError as e:
            assert e.status == gm.GM_ERR_CAPACITY
            cap = int(host(cnt)[0]) + 1
    fid = torch.full((cam.height, cam.width), -7, dtype=torch.int32, device="cuda")
    gm.gm_zbuffer(c, V, F, tr, ids, fid)
    md = torch.empty(cam.height, cam.width, dtype=torch.float32, device="cuda")
    mrgb = torch.empty(cam.height, cam.width, 3, dtype=torch.float32, device="cuda")
    tfar = torch.empty(T, dtype=torch.float32, device="cuda")
    tfull = torch.empty(T, dtype=torch.uint8, device="cuda")
    gm.gm_interp_mesh(c, V, F, vcol, fid, md, mrgb, tfar, tfull)
    return dict(K=K, tile_range=host(tr), tri_ids=host(ids)[:K], face_id=host(fid), mesh_depth=host(md),
                mesh_rgb=host(mrgb), tile_far=host(tfar), tile_full=host(tfull), counters=host(cnt))


def run_zbuffer_direct(cam, mesh):
    """GPU gm_zbuffer_direct: face ids [H][W] as numpy."""
    c = gm.make_camera(cam)
    V, F = dev(mesh.verts, torch.float32), dev(mesh.faces, torch.int32)
    nb = gm.gm_zbuffer_direct_workspace_size(len(mesh.faces), cam.width, cam.height)
    ws = torch.empty((nb + 15) // 16 * 16, dtype=torch.uint8, device="cuda")
    fid = torch.full((cam.height, cam.width), -7, dtype=torch.int32, device="cuda")
    gm.gm_zbuffer_direct(c, V, F, fid, ws)
    return host(fid)


def run_mesh_edges(F, nV):
    """GPU gm_mesh_edges: adjacency [nF][3] as numpy."""
    Fd = dev(F, torch.int32)
    adj = torch.full((max(len(F), 1), 3), -9, dtype=torch.int32, device="cuda")
    ws = torch.empty(gm.gm_mesh_edges_workspace_size(len(F)) + 16, dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(4, dtype=torch.int32, device="cuda")
    gm.gm_mesh_edges(Fd, nV, adj, cnt, ws)
    assert int(host(cnt)[2]) == 0
    return host(adj)[:len(F)]


def run_antialias(cam, mesh, m):
    """GPU gm_antialias over the GPU mesh images m (run_mesh): the layer and the
    per-tile bounds, plus the adjacency used."""
    c = gm.make_camera(cam)
    adj = run_mesh_edges(mesh.faces, len(mesh.verts))
    H, W, T = cam.height, cam.width, n_tiles(cam)
    cov = torch.full((H, W), -3.0, dtype=torch.float32, device="cuda")
    rgb = torch.full((H, W, 3), -3.0, dtype=torch.float32, device="cuda")
    depth = torch.full((H, W), -3.0, dtype=torch.float32, device="cuda")
    tf = torch.full((T,), -3.0, dtype=torch.float32, device="cuda")
    tu = torch.full((T,), 7, dtype=torch.uint8, device="cuda")
    gm.gm_antialias(c, dev(mesh.verts, torch.float32), dev(mesh.faces, torch.int32), dev(adj, torch.int32),
                    dev(m["face_id"], torch.int32), dev(m["mesh_depth"], torch.float32),
                    dev(m["mesh_rgb"], torch.float32), cov, rgb, depth, tf, tu)
    return dict(adj=adj, cov=host(cov), rgb_aa=host(rgb), depth_aa=host(depth), tile_far=host(tf),
                tile_full=host(tu))


def run_composite_aa(cam, bg, tile_range, gids, splats, aa, softness=0.0, depth_model=None, soft_split=0):
    """GPU composite over the antialiased layer aa (run_antialias)."""
    c = gm.make_camera(cam)
    o = gm.make_opts(bg, True, -1, True, softness, soft_split)
    H, W = cam.height, cam.width
    out = {k: torch.full(s, -3.0, dtype=torch.float32, device="cuda")
           for k, s in [("rgb", (H, W, 3)), ("depth", (H, W)), ("alpha", (H, W)), ("T", (H, W))]}
    nc = torch.full((H, W), -3, dtype=torch.int32, device="cuda")
    buf = dict(cov=dev(aa["cov"], torch.float32), back=torch.zeros(H, W, 4, dtype=torch.float32, device="cuda"),
               T_back=torch.zeros(H, W, dtype=torch.float32, device="cuda"),
               n_back=torch.zeros(H, W, dtype=torch.int32, device="cuda"),
               v_cov=torch.zeros(H, W, dtype=torch.float32, device="cuda"),
               v_rgb=torch.zeros(H, W, 3, dtype=torch.float32, device="cuda"))
    layer = gm.make_aa_layer(buf["cov"], buf["back"], buf["T_back"], buf["n_back"], buf["v_cov"], buf["v_rgb"])
    args = [dev(tile_range, torch.int32), dev(gids if len(gids) else np.zeros(1, np.int32), torch.int32),
            dev(splats if len(splats) else np.zeros((1, 12), np.float32), torch.float32),
            dev(aa["depth_aa"], torch.float32), dev(aa["rgb_aa"], torch.float32), None]
    dm = None
    if depth_model is not None:
        dm = dev(depth_model if len(depth_model) else np.zeros((1, 4), np.float32), torch.float32)
    gm.gm_composite_hybrid_fwd(c, o, *args, out["rgb"], out["depth"], out["alpha"], out["T"], nc, depth_model=dm,
                               aa=layer)
    res = {k: host(v) for k, v in out.items()}
    res["n_contrib"] = host(nc)
    res.update(back=host(buf["back"]), T_back=host(buf["T_back"]), n_back=host(buf["n_back"]))
    res["_args"] = args
    res["_dev"] = dict(T=out["T"], n_contrib=nc)
    res["_soft"] = (softness, dm, soft_split)
    res["_aa"] = (layer, buf)
    res["_depth_aa"] = args[3]
    return res


def run_backward_aa(cam, bg, fwd, grads, N, mesh, m, adj):
    """GPU backward over the antialiased layer: composite (Gaussians + layer),
    then gm_antialias_bwd and gm_interp_mesh_bwd.  Returns v_splats (+ the depth
    model's), v_verts, v_vcol and the layer gradients."""
    c = gm.make_camera(cam)
    softness, dm, split = fwd["_soft"]
    o = gm.make_opts(bg, True, -1, True, softness, split)
    layer, buf = fwd["_aa"]
    H, W = cam.height, cam.width
    v_splats = torch.zeros(max(N, 1), 12, dtype=torch.float32, device="cuda")
    v_dm = torch.zeros(max(N, 1), 4, dtype=torch.float32, device="cuda") if softness > 0 else None
    v_md = torch.full((H, W), 5.0, dtype=torch.float32, device="cuda")
    g_rgb, g_depth, g_alpha = (dev(x, torch.float32) for x in grads)
    gm.gm_composite_hybrid_bwd(c, o, *fwd["_args"], fwd["_dev"]["T"], fwd["_dev"]["n_contrib"], g_rgb, g_depth,
                               g_alpha, v_splats, depth_model=dm, v_depth_model=v_dm, v_mesh_depth=v_md, aa=layer)
    V, F, vcol = dev(mesh.verts, torch.float32), dev(mesh.faces, torch.int32), dev(mesh.vcol, torch.float32)
    v_verts, v_vcol = torch.zeros_like(V), torch.zeros_like(vcol)
    v_c = torch.full((H, W, 3), 7.0, dtype=torch.float32, device="cuda")
    v_d = torch.full((H, W), 7.0, dtype=torch.float32, device="cuda")
    fid = dev(m["face_id"], torch.int32)
    gm.gm_antialias_bwd(c, V, F, dev(adj, torch.int32), fid, dev(m["mesh_depth"], torch.float32),
                        dev(m["mesh_rgb"], torch.float32), buf["cov"], fwd["_depth_aa"], buf["v_cov"], buf["v_rgb"],
                        v_md, v_c, v_d, v_verts)
    gm.gm_interp_mesh_bwd(c, V, F, vcol, fid, v_c, v_d, v_verts, v_vcol)
    out = dict(v_splats=host(v_splats)[:N], v_verts=host(v_verts), v_vcol=host(v_vcol), v_cov=host(buf["v_cov"]),
               v_rgb_aa=host(buf["v_rgb"]), v_depth_aa=host(v_md), v_mesh_rgb=host(v_c), v_mesh_depth=host(v_d))
    if v_dm is not None:
        out["v_depth_model"] = host(v_dm)[:N]
    return out


def run_project(cam, g, bg=(1, 1, 1), depth_model=False, softness=0.0, soft_split=0):
    """GPU projection: splats, radii, tiles_touched (+ the soft split's depth
    model [N][4] when depth_model is set; with softness > 0 the records carry
    the soft cull's hide depth in field 10)."""
    c = gm.make_camera(cam)
    o = gm.make_opts(bg, True, g.sh_degree, True, softness, soft_split)
    N = len(g.means)
    splats = torch.full((N, 12), 7.0, dtype=torch.float32, device="cuda")
    radii = torch.full((N,), -3, dtype=torch.int32, device="cuda")
    touched = torch.full((N,), -3, dtype=torch.int32, device="cuda")
    dm = torch.full((max(N, 1), 4), 7.0, dtype=torch.float32, device="cuda") if depth_model else None
    gm.gm_project_gaussians(c, o, dev(g.means, torch.float32), dev(g.log_scales, torch.float32),
                            dev(g.quats, torch.float32), dev(g.logits, torch.float32), dev(g.colors, torch.float32),
                            splats, radii, touched, dm)
    if depth_model:
        return host(splats), host(radii), host(touched), host(dm)[:N]
    return host(splats), host(radii), host(touched)


def run_bin(cam, splats, radii, tile_far=None, tile_full=None, cull=False, cap=None, sync=True, tile_test=False,
            softness=0.0):
    c = gm.make_camera(cam)
    o = gm.make_opts((1, 1, 1), cull, -1, tile_test, softness)
    N = len(radii)
    T = n_tiles(cam)
    tf = dev(np.full(T, np.inf, np.float32) if tile_far is None else tile_far, torch.float32)
    tu = dev(np.zeros(T, np.uint8) if tile_full is None else tile_full, torch.uint8)
    tr = torch.full((T, 2), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((4,), -9, dtype=torch.int32, device="cuda")
    if cap is None:
        cap = int(np.asarray(radii > 0).sum() * 4) + 64
    while True:
        keys = torch.zeros(cap, dtype=torch.int64, device="cuda")
        gids = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
        ws = torch.empty(gm.gm_bin_sort_gaussians_workspace_size(N, cap, cam.width, cam.height), dtype=torch.uint8,
                         device="cuda")
        try:
            K = gm.gm_bin_sort_gaussians(c, o, dev(splats, torch.float32), dev(radii, torch.int32), tf, tu, keys,
                                         gids, tr, cap, cnt, ws, sync=sync)
            break
        except gm.GmError as e:
            assert e.status == gm.GM_ERR_CAPACITY
            cap = int(host(cnt)[0]) + 1
    cn = host(cnt)
    K = int(cn[0]) if K is None else K
    k = min(K, cap)
    return dict(K=K, keys=host(keys)[:k].view(np.uint64), gids=host(gids)[:k], tile_range=host(tr), counters=cn,
                cap=cap)


def run_composite(cam, bg, tile_range, gids, splats, mesh_depth, mesh_rgb, face_id, softness=0.0,
                  depth_model=None, soft_split=0):
    c = gm.make_camera(cam)
    o = gm.make_opts(bg, True, -1, True, softness, soft_split)
    H, W = cam.height, cam.width
    out = {k: torch.full(s, -3.0, dtype=torch.float32, device="cuda")
           for k, s in [("rgb", (H, W, 3)), ("depth", (H, W)), ("alpha", (H, W)), ("T", (H, W))]}
    nc = torch.full((H, W), -3, dtype=torch.int32, device="cuda")
    args = [dev(tile_range, torch.int32), dev(gids if len(gids) else np.zeros(1, np.int32), torch.int32),
            dev(splats if len(splats) else np.zeros((1, 12), np.float32), torch.float32),
            dev(mesh_depth, torch.float32), dev(mesh_rgb, torch.float32), dev(face_id, torch.int32)]
    dm = None
    if depth_model is not None:
        dm = dev(depth_model if len(depth_model) else np.zeros((1, 4), np.float32), torch.float32)
    gm.gm_composite_hybrid_fwd(c, o, *args, out["rgb"], out["depth"], out["alpha"], out["T"], nc, depth_model=dm)
    res = {k: host(v) for k, v in out.items()}
    res["n_contrib"] = host(nc)
    res["_args"] = args
    res["_dev"] = dict(T=out["T"], n_contrib=nc)
    res["_soft"] = (softness, dm, soft_split)
    return res


def run_composite_bwd(cam, bg, fwd, grads, N, mesh=None, mesh_grads=False):
    """GPU composite backward over the saved state of run_composite (its
    softness and depth model included).  Returns v_splats (+ v_verts / v_vcol
    with mesh_grads; + v_depth_model and v_mesh_depth with the soft split)."""
    c = gm.make_camera(cam)
    softness, dm, split = fwd.get("_soft", (0.0, None, 0))
    o = gm.make_opts(bg, True, -1, True, softness, split)
    soft = softness > 0.0
    v_splats = torch.zeros(max(N, 1), 12, dtype=torch.float32, device="cuda")
    v_dm = torch.zeros(max(N, 1), 4, dtype=torch.float32, device="cuda") if soft else None
    v_md = torch.full((cam.height, cam.width), 5.0, dtype=torch.float32, device="cuda") if soft else None
    g_rgb, g_depth, g_alpha = (dev(x, torch.float32) for x in grads)
    V = F = vcol = v_verts = v_vcol = None
    if mesh_grads:
        V, F, vcol = dev(mesh.verts, torch.float32), dev(mesh.faces, torch.int32), dev(mesh.vcol, torch.float32)
        v_verts = torch.zeros_like(V)
        v_vcol = torch.zeros_like(vcol)
    gm.gm_composite_hybrid_bwd(c, o, *fwd["_args"], fwd["_dev"]["T"], fwd["_dev"]["n_contrib"], g_rgb, g_depth,
                               g_alpha, v_splats, V, F, vcol, v_verts, v_vcol, depth_model=dm, v_depth_model=v_dm,
                               v_mesh_depth=v_md)
    out = dict(v_splats=host(v_splats)[:N])
    if soft:
        out.update(v_depth_model=host(v_dm)[:N], v_mesh_depth=host(v_md))
    if mesh_grads:
        out.update(v_verts=host(v_verts), v_vcol=host(v_vcol))
    return out


def lists_from_bins(cam, keys, gids):
    """(tile_start[T+1], entries) CSR lists from sorted GPU keys."""
    T = n_tiles(cam)
    start = np.zeros(T + 1, np.int64)
    if len(keys):
        np.add.at(start, (keys >> np.uint64(32)).astype(np.int64) + 1, 1)
    return np.cumsum(start), np.asarray(gids, np.int32)


# The kernels evaluate exp(-sigma) as 2^l with l from a conic pre-scaled by
# -log2(e)/2: the rounding of l (a few ulp of |l| <= 8 near alpha = 1/255) and
# ex2's own 2 ulp keep alpha within 8e-6 relative of the oracle's.
def tie_pixels(margins, alpha_band=8e-6, stop_band=1e-4, sigma_band=1e-5, clamp_band=None):
    m = margins
    t = (m[..., 1] < alpha_band) | (m[..., 3] < stop_band) | (m[..., 4] < sigma_band)
    if clamp_band is not None:
        t |= m[..., 2] < clamp_band
    return t


def input_ulp_perturbations(cam, V, draws=3, seed=0):
    """World vertex sets moved by about one fp32 rounding of the camera-space
    coordinates: each coordinate by 2 eps (|V| + |camera centre|) with a random
    sign.  The oracle evaluated on them bounds how far any fp32 evaluation of
    an ill-conditioned quantity (an edge-on triangle) can land from the exact
    value."""
    rng = np.random.default_rng(seed)
    C = -cam.R.astype(np.float64).T @ cam.t.astype(np.float64)
    scale = 2 * EPS32 * (np.abs(V.astype(np.float64)) + np.linalg.norm(C))
    out = []
    for _ in range(draws):
        r = rng.choice([-1.0, 1.0], size=V.shape)
        out.append((V.astype(np.float64) + scale * r).astype(np.float32))
    return out


def run_project_bwd(cam, g, v_splats, accumulate_into=None, v_depth_model=None):
    """GPU projection, then its backward for the upstream v_splats.  Returns
    radii and the gradients (v_means, v_log_scales, v_quats, v_logits, v_colors)
    as numpy; accumulate_into = previous gradients to add to (accumulate mode)."""
    c = gm.make_camera(cam)
    o = gm.make_opts((1, 1, 1), True, g.sh_degree)
    N = len(g.means)
    args = [dev(g.means, torch.float32), dev(g.log_scales, torch.float32), dev(g.quats, torch.float32),
            dev(g.logits, torch.float32), dev(g.colors, torch.float32)]
    splats = torch.zeros((N, 12), dtype=torch.float32, device="cuda")
    radii = torch.zeros((N,), dtype=torch.int32, device="cuda")
    touched = torch.zeros((N,), dtype=torch.int32, device="cuda")
    gm.gm_project_gaussians(c, o, *args, splats, radii, touched)
    if accumulate_into is None:
        outs = [torch.full(a.shape, 3.0, dtype=torch.float32, device="cuda") for a in args]
    else:
        outs = [dev(x, torch.float32).clone() for x in accumulate_into]
    vdm = None if v_depth_model is None else dev(v_depth_model, torch.float32)
    gm.gm_project_gaussians_bwd(c, o, *args, radii, dev(v_splats, torch.float32), *outs,
                                accumulate=accumulate_into is not None, v_depth_model=vdm)
    return host(radii), [host(x) for x in outs]

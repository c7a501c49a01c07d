"""CPU oracle of the hybrid mesh + 3D Gaussian renderer -- TEST INFRASTRUCTURE.

Thin ctypes wrapper around ``gm_oracle.c`` (a plain, slow C restatement of
each step of the renderer, see the header of that file).  Only the tests,
the smoke check and the CPU-baseline leg of the benchmark may import this
package; the CUDA library and its Python binding never do.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gm_oracle.c")
_LIB = os.path.join(_HERE, "liborc.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-Wall", "-Wextra", "-shared", "-fPIC"]

S_STRIDE = 12
FD_STATUS = {0: "ok", 1: "flip", 2: "precision", 3: "tie", 4: "order", 5: "unused", 6: "nonsmooth"}


def build(force: bool = False) -> str:
    """Compile gm_oracle.c into liborc.so next to it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cam(C.Structure):
    _fields_ = [("width", C.c_int32), ("height", C.c_int32),
                ("fx", C.c_float), ("fy", C.c_float), ("cx", C.c_float), ("cy", C.c_float),
                ("near_plane", C.c_float), ("far_plane", C.c_float),
                ("R", C.c_float * 9), ("t", C.c_float * 3)]


def _cam(cam) -> _Cam:
    c = _Cam()
    c.width, c.height = int(cam.width), int(cam.height)
    c.fx, c.fy, c.cx, c.cy = cam.fx, cam.fy, cam.cx, cam.cy
    c.near_plane, c.far_plane = cam.near, cam.far
    R = np.asarray(cam.R, np.float32).reshape(9)
    t = np.asarray(cam.t, np.float32).reshape(3)
    for k in range(9):
        c.R[k] = float(R[k])
    for k in range(3):
        c.t[k] = float(t[k])
    return c


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _lib.orc_bin_triangles.restype = C.c_int64
        _lib.orc_bin_gaussians.restype = C.c_int64
        _lib.orc_tile_lists.restype = C.c_int64
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def n_tiles(cam):
    return ((cam.width + 15) // 16) * ((cam.height + 15) // 16)


# ---------------------------------------------------------------- mesh ----

def bin_triangles(cam, V, F):
    V, F = _c(V, np.float32), _c(F, np.int32)
    T = n_tiles(cam)
    counts = np.zeros(T, np.int32)
    c = _cam(cam)
    K = lib().orc_bin_triangles(C.byref(c), _p(V), _p(F), C.c_int32(len(F)), _p(counts), None, C.c_int64(0))
    ids = np.zeros(max(K, 1), np.int32)
    lib().orc_bin_triangles(C.byref(c), _p(V), _p(F), C.c_int32(len(F)), _p(counts), _p(ids), C.c_int64(K))
    return counts, ids[:K]


def zbuffer(cam, V, F, pixels=None):
    V, F = _c(V, np.float32), _c(F, np.int32)
    n = cam.width * cam.height if pixels is None else len(pixels)
    pix = None if pixels is None else _c(pixels, np.int32)
    fid = np.zeros(n, np.int32)
    best = np.zeros(n, np.float32)
    second = np.zeros(n, np.float32)
    lib().orc_zbuffer(C.byref(_cam(cam)), _p(V), _p(F), C.c_int32(len(F)), _p(pix), C.c_int64(n),
                      _p(fid), _p(best), _p(second))
    return fid, best, second


def interp_mesh(cam, V, F, vcol, face_id, pixels=None):
    V, F, vcol = _c(V, np.float32), _c(F, np.int32), _c(vcol, np.float32)
    face_id = _c(face_id, np.int32).reshape(-1)
    n = len(face_id)
    pix = None if pixels is None else _c(pixels, np.int32)
    depth = np.zeros(n, np.float32)
    rgb = np.zeros((n, 3), np.float32)
    lib().orc_interp_mesh(C.byref(_cam(cam)), _p(V), _p(F), _p(vcol), _p(pix), C.c_int64(n),
                          _p(face_id), _p(depth), _p(rgb))
    return depth, rgb


def _opt(a, dt):
    return None if a is None else _c(a, dt)


def mesh_edges(F):
    """Edge adjacency [nF][3]: the face across edge k (corners k+1, k+2) of each
    face, -1 none, -2 shared by more than two faces."""
    F = _c(F, np.int32)
    adj = np.zeros((len(F), 3), np.int32)
    lib().orc_mesh_edges(_p(F), C.c_int32(len(F)), _p(adj))
    return adj


def antialias(cam, V, F, adj, face_id, mesh_depth, mesh_rgb, pixels=None):
    """Antialiased mesh layer from full-frame face ids, depth and colour: cov
    [H][W], premultiplied colour [H][W][3], split depth [H][W] and the pair
    decision codes [H][W][4] (written at the listed pixels, all when None)."""
    H, W = cam.height, cam.width
    cov = np.zeros((H, W), np.float32)
    rgb = np.zeros((H, W, 3), np.float32)
    depth = np.full((H, W), np.inf, np.float32)
    codes = np.zeros((H, W, 4), np.int32)
    pix = None if pixels is None else _c(pixels, np.int32)
    lib().orc_antialias(C.byref(_cam(cam)), _p(_c(V, np.float32)), _p(_c(F, np.int32)), _p(_c(adj, np.int32)),
                        _p(_c(face_id, np.int32)), _p(_c(mesh_depth, np.float32)), _p(_c(mesh_rgb, np.float32)),
                        _p(pix), C.c_int64(0 if pixels is None else len(pixels)), _p(cov), _p(rgb), _p(depth),
                        _p(codes))
    return cov, rgb, depth, codes


def tile_bounds_cov(cam, cov, depth):
    T = n_tiles(cam)
    far = np.zeros(T, np.float32)
    full = np.zeros(T, np.uint8)
    lib().orc_tile_bounds_cov(C.byref(_cam(cam)), _p(_c(cov, np.float32)), _p(_c(depth, np.float32)), _p(far),
                              _p(full))
    return far, full


def tile_depth_bounds(cam, mesh_depth):
    md = _c(mesh_depth, np.float32).reshape(-1)
    T = n_tiles(cam)
    far = np.zeros(T, np.float32)
    full = np.zeros(T, np.uint8)
    lib().orc_tile_depth_bounds(C.byref(_cam(cam)), _p(md), _p(far), _p(full))
    return far, full


# ----------------------------------------------------------- Gaussians ----

def project(cam, g):
    N = len(g.means)
    means, ls = _c(g.means, np.float32), _c(g.log_scales, np.float32)
    q, lo, col = _c(g.quats, np.float32), _c(g.logits, np.float32), _c(g.colors, np.float32)
    splats = np.zeros((N, S_STRIDE), np.float32)
    radii = np.zeros(N, np.int32)
    touched = np.zeros(N, np.int32)
    margin = np.zeros(N, np.float64)
    lib().orc_project_gaussians(C.byref(_cam(cam)), C.c_int32(g.sh_degree), C.c_int32(N),
                                _p(means), _p(ls), _p(q), _p(lo), _p(col),
                                _p(splats), _p(radii), _p(touched), _p(margin), None)
    return splats, radii, touched, margin


def project_depth_model(cam, g):
    """Soft-split depth model [N][4] = (g_u, g_v, sigma_z, 0) of each Gaussian
    (zeros where culled); see depth_model_f64."""
    N = len(g.means)
    splats = np.zeros((N, S_STRIDE), np.float32)
    radii = np.zeros(N, np.int32)
    touched = np.zeros(N, np.int32)
    margin = np.zeros(N, np.float64)
    dm = np.zeros((N, 4), np.float32)
    lib().orc_project_gaussians(C.byref(_cam(cam)), C.c_int32(g.sh_degree), C.c_int32(N),
                                _p(_c(g.means, np.float32)), _p(_c(g.log_scales, np.float32)),
                                _p(_c(g.quats, np.float32)), _p(_c(g.logits, np.float32)),
                                _p(_c(g.colors, np.float32)), _p(splats), _p(radii), _p(touched), _p(margin), _p(dm))
    return dm


PROJ_PARAMS = ("mean", "log_scale", "quat", "logit", "color")


def proj_nparams(sh_degree):
    """Parameters of one Gaussian in the projection gradient's numbering:
    mean 0-2, log-scale 3-5, quaternion (w, x, y, z) 6-9, logit 10, colour
    coefficient k of channel ch at 11 + 3 k + ch."""
    return 11 + 3 * ((sh_degree + 1) ** 2 if sh_degree >= 0 else 1)


def project_fd(cam, g, v_splats, gids, params, hs, v_depth_model=None):
    """dL/d(3D parameter) by central differences (double, Richardson) for
    L = sum over record fields of v_splats . record (+ v_depth_model . depth
    model); see orc_project_fd."""
    n = len(gids)
    grad = np.zeros(n, np.float64)
    status = np.zeros(n, np.int32)
    vd = None if v_depth_model is None else _c(v_depth_model, np.float32)
    lib().orc_project_fd(C.byref(_cam(cam)), C.c_int32(g.sh_degree), _p(_c(g.means, np.float32)),
                         _p(_c(g.log_scales, np.float32)), _p(_c(g.quats, np.float32)),
                         _p(_c(g.logits, np.float32)), _p(_c(g.colors, np.float32)),
                         _p(_c(v_splats, np.float32)), _p(vd), C.c_int32(n), _p(_c(gids, np.int32)),
                         _p(_c(params, np.int32)), _p(_c(hs, np.float64)), _p(grad), _p(status))
    return grad, status


def sh_basis(deg, direction):
    d = _c(direction, np.float64)
    Y = np.zeros(16, np.float64)
    lib().orc_sh_basis(C.c_int(deg), _p(d), _p(Y))
    return Y[: (deg + 1) ** 2]


def bin_gaussians(cam, splats, radii, tile_far=None, tile_full=None, cull=False):
    splats, radii = _c(splats, np.float32), _c(radii, np.int32)
    N = len(radii)
    T = n_tiles(cam)
    tf = _c(np.full(T, np.inf) if tile_far is None else tile_far, np.float32)
    tu = _c(np.zeros(T) if tile_full is None else tile_full, np.uint8)
    c = _cam(cam)
    pre = C.c_int64(0)
    K = lib().orc_bin_gaussians(C.byref(c), C.c_int32(N), _p(splats), _p(radii), _p(tf), _p(tu),
                                C.c_int32(int(cull)), None, None, C.c_int64(0), C.byref(pre))
    keys = np.zeros(max(K, 1), np.uint64)
    gids = np.zeros(max(K, 1), np.int32)
    lib().orc_bin_gaussians(C.byref(c), C.c_int32(N), _p(splats), _p(radii), _p(tf), _p(tu),
                            C.c_int32(int(cull)), _p(keys), _p(gids), C.c_int64(K), C.byref(pre))
    return keys[:K], gids[:K], int(pre.value)


def tile_lists(cam, splats, radii, tiles=None):
    """CSR lists (tile_start[T+1], entries) over all tiles, or only ``tiles``."""
    splats, radii = _c(splats, np.float32), _c(radii, np.int32)
    T = n_tiles(cam)
    mask = None
    if tiles is not None:
        mask = np.zeros(T, np.uint8)
        mask[np.asarray(tiles, np.int64)] = 1
    start = np.zeros(T + 1, np.int64)
    c = _cam(cam)
    K = lib().orc_tile_lists(C.byref(c), C.c_int32(len(radii)), _p(splats), _p(radii), _p(mask), _p(start), None,
                             C.c_int64(0))
    entries = np.zeros(max(K, 1), np.int32)
    lib().orc_tile_lists(C.byref(c), C.c_int32(len(radii)), _p(splats), _p(radii), _p(mask), _p(start),
                         _p(entries), C.c_int64(K))
    return start, entries


SPLIT_PHI, SPLIT_LOGISTIC = 0, 1


def _soft(depth_model, softness):
    if depth_model is None or not softness > 0.0:
        return None, C.c_double(0.0)
    return _c(depth_model, np.float32), C.c_double(float(softness))


def composite_fwd(cam, bg, splats, lists, mesh_depth, mesh_rgb, face_id, tiles=None, depth_model=None,
                  softness=0.0, split=SPLIT_PHI, mesh_cov=None):
    """Full-frame outputs; only pixels of ``tiles`` (all when None) are written.
    With depth_model and softness > 0: the soft split (front fraction Phi, or
    its logistic approximation with split=SPLIT_LOGISTIC).  With mesh_cov: the
    antialiased mesh layer (mesh_rgb premultiplied, mesh_depth the split depth)."""
    dm, sf = _soft(depth_model, softness)
    start, entries = lists
    H, W = cam.height, cam.width
    out = {
        "rgb": np.zeros((H, W, 3), np.float32), "depth": np.zeros((H, W), np.float32),
        "alpha": np.zeros((H, W), np.float32), "T": np.zeros((H, W), np.float32),
        "n_contrib": np.zeros((H, W), np.int32), "margins": np.full((H, W, 5), np.inf),
    }
    bgv = _c(bg, np.float32)
    tl = None if tiles is None else _c(tiles, np.int32)
    lib().orc_composite_fwd(
        C.byref(_cam(cam)), _p(bgv), _p(_c(splats, np.float32)), _p(_c(start, np.int64)),
        _p(_c(entries, np.int32)), _p(_c(mesh_depth, np.float32)), _p(_c(mesh_rgb, np.float32)),
        _p(_c(face_id, np.int32)), _p(_opt(mesh_cov, np.float32)), _p(tl),
        C.c_int32(0 if tiles is None else len(tiles)),
        _p(out["rgb"]), _p(out["depth"]), _p(out["alpha"]), _p(out["T"]), _p(out["n_contrib"]),
        _p(out["margins"]), _p(dm), sf, C.c_int32(split))
    return out


def composite_fd(cam, bg, splats, radii, lists, mesh_depth, mesh_rgb, face_id, grads,
                 gids, fields, hs, tie_band=1e-5, depth_model=None, softness=0.0, split=SPLIT_PHI, mesh_cov=None):
    """fields 0..9: record fields; 12, 13, 14: depth model g_u, g_v, sigma_z.
    With mesh_cov: over the antialiased mesh layer (as composite_fwd)."""
    dm, sf = _soft(depth_model, softness)
    start, entries = lists
    g_rgb, g_depth, g_alpha = (_c(x, np.float32) for x in grads)
    n = len(gids)
    grad = np.zeros(n, np.float64)
    status = np.zeros(n, np.int32)
    lib().orc_composite_fd(
        C.byref(_cam(cam)), _p(_c(bg, np.float32)), _p(_c(splats, np.float32)), _p(_c(radii, np.int32)),
        _p(_c(start, np.int64)), _p(_c(entries, np.int32)), _p(_c(mesh_depth, np.float32)),
        _p(_c(mesh_rgb, np.float32)), _p(_c(face_id, np.int32)), _p(_opt(mesh_cov, np.float32)), _p(g_rgb),
        _p(g_depth), _p(g_alpha),
        C.c_int32(n), _p(_c(gids, np.int32)), _p(_c(fields, np.int32)), _p(_c(hs, np.float64)),
        C.c_double(tie_band), _p(grad), _p(status), _p(dm), sf, C.c_int32(split))
    return grad, status


def mesh_fd(cam, bg, V, F, vcol, face_id, splats, lists, mesh_depth, mesh_rgb, grads,
            vids, fields, hs, tie_band=1e-5, depth_model=None, softness=0.0, split=SPLIT_PHI, adj=None):
    """dL/d(vertex position 0..2, colour 3..5); with adj (mesh_edges) through the
    antialiased layer as well.  mesh_depth / mesh_rgb: the interpolated images."""
    dm, sf = _soft(depth_model, softness)
    start, entries = lists
    V, F, vcol = _c(V, np.float32), _c(F, np.int32), _c(vcol, np.float32)
    g_rgb, g_depth, g_alpha = (_c(x, np.float32) for x in grads)
    n = len(vids)
    grad = np.zeros(n, np.float64)
    status = np.zeros(n, np.int32)
    lib().orc_mesh_fd(
        C.byref(_cam(cam)), _p(_c(bg, np.float32)), _p(V), C.c_int32(len(V)), _p(F), C.c_int32(len(F)),
        _p(vcol), _p(_c(face_id, np.int32)), _p(_opt(adj, np.int32)), _p(_c(splats, np.float32)),
        _p(_c(start, np.int64)),
        _p(_c(entries, np.int32)), _p(_c(mesh_depth, np.float32)), _p(_c(mesh_rgb, np.float32)),
        _p(g_rgb), _p(g_depth), _p(g_alpha), C.c_int32(n), _p(_c(vids, np.int32)),
        _p(_c(fields, np.int32)), _p(_c(hs, np.float64)), C.c_double(tie_band), _p(grad), _p(status), _p(dm), sf,
        C.c_int32(split))
    return grad, status


def composite_one(px, py, splats, order, D=np.inf, covered=False, cm=(0, 0, 0), bg=(1, 1, 1), f32=True,
                  depth_model=None, softness=0.0, split=SPLIT_PHI, cov=None):
    """One pixel over an explicit ordered list of splat ids: rgb, depth, alpha, T,
    n_contrib.  The mesh layer: covered (0/1) with colour cm, or, with cov, a
    coverage in [0, 1] with premultiplied colour cm."""
    dm, sf = _soft(depth_model, softness)
    out = np.zeros(7, np.float64)
    lst = _c(order, np.int32)
    a = float(cov) if cov is not None else (1.0 if covered else 0.0)
    M = np.asarray(cm, np.float64) if (cov is not None or covered) else np.zeros(3)
    lib().orc_composite_one(C.c_int32(int(f32)), C.c_double(px), C.c_double(py), _p(lst), C.c_int64(len(lst)),
                            _p(_c(splats, np.float32)), C.c_double(D), C.c_double(a),
                            _p(_c(M, np.float64)), _p(_c(bg, np.float64)), _p(out), _p(dm), sf, C.c_int32(split))
    return {"rgb": out[:3], "depth": out[3], "alpha": out[4], "T": out[5], "n_contrib": int(out[6])}


# ------------------------------------------------------------ pipeline ----

def render(scene, cam=None, tiles=None, softness=0.0, split=SPLIT_PHI, antialias_edges=False):
    """Whole forward pass from raw inputs for the listed tiles (all when None),
    with the soft split when softness > 0 and the antialiased mesh layer when
    antialias_edges is set (the z-buffer and interpolation then also cover a
    one-pixel ring around the tiles, whose pairs the antialiasing reads).

    Returns a dict of full-frame arrays (pixels outside ``tiles`` are zero)
    with every intermediate the parity tests look at."""
    cam = scene.camera if cam is None else cam
    W, H = cam.width, cam.height
    TW = (W + 15) // 16
    if tiles is None:
        pixels = None
        tiles_arr = None
        mesh_pixels = None
    else:
        tiles_arr = np.asarray(tiles, np.int32)
        pix = []
        for t in tiles_arr:
            tx, ty = t % TW, t // TW
            ys = np.arange(ty * 16, min(ty * 16 + 16, H))
            xs = np.arange(tx * 16, min(tx * 16 + 16, W))
            pix.append((ys[:, None] * W + xs[None, :]).reshape(-1))
        pixels = np.concatenate(pix).astype(np.int32)
        mesh_pixels = pixels
        if antialias_edges:
            ring = [pixels]
            i, j = pixels % W, pixels // W
            for di, dj in ((-1, 0), (1, 0), (0, -1), (0, 1)):
                ok = (i + di >= 0) & (i + di < W) & (j + dj >= 0) & (j + dj < H)
                ring.append(((j + dj) * W + (i + di))[ok])
            mesh_pixels = np.unique(np.concatenate(ring)).astype(np.int32)
    m = scene.mesh
    fid_s, best_s, second_s = zbuffer(cam, m.verts, m.faces, mesh_pixels)
    depth_s, rgb_s = interp_mesh(cam, m.verts, m.faces, m.vcol, fid_s, mesh_pixels)
    face_id = np.full(W * H, -1, np.int32)
    mesh_depth = np.full(W * H, np.inf, np.float32)
    mesh_rgb = np.zeros((W * H, 3), np.float32)
    best = np.full(W * H, np.inf, np.float32)
    second = np.full(W * H, np.inf, np.float32)
    sel = np.arange(W * H) if mesh_pixels is None else mesh_pixels
    face_id[sel], mesh_depth[sel], mesh_rgb[sel] = fid_s, depth_s, rgb_s
    best[sel], second[sel] = best_s, second_s
    splats, radii, touched, margin = project(cam, scene.gaussians)
    lists = tile_lists(cam, splats, radii, tiles_arr)
    dm = project_depth_model(cam, scene.gaussians) if softness > 0.0 else None
    layer = {}
    if antialias_edges:
        adj = mesh_edges(m.faces)
        cov, rgb_aa, depth_aa, codes = antialias(cam, m.verts, m.faces, adj, face_id, mesh_depth, mesh_rgb, pixels)
        layer = dict(adj=adj, cov=cov, rgb_aa=rgb_aa, depth_aa=depth_aa, aa_codes=codes)
        out = composite_fwd(cam, scene.bg, splats, lists, depth_aa, rgb_aa, face_id, tiles_arr,
                            depth_model=dm, softness=softness, split=split, mesh_cov=cov)
    else:
        out = composite_fwd(cam, scene.bg, splats, lists, mesh_depth, mesh_rgb, face_id, tiles_arr,
                            depth_model=dm, softness=softness, split=split)
    out.update(face_id=face_id.reshape(H, W), mesh_depth=mesh_depth.reshape(H, W),
               mesh_rgb=mesh_rgb.reshape(H, W, 3), zbest=best.reshape(H, W),
               zsecond=second.reshape(H, W), splats=splats, radii=radii,
               tiles_touched=touched, radius_margin=margin, lists=lists, pixels=pixels, depth_model=dm, **layer)
    return out

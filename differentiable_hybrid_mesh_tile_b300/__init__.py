"""Python binding of libgm, the B300 CUDA library for tile-based forward and
backward rendering of scenes holding a triangle mesh and 3D Gaussians (the
hybrid renderer of "A Lightweight and Differentiable Renderer for Joint Mesh
and 3D Gaussian Splat Scenes").

The ``gm_*`` functions mirror the C ABI of ``include/gm.h`` one to one: they
check and marshal torch CUDA tensors into raw device pointers and the current
CUDA stream, and raise :class:`GmError` on a non-zero status.  Every step of
the computation runs in the library's kernels; there is no CPU path, and the
import fails loudly when ``libgm.so`` has not been built.

:class:`HybridRenderer` sequences the seven calls for one camera and owns the
device buffers between them (allocation and ordering only).
"""

from __future__ import annotations

import ctypes as C
import os
import re
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgm.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "gm.h")

GM_OK, GM_ERR_INVALID_ARG, GM_ERR_CAPACITY, GM_ERR_CUDA, GM_ERR_TIMEOUT, GM_ERR_INTERNAL = range(6)
GM_CNT_K, GM_CNT_K_PRECULL, GM_CNT_FLAGS = 0, 1, 2
GM_FLAG_OVERFLOW, GM_FLAG_TIMEOUT = 1, 2
GM_SPLIT_PHI, GM_SPLIT_LOGISTIC = 0, 1
TILE = 16
SPLAT_STRIDE = 12


class GmError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__("%s failed with status %d: %s" % (where, status, msg))
        self.status = status


class gm_camera(C.Structure):
    _fields_ = [("width", C.c_int32), ("height", C.c_int32),
                ("fx", C.c_float), ("fy", C.c_float), ("cx", C.c_float), ("cy", C.c_float),
                ("near_plane", C.c_float), ("far_plane", C.c_float),
                ("R", C.c_float * 9), ("t", C.c_float * 3)]


class gm_opts(C.Structure):
    _fields_ = [("bg", C.c_float * 3), ("cull_occluded", C.c_int32), ("sh_degree", C.c_int32),
                ("tile_test", C.c_int32), ("softness", C.c_float), ("soft_split", C.c_int32)]


class gm_aa_layer(C.Structure):
    _fields_ = [("cov", C.c_void_p), ("back", C.c_void_p), ("T_back", C.c_void_p), ("n_back", C.c_void_p),
                ("v_cov", C.c_void_p), ("v_rgb", C.c_void_p)]


class gm_staged(C.Structure):
    """Staged-record buffer of the tile lists (gm.h: gm_staged)."""
    _fields_ = [("recs", C.c_void_p), ("cap", C.c_int32)]


_VP = C.c_void_p
_I32 = C.c_int32
_SIGS = {
    "gm_bin_triangles_workspace_size": (C.c_size_t, [_I32, _I32, _I32, _I32]),
    "gm_bin_triangles": (C.c_int, [_VP, _VP, _I32, _VP, _I32, _VP, _VP, _I32, _VP, _VP, _VP, C.c_size_t, _VP]),
    "gm_zbuffer": (C.c_int, [_VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP, _VP]),
    "gm_zbuffer_direct_workspace_size": (C.c_size_t, [_I32, _I32, _I32]),
    "gm_zbuffer_direct": (C.c_int, [_VP, _VP, _I32, _VP, _I32, _VP, _VP, C.c_size_t, _VP]),
    "gm_interp_mesh": (C.c_int, [_VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "gm_project_gaussians": (C.c_int, [_VP, _VP, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "gm_project_gaussians_bwd": (C.c_int, [_VP, _VP, _I32] + [_VP] * 8 + [_I32] + [_VP] * 6),
    "gm_project_gaussians_views": (C.c_int, [_VP, _I32, _VP, _I32] + [_VP] * 9 + [_VP]),
    "gm_project_gaussians_bwd_views": (C.c_int, [_VP, _I32, _VP, _I32] + [_VP] * 8 + [_I32] + [_VP] * 6),
    "gm_bin_sort_gaussians_workspace_size": (C.c_size_t, [_I32, _I32, _I32, _I32]),
    "gm_bin_sort_gaussians": (C.c_int, [_VP, _VP, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP,
                                        C.c_size_t, _VP]),
    "gm_bin_gaussians": (C.c_int, [_VP, _VP, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP,
                                   C.c_size_t, _VP]),
    "gm_sort_gaussians_by_depth": (C.c_int, [_VP, _I32, _VP, _VP, _I32, _VP, _VP, C.c_size_t, _VP]),
    "gm_composite_hybrid_fwd": (C.c_int, [_VP, _VP, _I32] + [_VP] * 16),
    "gm_composite_hybrid_bwd": (C.c_int, [_VP, _VP, _I32] + [_VP] * 16 + [_I32, _VP, _I32] + [_VP] * 7),
    "gm_staged_bytes": (C.c_size_t, [_I32, C.c_float]),
    "gm_get_copy_status": (C.c_int, [C.POINTER(C.c_uint32), _I32]),
    "gm_mesh_edges_workspace_size": (C.c_size_t, [_I32]),
    "gm_mesh_edges": (C.c_int, [_VP, _I32, _I32, _VP, _VP, _VP, C.c_size_t, _VP]),
    "gm_antialias": (C.c_int, [_VP, _VP, _I32, _VP, _I32] + [_VP] * 10),
    "gm_antialias_bwd": (C.c_int, [_VP, _VP, _I32, _VP, _I32] + [_VP] * 13),
    "gm_interp_mesh_bwd": (C.c_int, [_VP, _VP, _I32, _VP, _I32] + [_VP] * 7),
    "gm_bin_triangles_noalloc": (C.c_int, [_VP, _VP, _I32, _VP, _I32, _VP, _VP, _I32, _VP, _VP, _VP]),
    "gm_set_wait_limit": (C.c_int, [C.c_uint32]),
    "gm_get_wait_limit": (C.c_int, [C.POINTER(C.c_uint32)]),
    "gm_last_error": (C.c_char_p, []),
}

_lib = None


def lib():
    """The loaded libgm.so (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libgm.so not built: run differentiable_hybrid_mesh_tile_b300/build.py "
                              "(or __graft_entry__.build()); there is no CPU fallback")
        _lib = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(_lib, name)
            fn.restype = res
            fn.argtypes = args
    return _lib


def header_functions():
    """Names of the functions include/gm.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(gm_\w+)\s*\(", text, re.M)))


# ------------------------------------------------------------ marshalling --

def make_camera(cam) -> gm_camera:
    c = gm_camera()
    c.width, c.height = int(cam.width), int(cam.height)
    c.fx, c.fy, c.cx, c.cy = float(cam.fx), float(cam.fy), float(cam.cx), float(cam.cy)
    c.near_plane, c.far_plane = float(cam.near), float(cam.far)
    R = [float(x) for x in torch.as_tensor(cam.R, dtype=torch.float32).reshape(9)]
    t = [float(x) for x in torch.as_tensor(cam.t, dtype=torch.float32).reshape(3)]
    for k in range(9):
        c.R[k] = R[k]
    for k in range(3):
        c.t[k] = t[k]
    return c


def make_opts(bg=(1.0, 1.0, 1.0), cull_occluded=True, sh_degree=-1, tile_test=True, softness=0.0,
              soft_split=0) -> gm_opts:
    o = gm_opts()
    for k in range(3):
        o.bg[k] = float(bg[k])
    o.cull_occluded = int(bool(cull_occluded))
    o.sh_degree = int(sh_degree)
    o.tile_test = int(bool(tile_test))
    o.softness = float(softness)
    o.soft_split = int(soft_split)
    return o


def _p(t: Optional[torch.Tensor], dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError("expected %s, got %s" % (dtype, t.dtype))
    return C.c_void_p(t.data_ptr())


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, where: str):
    if status != GM_OK:
        raise GmError(status, where, lib().gm_last_error().decode())


F32, I32, U8, I64 = torch.float32, torch.int32, torch.uint8, torch.int64


# -------------------------------------------------------- the seven calls --

def gm_bin_triangles_workspace_size(nF: int, cap: int, width: int, height: int) -> int:
    return int(lib().gm_bin_triangles_workspace_size(nF, cap, width, height))


def gm_bin_triangles(cam: gm_camera, V, F, tile_range, tri_ids, cap: int, counters, ws, sync: bool = True):
    """Returns the needed number of entries when ``sync`` (K read back to the
    host), else None; raises GmError(GM_ERR_CAPACITY) when K > cap."""
    k = C.c_int32(0)
    st = lib().gm_bin_triangles(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0], _p(tile_range, I32),
                                _p(tri_ids, I32), cap, _p(counters, I32), C.byref(k) if sync else None,
                                _p(ws), ws.numel() * ws.element_size(), _stream())
    if st == GM_ERR_CAPACITY:
        raise GmError(st, "gm_bin_triangles", "capacity %d < needed %d" % (cap, k.value))
    _check(st, "gm_bin_triangles")
    return k.value if sync else None


def gm_bin_triangles_noalloc(cam: gm_camera, V, F, tile_range, tri_ids, cap: int, counters, sync: bool = True):
    """gm_bin_triangles for callers that may not allocate device memory: the
    scratch is the library's static device array (GM_NOALLOC_TRI_SCRATCH_BYTES),
    so no workspace is passed.  Overlapping calls share that array and race."""
    k = C.c_int32(0)
    st = lib().gm_bin_triangles_noalloc(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0],
                                        _p(tile_range, I32), _p(tri_ids, I32), cap, _p(counters, I32),
                                        C.byref(k) if sync else None, _stream())
    if st == GM_ERR_CAPACITY:
        raise GmError(st, "gm_bin_triangles_noalloc", "capacity %d < needed %d" % (cap, k.value))
    _check(st, "gm_bin_triangles_noalloc")
    return k.value if sync else None


GM_WAIT_LIMIT_DEFAULT = 1 << 22


def gm_set_wait_limit(polls: int):
    """Bound on the polls of the sorts' inter-block waits on the current device
    (gm.h: gm_set_wait_limit); set it only while no libgm kernel runs."""
    _check(lib().gm_set_wait_limit(C.c_uint32(int(polls))), "gm_set_wait_limit")


def gm_get_wait_limit() -> int:
    v = C.c_uint32(0)
    _check(lib().gm_get_wait_limit(C.byref(v)), "gm_get_wait_limit")
    return int(v.value)


def gm_zbuffer(cam: gm_camera, V, F, tile_range, tri_ids, face_id):
    _check(lib().gm_zbuffer(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0], _p(tile_range, I32),
                            _p(tri_ids, I32), _p(face_id, I32), _stream()), "gm_zbuffer")


def gm_zbuffer_direct_workspace_size(nF: int, width: int, height: int) -> int:
    return int(lib().gm_zbuffer_direct_workspace_size(nF, width, height))


def gm_zbuffer_direct(cam: gm_camera, V, F, face_id, ws):
    _check(lib().gm_zbuffer_direct(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0], _p(face_id, I32),
                                   _p(ws), ws.numel() * ws.element_size(), _stream()), "gm_zbuffer_direct")


def gm_interp_mesh(cam: gm_camera, V, F, vcol, face_id, mesh_depth, mesh_rgb, tile_far, tile_full):
    _check(lib().gm_interp_mesh(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0], _p(vcol, F32),
                                _p(face_id, I32), _p(mesh_depth, F32), _p(mesh_rgb, F32), _p(tile_far, F32),
                                _p(tile_full, U8), _stream()), "gm_interp_mesh")


def gm_project_gaussians(cam: gm_camera, opts: gm_opts, means, log_scales, quats, logits, colors, splats, radii,
                         tiles_touched, depth_model=None):
    _check(lib().gm_project_gaussians(C.byref(cam), C.byref(opts), means.shape[0], _p(means, F32),
                                      _p(log_scales, F32), _p(quats, F32), _p(logits, F32), _p(colors, F32),
                                      _p(splats, F32), _p(radii, I32), _p(tiles_touched, I32),
                                      _p(depth_model, F32), _stream()),
           "gm_project_gaussians")


def _cam_array(cams):
    arr = (gm_camera * len(cams))()
    for k, c in enumerate(cams):
        arr[k] = c
    return arr


def gm_project_gaussians_views(cams, opts: gm_opts, means, log_scales, quats, logits, colors, splats, radii,
                               tiles_touched, depth_model=None):
    """cams: a list of gm_camera; splats [V][N][12], radii / tiles_touched [V][N],
    depth_model [V][N][4] or None."""
    arr = _cam_array(cams)
    _check(lib().gm_project_gaussians_views(arr, len(cams), C.byref(opts), means.shape[0], _p(means, F32),
                                            _p(log_scales, F32), _p(quats, F32), _p(logits, F32), _p(colors, F32),
                                            _p(splats, F32), _p(radii, I32), _p(tiles_touched, I32),
                                            _p(depth_model, F32), _stream()),
           "gm_project_gaussians_views")


def gm_project_gaussians_bwd_views(cams, opts: gm_opts, means, log_scales, quats, logits, colors, radii, v_splats,
                                   v_means, v_log_scales, v_quats, v_logits, v_colors, accumulate=False,
                                   v_depth_model=None):
    arr = _cam_array(cams)
    _check(lib().gm_project_gaussians_bwd_views(arr, len(cams), C.byref(opts), means.shape[0], _p(means, F32),
                                                _p(log_scales, F32), _p(quats, F32), _p(logits, F32),
                                                _p(colors, F32), _p(radii, I32), _p(v_splats, F32),
                                                _p(v_depth_model, F32), int(bool(accumulate)), _p(v_means, F32), _p(v_log_scales, F32),
                                                _p(v_quats, F32), _p(v_logits, F32), _p(v_colors, F32), _stream()),
           "gm_project_gaussians_bwd_views")


def gm_project_gaussians_bwd(cam: gm_camera, opts: gm_opts, means, log_scales, quats, logits, colors, radii,
                             v_splats, v_means, v_log_scales, v_quats, v_logits, v_colors, accumulate=False,
                             v_depth_model=None):
    _check(lib().gm_project_gaussians_bwd(C.byref(cam), C.byref(opts), means.shape[0], _p(means, F32),
                                          _p(log_scales, F32), _p(quats, F32), _p(logits, F32), _p(colors, F32),
                                          _p(radii, I32), _p(v_splats, F32), _p(v_depth_model, F32),
                                          int(bool(accumulate)), _p(v_means, F32),
                                          _p(v_log_scales, F32), _p(v_quats, F32), _p(v_logits, F32),
                                          _p(v_colors, F32), _stream()),
           "gm_project_gaussians_bwd")


def gm_bin_sort_gaussians_workspace_size(N: int, cap: int, width: int, height: int) -> int:
    return int(lib().gm_bin_sort_gaussians_workspace_size(N, cap, width, height))


def gm_bin_sort_gaussians(cam: gm_camera, opts: gm_opts, splats, radii, tile_far, tile_full, keys, gids, tile_range,
                          cap: int, counters, ws, sync: bool = True):
    k = C.c_int32(0)
    st = lib().gm_bin_sort_gaussians(C.byref(cam), C.byref(opts), radii.shape[0], _p(splats, F32), _p(radii, I32),
                                     _p(tile_far, F32), _p(tile_full, U8), _p(keys, I64), _p(gids, I32),
                                     _p(tile_range, I32), cap, _p(counters, I32), C.byref(k) if sync else None,
                                     _p(ws), ws.numel() * ws.element_size(), _stream())
    if st == GM_ERR_CAPACITY:
        raise GmError(st, "gm_bin_sort_gaussians", "capacity %d < needed %d" % (cap, k.value))
    _check(st, "gm_bin_sort_gaussians")
    return k.value if sync else None


def _aa_ref(aa):
    return None if aa is None else C.byref(aa)


def make_aa_layer(cov, back, T_back, n_back, v_cov=None, v_rgb=None) -> gm_aa_layer:
    """gm_aa_layer over torch CUDA tensors (the antialiased layer's coverage and
    the back-chain buffers; v_cov / v_rgb for the backward)."""
    a = gm_aa_layer()
    a.cov, a.back, a.T_back, a.n_back = _p(cov, F32), _p(back, F32), _p(T_back, F32), _p(n_back, I32)
    a.v_cov, a.v_rgb = _p(v_cov, F32), _p(v_rgb, F32)
    return a


def gm_mesh_edges_workspace_size(nF: int) -> int:
    return int(lib().gm_mesh_edges_workspace_size(nF))


def gm_mesh_edges(F, nV, adj, counters, ws):
    _check(lib().gm_mesh_edges(_p(F, I32), F.shape[0], int(nV), _p(adj, I32), _p(counters, I32), _p(ws),
                               ws.numel() * ws.element_size(), _stream()), "gm_mesh_edges")


def gm_antialias(cam: gm_camera, V, F, adj, face_id, mesh_depth, mesh_rgb, cov, rgb_aa, depth_aa, tile_far,
                 tile_full):
    _check(lib().gm_antialias(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0], _p(adj, I32),
                              _p(face_id, I32), _p(mesh_depth, F32), _p(mesh_rgb, F32), _p(cov, F32), _p(rgb_aa, F32),
                              _p(depth_aa, F32), _p(tile_far, F32), _p(tile_full, U8), _stream()), "gm_antialias")


def gm_antialias_bwd(cam: gm_camera, V, F, adj, face_id, mesh_depth, mesh_rgb, cov, depth_aa, v_cov, v_rgb_aa,
                     v_depth_aa, v_mesh_rgb, v_mesh_depth, v_verts):
    _check(lib().gm_antialias_bwd(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0], _p(adj, I32),
                                  _p(face_id, I32), _p(mesh_depth, F32), _p(mesh_rgb, F32), _p(cov, F32),
                                  _p(depth_aa, F32), _p(v_cov, F32),
                                  _p(v_rgb_aa, F32), _p(v_depth_aa, F32), _p(v_mesh_rgb, F32), _p(v_mesh_depth, F32),
                                  _p(v_verts, F32), _stream()), "gm_antialias_bwd")


def gm_interp_mesh_bwd(cam: gm_camera, V, F, vcol, face_id, v_mesh_rgb, v_mesh_depth, v_verts, v_vcol):
    _check(lib().gm_interp_mesh_bwd(C.byref(cam), _p(V, F32), V.shape[0], _p(F, I32), F.shape[0], _p(vcol, F32),
                                    _p(face_id, I32), _p(v_mesh_rgb, F32), _p(v_mesh_depth, F32), _p(v_verts, F32),
                                    _p(v_vcol, F32), _stream()), "gm_interp_mesh_bwd")


def gm_sort_gaussians_by_depth(cam: gm_camera, splats, radii, cap: int, counters, ws):
    _check(lib().gm_sort_gaussians_by_depth(C.byref(cam), radii.shape[0], _p(splats, F32), _p(radii, I32), cap,
                                            _p(counters, I32), _p(ws), ws.numel() * ws.element_size(), _stream()),
           "gm_sort_gaussians_by_depth")


def gm_bin_gaussians(cam: gm_camera, opts: gm_opts, splats, radii, tile_far, tile_full, keys, gids, tile_range,
                     cap: int, counters, ws, sync: bool = True):
    """The second half of gm_bin_sort_gaussians (after gm_sort_gaussians_by_depth
    on the same workspace)."""
    k = C.c_int32(0)
    st = lib().gm_bin_gaussians(C.byref(cam), C.byref(opts), radii.shape[0], _p(splats, F32), _p(radii, I32),
                                _p(tile_far, F32), _p(tile_full, U8), _p(keys, I64), _p(gids, I32),
                                _p(tile_range, I32), cap, _p(counters, I32), C.byref(k) if sync else None,
                                _p(ws), ws.numel() * ws.element_size(), _stream())
    if st == GM_ERR_CAPACITY:
        raise GmError(st, "gm_bin_gaussians", "capacity %d < needed %d" % (cap, k.value))
    _check(st, "gm_bin_gaussians")
    return k.value if sync else None


def gm_staged_bytes(cap: int, softness: float = 0.0) -> int:
    return int(lib().gm_staged_bytes(int(cap), float(softness)))


def make_staged(recs, cap: int) -> gm_staged:
    """gm_staged over a 16-byte aligned device buffer of gm_staged_bytes(cap, softness) bytes."""
    s = gm_staged()
    s.recs = _p(recs)
    s.cap = int(cap)
    return s


def gm_get_copy_status(clear: bool = False) -> int:
    v = C.c_uint32(0)
    _check(lib().gm_get_copy_status(C.byref(v), int(bool(clear))), "gm_get_copy_status")
    return int(v.value)


def _staged_ref(st):
    return None if st is None else C.byref(st)


def gm_composite_hybrid_fwd(cam: gm_camera, opts: gm_opts, tile_range, gids, splats, mesh_depth, mesh_rgb, face_id,
                            out_rgb, out_depth, out_alpha, T_final, n_contrib, stats=None, depth_model=None,
                            aa=None, staged=None):
    _check(lib().gm_composite_hybrid_fwd(C.byref(cam), C.byref(opts), splats.shape[0], _p(tile_range, I32),
                                         _p(gids, I32), _p(splats, F32), _p(depth_model, F32),
                                         _p(mesh_depth, F32), _p(mesh_rgb, F32), _p(face_id, I32),
                                         _p(out_rgb, F32), _p(out_depth, F32), _p(out_alpha, F32), _p(T_final, F32),
                                         _p(n_contrib, I32), _aa_ref(aa), _staged_ref(staged), _p(stats, I64),
                                         _stream()),
           "gm_composite_hybrid_fwd")


def gm_composite_hybrid_bwd(cam: gm_camera, opts: gm_opts, tile_range, gids, splats, mesh_depth, mesh_rgb, face_id,
                            T_final, n_contrib, g_rgb, g_depth, g_alpha, v_splats, V=None, F=None, vcol=None,
                            v_verts=None, v_vcol=None, stats=None, depth_model=None, v_depth_model=None,
                            v_mesh_depth=None, aa=None, staged=None):
    nV = 0 if V is None else V.shape[0]
    nF = 0 if F is None else F.shape[0]
    _check(lib().gm_composite_hybrid_bwd(C.byref(cam), C.byref(opts), splats.shape[0], _p(tile_range, I32),
                                         _p(gids, I32), _p(splats, F32), _p(depth_model, F32),
                                         _p(mesh_depth, F32), _p(mesh_rgb, F32), _p(face_id, I32),
                                         _p(T_final, F32), _p(n_contrib, I32), _p(g_rgb, F32), _p(g_depth, F32),
                                         _p(g_alpha, F32), _p(v_splats, F32), _p(v_depth_model, F32),
                                         _p(v_mesh_depth, F32), _p(V, F32), nV, _p(F, I32), nF,
                                         _p(vcol, F32), _p(v_verts, F32), _p(v_vcol, F32), _aa_ref(aa),
                                         _staged_ref(staged), _p(stats, I64), _stream()),
           "gm_composite_hybrid_bwd")


# ------------------------------------------------------------- renderer --

class HybridRenderer:
    """One camera's forward / backward pass through the seven calls.

    ``upload`` copies a scene's mesh and Gaussians to the device; ``forward``
    renders (rgb, depth, alpha); ``backward`` takes dL/d(rgb, depth, alpha)
    and returns dL/d(splats) and dL/d(vertex positions, colours).  Buffers
    are kept between calls; the tile-entry capacities grow on demand (a
    GM_ERR_CAPACITY status triggers one reallocation and a retry).  With
    ``sync=False`` the binning calls do not read K back, so a whole step can
    be captured in a CUDA graph; the caller then checks ``overflowed()``.

    With ``concurrent=True`` the calls that do not depend on each other run on
    a second stream: the Gaussian projection beside the mesh binning,
    z-buffer and interpolation, and the mesh backward beside the composite
    backward (joined back into the caller's stream before anything reads
    their results; a captured graph keeps the two branches).

    ``antialias=True`` adds the analytic edge antialiasing of the mesh layer
    (``gm_antialias``; edge adjacency from ``gm_mesh_edges`` at upload): the
    Gaussians composite over a layer of fractional coverage at silhouettes and
    the backward pass adds the silhouette vertex gradients
    (``gm_antialias_bwd``, then ``gm_interp_mesh_bwd``), all on the caller's
    stream.

    ``zbuffer="direct"`` (default) finds the face ids with ``gm_zbuffer_direct``
    (no triangle lists); ``zbuffer="tile"`` with ``gm_bin_triangles`` and
    ``gm_zbuffer``.  Both give the same face ids.

    ``staged=True`` (default) gives the forward composite a staged-record
    buffer (``gm_staged``) that the backward composite then reads with bulk
    copies; ``staged=False`` makes the backward gather the records itself.

    ``softness > 0`` selects the soft split at the mesh surface (front
    fraction ``soft_split``: GM_SPLIT_PHI or GM_SPLIT_LOGISTIC): the
    projection also writes each Gaussian's depth model (``depth_model``), the
    backward pass writes its gradient (``v_depth_model``) and dL/d mesh depth
    through the split (``v_mesh_depth``), and the mesh backward then runs
    after the Gaussian backward on one stream (it reads ``v_mesh_depth``).
    """

    def __init__(self, cam, bg=(1.0, 1.0, 1.0), cull_occluded=True, device="cuda", headroom=1.25,
                 concurrent=True, tile_test=True, softness=0.0, soft_split=GM_SPLIT_PHI, antialias=False,
                 zbuffer="direct", staged=True):
        self.cam_desc = cam
        self.use_staged = bool(staged)
        self.staged = None
        self.cam = make_camera(cam)
        self.W, self.H = int(cam.width), int(cam.height)
        self.TW, self.TH = (self.W + TILE - 1) // TILE, (self.H + TILE - 1) // TILE
        self.T = self.TW * self.TH
        self.bg = tuple(float(x) for x in bg)
        self.cull = bool(cull_occluded)
        self.dev = torch.device(device)
        self.headroom = headroom
        self.concurrent = bool(concurrent)
        self.tile_test = bool(tile_test)
        self.softness = float(softness)
        if not self.softness >= 0.0:
            raise ValueError("softness must be >= 0")
        self.soft = self.softness > 0.0
        self.soft_split = int(soft_split)
        self.antialias = bool(antialias)
        if zbuffer not in ("direct", "tile"):
            raise ValueError("zbuffer must be 'direct' or 'tile'")
        self.zbuffer = zbuffer
        self.K_tri = None
        self._side = None
        self.tri_cap = 0
        self.g_cap = 0
        self.sh_degree = -1
        d = self.dev
        H, W = self.H, self.W
        self.tri_range = torch.zeros(self.T, 2, dtype=I32, device=d)
        self.g_range = torch.zeros(self.T, 2, dtype=I32, device=d)
        self.tri_counters = torch.zeros(4, dtype=I32, device=d)
        self.g_counters = torch.zeros(4, dtype=I32, device=d)
        self.face_id = torch.empty(H, W, dtype=I32, device=d)
        self.mesh_depth = torch.empty(H, W, dtype=F32, device=d)
        self.mesh_rgb = torch.empty(H, W, 3, dtype=F32, device=d)
        self.tile_far = torch.empty(self.T, dtype=F32, device=d)
        self.tile_full = torch.empty(self.T, dtype=U8, device=d)
        self.out_rgb = torch.empty(H, W, 3, dtype=F32, device=d)
        self.out_depth = torch.empty(H, W, dtype=F32, device=d)
        self.out_alpha = torch.empty(H, W, dtype=F32, device=d)
        self.T_final = torch.empty(H, W, dtype=F32, device=d)
        self.n_contrib = torch.empty(H, W, dtype=I32, device=d)
        self.v_mesh_depth = torch.zeros(H, W, dtype=F32, device=d) if self.soft or self.antialias else None
        self.depth_model = self.v_depth_model = None
        if self.antialias:
            self.cov = torch.zeros(H, W, dtype=F32, device=d)
            self.rgb_aa = torch.zeros(H, W, 3, dtype=F32, device=d)
            self.depth_aa = torch.zeros(H, W, dtype=F32, device=d)
            self.back = torch.zeros(H, W, 4, dtype=F32, device=d)
            self.T_back = torch.zeros(H, W, dtype=F32, device=d)
            self.n_back = torch.zeros(H, W, dtype=I32, device=d)
            self.v_cov = torch.zeros(H, W, dtype=F32, device=d)
            self.v_rgb_aa = torch.zeros(H, W, 3, dtype=F32, device=d)
            self.v_mesh_rgb = torch.zeros(H, W, 3, dtype=F32, device=d)
            self.v_interp_depth = torch.zeros(H, W, dtype=F32, device=d)
            self.aa = make_aa_layer(self.cov, self.back, self.T_back, self.n_back, self.v_cov, self.v_rgb_aa)
        else:
            self.aa = None

    def set_camera(self, cam):
        assert int(cam.width) == self.W and int(cam.height) == self.H
        self.cam_desc = cam
        self.cam = make_camera(cam)

    @property
    def opts(self) -> gm_opts:
        return make_opts(self.bg, self.cull, self.sh_degree, self.tile_test, self.softness, self.soft_split)

    def upload(self, mesh, gaussians):
        d = self.dev

        def t(x, dt):
            return torch.as_tensor(x).to(device=d, dtype=dt).contiguous()

        self.V, self.F, self.vcol = t(mesh.verts, F32), t(mesh.faces, I32), t(mesh.vcol, F32)
        self.means, self.log_scales = t(gaussians.means, F32), t(gaussians.log_scales, F32)
        self.quats, self.logits = t(gaussians.quats, F32), t(gaussians.logits, F32)
        self.colors = t(gaussians.colors, F32)
        self.sh_degree = int(gaussians.sh_degree)
        self._alloc_gauss(int(self.means.shape[0]))
        self._alloc_mesh_ws()
        if self.antialias:
            self.adj = torch.empty(self.F.shape[0], 3, dtype=I32, device=d)
            nb = gm_mesh_edges_workspace_size(int(self.F.shape[0]))
            ws = torch.empty((nb + 15) // 16 * 16 + 16, dtype=U8, device=d)
            cnt = torch.zeros(4, dtype=I32, device=d)
            gm_mesh_edges(self.F, self.V.shape[0], self.adj, cnt, ws)
            if int(cnt[GM_CNT_FLAGS].item()) & GM_FLAG_TIMEOUT:
                raise GmError(GM_ERR_TIMEOUT, "gm_mesh_edges", "a sort wait gave up")

    def _alloc_gauss(self, N):
        d = self.dev
        self.N = N
        self.splats = torch.zeros(N, SPLAT_STRIDE, dtype=F32, device=d)
        self.radii = torch.zeros(N, dtype=I32, device=d)
        self.tiles_touched = torch.zeros(N, dtype=I32, device=d)
        self.v_splats = torch.zeros(N, SPLAT_STRIDE, dtype=F32, device=d)
        if self.soft:
            self.depth_model = torch.zeros(N, 4, dtype=F32, device=d)
            self.v_depth_model = torch.zeros(N, 4, dtype=F32, device=d)
        self._alloc_g(max(self.g_cap, 1))

    def _alloc_g(self, cap):
        d = self.dev
        self.g_cap = cap
        self.keys = torch.empty(cap, dtype=I64, device=d)
        self.gids = torch.empty(cap, dtype=I32, device=d)
        nb = gm_bin_sort_gaussians_workspace_size(self.N, cap, self.W, self.H)
        self.g_ws = torch.empty((nb + 15) // 16 * 16, dtype=U8, device=d)
        if self.use_staged:
            nb = gm_staged_bytes(cap, self.softness)
            self.staged_buf = torch.empty((nb + 15) // 16 * 16, dtype=U8, device=d)
            self.staged = make_staged(self.staged_buf, cap)

    def _alloc_mesh_ws(self):
        """Triangle-list buffers (tile z-buffer) or the direct z-buffer's workspace."""
        if self.zbuffer == "tile":
            self._alloc_tri(max(self.tri_cap, 1))
        else:
            nb = gm_zbuffer_direct_workspace_size(int(self.F.shape[0]), self.W, self.H)
            self.zb_ws = torch.empty((nb + 15) // 16 * 16, dtype=U8, device=self.dev)

    def _alloc_tri(self, cap):
        d = self.dev
        self.tri_cap = cap
        self.tri_ids = torch.empty(cap, dtype=I32, device=d)
        nb = gm_bin_triangles_workspace_size(int(self.F.shape[0]), cap, self.W, self.H)
        self.tri_ws = torch.empty((nb + 15) // 16 * 16, dtype=U8, device=d)

    def _grow(self, needed):
        return max(int(needed * self.headroom) + 16, 16)

    def _side_stream(self):
        if self._side is None:
            self._side = torch.cuda.Stream(device=self.dev)
        return self._side

    def _zbuffer(self, sync: bool):
        """face_id: gm_zbuffer_direct, or triangle lists (grown on demand) and gm_zbuffer."""
        cam = self.cam
        if self.zbuffer == "direct":
            gm_zbuffer_direct(cam, self.V, self.F, self.face_id, self.zb_ws)
            return
        for attempt in range(2):
            try:
                self.K_tri = gm_bin_triangles(cam, self.V, self.F, self.tri_range, self.tri_ids, self.tri_cap,
                                              self.tri_counters, self.tri_ws, sync=sync)
                break
            except GmError as e:
                if e.status != GM_ERR_CAPACITY or attempt:
                    raise
                self._alloc_tri(self._grow(int(self.tri_counters[GM_CNT_K].item())))
        gm_zbuffer(cam, self.V, self.F, self.tri_range, self.tri_ids, self.face_id)

    def forward(self, sync: bool = True):
        cam, opts = self.cam, self.opts
        main = torch.cuda.current_stream(self.dev)
        side = self._side_stream() if self.concurrent else main
        if self.concurrent:
            side.wait_stream(main)
        with torch.cuda.stream(side):
            # the projection and the Gaussians' depth pre-sort need no mesh: they run
            # beside the mesh layer
            gm_project_gaussians(cam, opts, self.means, self.log_scales, self.quats, self.logits, self.colors,
                                 self.splats, self.radii, self.tiles_touched, self.depth_model)
            gm_sort_gaussians_by_depth(cam, self.splats, self.radii, self.g_cap, self.g_counters, self.g_ws)
        self._zbuffer(sync)
        gm_interp_mesh(cam, self.V, self.F, self.vcol, self.face_id, self.mesh_depth, self.mesh_rgb, self.tile_far,
                       self.tile_full)
        if self.antialias:
            gm_antialias(cam, self.V, self.F, self.adj, self.face_id, self.mesh_depth, self.mesh_rgb, self.cov,
                         self.rgb_aa, self.depth_aa, self.tile_far, self.tile_full)
        if self.concurrent:
            main.wait_stream(side)
        for attempt in range(2):
            try:
                if attempt:  # a new workspace: its depth pre-sort again
                    gm_sort_gaussians_by_depth(cam, self.splats, self.radii, self.g_cap, self.g_counters, self.g_ws)
                k = gm_bin_gaussians(cam, opts, self.splats, self.radii, self.tile_far, self.tile_full,
                                     self.keys, self.gids, self.g_range, self.g_cap, self.g_counters,
                                     self.g_ws, sync=sync)
                self.K_gauss = k
                break
            except GmError as e:
                if e.status != GM_ERR_CAPACITY or attempt:
                    raise
                self._alloc_g(self._grow(int(self.g_counters[GM_CNT_K].item())))
        md, mc = (self.depth_aa, self.rgb_aa) if self.antialias else (self.mesh_depth, self.mesh_rgb)
        gm_composite_hybrid_fwd(cam, opts, self.g_range, self.gids, self.splats, md, mc,
                                self.face_id, self.out_rgb, self.out_depth, self.out_alpha, self.T_final,
                                self.n_contrib, depth_model=self.depth_model, aa=self.aa, staged=self.staged)
        return self.out_rgb, self.out_depth, self.out_alpha

    def _ensure_mesh_grads(self):
        if not hasattr(self, "v_verts") or self.v_verts.shape != self.V.shape:
            self.v_verts = torch.zeros_like(self.V)
            self.v_vcol = torch.zeros_like(self.vcol)

    def backward(self, g_rgb, g_depth, g_alpha, mesh_grads: bool = True):
        cam, opts = self.cam, self.opts
        main = torch.cuda.current_stream(self.dev)
        if self.antialias:
            # Gaussians and the layer, then the layer to the interpolated colour / depth and
            # the silhouettes, then the interpolation: one stream
            self.v_splats.zero_()
            if self.soft:
                self.v_depth_model.zero_()
            gm_composite_hybrid_bwd(cam, opts, self.g_range, self.gids, self.splats, self.depth_aa, self.rgb_aa,
                                    self.face_id, self.T_final, self.n_contrib, g_rgb, g_depth, g_alpha,
                                    self.v_splats, depth_model=self.depth_model, v_depth_model=self.v_depth_model,
                                    v_mesh_depth=self.v_mesh_depth, aa=self.aa, staged=self.staged)
            if not mesh_grads:
                return self.v_splats, None, None
            self._ensure_mesh_grads()
            self.v_verts.zero_()
            self.v_vcol.zero_()
            gm_antialias_bwd(cam, self.V, self.F, self.adj, self.face_id, self.mesh_depth, self.mesh_rgb, self.cov,
                             self.depth_aa, self.v_cov, self.v_rgb_aa, self.v_mesh_depth, self.v_mesh_rgb,
                             self.v_interp_depth, self.v_verts)
            gm_interp_mesh_bwd(cam, self.V, self.F, self.vcol, self.face_id, self.v_mesh_rgb, self.v_interp_depth,
                               self.v_verts, self.v_vcol)
            return self.v_splats, self.v_verts, self.v_vcol
        if self.soft:
            # the mesh part reads dL/dD that the Gaussian part writes: one call, one stream
            if mesh_grads:
                if not hasattr(self, "v_verts") or self.v_verts.shape != self.V.shape:
                    self.v_verts = torch.zeros_like(self.V)
                    self.v_vcol = torch.zeros_like(self.vcol)
                self.v_verts.zero_()
                self.v_vcol.zero_()
            self.v_splats.zero_()
            self.v_depth_model.zero_()
            mesh = (self.V, self.F, self.vcol, self.v_verts, self.v_vcol) if mesh_grads else (None,) * 5
            gm_composite_hybrid_bwd(cam, opts, self.g_range, self.gids, self.splats, self.mesh_depth, self.mesh_rgb,
                                    self.face_id, self.T_final, self.n_contrib, g_rgb, g_depth, g_alpha,
                                    self.v_splats, *mesh, depth_model=self.depth_model,
                                    v_depth_model=self.v_depth_model, v_mesh_depth=self.v_mesh_depth,
                                    staged=self.staged)
            return (self.v_splats,) + ((self.v_verts, self.v_vcol) if mesh_grads else (None, None))
        if mesh_grads:
            if not hasattr(self, "v_verts") or self.v_verts.shape != self.V.shape:
                self.v_verts = torch.zeros_like(self.V)
                self.v_vcol = torch.zeros_like(self.vcol)
            side = self._side_stream() if self.concurrent else main
            if self.concurrent:
                side.wait_stream(main)
            with torch.cuda.stream(side):
                self.v_verts.zero_()
                self.v_vcol.zero_()
                gm_composite_hybrid_bwd(cam, opts, self.g_range, self.gids, self.splats, self.mesh_depth,
                                        self.mesh_rgb, self.face_id, self.T_final, self.n_contrib, g_rgb, g_depth,
                                        g_alpha, None, self.V, self.F, self.vcol, self.v_verts, self.v_vcol)
        self.v_splats.zero_()
        gm_composite_hybrid_bwd(cam, opts, self.g_range, self.gids, self.splats, self.mesh_depth, self.mesh_rgb,
                                self.face_id, self.T_final, self.n_contrib, g_rgb, g_depth, g_alpha, self.v_splats,
                                staged=self.staged)
        if mesh_grads and self.concurrent:
            main.wait_stream(side)
        if mesh_grads:
            return self.v_splats, self.v_verts, self.v_vcol
        return self.v_splats, None, None

    def capture_step(self, g_rgb, g_depth, g_alpha, mesh_grads: bool = True):
        """Records one forward + backward pass (the seven calls, no host
        synchronisation) into a CUDA graph and returns it; ``graph.replay()``
        then re-runs the step on the current inputs.  Call after a sizing
        ``forward(sync=True)`` so the capacities fit, and check
        ``overflowed()`` after replays."""
        if not hasattr(self, "v_verts"):
            self.backward(g_rgb, g_depth, g_alpha, mesh_grads)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm the capture stream once
            self.forward(sync=False)
            self.backward(g_rgb, g_depth, g_alpha, mesh_grads)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.forward(sync=False)
            self.backward(g_rgb, g_depth, g_alpha, mesh_grads)
        return graph

    def overflowed(self) -> bool:
        f = int(self.tri_counters[GM_CNT_FLAGS].item()) | int(self.g_counters[GM_CNT_FLAGS].item())
        return bool(f & (GM_FLAG_OVERFLOW | GM_FLAG_TIMEOUT))


class MultiViewRenderer:
    """Several cameras of one scene rendered and differentiated as one batch.

    The projection and its backward run once for all views
    (``gm_project_gaussians_views`` / ``_bwd_views``); each view's binning,
    z-buffer, interpolation and compositing run on one of ``streams`` CUDA
    streams, so the views overlap on the GPU.  ``backward`` sums the Gaussian
    parameter gradients over the views (in view order) and accumulates the
    mesh gradients of all views; ``capture_step`` records the whole batch as
    one CUDA graph.  Per-view buffers are those of one ``HybridRenderer`` per
    camera (``views[k]``), whose ``splats`` / ``radii`` / ``v_splats`` are
    slices of the batch arrays.
    """

    def __init__(self, cams, bg=(1.0, 1.0, 1.0), cull_occluded=True, device="cuda", tile_test=True, streams=4,
                 softness=0.0, soft_split=GM_SPLIT_PHI, antialias=False, zbuffer="direct", staged=True):
        self.views = [HybridRenderer(c, bg=bg, cull_occluded=cull_occluded, device=device, concurrent=False,
                                     tile_test=tile_test, softness=softness, soft_split=soft_split,
                                     antialias=antialias, zbuffer=zbuffer, staged=staged) for c in cams]
        self.antialias = bool(antialias)
        self.soft = self.views[0].soft
        self.V = len(self.views)
        self.dev = torch.device(device)
        self.n_streams = max(1, min(int(streams), self.V))
        self._streams = None

    @property
    def cams(self):
        return [v.cam for v in self.views]

    @property
    def opts(self) -> gm_opts:
        return self.views[0].opts

    def _pool(self):
        if self._streams is None:
            self._streams = [torch.cuda.Stream(device=self.dev) for _ in range(self.n_streams)]
        return self._streams

    def upload(self, mesh, gaussians):
        """Copies the scene once; sizes every view's tile-entry buffers with one
        synchronous forward pass per view."""
        v0 = self.views[0]
        v0.upload(mesh, gaussians)
        N, d = v0.N, self.dev
        self.N = N
        self.splats = torch.zeros(self.V, N, SPLAT_STRIDE, dtype=F32, device=d)
        self.radii = torch.zeros(self.V, N, dtype=I32, device=d)
        self.tiles_touched = torch.zeros(self.V, N, dtype=I32, device=d)
        self.v_splats = torch.zeros(self.V, N, SPLAT_STRIDE, dtype=F32, device=d)
        self.depth_model = torch.zeros(self.V, N, 4, dtype=F32, device=d) if self.soft else None
        self.v_depth_model = torch.zeros(self.V, N, 4, dtype=F32, device=d) if self.soft else None
        for k, r in enumerate(self.views):
            if k:
                for name in ("V", "F", "vcol", "means", "log_scales", "quats", "logits", "colors", "sh_degree"):
                    setattr(r, name, getattr(v0, name))
                if self.antialias:
                    r.adj = v0.adj
                r.N = N
                r._alloc_g(max(r.g_cap, 1))
                r._alloc_mesh_ws()
            r.splats, r.radii, r.tiles_touched = self.splats[k], self.radii[k], self.tiles_touched[k]
            r.v_splats = self.v_splats[k]
            if self.soft:
                r.depth_model, r.v_depth_model = self.depth_model[k], self.v_depth_model[k]
            r.forward(sync=True)
        self.v_verts = torch.zeros_like(v0.V)
        self.v_vcol = torch.zeros_like(v0.vcol)
        self.v_means = torch.zeros_like(v0.means)
        self.v_log_scales = torch.zeros_like(v0.log_scales)
        self.v_quats = torch.zeros_like(v0.quats)
        self.v_logits = torch.zeros_like(v0.logits)
        self.v_colors = torch.zeros_like(v0.colors)
        torch.cuda.synchronize(self.dev)

    def forward(self):
        """All views' (rgb, depth, alpha), without host synchronisation (check
        ``overflowed()``)."""
        main = torch.cuda.current_stream(self.dev)
        pool = self._pool()
        start = torch.cuda.Event()
        start.record(main)
        v0 = self.views[0]
        gm_project_gaussians_views(self.cams, self.opts, v0.means, v0.log_scales, v0.quats, v0.logits, v0.colors,
                                   self.splats, self.radii, self.tiles_touched, self.depth_model)
        projected = torch.cuda.Event()
        projected.record(main)
        for k, r in enumerate(self.views):
            s = pool[k % len(pool)]
            s.wait_event(start)
            with torch.cuda.stream(s):
                cam, opts = r.cam, r.opts
                r._zbuffer(sync=False)
                gm_interp_mesh(cam, r.V, r.F, r.vcol, r.face_id, r.mesh_depth, r.mesh_rgb, r.tile_far, r.tile_full)
                if r.antialias:
                    gm_antialias(cam, r.V, r.F, r.adj, r.face_id, r.mesh_depth, r.mesh_rgb, r.cov, r.rgb_aa,
                                 r.depth_aa, r.tile_far, r.tile_full)
                s.wait_event(projected)
                gm_bin_sort_gaussians(cam, opts, r.splats, r.radii, r.tile_far, r.tile_full, r.keys, r.gids,
                                      r.g_range, r.g_cap, r.g_counters, r.g_ws, sync=False)
                md, mc = (r.depth_aa, r.rgb_aa) if r.antialias else (r.mesh_depth, r.mesh_rgb)
                gm_composite_hybrid_fwd(cam, opts, r.g_range, r.gids, r.splats, md, mc, r.face_id,
                                        r.out_rgb, r.out_depth, r.out_alpha, r.T_final, r.n_contrib,
                                        depth_model=r.depth_model, aa=r.aa, staged=r.staged)
        for s in pool:
            main.wait_stream(s)
        return [(r.out_rgb, r.out_depth, r.out_alpha) for r in self.views]

    def backward(self, grads):
        """grads: per view (g_rgb, g_depth, g_alpha).  Returns the gradients of
        (means, log_scales, quats, logits, colors) summed over the views and of
        (vertex positions, vertex colours) accumulated over the views."""
        main = torch.cuda.current_stream(self.dev)
        pool = self._pool()
        self.v_splats.zero_()
        if self.soft:
            self.v_depth_model.zero_()
        self.v_verts.zero_()
        self.v_vcol.zero_()
        start = torch.cuda.Event()
        start.record(main)
        for k, (r, (g_rgb, g_depth, g_alpha)) in enumerate(zip(self.views, grads)):
            s = pool[k % len(pool)]
            s.wait_event(start)
            with torch.cuda.stream(s):
                if r.antialias:
                    gm_composite_hybrid_bwd(r.cam, r.opts, r.g_range, r.gids, r.splats, r.depth_aa, r.rgb_aa,
                                            r.face_id, r.T_final, r.n_contrib, g_rgb, g_depth, g_alpha, r.v_splats,
                                            depth_model=r.depth_model, v_depth_model=r.v_depth_model,
                                            v_mesh_depth=r.v_mesh_depth, aa=r.aa, staged=r.staged)
                    gm_antialias_bwd(r.cam, r.V, r.F, r.adj, r.face_id, r.mesh_depth, r.mesh_rgb, r.cov,
                                     r.depth_aa, r.v_cov, r.v_rgb_aa, r.v_mesh_depth, r.v_mesh_rgb, r.v_interp_depth,
                                     self.v_verts)
                    gm_interp_mesh_bwd(r.cam, r.V, r.F, r.vcol, r.face_id, r.v_mesh_rgb, r.v_interp_depth,
                                       self.v_verts, self.v_vcol)
                    continue
                gm_composite_hybrid_bwd(r.cam, r.opts, r.g_range, r.gids, r.splats, r.mesh_depth, r.mesh_rgb,
                                        r.face_id, r.T_final, r.n_contrib, g_rgb, g_depth, g_alpha, r.v_splats,
                                        r.V, r.F, r.vcol, self.v_verts, self.v_vcol, depth_model=r.depth_model,
                                        v_depth_model=r.v_depth_model, v_mesh_depth=r.v_mesh_depth,
                                        staged=r.staged)
        for s in pool:
            main.wait_stream(s)
        v0 = self.views[0]
        gm_project_gaussians_bwd_views(self.cams, self.opts, v0.means, v0.log_scales, v0.quats, v0.logits, v0.colors,
                                       self.radii, self.v_splats, self.v_means, self.v_log_scales, self.v_quats,
                                       self.v_logits, self.v_colors, v_depth_model=self.v_depth_model)
        return (self.v_means, self.v_log_scales, self.v_quats, self.v_logits, self.v_colors, self.v_verts,
                self.v_vcol)

    def capture_step(self, grads):
        """Records forward + backward of all views into one CUDA graph."""
        side = torch.cuda.Stream(device=self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(side):  # warm the capture stream once
            self.forward()
            self.backward(grads)
        torch.cuda.current_stream(self.dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.forward()
            self.backward(grads)
        return graph

    def overflowed(self) -> bool:
        return any(r.overflowed() for r in self.views)


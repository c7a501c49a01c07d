"""The C ABI library loads and exports every function include/gm.h declares;
argument checks answer GM_ERR_INVALID_ARG before any CUDA work (no GPU
needed: these calls return before touching the device)."""

import ctypes as C

import pytest

import differentiable_hybrid_mesh_tile_b300 as gm
from differentiable_hybrid_mesh_tile_b300 import build as gm_build


@pytest.fixture(scope="module")
def lib():
    gm_build.build()
    return gm.lib()


def test_exports_every_declared_function(lib):
    names = gm.header_functions()
    assert len(names) >= 10
    for n in ["gm_bin_triangles", "gm_zbuffer", "gm_interp_mesh", "gm_project_gaussians",
              "gm_bin_sort_gaussians", "gm_composite_hybrid_fwd", "gm_composite_hybrid_bwd", "gm_last_error"]:
        assert n in names
    raw = C.CDLL(gm.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_workspace_queries_are_host_only(lib):
    a = gm.gm_bin_triangles_workspace_size(1000, 5000, 64, 64)
    b = gm.gm_bin_triangles_workspace_size(1000, 50000, 64, 64)
    assert 0 < a < b
    c = gm.gm_bin_sort_gaussians_workspace_size(100000, 400000, 512, 512)
    assert c > 400000 * 12


def _cam(**kw):
    c = gm.gm_camera()
    c.width, c.height, c.fx, c.fy, c.cx, c.cy = 64, 48, 50.0, 50.0, 32.0, 24.0
    c.near_plane, c.far_plane = 0.01, 100.0
    for k in range(9):
        c.R[k] = 1.0 if k in (0, 4, 8) else 0.0
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("bad", [dict(width=0), dict(fx=-1.0), dict(near_plane=0.0), dict(far_plane=0.001),
                                 dict(fy=float("nan"))])
def test_bad_camera_rejected(lib, bad):
    cam = _cam(**bad)
    st = lib.gm_zbuffer(C.byref(cam), None, 0, None, 0, C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), None)
    assert st == gm.GM_ERR_INVALID_ARG
    assert len(lib.gm_last_error()) > 0


def test_null_and_size_checks(lib):
    cam = _cam()
    opts = gm.make_opts()
    # NULL camera
    assert lib.gm_interp_mesh(None, None, 0, None, 0, None, None, None, None, None, None, None) == gm.GM_ERR_INVALID_ARG
    # negative N
    st = lib.gm_project_gaussians(C.byref(cam), C.byref(opts), -1, *([None] * 10))
    assert st == gm.GM_ERR_INVALID_ARG
    # sh degree out of range
    bad = gm.make_opts(sh_degree=4)
    st = lib.gm_project_gaussians(C.byref(cam), C.byref(bad), 0, *([None] * 10))
    assert st == gm.GM_ERR_INVALID_ARG and b"sh_degree" in lib.gm_last_error()
    # misaligned splats
    st = lib.gm_project_gaussians(C.byref(cam), C.byref(opts), 4, *([C.c_void_p(256)] * 5), C.c_void_p(260),
                                  C.c_void_p(256), C.c_void_p(256), None, None)
    assert st == gm.GM_ERR_INVALID_ARG
    # workspace too small
    st = lib.gm_bin_sort_gaussians(C.byref(cam), C.byref(opts), 10, C.c_void_p(256), C.c_void_p(256),
                                   C.c_void_p(256), C.c_void_p(256), C.c_void_p(256), C.c_void_p(256),
                                   C.c_void_p(256), 100, C.c_void_p(256), None, C.c_void_p(256), 10, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"workspace" in lib.gm_last_error()
    # cull without tile bounds
    st = lib.gm_bin_sort_gaussians(C.byref(cam), C.byref(opts), 10, C.c_void_p(256), C.c_void_p(256), None, None,
                                   C.c_void_p(256), C.c_void_p(256), C.c_void_p(256), 100, C.c_void_p(256), None,
                                   C.c_void_p(256), 1 << 30, None)
    assert st == gm.GM_ERR_INVALID_ARG
    # incomplete mesh-gradient arguments
    st = lib.gm_composite_hybrid_bwd(C.byref(cam), C.byref(opts), 4, *([C.c_void_p(256)] * 13), None, None,
                                     None, 3, None, 1, None, C.c_void_p(256), None, None, None, None, None)
    assert st == gm.GM_ERR_INVALID_ARG
    # soft split: negative softness; Gaussian gradients without the depth model or its gradient;
    # mesh gradients without dL/d mesh depth
    neg = gm.make_opts(softness=-1.0)
    st = lib.gm_composite_hybrid_fwd(C.byref(cam), C.byref(neg), 4, *([C.c_void_p(256)] * 12), None, None, None,
                                     None)
    assert st == gm.GM_ERR_INVALID_ARG and b"softness" in lib.gm_last_error()
    soft = gm.make_opts(softness=1.0)
    st = lib.gm_composite_hybrid_fwd(C.byref(cam), C.byref(soft), 4, C.c_void_p(256), C.c_void_p(256),
                                     C.c_void_p(256), None, *([C.c_void_p(256)] * 8), None, None, None, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"depth_model" in lib.gm_last_error()
    st = lib.gm_composite_hybrid_bwd(C.byref(cam), C.byref(soft), 4, *([C.c_void_p(256)] * 13), None, None,
                                     None, 0, None, 0, None, None, None, None, None, None, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"depth_model" in lib.gm_last_error()
    st = lib.gm_composite_hybrid_bwd(C.byref(cam), C.byref(soft), 4, *([C.c_void_p(256)] * 12), None, None,
                                     None, C.c_void_p(256), 3, C.c_void_p(256), 1, C.c_void_p(256),
                                     C.c_void_p(256), C.c_void_p(256), None, None, None, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"v_mesh_depth" in lib.gm_last_error()
    bad_split = gm.make_opts(softness=1.0, soft_split=2)
    st = lib.gm_composite_hybrid_fwd(C.byref(cam), C.byref(bad_split), 4, *([C.c_void_p(256)] * 12), None, None,
                                     None, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"soft_split" in lib.gm_last_error()
    # antialiased layer: misaligned back buffer; mesh arguments given with the layer
    aa = gm.gm_aa_layer()
    aa.cov, aa.back, aa.T_back, aa.n_back, aa.v_cov, aa.v_rgb = 256, 264, 256, 256, 256, 256
    st = lib.gm_composite_hybrid_fwd(C.byref(cam), C.byref(opts), 4, *([C.c_void_p(256)] * 12), C.byref(aa), None,
                                     None, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"back" in lib.gm_last_error()
    aa.back = 256
    st = lib.gm_composite_hybrid_bwd(C.byref(cam), C.byref(opts), 4, *([C.c_void_p(256)] * 16), 3,
                                     C.c_void_p(256), 1, C.c_void_p(256), C.c_void_p(256), C.c_void_p(256),
                                     C.byref(aa), None, None, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"gm_antialias_bwd" in lib.gm_last_error()
    # staged records: misaligned buffer
    stg = gm.gm_staged()
    stg.recs, stg.cap = 264, 100
    st = lib.gm_composite_hybrid_fwd(C.byref(cam), C.byref(opts), 4, *([C.c_void_p(256)] * 12), None,
                                     C.byref(stg), None, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"staged" in lib.gm_last_error()
    assert gm.gm_staged_bytes(1000, 0.0) == 56000 and gm.gm_staged_bytes(1000, 1.0) == 64000
    # edge adjacency: workspace too small; antialiasing without adjacency
    st = lib.gm_mesh_edges(C.c_void_p(256), 10, 12, C.c_void_p(256), C.c_void_p(256), C.c_void_p(256), 16, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"workspace" in lib.gm_last_error()
    st = lib.gm_antialias(C.byref(cam), C.c_void_p(256), 3, C.c_void_p(256), 1, None, *([C.c_void_p(256)] * 8), None)
    assert st == gm.GM_ERR_INVALID_ARG and b"adj" in lib.gm_last_error()
    # direct z-buffer: workspace too small
    st = lib.gm_zbuffer_direct(C.byref(cam), C.c_void_p(256), 3, C.c_void_p(256), 1, C.c_void_p(256),
                               C.c_void_p(256), 64, None)
    assert st == gm.GM_ERR_INVALID_ARG and b"workspace" in lib.gm_last_error()
    assert gm.gm_zbuffer_direct_workspace_size(10, 64, 48) >= 8 * 64 * 48 + 10 * 100
    # misaligned v_depth_model in the projection backward
    st = lib.gm_project_gaussians_bwd(C.byref(cam), C.byref(opts), 4, *([C.c_void_p(256)] * 7), C.c_void_p(260),
                                      0, *([C.c_void_p(256)] * 5), None)
    assert st == gm.GM_ERR_INVALID_ARG and b"v_depth_model" in lib.gm_last_error()


def test_no_cpu_fallback_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(gm, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(gm, "_lib", None)
    with pytest.raises(ImportError):
        gm.lib()


def test_header_constants_match_binding():
    """Every GM_* integer constant the header defines has the same value in the binding."""
    import re
    text = open(gm.HEADER).read()
    found = dict((k, int(v)) for k, v in re.findall(r"^#define\s+(GM_\w+)\s+(\d+)\s*$", text, re.M))
    assert "GM_SPLIT_LOGISTIC" in found and "GM_FLAG_TIMEOUT" in found
    for name, value in found.items():
        if hasattr(gm, name):
            assert getattr(gm, name) == value, name
    # the option struct's fields in header order
    body = re.search(r"typedef struct gm_opts \{(.*?)\} gm_opts;", text, re.S).group(1)
    names = re.findall(r"^\s*(?:float|int32_t)\s+(\w+)(?:\[\d+\])?;", body, re.M)
    assert names == [f[0] for f in gm.gm_opts._fields_]


def test_renderer_rejects_unknown_zbuffer():
    """The renderers take zbuffer="direct" (no triangle lists) or "tile"; anything
    else is refused before any device memory is touched."""
    from differentiable_hybrid_mesh_tile_b300 import scenes
    cam = scenes.look_at((0, 0, 3), (0, 0, 0), 64, 48, 50, 50)
    with pytest.raises(ValueError):
        gm.HybridRenderer(cam, zbuffer="lists")

"""gm_bin_triangles_noalloc -- the triangle binning entry point for callers
that may not allocate device memory (e.g. a plugin inside a host application
that owns all device memory through its own pool) -- against the regular
gm_bin_triangles, which takes a caller-allocated workspace.

The outputs are integers (tile ranges, face ids, counts), so they must be
equal bit for bit.  Two calls in a row check that the shared static scratch
array is cleared where it must start at zero.  This file is collected last;
it passes alone in a fresh process and after the other tests."""

import numpy as np
import pytest
import torch

import differentiable_hybrid_mesh_tile_b300 as gm
from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _cases():
    tiny = scenes.tiny()
    sph = scenes.sphere512()
    ragged = scenes.look_at((0.3, 0.5, 2.6), (0, 0, 0), 101, 77, 90, 95, 47.3, 40.1)
    soup = scenes.soup1080(n_gauss=10, n_tri=100_000)
    return [("tiny", tiny.camera, tiny.mesh), ("sphere512", sph.camera, sph.mesh),
            ("ragged", ragged, tiny.mesh), ("soup_100k", soup.camera, soup.mesh)]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_noalloc_matches_workspace_path_twice(case):
    H.need_gpu()
    name, cam, mesh = case
    c = gm.make_camera(cam)
    V, F = H.dev(mesh.verts, torch.float32), H.dev(mesh.faces, torch.int32)
    T = H.n_tiles(cam)
    ref = H.run_mesh(cam, mesh)
    cap = ref["K"] + 100
    for call in range(2):
        tr = torch.full((T, 2), -3, dtype=torch.int32, device="cuda")
        ids = torch.full((cap,), -3, dtype=torch.int32, device="cuda")
        cnt = torch.full((4,), -3, dtype=torch.int32, device="cuda")
        K = gm.gm_bin_triangles_noalloc(c, V, F, tr, ids, cap, cnt)
        assert K == ref["K"], (name, call)
        np.testing.assert_array_equal(H.host(tr), ref["tile_range"])
        np.testing.assert_array_equal(H.host(ids)[:K], ref["tri_ids"])
        np.testing.assert_array_equal(H.host(cnt), ref["counters"])
        assert np.all(H.host(ids)[K:] == -3)


def test_noalloc_rejects_oversized_requests():
    H.need_gpu()
    s = scenes.tiny()
    c = gm.make_camera(s.camera)
    V, F = H.dev(s.mesh.verts, torch.float32), H.dev(s.mesh.faces, torch.int32)
    tr = torch.zeros(H.n_tiles(s.camera), 2, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(4, dtype=torch.int32, device="cuda")
    big = 50_000_000  # 50M entries of scratch cannot fit in the static array
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(gm.GmError) as e:
        gm.gm_bin_triangles_noalloc(c, V, F, tr, ids, big, cnt)
    assert e.value.status == gm.GM_ERR_INVALID_ARG and "static scratch" in str(e.value)

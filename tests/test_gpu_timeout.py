"""The bounded inter-block waits of the scans and radix sorts give up cleanly.

Failure detection without a GPU fault: with the wait limit set to 0 polls
(gm_set_wait_limit), a block whose predecessor has not yet published its
descriptor gives up at once, sets GM_FLAG_TIMEOUT in the call's counters and
carries on with a prefix that is at most the true one.  The call must then
report GM_ERR_TIMEOUT (synchronous mode) or the flag (asynchronous mode),
write nothing outside its buffers (canaries past the capacity, past the tile
ranges, past the counters and past the workspace stay intact), and leave the
context usable: with the limit restored, the same call gives the exact bins
again.  Nothing downstream reads the broken bins.

Whether a block finds an unpublished predecessor depends on how the
partitions are scheduled, so the call is repeated (up to eight times, on an
input of several hundred partitions) until a give-up has been seen."""

import numpy as np
import pytest
import torch

import differentiable_hybrid_mesh_tile_b300 as gm
from differentiable_hybrid_mesh_tile_b300 import scenes
import gpu_helpers as H

pytestmark = pytest.mark.gpu

CANARY_KEY = 0x5A5A5A5A5A5A5A5A
CANARY_ID = -77
PAD = 4096


def _inputs():
    s = scenes.soup1080(n_gauss=200_000, n_tri=10)
    cam = s.camera
    sp, rad, _ = H.run_project(cam, s.gaussians)
    return cam, sp, rad


def _bin_with_canaries(cam, sp, rad, cap, sync):
    """gm_bin_sort_gaussians (no cull, rectangle bins) into buffers that extend
    PAD elements past what the call is given, filled with canaries."""
    c = gm.make_camera(cam)
    o = gm.make_opts((1, 1, 1), False, -1, False)
    T = H.n_tiles(cam)
    keys = torch.full((cap + PAD,), CANARY_KEY, dtype=torch.int64, device="cuda")
    gids = torch.full((cap + PAD,), CANARY_ID, dtype=torch.int32, device="cuda")
    tr = torch.full((T + PAD, 2), CANARY_ID, dtype=torch.int32, device="cuda")
    cnt = torch.full((4 + PAD,), CANARY_ID, dtype=torch.int32, device="cuda")
    cnt[:4] = 0
    nb = gm.gm_bin_sort_gaussians_workspace_size(len(rad), cap, cam.width, cam.height)
    nb = (nb + 15) // 16 * 16
    ws = torch.full((nb + PAD,), 0xA5, dtype=torch.uint8, device="cuda")
    status = gm.GM_OK
    try:
        gm.gm_bin_sort_gaussians(c, o, H.dev(sp, torch.float32), H.dev(rad, torch.int32), None, None, keys[:cap],
                                 gids[:cap], tr[:T], cap, cnt[:4], ws[:nb], sync=sync)
    except gm.GmError as e:
        status = e.status
    torch.cuda.synchronize()
    k, g, r, n, w = (H.host(x) for x in (keys, gids, tr, cnt, ws))
    intact = (np.all(k[cap:].view(np.uint64) == np.uint64(CANARY_KEY)) and np.all(g[cap:] == CANARY_ID)
              and np.all(r[T:] == CANARY_ID) and np.all(n[4:] == CANARY_ID) and np.all(w[nb:] == 0xA5))
    return status, n[:4], intact, (k[:cap].view(np.uint64), g[:cap], r[:T])


def test_wait_limit_zero_times_out_inside_buffers(orc):
    H.need_gpu()
    cam, sp, rad = _inputs()
    ref = H.run_bin(cam, sp, rad, tile_test=False)
    K = ref["K"]
    cap = K + 1000
    assert K > 300 * 2048, K  # several hundred sort partitions
    assert gm.gm_get_wait_limit() == gm.GM_WAIT_LIMIT_DEFAULT
    seen_sync = seen_async = False
    try:
        gm.gm_set_wait_limit(0)
        assert gm.gm_get_wait_limit() == 0
        for attempt in range(8):
            st, cn, intact, _ = _bin_with_canaries(cam, sp, rad, cap, sync=True)
            assert intact, "a write left the buffers (synchronous call, attempt %d)" % attempt
            assert st in (gm.GM_OK, gm.GM_ERR_TIMEOUT), st
            if st == gm.GM_ERR_TIMEOUT:
                assert cn[2] & gm.GM_FLAG_TIMEOUT
                seen_sync = True
            st, cn, intact, _ = _bin_with_canaries(cam, sp, rad, cap, sync=False)
            assert intact, "a write left the buffers (asynchronous call, attempt %d)" % attempt
            assert st == gm.GM_OK  # no host read-back: the flag carries the failure
            seen_async |= bool(cn[2] & gm.GM_FLAG_TIMEOUT)
            if seen_sync and seen_async:
                break
    finally:
        gm.gm_set_wait_limit(gm.GM_WAIT_LIMIT_DEFAULT)
    print("wait limit 0: GM_ERR_TIMEOUT seen %s, GM_FLAG_TIMEOUT seen %s" % (seen_sync, seen_async))
    assert seen_sync and seen_async
    assert gm.gm_get_wait_limit() == gm.GM_WAIT_LIMIT_DEFAULT
    # the context is still usable and the restored limit gives the exact bins
    st, cn, intact, (k, g, r) = _bin_with_canaries(cam, sp, rad, cap, sync=True)
    assert st == gm.GM_OK and intact and cn[2] == 0 and cn[0] == K
    np.testing.assert_array_equal(k[:K], ref["keys"])
    np.testing.assert_array_equal(g[:K], ref["gids"])
    np.testing.assert_array_equal(r, ref["tile_range"])
    keys, gids, _ = orc.bin_gaussians(cam, sp, rad)
    np.testing.assert_array_equal(k[:K], keys)
    np.testing.assert_array_equal(g[:K], gids)

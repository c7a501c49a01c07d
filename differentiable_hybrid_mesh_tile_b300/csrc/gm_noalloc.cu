// gm_bin_triangles_noalloc: triangle binning whose scratch memory is a
// file-scope static device array instead of a caller-provided workspace.
//
// Who needs it: callers that are not allowed to allocate device memory at
// all -- for example a plugin or engine embedded in a host application that
// owns every byte of device memory through its own pool and budget, where a
// library call to cudaMalloc would either fail against that budget or stall
// the whole device while the host application is running.  Such callers can
// still pass their own input and output buffers; this entry point needs
// nothing else.
//
// Cost: every GPU that loads libgm holds kScratchBytes of device memory for
// the array until the process exits, whether or not this entry point is
// called.
#include <mutex>

#include "gm_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)GM_NOALLOC_TRI_SCRATCH_BYTES;

// Scratch of gm_bin_triangles_noalloc: scan descriptors, per-face counts and
// offsets, key buffers and radix-sort state, carved exactly as the
// caller-workspace path carves its workspace.
static __device__ __align__(256) unsigned char g_tri_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_tri_scratch on the current device.  In host code the
// symbol's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress once per device (with that device current) and
// cached.
int scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return gm::set_last_error(GM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return gm::set_last_error(GM_ERR_INVALID_ARG, "device %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_tri_scratch);
        if (e != cudaSuccess || !p)
            return gm::set_last_error(GM_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GM_OK;
}

}  // namespace

extern "C" {

int gm_bin_triangles_noalloc(const gm_camera* cam, const float* V, int32_t nV, const int32_t* F, int32_t nF,
                             int32_t* tile_range, int32_t* tri_ids, int32_t cap, int32_t* counters,
                             int32_t* K_host, void* stream)
{
    const size_t need = gm_bin_triangles_workspace_size(nF < 0 ? 0 : nF, cap < 0 ? 0 : cap, 0, 0);
    if (nF >= 0 && cap >= 0 && need > kScratchBytes)
        return gm::set_last_error(GM_ERR_INVALID_ARG,
                                  "gm_bin_triangles_noalloc: %d faces with capacity %d need %zu bytes of scratch, "
                                  "the static scratch holds %zu; use gm_bin_triangles with a workspace",
                                  nF, cap, need, kScratchBytes);
    void* ws = nullptr;
    if (int st = scratch_address(&ws)) return st;
    // Argument checks, clearing of the scratch parts that must start at zero,
    // and the launches are those of gm_bin_triangles.
    return gm_bin_triangles(cam, V, nV, F, nF, tile_range, tri_ids, cap, counters, K_host, ws, kScratchBytes,
                            stream);
}

}  // extern "C"

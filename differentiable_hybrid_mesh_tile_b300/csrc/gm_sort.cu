// Device-wide exclusive scan and stable LSD radix sort (onesweep style) used
// by the triangle and Gaussian tile binning.
//
// Scan: one pass; each block takes a partition ticket, scans it, publishes its
// aggregate and looks back over earlier partitions for its prefix (decoupled
// look-back).  Sort: one histogram pass over all digits, then one kernel per
// 8-bit digit that ranks a partition in shared memory (warp multisplit),
// gets each digit's global offset by look-back over earlier partitions and
// writes the partition out digit-run by digit-run.  Every inter-block wait is
// bounded: after wait_limit() polls (SPIN_LIMIT unless gm_set_wait_limit
// changed it; passed to each launch) the block sets GM_FLAG_TIMEOUT in the
// caller's counters and carries on, so no launch can hang.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <utility>

#include <cuda/atomic>

#include "gm_internal.cuh"
#include "gm_lookback.cuh"

namespace gm {
namespace {

__global__ void __launch_bounds__(SCAN_THREADS)
k_scan(const int32_t* __restrict__ in, const int32_t* __restrict__ idx, int32_t* __restrict__ out, int n,
       uint32_t* desc, uint32_t* ticket, int32_t* counters, uint32_t limit)
{
    __shared__ uint32_t s_warp[SCAN_THREADS / 32];
    __shared__ int s_part;
    __shared__ uint32_t s_excl;
    if (threadIdx.x == 0) s_part = (int)atomicAdd(ticket, 1u);
    __syncthreads();
    const int p = s_part;
    const int64_t base = (int64_t)p * SCAN_PART + (int64_t)threadIdx.x * SCAN_IPT;
    uint32_t v[SCAN_IPT];
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < SCAN_IPT; ++i) {
        int64_t e = base + i;
        // a gathered index outside [0, n) (possible only when the sort that
        // produced idx gave up a bounded wait) counts as zero
        const int64_t j = e < n ? (idx ? (int64_t)idx[e] : e) : -1;
        v[i] = (j >= 0 && j < n) ? (uint32_t)in[j] : 0u;
        sum += v[i];
    }
    uint32_t total;
    uint32_t ex = block_excl_scan<SCAN_THREADS>(sum, s_warp, total);
    if (threadIdx.x == 0) {
        if (p == 0) {
            st_relaxed(desc, F_PRE | (total & V_MASK));
            s_excl = 0;
        } else {
            st_relaxed(desc + p, F_AGG | (total & V_MASK));
            uint32_t e = look_back(desc, p, 1, counters, limit);
            st_relaxed(desc + p, F_PRE | ((e + total) & V_MASK));
            s_excl = e;
        }
    }
    __syncthreads();
    uint32_t run = s_excl + ex;
#pragma unroll
    for (int i = 0; i < SCAN_IPT; ++i) {
        int64_t e = base + i;
        if (e < n) out[e] = (int32_t)run;
        run += v[i];
    }
    if (p == gridDim.x - 1 && threadIdx.x == SCAN_THREADS - 1) counters[GM_CNT_K] = (int32_t)(s_excl + total);
}

// Histograms of every digit pass in one read of the keys; also clears the
// look-back descriptors of the partitions the passes will use.
__global__ void __launch_bounds__(256)
k_hist(const uint64_t* __restrict__ keys, const int32_t* __restrict__ n_dev, int cap, int begin_bit,
       int passes, uint32_t* __restrict__ hist, uint32_t* __restrict__ desc, int max_parts)
{
    __shared__ uint32_t sh[SORT_MAX_PASSES * 256];
    for (int i = threadIdx.x; i < passes * 256; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const int n = min(*n_dev, cap);
    const int nparts = (n + SORT_PART - 1) / SORT_PART;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)passes * nparts * 256; i += stride) {
        int64_t p = i / ((int64_t)nparts * 256), r = i % ((int64_t)nparts * 256);
        desc[p * max_parts * 256 + r] = 0u;
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t k = keys[i];
        for (int p = 0; p < passes; ++p)
            atomicAdd(&sh[p * 256 + (uint32_t)((k >> (begin_bit + 8 * p)) & 0xffu)], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < passes * 256; i += blockDim.x)
        if (sh[i]) atomicAdd(hist + i, sh[i]);
}

__global__ void __launch_bounds__(256) k_hist_scan(uint32_t* hist, int passes)
{
    __shared__ uint32_t s_warp[8];
    for (int p = 0; p < passes; ++p) {
        uint32_t v = hist[p * 256 + threadIdx.x];
        uint32_t total;
        uint32_t e = block_excl_scan<256>(v, s_warp, total);
        hist[p * 256 + threadIdx.x] = e;
    }
}

struct OnesweepSmem {
    uint64_t keys[SORT_PART];
    int32_t vals[SORT_PART];
    uint32_t whist[SORT_THREADS / 32][256];
    uint32_t lstart[256];
    uint32_t gofs[256];
    uint32_t s_warp[SORT_THREADS / 32];
    int part;
};

__global__ void __launch_bounds__(SORT_THREADS, 4)
k_onesweep(const uint64_t* __restrict__ kin, const int32_t* __restrict__ vin, uint64_t* __restrict__ kout,
           int32_t* __restrict__ vout, const int32_t* __restrict__ n_dev, int32_t* counters, int cap, int shift,
           const uint32_t* __restrict__ digit_start, uint32_t* desc, uint32_t* ticket, uint32_t limit)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    OnesweepSmem& S = *reinterpret_cast<OnesweepSmem*>(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = min(*n_dev, cap);
    const int nparts = (n + SORT_PART - 1) / SORT_PART;
    const uint32_t lt_mask = (1u << lane) - 1u;

    for (;;) {
        if (threadIdx.x == 0) S.part = (int)atomicAdd(ticket, 1u);
        for (int i = threadIdx.x; i < (SORT_THREADS / 32) * 256; i += SORT_THREADS) (&S.whist[0][0])[i] = 0;
        __syncthreads();
        const int p = S.part;
        if (p >= nparts) break;
        const int64_t pbase = (int64_t)p * SORT_PART;
        const int n_valid = (int)min((int64_t)SORT_PART, (int64_t)n - pbase);
        const int64_t wbase = pbase + (int64_t)warp * (32 * SORT_IPT);

        uint64_t key[SORT_IPT];
        int32_t val[SORT_IPT];
        uint32_t rank[SORT_IPT];  // digit << 16 | offset within the warp's run of that digit
#pragma unroll
        for (int i = 0; i < SORT_IPT; ++i) {
            int64_t idx = wbase + i * 32 + lane;
            bool ok = idx < n;
            key[i] = ok ? kin[idx] : ~0ull;
            val[i] = ok ? vin[idx] : 0;
        }
        // warp multisplit, in item order i * 32 + lane (stable)
#pragma unroll
        for (int i = 0; i < SORT_IPT; ++i) {
            uint32_t d = (uint32_t)(key[i] >> shift) & 0xffu;
            if (key[i] == ~0ull) d = 0xffu;
            // lanes holding the same digit: eight ballots, one per digit bit
            // (cheaper here than match.any, which queues on a narrow pipe)
            uint32_t peers = 0xffffffffu;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const uint32_t bit = (d >> b) & 1u;
                const uint32_t bal = __ballot_sync(0xffffffffu, bit);
                peers &= bit ? bal : ~bal;
            }
            uint32_t before = S.whist[warp][d];
            __syncwarp();
            if (lane == 31 - __clz(peers)) S.whist[warp][d] = before + __popc(peers);
            __syncwarp();
            rank[i] = (d << 16) | (before + __popc(peers & lt_mask));
        }
        __syncthreads();
        // per digit: warp offsets, partition count, look-back for the global offset
        {
            const int d = threadIdx.x;
            uint32_t run = 0;
#pragma unroll
            for (int w = 0; w < SORT_THREADS / 32; ++w) {
                uint32_t c = S.whist[w][d];
                S.whist[w][d] = run;
                run += c;
            }
            uint32_t count = run;
            if (d == 255) count -= (uint32_t)(SORT_PART - n_valid);  // padding items sort last
            uint32_t* slot = desc + (int64_t)p * 256 + d;
            uint32_t excl = 0;
            if (p == 0) {
                st_relaxed(slot, F_PRE | count);
            } else {
                st_relaxed(slot, F_AGG | count);
                excl = look_back(desc + d, p, 256, counters, limit);
                st_relaxed(slot, F_PRE | ((excl + count) & V_MASK));
            }
            S.gofs[d] = digit_start[d] + excl;
            uint32_t tot;
            S.lstart[d] = block_excl_scan<SORT_THREADS>(run, S.s_warp, tot);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < SORT_IPT; ++i) {
            uint32_t d = rank[i] >> 16;
            uint32_t pos = S.lstart[d] + S.whist[warp][d] + (rank[i] & 0xffffu);
            S.keys[pos] = key[i];
            S.vals[pos] = val[i];
        }
        __syncthreads();
        for (int pos = threadIdx.x; pos < n_valid; pos += SORT_THREADS) {
            uint64_t k = S.keys[pos];
            uint32_t d = (uint32_t)(k >> shift) & 0xffu;
            uint32_t g = S.gofs[d] + ((uint32_t)pos - S.lstart[d]);
            if (g < (uint32_t)n) {  // always true unless a bounded wait gave up
                kout[g] = k;
                vout[g] = S.vals[pos];
            }
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256)
k_tile_ranges(const uint64_t* __restrict__ keys, const int32_t* __restrict__ counters, int cap, int n_tiles,
              int2* __restrict__ range)
{
    const int n = min(counters[GM_CNT_K], cap);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        uint32_t t = (uint32_t)(keys[i] >> 32);
        if (t >= (uint32_t)n_tiles) continue;
        if (i == 0 || (uint32_t)(keys[i - 1] >> 32) != t) range[t].x = (int)i;
        if (i == n - 1 || (uint32_t)(keys[i + 1] >> 32) != t) range[t].y = (int)(i + 1);
    }
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

namespace {

// Per-device state of the host side: SM count and whether k_onesweep's
// dynamic shared-memory limit has been raised (a function attribute is set per
// device).  Guarded by one mutex: host threads may call from several devices.
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {};
bool g_onesweep_attr[kMaxDevices] = {};
std::mutex g_dev_mu;

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// raises k_onesweep's dynamic shared-memory limit on the current device once
cudaError_t onesweep_attr()
{
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (g_onesweep_attr[dev]) return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(k_onesweep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(OnesweepSmem));
    if (e == cudaSuccess) g_onesweep_attr[dev] = true;
    return e;
}

}  // namespace

int num_sms()
{
    const int dev = current_device();
    if (dev < 0) return 148;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (g_sms[dev] <= 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
        g_sms[dev] = sms;
    }
    return g_sms[dev];
}

namespace {
std::atomic<uint32_t> g_wait_limit{SPIN_LIMIT};
}  // namespace

void set_wait_limit(uint32_t polls) { g_wait_limit.store(polls); }

uint32_t wait_limit() { return g_wait_limit.load(); }

static int scan_parts(int64_t n) { return (int)((n + SCAN_PART - 1) / SCAN_PART); }
static int sort_parts(int64_t cap) { return (int)((cap + SORT_PART - 1) / SORT_PART); }

size_t scan_ws_bytes(int64_t n) { return align256(sizeof(uint32_t) * (scan_parts(n) + 1)) + 256; }

size_t carve_scan_ws(void* base, int64_t n, ScanWs& ws)
{
    uint8_t* b = (uint8_t*)base;
    ws.parts = scan_parts(n);
    ws.ticket = (uint32_t*)b;
    ws.desc = (uint32_t*)(b + 256);
    return scan_ws_bytes(n);
}

size_t scan_zero_bytes(const ScanWs& ws) { return 256 + sizeof(uint32_t) * (size_t)ws.parts; }

size_t sort_ws_bytes(int64_t cap)
{
    int64_t c = cap > 0 ? cap : 1;
    return align256(sizeof(uint32_t) * SORT_MAX_PASSES * 256) + align256(sizeof(uint32_t) * SORT_MAX_PASSES) +
           align256(sizeof(uint32_t) * (size_t)SORT_MAX_PASSES * sort_parts(c) * 256) +
           align256(sizeof(uint64_t) * c) + align256(sizeof(int32_t) * c);
}

size_t carve_sort_ws(void* base, int64_t cap, SortWs& ws)
{
    int64_t c = cap > 0 ? cap : 1;
    uint8_t* b = (uint8_t*)base;
    ws.max_parts = sort_parts(c);
    ws.hist = (uint32_t*)b;
    b += align256(sizeof(uint32_t) * SORT_MAX_PASSES * 256);
    ws.tickets = (uint32_t*)b;
    b += align256(sizeof(uint32_t) * SORT_MAX_PASSES);
    ws.desc = (uint32_t*)b;
    b += align256(sizeof(uint32_t) * (size_t)SORT_MAX_PASSES * ws.max_parts * 256);
    ws.keys_alt = (uint64_t*)b;
    b += align256(sizeof(uint64_t) * c);
    ws.vals_alt = (int32_t*)b;
    return sort_ws_bytes(cap);
}

cudaError_t exclusive_scan(const int32_t* counts, const int32_t* idx, int32_t* offsets, int n, int32_t* counters,
                           const ScanWs& ws, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(ws.ticket, 0, scan_zero_bytes(ws), s);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaMemsetAsync(counters + GM_CNT_K, 0, sizeof(int32_t), s);
    k_scan<<<scan_parts(n), SCAN_THREADS, 0, s>>>(counts, idx, offsets, n, ws.desc, ws.ticket, counters,
                                                  wait_limit());
    return cudaGetLastError();
}

int sort_passes(int begin_bit, int end_bit)
{
    return end_bit > begin_bit ? (end_bit - begin_bit + 7) / 8 : 0;
}

cudaError_t clear_sort_hist(const SortWs& ws, cudaStream_t s)
{
    return cudaMemsetAsync(ws.hist, 0, (uint8_t*)ws.desc - (uint8_t*)ws.hist, s);  // histograms and tickets
}

cudaError_t radix_sort(uint64_t* k0, int32_t* v0, uint64_t* k1, int32_t* v1, int cap, int begin_bit, int end_bit,
                       const int32_t* n_dev, int32_t* counters, const SortWs& ws, cudaStream_t s, bool have_hist)
{
    const int passes = sort_passes(begin_bit, end_bit);
    if (passes == 0 || cap <= 0) return cudaSuccess;
    if (passes > SORT_MAX_PASSES) return cudaErrorInvalidValue;
    cudaError_t e = cudaSuccess;
    const int sms = num_sms();
    if (!have_hist) {
        if ((e = clear_sort_hist(ws, s)) != cudaSuccess) return e;
        int hgrid = (int)std::min<int64_t>(((int64_t)cap + 255) / 256, (int64_t)sms * 4);
        k_hist<<<hgrid, 256, 0, s>>>(k0, n_dev, cap, begin_bit, passes, ws.hist, ws.desc, ws.max_parts);
    }
    k_hist_scan<<<1, 256, 0, s>>>(ws.hist, passes);
    e = onesweep_attr();
    if (e != cudaSuccess) return e;
    const int grid = std::min(ws.max_parts, sms * 4);
    uint64_t* kin = k0; int32_t* vin = v0;
    uint64_t* kout = k1; int32_t* vout = v1;
    for (int p = 0; p < passes; ++p) {
        k_onesweep<<<grid, SORT_THREADS, sizeof(OnesweepSmem), s>>>(
            kin, vin, kout, vout, n_dev, counters, cap, begin_bit + 8 * p, ws.hist + p * 256,
            ws.desc + (size_t)p * ws.max_parts * 256, ws.tickets + p, wait_limit());
        std::swap(kin, kout);
        std::swap(vin, vout);
    }
    return cudaGetLastError();
}

cudaError_t tile_ranges(const uint64_t* keys, int cap, const int32_t* counters, int32_t* tile_range, int n_tiles,
                        cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(tile_range, 0, sizeof(int32_t) * 2 * (size_t)n_tiles, s);
    if (e != cudaSuccess || cap <= 0) return e;
    int grid = (int)std::min<int64_t>(((int64_t)cap + 255) / 256, (int64_t)num_sms() * 8);
    k_tile_ranges<<<grid, 256, 0, s>>>(keys, counters, cap, n_tiles, reinterpret_cast<int2*>(tile_range));
    return cudaGetLastError();
}

}  // namespace gm

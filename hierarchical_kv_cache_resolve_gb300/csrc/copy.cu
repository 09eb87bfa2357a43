// Copy-only kernels.
//
// prefetch_copy_kernel: the copy half of exact layer-wise prefetch
// ("Inference Systems Infrastructure Notes (6): HiSparse", section 4 "Exact
// Layer-Wise Prefetching"): replays a plan -- (position, slot) pairs of each
// request -- by copying host records into the planned slots, touching no
// metadata.  Grid (X, n_req): blockIdx.y picks the plan entry, the X CTAs of
// a row split its 16-byte chunks.
//
// gather_probe_kernel: the scattered-record GPU-load microbenchmark used to
// measure the host link with the same access pattern as the miss fetch.
#include "hs.h"
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kUnroll = 8;

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kThreads)
    prefetch_copy_kernel(DevPool p, int layer, int n_req, int k, const uint8_t *__restrict__ plan,
                         int plan_layer) {
    const int i = blockIdx.y;
    const PlanHeader *ph = reinterpret_cast<const PlanHeader *>(plan);
    const int32_t *eh = reinterpret_cast<const int32_t *>(plan + 16 + (size_t)i * plan_entry_bytes(k));
    const int m = eh[0], r = eh[1];
    const bool ok = ph->magic == kPlanMagic && ph->n_req == n_req && ph->k == k &&
                    (ph->layer == layer || ph->layer == plan_layer) && m >= 0 && m <= k &&
                    r >= 0 && r < p.R;
    if (!ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status, HS_STATUS_PLAN);
        return;
    }
    const int32_t *ppos = eh + 4;
    const int32_t *pslot = ppos + k;
    const int W = p.W, B = p.B, CW = W >> 4;
    const uint8_t *host_pair = p.host + host_region(r, layer, p.R, p.L, W);
    uint8_t *cache_pair = p.cache + ((int64_t)layer * p.R + r) * B * (int64_t)W;

    if (blockIdx.x == 0) {
        // count what is copied (valid pairs) once per entry
        __shared__ unsigned int nvalid;
        if (threadIdx.x == 0) nvalid = 0;
        __syncthreads();
        unsigned int c = 0;
        for (int j = threadIdx.x; j < m; j += kThreads) {
            const int32_t pos = ppos[j], s = pslot[j];
            c += (pos >= 0 && (int64_t)pos < p.L && s >= 0 && s < B) ? 1u : 0u;
        }
        atomicAdd(&nvalid, c);
        __syncthreads();
        if (threadIdx.x == 0) {
            atomicAdd(&p.counters[(int64_t)layer * CTR_COUNT + CTR_PREFETCHED],
                      (unsigned long long)nvalid * (unsigned long long)W);
            if (nvalid != (unsigned)m) atomicOr(p.status, HS_STATUS_PLAN);
        }
    }

    const int Q = m * CW;
    const int G = gridDim.x * kThreads;
    for (int q0 = blockIdx.x * kThreads + threadIdx.x; q0 < Q; q0 += G * kUnroll) {
        uint4 v[kUnroll];
        int64_t doff[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int q = q0 + u * G;
            doff[u] = -1;
            if (q < Q) {
                const int j = q / CW;
                const int part = q - j * CW;
                const int32_t pos = ppos[j], s = pslot[j];
                if (pos >= 0 && (int64_t)pos < p.L && s >= 0 && s < B) {
                    v[u] = ld_nc_v4(host_pair + (int64_t)pos * W + part * 16);
                    doff[u] = (int64_t)s * W + part * 16;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (doff[u] >= 0) *reinterpret_cast<uint4 *>(cache_pair + doff[u]) = v[u];
    }
}

// Reads every byte of [p, p + bytes) once from the device (16-byte loads;
// `bytes` a multiple of 16, p 16-byte aligned).  The words are folded into
// a value that is stored to `sink` only if it equals a constant, so that no
// compiler stage may drop the reads as dead; `sink` is a word no one else
// reads.
__global__ void touch_kernel(const uint8_t *__restrict__ p, size_t bytes, uint32_t *sink) {
    const size_t n = bytes / 16;
    uint32_t acc = 0;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const uint4 v = ld_nc_v4(p + i * 16);
        acc = acc * 31u + (v.x ^ v.y ^ v.z ^ v.w);
    }
    if (acc == 0x9E3779B9u) *sink = acc;
}

__global__ void init_lru_kernel(uint16_t *lru, int64_t n, int B) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x)
        lru[e] = (uint16_t)(e % B);
}

__global__ void __launch_bounds__(kThreads)
    gather_probe_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                        const int32_t *__restrict__ idx, int64_t n_rec, int W) {
    const int64_t CW = W >> 4;
    const int64_t Q = n_rec * CW;
    const int64_t G = (int64_t)gridDim.x * kThreads;
    for (int64_t q0 = blockIdx.x * (int64_t)kThreads + threadIdx.x; q0 < Q; q0 += G * kUnroll) {
        uint4 v[kUnroll];
        int64_t doff[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t q = q0 + u * G;
            doff[u] = -1;
            if (q < Q) {
                const int64_t j = q / CW;
                const int64_t part = q - j * CW;
                v[u] = ld_nc_v4(src + (int64_t)idx[j] * W + part * 16);
                doff[u] = j * W + part * 16;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (doff[u] >= 0) *reinterpret_cast<uint4 *>(dst + doff[u]) = v[u];
    }
}

}  // namespace

// Dynamic shared memory a confined copy asks for (unused by the kernel):
// more than half of an SM's, so that no two of its CTAs share an SM.
constexpr int kConfinedSmem = 120 * 1024;

cudaError_t prepare_copy_kernel() {
    return cudaFuncSetAttribute(prefetch_copy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kConfinedSmem);
}

cudaError_t launch_prefetch_copy(const DevPool &p, int layer, int n_req, int k, const void *plan,
                                 int sm_count, cudaStream_t st, int plan_layer, bool confined) {
    // about two CTAs per SM in total, at least one per request row; or,
    // confined, one CTA per SM and every SM on one request's records
    int x = confined ? sm_count / n_req : (2 * sm_count + n_req - 1) / n_req;
    const int max_x = (k * (p.W >> 4) + kThreads - 1) / kThreads;
    if (x > max_x) x = max_x;
    if (x < 1) x = 1;
    prefetch_copy_kernel<<<dim3(x, n_req), kThreads, confined ? kConfinedSmem : 0, st>>>(
        p, layer, n_req, k, static_cast<const uint8_t *>(plan), plan_layer);
    return cudaGetLastError();
}

cudaError_t launch_touch(const void *p, size_t bytes, uint32_t *sink, int sm_count,
                         cudaStream_t st) {
    if (bytes < 16) return cudaSuccess;
    touch_kernel<<<(sm_count > 0 ? sm_count : 1) * 4, kThreads, 0, st>>>(
        static_cast<const uint8_t *>(p), bytes, sink);
    return cudaGetLastError();
}

cudaError_t launch_init_lru(uint16_t *lru, int64_t pairs, int B, cudaStream_t st) {
    const int64_t n = pairs * B;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    init_lru_kernel<<<blocks, 256, 0, st>>>(lru, n, B);
    return cudaGetLastError();
}

cudaError_t launch_gather_probe(const uint8_t *src, uint8_t *dst, const int32_t *idx, int64_t n_rec,
                                int W, int sm_count, cudaStream_t st) {
    gather_probe_kernel<<<2 * sm_count, kThreads, 0, st>>>(src, dst, idx, n_rec, W);
    return cudaGetLastError();
}

}  // namespace hs

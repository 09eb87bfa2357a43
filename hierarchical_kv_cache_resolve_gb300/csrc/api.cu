// Host side of the C ABI declared in include/hs.h: pool allocation,
// argument checks, launches, counters and the link probe.
#include <algorithm>
#include <chrono>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <random>
#include <vector>

#include "hs.h"
#include "hs_internal.cuh"

struct hs_pool {
    hs_pool_desc desc;
    std::vector<int32_t> anchor;
    int device = 0;
    int sm_count = 0;
    int cluster_override = 0;
    bool overlap = true;  // consecutive resolves may overlap (launch_overlap)
    double warmup_us = 0;  // the huge-page pool's warm-up at creation
    hs::HostBuffer host = {};
    size_t host_bytes = 0;
    hs::DevPool dp = {};
    size_t cache_bytes = 0, pt_bytes = 0, meta_pairs = 0;
};

namespace {

bool cuda_ok(cudaError_t e) { return e == cudaSuccess; }

void free_device(hs_pool *p) {
    cudaFree(p->dp.cache);
    cudaFree(p->dp.pt);
    cudaFree(p->dp.slot_pos);
    cudaFree(p->dp.stamp);
    cudaFree(p->dp.lru);
    cudaFree(p->dp.tcount);
    cudaFree(p->dp.busy);
    cudaFree(p->dp.counters);
    cudaFree(p->dp.status);
    cudaFree(p->dp.sink);
    hs::host_free(&p->host);
}

// The host allocation a probe uses for HS_HOST_ALLOC_AUTO (a pool picks
// by its size, see hs_create_pool).
int auto_host_alloc() { return HS_HOST_ALLOC_PINNED; }

int reset_state(hs_pool *p) {
    const size_t pairs = p->meta_pairs;
    const size_t B = (size_t)p->desc.slots;
    if (!cuda_ok(cudaMemset(p->dp.pt, 0xFF, p->pt_bytes)) ||
        !cuda_ok(cudaMemset(p->dp.slot_pos, 0xFF, pairs * B * 4)) ||
        !cuda_ok(cudaMemset(p->dp.stamp, 0, pairs * B * 4)) ||
        !cuda_ok(cudaMemset(p->dp.tcount, 0, pairs * 4)) ||
        !cuda_ok(cudaMemset(p->dp.busy, 0, pairs * 4)) ||
        !cuda_ok(cudaMemset(p->dp.counters, 0, (size_t)p->desc.n_layers * hs::CTR_COUNT * 8)) ||
        !cuda_ok(cudaMemset(p->dp.status, 0, 4)) ||
        !cuda_ok(hs::launch_init_lru(p->dp.lru, (int64_t)pairs, (int)B, 0)) ||
        !cuda_ok(cudaDeviceSynchronize()))
        return HS_ERR_CUDA;
    return HS_OK;
}

int pick_cluster(const hs_pool *p, int n_req);
int lead_share(const hs_pool *p, int k, int cluster);

// Every byte of the host records read once from the device, synthetic
// resolves over every (request, layer) pair, then the empty state again
// (hs_warm_pool): kWarmSteps steps, each a new set of k distinct positions
// per request, so that every selection misses and every slot is written.
constexpr int kWarmSteps = 16;
int warm_pool(hs_pool *p) {
    const int R = p->desc.n_requests, NL = p->desc.n_layers;
    const int64_t L = p->desc.n_positions;
    const int k = (int)std::min<int64_t>(p->desc.max_k, L);
    const int64_t G = std::max<int64_t>(1, L / k), D = std::max<int64_t>(1, G / 7);
    std::vector<int32_t> sel((size_t)R * k);
    int32_t *dsel = nullptr, *dout = nullptr;
    int rc = HS_OK;
    if (!cuda_ok(cudaMalloc(&dsel, sel.size() * 4)) || !cuda_ok(cudaMalloc(&dout, sel.size() * 4))) {
        rc = HS_ERR_NOMEM;
    } else {
        // every byte of the records read once, then the synthetic steps
        if (!cuda_ok(hs::launch_touch(p->host.dev, p->host_bytes, p->dp.sink, p->sm_count, 0)))
            rc = HS_ERR_CUDA;
        const int cluster = pick_cluster(p, R);
        for (int step = 0; step < kWarmSteps && rc == HS_OK; ++step) {
            // positions (base_r + step * D + i * G) mod L: distinct, since k * G <= L
            for (int r = 0; r < R; ++r) {
                const int64_t base = ((int64_t)r * 7919) % L;
                for (int i = 0; i < k; ++i)
                    sel[(size_t)r * k + i] = (int32_t)((base + step * D + (int64_t)i * G) % L);
            }
            if (!cuda_ok(cudaMemcpy(dsel, sel.data(), sel.size() * 4, cudaMemcpyHostToDevice))) {
                rc = HS_ERR_CUDA;
                break;
            }
            for (int l = 0; l < NL && rc == HS_OK; ++l)
                if (!cuda_ok(hs::launch_resolve(p->dp, l, R, nullptr, dsel, k, dout, nullptr, cluster,
                                                0, p->anchor[l], nullptr, p->overlap,
                                                lead_share(p, k, cluster))))
                    rc = HS_ERR_CUDA;
        }
        if (rc == HS_OK && !cuda_ok(cudaDeviceSynchronize())) rc = HS_ERR_CUDA;
    }
    cudaFree(dsel);
    cudaFree(dout);
    if (rc != HS_OK) return rc;
    return reset_state(p);
}

// Cluster size for a resolve over n_req requests: the largest power of two
// up to 8 that keeps the grid in one wave (a resolve CTA occupies an SM),
// and 7 rather than 8 with launch overlap: measured on GB300 (8 requests,
// 4 layers, launches overlapping), clusters of 7 moved the misses at 0.73
// of the link against 0.71 for clusters of 8 in every one of four rounds,
// while clusters of 6 fell to 0.62.
int pick_cluster(const hs_pool *p, int n_req) {
    if (p->cluster_override > 0) return p->cluster_override;
    int c = hs::kMaxCluster;
    while (c > 1 && (int64_t)n_req * c > (int64_t)p->sm_count) c >>= 1;
    if (c == 8 && p->overlap) c = 7;
    return c;
}

// Selections whose misses the leader CTA fetches itself: without launch
// overlap its decision is never hidden under an earlier launch, and it
// would otherwise idle while its followers move the records; it takes an
// equal share of the selection.
int lead_share(const hs_pool *p, int k, int cluster) {
    return (p->overlap || cluster < 2) ? 0 : k / cluster;
}

bool check_common(const hs_pool *p, int32_t layer, int32_t n_req, int32_t k) {
    return p && layer >= 0 && layer < p->desc.n_layers && n_req >= 0 &&
           n_req <= p->desc.n_requests && k >= 1 && k <= p->desc.max_k;
}

// int32 arrays are read and written with 4-byte accesses
bool misaligned4(const void *a) { return (reinterpret_cast<uintptr_t>(a) & 3u) != 0; }

}  // namespace

static_assert(HS_STAMP_ENTRY == hs::S_ENTRY && HS_STAMP_LOADED == hs::S_LOADED &&
                  HS_STAMP_HASHED == hs::S_HASHED && HS_STAMP_PROBED == hs::S_PROBED &&
                  HS_STAMP_DECIDED == hs::S_DECIDED && HS_STAMP_CHECKED == hs::S_CHECKED &&
                  HS_STAMP_VERDICT == hs::S_VERDICT && HS_STAMP_COMMITTED == hs::S_COMMITTED &&
                  HS_STAMP_F_ISSUE == hs::S_F_ISSUE && HS_STAMP_F_ISSUED == hs::S_F_ISSUED &&
                  HS_STAMP_F_WAITED == hs::S_F_WAITED && HS_STAMP_F_LANDED == hs::S_F_LANDED &&
                  HS_STAMP_F_STORED == hs::S_F_STORED && HS_STAMP_ATTEMPTS == hs::S_ATTEMPTS &&
                  HS_STAMP_EXIT == hs::S_EXIT && HS_STAMP_LEAD_FETCHED == hs::S_LEAD_FETCHED,
              "stamp slots of hs.h and the kernel differ");

extern "C" {

const char *hs_strerror(int code) {
    switch (code) {
        case HS_OK: return "ok";
        case HS_ERR_INVALID_ARG: return "invalid argument";
        case HS_ERR_CUDA: return "CUDA runtime error";
        case HS_ERR_NOMEM: return "out of memory or over the configured host limit";
        case HS_ERR_DEVICE_INPUT: return "a kernel flagged invalid device input";
        case HS_ERR_TIMEOUT: return "timeout";
        case HS_ERR_UNSUPPORTED: return "sizes not supported by this build";
        default: return "unknown error";
    }
}

int32_t hs_kernels_per_call(void) { return 1; }

size_t hs_plan_bytes(int32_t n_req, int32_t k) {
    if (n_req < 0 || k < 0) return 0;
    return hs::plan_bytes(n_req, k);
}

int hs_create_pool(const hs_pool_desc *desc, hs_pool **out) {
    if (!out) return HS_ERR_INVALID_ARG;
    *out = nullptr;
    if (!desc) return HS_ERR_INVALID_ARG;
    const hs_pool_desc d = *desc;
    if (d.n_requests < 1 || d.n_layers < 1 || d.n_positions < 1 ||
        d.n_positions > INT32_MAX || d.record_bytes < 16 || d.record_bytes % 16 != 0 ||
        d.slots < 1 || d.slots > 32767 || d.max_k < 1 || d.max_k > d.slots ||
        d.host_alloc < HS_HOST_ALLOC_AUTO || d.host_alloc > HS_HOST_ALLOC_THP_REGISTERED ||
        d.launch_overlap < HS_OVERLAP_AUTO || d.launch_overlap > HS_OVERLAP_OFF)
        return HS_ERR_INVALID_ARG;
    // index arithmetic limits of the kernels (32-bit chunk counters and
    // published row indices)
    if ((int64_t)d.n_requests * d.slots > INT32_MAX ||
        (int64_t)2 * d.max_k * (d.record_bytes / 16) > INT32_MAX / 2)
        return HS_ERR_UNSUPPORTED;
    if (d.layer_anchor) {
        for (int l = 0; l < d.n_layers; ++l) {
            const int a = d.layer_anchor[l];
            if (a < 0 || a > l || d.layer_anchor[a] != a) return HS_ERR_INVALID_ARG;
        }
    }
    const size_t host_bytes = (size_t)d.n_requests * d.n_layers * (size_t)d.n_positions * d.record_bytes;
    if (d.host_limit_bytes && host_bytes > d.host_limit_bytes) return HS_ERR_NOMEM;

    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev))) return HS_ERR_CUDA;
    int smem_optin = 0, sms = 0;
    if (!cuda_ok(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) ||
        !cuda_ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
        return HS_ERR_CUDA;
    const size_t need = hs::resolve_smem_bytes(d.slots, d.max_k, true, d.n_positions);
    if (need > (size_t)smem_optin) return HS_ERR_UNSUPPORTED;

    hs_pool *p = new (std::nothrow) hs_pool();
    if (!p) return HS_ERR_NOMEM;
    p->desc = d;
    p->anchor.resize(d.n_layers);
    for (int l = 0; l < d.n_layers; ++l) p->anchor[l] = d.layer_anchor ? d.layer_anchor[l] : l;
    p->desc.layer_anchor = p->anchor.data();
    p->device = dev;
    p->sm_count = sms;
    p->overlap = d.launch_overlap == HS_OVERLAP_ON ||
                 (d.launch_overlap == HS_OVERLAP_AUTO && host_bytes <= HS_OVERLAP_AUTO_MAX_HOST_BYTES);
    p->desc.launch_overlap = p->overlap ? HS_OVERLAP_ON : HS_OVERLAP_OFF;
    if (const char *e = std::getenv("HS_CLUSTER")) {
        const int c = std::atoi(e);
        if (c >= 1 && c <= hs::kMaxCluster) p->cluster_override = c;
    }

    const size_t pairs = (size_t)d.n_requests * d.n_layers;
    const size_t B = (size_t)d.slots;
    p->meta_pairs = pairs;
    p->cache_bytes = pairs * B * d.record_bytes;
    p->pt_bytes = pairs * (size_t)d.n_positions * 4;
    p->host_bytes = host_bytes;

    int rc = HS_OK;
    if (d.host_alloc != HS_HOST_ALLOC_AUTO) {
        rc = hs::host_alloc(host_bytes, d.host_alloc, dev, &p->host);
    } else if (host_bytes > HS_OVERLAP_AUTO_MAX_HOST_BYTES) {
        // past the translation reach: huge pages if the kernel backs (nearly)
        // the whole pool with them, cudaHostAlloc otherwise
        rc = hs::host_alloc(host_bytes, HS_HOST_ALLOC_THP_REGISTERED, dev, &p->host);
        if (rc == HS_OK && p->host.huge_bytes < p->host.mapped / 10 * 9) hs::host_free(&p->host);
        if (rc != HS_OK || !p->host.host)
            rc = hs::host_alloc(host_bytes, HS_HOST_ALLOC_PINNED, dev, &p->host);
    } else {
        rc = hs::host_alloc(host_bytes, HS_HOST_ALLOC_PINNED, dev, &p->host);
    }
    if (rc != HS_OK) goto fail;
    p->desc.host_alloc = p->host.kind;
    p->dp.host = static_cast<const uint8_t *>(p->host.dev);
    if (!cuda_ok(cudaMalloc(&p->dp.cache, p->cache_bytes)) ||
        !cuda_ok(cudaMalloc(&p->dp.pt, p->pt_bytes)) ||
        !cuda_ok(cudaMalloc(&p->dp.slot_pos, pairs * B * 4)) ||
        !cuda_ok(cudaMalloc(&p->dp.stamp, pairs * B * 4)) ||
        !cuda_ok(cudaMalloc(&p->dp.lru, pairs * B * 2)) ||
        !cuda_ok(cudaMalloc(&p->dp.tcount, pairs * 4)) ||
        !cuda_ok(cudaMalloc(&p->dp.busy, pairs * 4)) ||
        !cuda_ok(cudaMalloc(&p->dp.counters, (size_t)d.n_layers * hs::CTR_COUNT * 8)) ||
        !cuda_ok(cudaMalloc(&p->dp.status, 4)) || !cuda_ok(cudaMalloc(&p->dp.sink, 4))) {
        cudaGetLastError();
        rc = HS_ERR_NOMEM;
        goto fail;
    }
    p->dp.R = d.n_requests;
    p->dp.NL = d.n_layers;
    p->dp.B = d.slots;
    p->dp.W = d.record_bytes;
    p->dp.L = d.n_positions;
    // the kernels' dynamic shared memory limit is a per-function setting
    // shared by every pool: raise it to the device maximum, never lower it
    if (!cuda_ok(hs::prepare_kernels((size_t)smem_optin))) { rc = HS_ERR_CUDA; goto fail; }
    rc = reset_state(p);
    if (rc != HS_OK) goto fail;
    *out = p;
    return HS_OK;
fail:
    free_device(p);
    delete p;
    return rc;
}

int hs_destroy_pool(hs_pool *pool) {
    if (!pool) return HS_OK;
    cudaDeviceSynchronize();
    free_device(pool);
    delete pool;
    return HS_OK;
}

int hs_host_records(hs_pool *pool, int32_t req, int32_t layer, void **host_ptr) {
    if (!pool || !host_ptr || req < 0 || req >= pool->desc.n_requests || layer < 0 ||
        layer >= pool->desc.n_layers)
        return HS_ERR_INVALID_ARG;
    *host_ptr = static_cast<uint8_t *>(pool->host.host) +
                hs::host_region(req, layer, pool->desc.n_requests, pool->desc.n_positions,
                                pool->desc.record_bytes);
    return HS_OK;
}

int hs_touch_records(hs_pool *pool, int32_t req, int32_t layer, void *stream) {
    if (!pool || req < -1 || req >= pool->desc.n_requests || layer < -1 ||
        layer >= pool->desc.n_layers)
        return HS_ERR_INVALID_ARG;
    const size_t per = (size_t)pool->desc.n_positions * pool->desc.record_bytes;
    const int R = pool->desc.n_requests, NL = pool->desc.n_layers;
    const uint8_t *base = static_cast<const uint8_t *>(pool->host.dev);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto region = [&](int r, int l) {
        return base + hs::host_region(r, l, R, pool->desc.n_positions, pool->desc.record_bytes);
    };
    // host[l][r][L][W]: all of a layer's requests, or all layers, are
    // contiguous; one (request, layer) region otherwise
    cudaError_t e = cudaSuccess;
    if (req < 0 && layer < 0) {
        e = hs::launch_touch(base, pool->host_bytes, pool->dp.sink, pool->sm_count, st);
    } else if (req < 0) {
        e = hs::launch_touch(region(0, layer), (size_t)R * per, pool->dp.sink, pool->sm_count, st);
    } else {
        for (int l = (layer < 0 ? 0 : layer); l < (layer < 0 ? NL : layer + 1) && e == cudaSuccess;
             ++l)
            e = hs::launch_touch(region(req, l), per, pool->dp.sink, pool->sm_count, st);
    }
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int hs_warm_pool(hs_pool *pool) {
    if (!pool) return HS_ERR_INVALID_ARG;
    const auto t0 = std::chrono::steady_clock::now();
    const int rc = warm_pool(pool);
    if (rc == HS_OK)
        pool->warmup_us =
            std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
    return rc;
}

int hs_device_host_numa(int32_t device) {
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (device < 0 || device >= n) return -1;
    return hs::device_host_numa(device);
}

int hs_pool_info(hs_pool *pool, hs_pool_info_t *out) {
    if (!pool || !out) return HS_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    out->host_alloc = pool->host.kind;
    out->device = pool->device;
    out->launch_overlap = pool->desc.launch_overlap;
    out->device_numa = hs::device_host_numa(pool->device);
    const uint8_t *h = static_cast<const uint8_t *>(pool->host.host);
    out->host_numa_first = hs::page_numa_node(h);
    out->host_numa_last = hs::page_numa_node(h + pool->host_bytes - 1);
    out->host_bytes = pool->host_bytes;
    out->host_mapped_bytes = pool->host.mapped;
    out->host_granularity = pool->host.granularity;
    out->host_huge_bytes = pool->host.huge_bytes;
    out->warmup_us = (uint64_t)pool->warmup_us;
    const size_t pairs = pool->meta_pairs, B = (size_t)pool->desc.slots;
    out->device_bytes = pool->cache_bytes + pool->pt_bytes + pairs * B * (4 + 4 + 2) + pairs * 8 +
                        (size_t)pool->desc.n_layers * hs::CTR_COUNT * 8 + 4;
    return HS_OK;
}

int hs_device_views(hs_pool *pool, int32_t layer, hs_views *out) {
    if (!pool || !out || layer < 0 || layer >= pool->desc.n_layers) return HS_ERR_INVALID_ARG;
    const size_t R = pool->desc.n_requests, B = pool->desc.slots;
    const size_t lp = (size_t)layer * R;
    out->cache = pool->dp.cache + lp * B * pool->desc.record_bytes;
    out->page_table = pool->dp.pt + lp * (size_t)pool->desc.n_positions;
    out->slot_pos = pool->dp.slot_pos + lp * B;
    out->stamps = pool->dp.stamp + lp * B;
    out->lru = pool->dp.lru + lp * B;
    out->resolves = pool->dp.tcount + lp;
    return HS_OK;
}

int hs_resolve(hs_pool *pool, int32_t layer, int32_t n_req, const int32_t *d_req_ids,
               const int32_t *d_sel, int32_t k, int32_t *d_out, const void *d_plan, void *stream) {
    if (!check_common(pool, layer, n_req, k) || !d_sel || !d_out) return HS_ERR_INVALID_ARG;
    if (d_plan && (reinterpret_cast<uintptr_t>(d_plan) & 15u)) return HS_ERR_INVALID_ARG;
    if (misaligned4(d_sel) || misaligned4(d_out) || misaligned4(d_req_ids)) return HS_ERR_INVALID_ARG;
    if (n_req == 0) return HS_OK;
    const int cluster = pick_cluster(pool, n_req);
    const cudaError_t e = hs::launch_resolve(pool->dp, layer, n_req, d_req_ids, d_sel, k, d_out, d_plan,
                                             cluster, static_cast<cudaStream_t>(stream),
                                             pool->anchor[layer], nullptr, pool->overlap,
                                             lead_share(pool, k, cluster));
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int hs_resolve_anchor(hs_pool *pool, int32_t layer, int32_t n_req, const int32_t *d_req_ids,
                      const int32_t *d_sel, int32_t k, int32_t *d_out, void *d_plan_out,
                      void *stream) {
    if (!check_common(pool, layer, n_req, k) || !d_sel || !d_out || !d_plan_out)
        return HS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_plan_out) & 15u) || misaligned4(d_sel) || misaligned4(d_out) ||
        misaligned4(d_req_ids))
        return HS_ERR_INVALID_ARG;
    if (n_req == 0) return HS_OK;
    const int cluster = pick_cluster(pool, n_req);
    const cudaError_t e = hs::launch_resolve(pool->dp, layer, n_req, d_req_ids, d_sel, k, d_out,
                                             nullptr, cluster, static_cast<cudaStream_t>(stream),
                                             -1, d_plan_out, pool->overlap,
                                             lead_share(pool, k, cluster));
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int hs_resolve_measure(hs_pool *pool, int32_t layer, int32_t n_req, const int32_t *d_req_ids,
                       const int32_t *d_sel, int32_t k, int32_t *d_out, int32_t flags,
                       uint64_t *d_times, void *stream) {
    if (!check_common(pool, layer, n_req, k) || !d_sel || !d_out) return HS_ERR_INVALID_ARG;
    if (misaligned4(d_sel) || misaligned4(d_out) || misaligned4(d_req_ids) ||
        (reinterpret_cast<uintptr_t>(d_times) & 7u) || (flags & ~HS_MEASURE_NO_FETCH))
        return HS_ERR_INVALID_ARG;
    if (n_req == 0) return HS_OK;
    const int cluster = pick_cluster(pool, n_req);
    const cudaError_t e = hs::launch_resolve_measure(
        pool->dp, layer, n_req, d_req_ids, d_sel, k, d_out, (flags & HS_MEASURE_NO_FETCH) != 0,
        reinterpret_cast<unsigned long long *>(d_times), cluster,
        static_cast<cudaStream_t>(stream), pool->overlap, lead_share(pool, k, cluster));
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int32_t hs_measure_stamp_slots(void) { return hs::kMaxCluster * hs::kStampSlots; }

int hs_prefetch_plan(hs_pool *pool, int32_t anchor_layer, int32_t target_layer, int32_t n_req,
                     const int32_t *d_req_ids, const int32_t *d_sel, int32_t k, void *d_plan,
                     void *stream) {
    if (!check_common(pool, target_layer, n_req, k) || !d_sel || !d_plan ||
        misaligned4(d_sel) || misaligned4(d_req_ids))
        return HS_ERR_INVALID_ARG;
    if (anchor_layer < 0 || anchor_layer >= pool->desc.n_layers ||
        pool->anchor[target_layer] != anchor_layer)
        return HS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_plan) & 15u) return HS_ERR_INVALID_ARG;
    if (n_req == 0) return HS_OK;
    const cudaError_t e = hs::launch_plan(pool->dp, target_layer, n_req, d_req_ids, d_sel, k, d_plan,
                                          static_cast<cudaStream_t>(stream));
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int hs_prefetch_copy(hs_pool *pool, int32_t target_layer, int32_t n_req, int32_t k,
                     const void *d_plan, void *stream) {
    if (!check_common(pool, target_layer, n_req, k) || !d_plan) return HS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_plan) & 15u) return HS_ERR_INVALID_ARG;
    if (n_req == 0) return HS_OK;
    const cudaError_t e = hs::launch_prefetch_copy(pool->dp, target_layer, n_req, k, d_plan,
                                                   pool->sm_count, static_cast<cudaStream_t>(stream),
                                                   pool->anchor[target_layer], !pool->overlap);
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int hs_stats(hs_pool *pool, int32_t layer, hs_stats_t *out) {
    if (!pool || !out || layer < -1 || layer >= pool->desc.n_layers) return HS_ERR_INVALID_ARG;
    if (!cuda_ok(cudaDeviceSynchronize())) return HS_ERR_CUDA;
    const int NL = pool->desc.n_layers;
    std::vector<unsigned long long> c((size_t)NL * hs::CTR_COUNT);
    uint32_t status = 0;
    if (!cuda_ok(cudaMemcpy(c.data(), pool->dp.counters, c.size() * 8, cudaMemcpyDeviceToHost)) ||
        !cuda_ok(cudaMemcpy(&status, pool->dp.status, 4, cudaMemcpyDeviceToHost)) ||
        !cuda_ok(cudaMemset(pool->dp.status, 0, 4)))
        return HS_ERR_CUDA;
    std::memset(out, 0, sizeof(*out));
    for (int l = 0; l < NL; ++l) {
        if (layer >= 0 && l != layer) continue;
        const unsigned long long *x = &c[(size_t)l * hs::CTR_COUNT];
        out->resolves += x[hs::CTR_RESOLVES];
        out->hits += x[hs::CTR_HITS];
        out->misses += x[hs::CTR_MISSES];
        out->fetched_bytes += x[hs::CTR_FETCHED];
        out->prefetched_bytes += x[hs::CTR_PREFETCHED];
        out->plan_hits += x[hs::CTR_PLAN_HITS];
        out->plan_mismatches += x[hs::CTR_PLAN_MISMATCH];
    }
    out->status = status;
    return status ? HS_ERR_DEVICE_INPUT : HS_OK;
}

int hs_reset(hs_pool *pool) {
    if (!pool) return HS_ERR_INVALID_ARG;
    if (!cuda_ok(cudaDeviceSynchronize())) return HS_ERR_CUDA;
    return reset_state(pool);
}

int hs_sparse_attention(const void *d_q, const void *d_cache, int64_t cache_rows,
                        const int32_t *d_idx, int32_t n_req, int32_t k, int32_t heads,
                        float scale, float *d_out, void *stream) {
    auto misaligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (!d_q || !d_cache || !d_idx || !d_out || cache_rows < 1 || n_req < 0 || n_req > 65535 ||
        k < 1 || heads < 16 || heads % 16 != 0 || heads / 16 > 65535 || misaligned(d_q) ||
        misaligned(d_cache) || misaligned(d_out))
        return HS_ERR_INVALID_ARG;
    if (n_req == 0) return HS_OK;
    const cudaError_t e = hs::launch_attention(d_q, d_cache, cache_rows, d_idx, n_req, k, heads,
                                               scale, d_out, static_cast<cudaStream_t>(stream));
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int hs_sparse_attention_heads(const void *d_q, const void *d_cache, int64_t cache_rows,
                              const int32_t *d_idx, int32_t n_req, int32_t k, int32_t heads,
                              float scale, float *d_out, void *stream) {
    auto misaligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (!d_q || !d_cache || !d_idx || !d_out || cache_rows < 1 || n_req < 0 || n_req > 65535 ||
        k < 1 || heads < 1 || heads > 8 || misaligned(d_q) || misaligned(d_cache) ||
        misaligned(d_out))
        return HS_ERR_INVALID_ARG;
    if (n_req == 0) return HS_OK;
    const cudaError_t e = hs::launch_attention_heads(d_q, d_cache, cache_rows, d_idx, n_req, k,
                                                     heads, scale, d_out,
                                                     static_cast<cudaStream_t>(stream));
    return cuda_ok(e) ? HS_OK : HS_ERR_CUDA;
}

int hs_attention_status(uint32_t *status) {
    if (!status) return HS_ERR_INVALID_ARG;
    if (!cuda_ok(cudaDeviceSynchronize())) return HS_ERR_CUDA;
    return cuda_ok(hs::attention_status(status)) ? HS_OK : HS_ERR_CUDA;
}

int hs_link_probe(size_t bytes, int32_t reps, int32_t record_bytes, int32_t host_alloc,
                  double *h2d_gbs, double *gather_gbs) {
    if (bytes < (size_t)record_bytes || reps < 1 || record_bytes < 16 || record_bytes % 16 ||
        host_alloc < HS_HOST_ALLOC_AUTO || host_alloc > HS_HOST_ALLOC_THP_REGISTERED)
        return HS_ERR_INVALID_ARG;
    const int64_t n_rec = (int64_t)(bytes / (size_t)record_bytes);
    if (n_rec > INT32_MAX) return HS_ERR_INVALID_ARG;
    bytes = (size_t)n_rec * record_bytes;
    // what one timed run moves: at most 1 GiB, gathered from all of `bytes`
    const size_t moved_cap = (size_t)1 << 30;
    const int64_t n_move = std::min<int64_t>(n_rec, (int64_t)(moved_cap / (size_t)record_bytes));
    const size_t moved = (size_t)n_move * record_bytes;
    int dev = 0, sms = 0;
    if (!cuda_ok(cudaGetDevice(&dev)) ||
        !cuda_ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
        return HS_ERR_CUDA;
    hs::HostBuffer hb = {};
    void *ddst = nullptr;
    int32_t *didx = nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    std::vector<int32_t> idx((size_t)n_move);
    int rc = hs::host_alloc(bytes, host_alloc ? host_alloc : auto_host_alloc(), dev, &hb);
    if (rc != HS_OK) return rc;
    if (n_move == n_rec) {
        for (int64_t i = 0; i < n_rec; ++i) idx[(size_t)i] = (int32_t)i;
        std::shuffle(idx.begin(), idx.end(), std::mt19937_64(12345));
    } else {
        std::mt19937_64 g(12345);
        std::uniform_int_distribution<int64_t> u(0, n_rec - 1);
        for (auto &x : idx) x = (int32_t)u(g);
    }
    if (!cuda_ok(cudaMalloc(&ddst, moved)) || !cuda_ok(cudaMalloc(&didx, (size_t)n_move * 4)) ||
        !cuda_ok(cudaMemcpy(didx, idx.data(), (size_t)n_move * 4, cudaMemcpyHostToDevice)) ||
        !cuda_ok(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking)) ||
        !cuda_ok(cudaEventCreate(&e0)) || !cuda_ok(cudaEventCreate(&e1))) {
        rc = HS_ERR_CUDA;
        goto done;
    }
    for (int which = 0; which < 2; ++which) {
        double *dst = which == 0 ? h2d_gbs : gather_gbs;
        if (!dst) continue;
        float best = 0.f;
        for (int it = 0; it < reps + 1; ++it) {  // first run is a warm-up
            cudaEventRecord(e0, st);
            cudaError_t e = which == 0
                                ? cudaMemcpyAsync(ddst, hb.host, moved, cudaMemcpyHostToDevice, st)
                                : hs::launch_gather_probe(static_cast<const uint8_t *>(hb.dev),
                                                          static_cast<uint8_t *>(ddst), didx, n_move,
                                                          record_bytes, sms, st);
            cudaEventRecord(e1, st);
            if (!cuda_ok(e) || !cuda_ok(cudaEventSynchronize(e1))) { rc = HS_ERR_CUDA; goto done; }
            float ms = 0.f;
            cudaEventElapsedTime(&ms, e0, e1);
            if (it > 0 && (best == 0.f || ms < best)) best = ms;
        }
        *dst = (double)moved / (best * 1e-3) / 1e9;
    }
done:
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (st) cudaStreamDestroy(st);
    cudaFree(didx);
    cudaFree(ddst);
    hs::host_free(&hb);
    return rc;
}

}  // extern "C"

// hs_resolve_noalloc: the resolve kernel over caller-owned layer state, with
// its scratch (per-request claim flags, counters, a spare status word) in a
// file-scope device array instead of pool memory, so that the call
// allocates nothing.
#include <cstdint>
#include <mutex>

#include <cuda.h>

#include "hs.h"
#include "hs_internal.cuh"

namespace {

constexpr size_t kHeaderBytes = 256;  // counters [0, 64), spare status word at 64
constexpr size_t kScratchBytes = kHeaderBytes + 4 * (size_t)HS_NOALLOC_MAX_REQUESTS;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mu;
unsigned char *g_scratch_addr[kMaxDevices];  // device address of the array, per device
unsigned long long g_ctx_id[kMaxDevices];    // the context that address belongs to
int g_sm_count[kMaxDevices];

// Unique id of the current context (cuCtxGetId, looked up through the
// runtime), 0 when it cannot be had.  A device reset makes a new primary
// context with a new id, in which the array has a new address.
unsigned long long current_context_id() {
    static CUresult (*get_current)(CUcontext *) = nullptr;
    static CUresult (*get_id)(CUcontext, unsigned long long *) = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa = cudaDriverEntryPointSymbolNotFound, qb = qa;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
                cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qa == cudaDriverEntryPointSuccess && qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CUresult (*)(CUcontext *)>(a);
            get_id = reinterpret_cast<CUresult (*)(CUcontext, unsigned long long *)>(b);
        }
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Once per device and context, with that device current: the array's
// device address (host code may not use the symbol itself) and the kernel
// configuration.  Redone when the device's context has changed (after a
// device reset), so no stale address is used.
int setup_current_device(unsigned char **scratch, int *sm_count) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    // 0 before the runtime has made the device's primary context current
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_addr[dev] || ctx == 0 || g_ctx_id[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return HS_ERR_CUDA;
        int smem_optin = 0, sms = 0;
        if (cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            hs::prepare_kernels((size_t)smem_optin) != cudaSuccess)
            return HS_ERR_CUDA;
        g_sm_count[dev] = sms;
        g_scratch_addr[dev] = static_cast<unsigned char *>(p);
        g_ctx_id[dev] = current_context_id();  // the lookup made the context current
    }
    *scratch = g_scratch_addr[dev];
    *sm_count = g_sm_count[dev];
    return HS_OK;
}

}  // namespace

extern "C" int hs_resolve_noalloc(const hs_layer_state *st, int32_t n_req, const int32_t *d_req_ids,
                                  const int32_t *d_sel, int32_t k, int32_t *d_out,
                                  uint32_t *d_status, void *stream) {
    if (!st || !d_sel || !d_out) return HS_ERR_INVALID_ARG;
    const hs_layer_state s = *st;
    if (s.n_requests < 1 || s.n_positions < 1 || s.n_positions > INT32_MAX ||
        s.record_bytes < 16 || s.record_bytes % 16 != 0 || s.slots < 1 || s.slots > 32767 ||
        k < 1 || k > s.slots || n_req < 0 || n_req > s.n_requests || !s.host_records ||
        !s.cache || !s.page_table || !s.slot_pos || !s.stamps || !s.lru || !s.resolves)
        return HS_ERR_INVALID_ARG;
    // the kernel reads records and writes slots with 16-byte accesses, the
    // int32 / u32 arrays with 4-byte and the LRU order with 2-byte ones: a
    // misaligned pointer would fault the GPU, so it is refused here
    auto off = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
    if (off(s.host_records, 16) || off(s.cache, 16) || off(s.page_table, 4) || off(s.slot_pos, 4) ||
        off(s.stamps, 4) || off(s.resolves, 4) || off(s.lru, 2) || off(d_sel, 4) || off(d_out, 4) ||
        off(d_req_ids, 4) || off(d_status, 4))
        return HS_ERR_INVALID_ARG;
    if (s.n_requests > HS_NOALLOC_MAX_REQUESTS) return HS_ERR_UNSUPPORTED;
    if ((int64_t)s.n_requests * s.slots > INT32_MAX ||
        (int64_t)2 * k * (s.record_bytes / 16) > INT32_MAX / 2)
        return HS_ERR_UNSUPPORTED;
    int dev = 0, smem_optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return HS_ERR_CUDA;
    if (hs::resolve_smem_bytes(s.slots, k, false, s.n_positions) > (uint32_t)smem_optin)
        return HS_ERR_UNSUPPORTED;
    if (n_req == 0) return HS_OK;

    unsigned char *scratch = nullptr;
    int sms = 0;
    const int rc = setup_current_device(&scratch, &sms);
    if (rc != HS_OK) return rc;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // counters, spare status word and this layer's claim flags start at zero
    if (cudaMemsetAsync(scratch, 0, kHeaderBytes + 4 * (size_t)s.n_requests, cs) != cudaSuccess)
        return HS_ERR_CUDA;

    hs::DevPool p = {};
    p.host = static_cast<const uint8_t *>(s.host_records);
    p.cache = static_cast<uint8_t *>(s.cache);
    p.pt = s.page_table;
    p.slot_pos = s.slot_pos;
    p.stamp = s.stamps;
    p.lru = s.lru;
    p.tcount = s.resolves;
    p.busy = reinterpret_cast<uint32_t *>(scratch + kHeaderBytes);
    p.counters = reinterpret_cast<unsigned long long *>(scratch);
    p.status = d_status ? d_status : reinterpret_cast<unsigned int *>(scratch + 64);
    p.R = s.n_requests;
    p.NL = 1;
    p.B = s.slots;
    p.W = s.record_bytes;
    p.L = s.n_positions;
    int cluster = hs::kMaxCluster;
    while (cluster > 1 && (int64_t)n_req * cluster > (int64_t)sms) cluster >>= 1;
    const cudaError_t e = hs::launch_resolve(p, 0, n_req, d_req_ids, d_sel, k, d_out, nullptr,
                                             cluster, cs);
    return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

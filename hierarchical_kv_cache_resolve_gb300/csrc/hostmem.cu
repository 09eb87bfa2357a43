// Host memory that the GPU reads directly: the authoritative tier of the
// two-level hierarchy ("Inference Systems Infrastructure Notes (6):
// HiSparse", section 2 "Two-Level Hierarchy": every KV record lives in
// pinned, device-mapped host memory).
//
// Three ways to provide it:
//   HS_HOST_ALLOC_PINNED   cudaHostAlloc(Mapped | Portable), allocated
//                          while the calling thread prefers the host NUMA
//                          node the device reports as its closest
//                          (cudaDevAttrHostNumaId), so the pinned pages
//                          come from that node;
//   HS_HOST_ALLOC_VMM_NUMA the virtual memory management API: one pinned
//                          physical allocation on the host NUMA node the
//                          device reports as its closest
//                          (cudaDevAttrHostNumaId), mapped at one virtual
//                          address range that both the device and the host
//                          may read and write;
//   HS_HOST_ALLOC_THP_REGISTERED anonymous memory in transparent huge pages,
//                          first touched on that node, pinned and mapped
//                          with cudaHostRegister.
// The driver API entry points are looked up through the runtime
// (cudaGetDriverEntryPointByVersion), so the library does not link
// libcuda itself.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <sys/mman.h>
#include <sys/syscall.h>
#include <unistd.h>

#include "hs.h"
#include "hs_internal.cuh"

namespace hs {
namespace {

struct Vmm {
    CUresult (*get_granularity)(size_t *, const CUmemAllocationProp *,
                                CUmemAllocationGranularity_flags) = nullptr;
    CUresult (*address_reserve)(CUdeviceptr *, size_t, size_t, CUdeviceptr,
                                unsigned long long) = nullptr;
    CUresult (*address_free)(CUdeviceptr, size_t) = nullptr;
    CUresult (*create)(CUmemGenericAllocationHandle *, size_t, const CUmemAllocationProp *,
                       unsigned long long) = nullptr;
    CUresult (*release)(CUmemGenericAllocationHandle) = nullptr;
    CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle,
                    unsigned long long) = nullptr;
    CUresult (*unmap)(CUdeviceptr, size_t) = nullptr;
    CUresult (*set_access)(CUdeviceptr, size_t, const CUmemAccessDesc *, size_t) = nullptr;
    bool ok = false;
};

template <class F>
bool entry(const char *name, F *fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return false;
    *fn = reinterpret_cast<F>(p);
    return true;
}

const Vmm &vmm() {
    static Vmm v;
    static std::once_flag once;
    std::call_once(once, [] {
        v.ok = entry("cuMemGetAllocationGranularity", &v.get_granularity) &&
               entry("cuMemAddressReserve", &v.address_reserve) &&
               entry("cuMemAddressFree", &v.address_free) && entry("cuMemCreate", &v.create) &&
               entry("cuMemRelease", &v.release) && entry("cuMemMap", &v.map) &&
               entry("cuMemUnmap", &v.unmap) && entry("cuMemSetAccess", &v.set_access);
    });
    return v;
}

CUmemAllocationProp numa_prop(int numa) {
    CUmemAllocationProp prop;
    std::memset(&prop, 0, sizeof(prop));
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_HOST_NUMA;
    prop.location.id = numa;
    prop.requestedHandleTypes = CU_MEM_HANDLE_TYPE_NONE;
    return prop;
}

int alloc_vmm(size_t bytes, int dev, HostBuffer *out) {
    const Vmm &v = vmm();
    if (!v.ok) return HS_ERR_UNSUPPORTED;
    int numa = -1;
    if (cudaDeviceGetAttribute(&numa, cudaDevAttrHostNumaId, dev) != cudaSuccess) return HS_ERR_CUDA;
    if (numa < 0) numa = 0;  // a system without NUMA has node 0 only
    const CUmemAllocationProp prop = numa_prop(numa);
    size_t gran = 0;
    if (v.get_granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_RECOMMENDED) != CUDA_SUCCESS ||
        gran == 0)
        return HS_ERR_UNSUPPORTED;
    const size_t size = (bytes + gran - 1) / gran * gran;
    // align the range to 1 GiB (or the granularity, if larger), so that the
    // mapping may use the largest pages the driver has
    const size_t align = gran > ((size_t)1 << 30) ? gran : ((size_t)1 << 30);
    CUdeviceptr va = 0;
    if (v.address_reserve(&va, size, align, 0, 0) != CUDA_SUCCESS) return HS_ERR_NOMEM;
    CUmemGenericAllocationHandle h = 0;
    if (v.create(&h, size, &prop, 0) != CUDA_SUCCESS) {
        v.address_free(va, size);
        return HS_ERR_NOMEM;
    }
    CUmemAccessDesc acc[2];
    std::memset(acc, 0, sizeof(acc));
    acc[0].location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    acc[0].location.id = dev;
    acc[0].flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    acc[1].location.type = CU_MEM_LOCATION_TYPE_HOST_NUMA;
    acc[1].location.id = numa;
    acc[1].flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    if (v.map(va, size, 0, h, 0) != CUDA_SUCCESS) {
        v.release(h);
        v.address_free(va, size);
        return HS_ERR_CUDA;
    }
    if (v.set_access(va, size, acc, 2) != CUDA_SUCCESS) {
        v.unmap(va, size);
        v.release(h);
        v.address_free(va, size);
        return HS_ERR_CUDA;
    }
    out->host = reinterpret_cast<void *>(va);
    out->dev = reinterpret_cast<const void *>(va);
    out->bytes = bytes;
    out->mapped = size;
    out->granularity = gran;
    out->handle = (unsigned long long)h;
    out->kind = HS_HOST_ALLOC_VMM_NUMA;
    out->numa = numa;
    return HS_OK;
}

// The calling thread's NUMA memory policy, replaced for the duration of an
// allocation by "prefer node `node`" (set_mempolicy(MPOL_PREFERRED)), so
// that the pages the driver pins for it come from the node closest to the
// device.  Does nothing where the kernel has no NUMA policy support.
class PreferNode {
  public:
    explicit PreferNode(int node) {
#if defined(SYS_get_mempolicy) && defined(SYS_set_mempolicy)
        if (node < 0 || node >= kBits) return;
        if (syscall(SYS_get_mempolicy, &old_mode_, old_mask_, (unsigned long)kBits + 1, nullptr,
                    0UL) != 0)
            return;
        unsigned long mask[kWords] = {};
        mask[node / 64] |= 1UL << (node % 64);
        const int kPreferred = 1;  // MPOL_PREFERRED
        active_ = syscall(SYS_set_mempolicy, kPreferred, mask, (unsigned long)kBits + 1) == 0;
#else
        (void)node;
#endif
    }
    ~PreferNode() {
#if defined(SYS_set_mempolicy)
        if (!active_) return;
        // the default policy takes no node mask
        if ((old_mode_ & 0xFF) == 0)
            syscall(SYS_set_mempolicy, old_mode_, nullptr, 0UL);
        else
            syscall(SYS_set_mempolicy, old_mode_, old_mask_, (unsigned long)kBits + 1);
#endif
    }

  private:
    static constexpr int kBits = 1024, kWords = kBits / 64;
    int old_mode_ = 0;
    unsigned long old_mask_[kWords] = {};
    bool active_ = false;
};

// Transparent-huge-page size of the kernel (PMD size), 2 MiB if unknown.
size_t thp_size() {
    size_t v = 0;
    if (FILE *f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
        unsigned long long x = 0;
        if (std::fscanf(f, "%llu", &x) == 1) v = (size_t)x;
        std::fclose(f);
    }
    return v >= 4096 ? v : ((size_t)2 << 20);
}

int alloc_thp_registered(size_t bytes, int dev, HostBuffer *out);

// Bytes of [p, p + n) that the kernel backs with transparent huge pages:
// the AnonHugePages of the mappings overlapping it (/proc/self/smaps).
size_t huge_backed_bytes(const void *p, size_t n) {
    FILE *f = std::fopen("/proc/self/smaps", "r");
    if (!f) return 0;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p), hi = lo + n;
    char line[512];
    bool cur = false;
    size_t kb = 0;
    while (std::fgets(line, sizeof line, f)) {
        unsigned long long a = 0, b = 0;
        char c = 0;
        if (std::sscanf(line, "%llx-%llx %c", &a, &b, &c) == 3) {  // a mapping's header line
            cur = a < hi && b > lo;
            continue;
        }
        unsigned long long v = 0;
        if (cur && std::sscanf(line, "AnonHugePages: %llu kB", &v) == 1) kb += (size_t)v;
    }
    std::fclose(f);
    return kb << 10;
}

}  // namespace

int device_host_numa(int dev) {
    int numa = -1;
    if (cudaDeviceGetAttribute(&numa, cudaDevAttrHostNumaId, dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return numa;
}

namespace {

// Anonymous memory in transparent huge pages (madvise on the mapping only),
// aligned to the huge-page size, first touched by threads preferring the
// device's NUMA node, then pinned and mapped for the device with
// cudaHostRegister.
int alloc_thp_registered(size_t bytes, int dev, HostBuffer *out) {
    const size_t hp = thp_size();
    const size_t size = (bytes + hp - 1) / hp * hp;
    void *raw = mmap(nullptr, size + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (raw == MAP_FAILED) return HS_ERR_NOMEM;
    uint8_t *p = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(raw) + hp - 1) / hp * hp);
    madvise(p, size, MADV_HUGEPAGE);
    const int numa = device_host_numa(dev);
    // first touch in parallel, one huge page at a time
    const size_t pages = size / hp;
    unsigned nt = std::thread::hardware_concurrency();
    if (nt < 1) nt = 1;
    if (nt > 64) nt = 64;
    if ((size_t)nt > pages) nt = (unsigned)pages;
    auto touch_share = [=](unsigned t) {
        PreferNode prefer(numa);
        for (size_t i = t; i < pages; i += nt) std::memset(p + i * hp, 0, hp);
    };
    std::vector<std::thread> th;
    unsigned started = 0;
    try {
        for (; started < nt; ++started) th.emplace_back(touch_share, started);
    } catch (...) {
        // no more threads: this one touches the shares left
    }
    for (unsigned t = started; t < nt; ++t) touch_share(t);
    for (auto &x : th) x.join();
    if (cudaHostRegister(p, size, cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess) {
        cudaGetLastError();
        munmap(raw, size + hp);
        return HS_ERR_NOMEM;
    }
    void *d = nullptr;
    if (cudaHostGetDevicePointer(&d, p, 0) != cudaSuccess) {
        cudaHostUnregister(p);
        munmap(raw, size + hp);
        return HS_ERR_CUDA;
    }
    out->host = p;
    out->dev = d;
    out->bytes = bytes;
    out->mapped = size;
    out->granularity = hp;
    out->huge_bytes = huge_backed_bytes(p, size);
    out->handle = reinterpret_cast<unsigned long long>(raw);
    out->kind = HS_HOST_ALLOC_THP_REGISTERED;
    out->numa = numa;
    return HS_OK;
}

}  // namespace

int host_alloc(size_t bytes, int kind, int dev, HostBuffer *out) {
    std::memset(out, 0, sizeof(*out));
    out->numa = -1;
    if (kind == HS_HOST_ALLOC_VMM_NUMA) return alloc_vmm(bytes, dev, out);
    if (kind == HS_HOST_ALLOC_THP_REGISTERED) return alloc_thp_registered(bytes, dev, out);
    if (kind != HS_HOST_ALLOC_PINNED) return HS_ERR_INVALID_ARG;
    void *h = nullptr, *d = nullptr;
    const int numa = device_host_numa(dev);
    cudaError_t e;
    {
        PreferNode prefer(numa);
        e = cudaHostAlloc(&h, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return HS_ERR_NOMEM;
    }
    out->numa = numa;
    if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
        cudaFreeHost(h);
        return HS_ERR_CUDA;
    }
    out->host = h;
    out->dev = d;
    out->bytes = bytes;
    out->mapped = bytes;
    out->kind = HS_HOST_ALLOC_PINNED;
    return HS_OK;
}

void host_free(HostBuffer *b) {
    if (!b->host) return;
    if (b->kind == HS_HOST_ALLOC_VMM_NUMA) {
        const Vmm &v = vmm();
        const CUdeviceptr va = reinterpret_cast<CUdeviceptr>(b->host);
        v.unmap(va, b->mapped);
        v.release((CUmemGenericAllocationHandle)b->handle);
        v.address_free(va, b->mapped);
    } else if (b->kind == HS_HOST_ALLOC_THP_REGISTERED) {
        cudaHostUnregister(b->host);
        munmap(reinterpret_cast<void *>(b->handle), b->mapped + b->granularity);
    } else {
        cudaFreeHost(b->host);
    }
    std::memset(b, 0, sizeof(*b));
    b->numa = -1;
}

// NUMA node of the page holding `addr` (get_mempolicy with MPOL_F_NODE |
// MPOL_F_ADDR), or -1 when the kernel does not say (no NUMA support, or a
// mapping it does not track per page).
int page_numa_node(const void *addr) {
#ifdef SYS_get_mempolicy
    int node = -1;
    const unsigned long kNode = 1, kAddr = 2;  // MPOL_F_NODE, MPOL_F_ADDR
    if (syscall(SYS_get_mempolicy, &node, nullptr, 0UL, addr, kNode | kAddr) == 0) return node;
#else
    (void)addr;
#endif
    return -1;
}

}  // namespace hs

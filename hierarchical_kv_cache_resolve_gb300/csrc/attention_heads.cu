// Decode attention over the published slots for token records made of
// per-head key and value blocks (the Quest-style token records: `heads`
// blocks of 128 bf16 keys, then `heads` blocks of 128 bf16 values, 512
// bytes per head).  It is the consumer side of the exactness claim of
// "Inference Systems Infrastructure Notes (6): HiSparse", section 5 "Why It
// Is Exact": only the placement of the records changes, so attention over
// the slots a resolve published equals attention over the selected
// positions read from the host pool.
//
// Work split: one thread-block cluster per request; its C CTAs split the k
// published rows into C contiguous ranges.  Warp w of a CTA is head w: per
// row it reads its 256-byte key block and 256-byte value block with one
// 8-byte load per lane each (four of the 128 dimensions per lane), forms
// the score with a warp reduction and keeps an online softmax (base 2) and
// its four output dimensions in registers.  The slot indices are staged in
// shared memory; rows go in batches of eight whose loads are issued
// together, and the next batch is issued before the current one is used.  The C partial results (max, sum,
// unnormalised output per head) are merged on chip through distributed
// shared memory: CTA c writes output elements [c * heads * 128 / C, ...).
//
// The contraction is one query against 128 dimensions per head and row,
// about half a multiply-add per gathered byte: HBM-bound on the CUDA cores,
// with nothing for a tensor-core tile to do.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cooperative_groups.h>

#include "hs.h"
#include "hs_internal.cuh"

namespace hs {
namespace {

namespace cg = cooperative_groups;

constexpr int kHeadDim = 128;
constexpr int kMaxHeadsMH = 8;       // warps per CTA
constexpr int kMaxSplitMH = 8;       // portable cluster size
constexpr int kBatch = 8;            // rows whose loads are issued together
constexpr int kMinRowsPerSplit = 64;
constexpr int kIdxChunk = 512;       // slot indices staged in shared memory at a time

__device__ __forceinline__ uint2 ld_nc_v2(const void *p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__global__ void __launch_bounds__(kMaxHeadsMH * 32)
    attn_heads_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ cache,
                      int64_t cache_rows, const int32_t *__restrict__ idx, int k, int heads,
                      int split_rows, float scale_log2, float *__restrict__ out) {
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ float2 ml_s[kMaxHeadsMH];                         // (max, sum) per head
    __shared__ __align__(16) float o_s[kMaxHeadsMH * kHeadDim];  // unnormalised output
    __shared__ float wts[kMaxHeadsMH][kMaxSplitMH];
    __shared__ float lsum[kMaxHeadsMH];
    __shared__ int32_t rows_s[kIdxChunk];

    const int lane = threadIdx.x & 31, h = threadIdx.x >> 5;
    const int split = blockIdx.x, nsplit = gridDim.x, r = blockIdx.y;
    const int row0 = split * split_rows;
    const int row1 = min(k, row0 + split_rows);
    const int64_t W = (int64_t)heads * 4 * kHeadDim;  // bytes per record
    const int koff = h * 2 * kHeadDim + lane * 8;
    const int voff = (heads + h) * 2 * kHeadDim + lane * 8;

    const uint2 qr = *reinterpret_cast<const uint2 *>(q + (((int64_t)r * heads + h) * kHeadDim + 4 * lane) * 2);
    const float q0 = bf_lo(qr.x), q1 = bf_hi(qr.x), q2 = bf_lo(qr.y), q3 = bf_hi(qr.y);

    float m = -INFINITY, l = 0.f;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    const int32_t *ir = idx + (int64_t)r * k;

    // issue the key and value loads of rows rows_s[b0 .. b0 + kBatch)
    auto load = [&](int b0, int n, uint2 *kv, uint2 *vv, bool *use) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int32_t row = b0 + u < n ? rows_s[b0 + u] : -1;
            use[u] = row >= 0 && (int64_t)row < cache_rows;  // the same for every lane
            kv[u] = make_uint2(0u, 0u);
            vv[u] = make_uint2(0u, 0u);
            if (use[u]) {
                const uint8_t *rec = cache + (int64_t)row * W;
                kv[u] = ld_nc_v2(rec + koff);
                vv[u] = ld_nc_v2(rec + voff);
            }
        }
    };
    // scores, online softmax (base 2) and output update for one batch
    auto consume = [&](const uint2 *kv, const uint2 *vv, const bool *use) {
        float s[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            s[u] = q0 * bf_lo(kv[u].x) + q1 * bf_hi(kv[u].x) + q2 * bf_lo(kv[u].y) +
                   q3 * bf_hi(kv[u].y);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int u = 0; u < kBatch; ++u) s[u] += __shfl_xor_sync(0xFFFFFFFFu, s[u], off);
        float mx = m;
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (use[u]) {
                s[u] *= scale_log2;
                mx = fmaxf(mx, s[u]);
            }
        if (mx != -INFINITY) {  // else nothing in this batch or before it
            const float corr = exp2f(m - mx);
            l *= corr;
            o0 *= corr;
            o1 *= corr;
            o2 *= corr;
            o3 *= corr;
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (use[u]) {
                    const float p = exp2f(s[u] - mx);
                    l += p;
                    o0 += p * bf_lo(vv[u].x);
                    o1 += p * bf_hi(vv[u].x);
                    o2 += p * bf_lo(vv[u].y);
                    o3 += p * bf_hi(vv[u].y);
                }
            m = mx;
        }
    };

    // the rows in chunks of kIdxChunk slot indices staged in shared memory;
    // within a chunk two batches alternate, each one's loads in flight while
    // the other is consumed
    for (int c0 = row0; c0 < row1; c0 += kIdxChunk) {
        const int n = min(kIdxChunk, row1 - c0);
        __syncthreads();  // the previous chunk's indices are no longer read
        for (int i = threadIdx.x; i < n; i += blockDim.x) rows_s[i] = __ldg(ir + c0 + i);
        __syncthreads();
        uint2 ka[kBatch], va[kBatch], kb[kBatch], vb[kBatch];
        bool ua[kBatch], ub[kBatch];
        load(0, n, ka, va, ua);
        for (int b0 = 0; b0 < n; b0 += 2 * kBatch) {
            load(b0 + kBatch, n, kb, vb, ub);
            consume(ka, va, ua);
            load(b0 + 2 * kBatch, n, ka, va, ua);
            consume(kb, vb, ub);
        }
    }
    if (h < heads) {
        *reinterpret_cast<float4 *>(o_s + h * kHeadDim + 4 * lane) = make_float4(o0, o1, o2, o3);
        if (lane == 0) ml_s[h] = make_float2(m, l);
    }
    cluster.sync();  // every split's partial result is visible to the cluster

    // ---- merge: O = sum_c O_c 2^(m_c - M) / L --------------------------
    if (threadIdx.x < heads) {
        const int hh = threadIdx.x;
        float M = -INFINITY;
        float2 mlc[kMaxSplitMH];
#pragma unroll
        for (int c = 0; c < kMaxSplitMH; ++c) {
            mlc[c] = c < nsplit ? cluster.map_shared_rank(ml_s, c)[hh] : make_float2(-INFINITY, 0.f);
            M = fmaxf(M, mlc[c].x);
        }
        float L = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxSplitMH; ++c) {
            const float w = mlc[c].x == -INFINITY ? 0.f : exp2f(mlc[c].x - M);
            wts[hh][c] = w;
            L += mlc[c].y * w;
        }
        lsum[hh] = L;
    }
    __syncthreads();
    const int total = heads * kHeadDim;
    const int per = total / nsplit;  // nsplit is a power of two <= 8
    for (int e = split * per + threadIdx.x; e < (split + 1) * per; e += blockDim.x) {
        const int hh = e / kHeadDim;
        // the splits' values first (remote loads in flight together), then
        // the sum in split order
        float v[kMaxSplitMH];
#pragma unroll
        for (int c = 0; c < kMaxSplitMH; ++c)
            v[c] = c < nsplit ? cluster.map_shared_rank(o_s, c)[e] : 0.f;
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxSplitMH; ++c)
            if (c < nsplit) acc += v[c] * wts[hh][c];
        const float L = lsum[hh];
        out[(int64_t)r * total + e] = L > 0.f ? acc / L : 0.f;
    }
    cluster.sync();  // no CTA leaves while another still reads its shared memory
}

// Splits per request: a power of two up to 8, at least 64 rows each, and no
// more CTAs than two per SM over the whole grid (the register budget of a
// 256-thread CTA allows two), so that the grid is one wave.
int nsplit_heads(int n_req, int k, int sms) {
    int c = 1;
    while (c < kMaxSplitMH && (int64_t)(2 * c) * kMinRowsPerSplit <= k &&
           (int64_t)n_req * 2 * c <= 2 * (int64_t)sms)
        c <<= 1;
    return c;
}

int device_sms() {
    static std::mutex mu;
    static int cached_dev = -1, cached = 0;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev != cached_dev) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached = v;
        cached_dev = dev;
    }
    return cached;
}

}  // namespace

cudaError_t launch_attention_heads(const void *q, const void *cache, int64_t cache_rows,
                                   const int32_t *idx, int n_req, int k, int heads, float scale,
                                   float *out, cudaStream_t st) {
    const int sms = device_sms();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int nsplit = nsplit_heads(n_req, k, sms);
    const int split_rows = (((k + nsplit - 1) / nsplit) + kBatch - 1) / kBatch * kBatch;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nsplit, n_req, 1);
    cfg.blockDim = dim3(heads * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_heads_kernel, static_cast<const uint8_t *>(q),
                              static_cast<const uint8_t *>(cache), cache_rows, idx, k, heads,
                              split_rows, scale * 1.4426950408889634f, out);
}

}  // namespace hs

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
// published rows into C contiguous ranges.  Warp w of a CTA is head w, and
// its two half-warps take every other row: per row a half-warp reads the
// head's 256-byte key block and 256-byte value block with one 16-byte load
// per lane each (eight of the 128 dimensions per lane), forms the score
// with a 16-lane reduction (one shuffle serves both halves' rows) and keeps
// an online softmax (base 2) and its eight output dimensions in registers;
// the two halves are combined at the end.  The slot indices are staged in
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

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
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
    // each half-warp takes every other row: lane (half, hl) holds dimensions
    // [8 hl, 8 hl + 8) of head h for the rows of its half
    const int half = lane >> 4, hl = lane & 15;
    const int koff = h * 2 * kHeadDim + hl * 16;
    const int voff = (heads + h) * 2 * kHeadDim + hl * 16;

    float qf[8];
    {
        const uint4 qr = *reinterpret_cast<const uint4 *>(
            q + (((int64_t)r * heads + h) * kHeadDim + 8 * hl) * 2);
        qf[0] = bf_lo(qr.x); qf[1] = bf_hi(qr.x); qf[2] = bf_lo(qr.y); qf[3] = bf_hi(qr.y);
        qf[4] = bf_lo(qr.z); qf[5] = bf_hi(qr.z); qf[6] = bf_lo(qr.w); qf[7] = bf_hi(qr.w);
    }

    float m = -INFINITY, l = 0.f;  // of this half's rows
    float o[8];
#pragma unroll
    for (int d = 0; d < 8; ++d) o[d] = 0.f;
    const int32_t *ir = idx + (int64_t)r * k;
    constexpr int kPairs = kBatch / 2;  // rows per half in a batch

    // issue the loads of rows rows_s[b0 + 2p + half], p < kPairs
    auto load = [&](int b0, int n, uint4 *kv, uint4 *vv, bool *use) {
#pragma unroll
        for (int p2 = 0; p2 < kPairs; ++p2) {
            const int j = b0 + 2 * p2 + half;
            const int32_t row = j < n ? rows_s[j] : -1;
            use[p2] = row >= 0 && (int64_t)row < cache_rows;  // the same within a half
            kv[p2] = make_uint4(0u, 0u, 0u, 0u);
            vv[p2] = make_uint4(0u, 0u, 0u, 0u);
            if (use[p2]) {
                const uint8_t *rec = cache + (int64_t)row * W;
                kv[p2] = ld_nc_v4(rec + koff);
                vv[p2] = ld_nc_v4(rec + voff);
            }
        }
    };
    // scores (a 16-lane reduction serves both halves' rows), online softmax
    // (base 2) and output update of this half for one batch
    auto consume = [&](const uint4 *kv, const uint4 *vv, const bool *use) {
        float s[kPairs];
#pragma unroll
        for (int p2 = 0; p2 < kPairs; ++p2) {
            const uint4 x = kv[p2];
            s[p2] = qf[0] * bf_lo(x.x) + qf[1] * bf_hi(x.x) + qf[2] * bf_lo(x.y) +
                    qf[3] * bf_hi(x.y) + qf[4] * bf_lo(x.z) + qf[5] * bf_hi(x.z) +
                    qf[6] * bf_lo(x.w) + qf[7] * bf_hi(x.w);
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
#pragma unroll
            for (int p2 = 0; p2 < kPairs; ++p2) s[p2] += __shfl_xor_sync(0xFFFFFFFFu, s[p2], off);
        float mx = m;
#pragma unroll
        for (int p2 = 0; p2 < kPairs; ++p2)
            if (use[p2]) {
                s[p2] *= scale_log2;
                mx = fmaxf(mx, s[p2]);
            }
        if (mx != -INFINITY) {  // else nothing of this half in this batch or before it
            const float corr = exp2f(m - mx);
            l *= corr;
#pragma unroll
            for (int d = 0; d < 8; ++d) o[d] *= corr;
#pragma unroll
            for (int p2 = 0; p2 < kPairs; ++p2)
                if (use[p2]) {
                    const float p = exp2f(s[p2] - mx);
                    const uint4 x = vv[p2];
                    l += p;
                    o[0] += p * bf_lo(x.x);
                    o[1] += p * bf_hi(x.x);
                    o[2] += p * bf_lo(x.y);
                    o[3] += p * bf_hi(x.y);
                    o[4] += p * bf_lo(x.z);
                    o[5] += p * bf_hi(x.z);
                    o[6] += p * bf_lo(x.w);
                    o[7] += p * bf_hi(x.w);
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
        uint4 ka[kPairs], va[kPairs], kb[kPairs], vb[kPairs];
        bool ua[kPairs], ub[kPairs];
        load(0, n, ka, va, ua);
        for (int b0 = 0; b0 < n; b0 += 2 * kBatch) {
            load(b0 + kBatch, n, kb, vb, ub);
            consume(ka, va, ua);
            load(b0 + 2 * kBatch, n, ka, va, ua);
            consume(kb, vb, ub);
        }
    }

    // the two halves' states of each head combined (lane hl and lane hl + 16
    // hold the same dimensions)
    {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, 16);
        const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, 16);
        const float M = fmaxf(m, m2);
        const float w1 = m == -INFINITY ? 0.f : exp2f(m - M);
        const float w2 = m2 == -INFINITY ? 0.f : exp2f(m2 - M);
        // the sums in half order, the same on both halves
        const float a1 = half == 0 ? w1 : w2, a2 = half == 0 ? w2 : w1;
        const float la = half == 0 ? l : l2, lb = half == 0 ? l2 : l;
        const float L = la * a1 + lb * a2;
#pragma unroll
        for (int d = 0; d < 8; ++d) {
            const float other = __shfl_xor_sync(0xFFFFFFFFu, o[d], 16);
            const float oa = half == 0 ? o[d] : other, ob = half == 0 ? other : o[d];
            o[d] = oa * a1 + ob * a2;
        }
        if (half == 0) {
            *reinterpret_cast<float4 *>(o_s + h * kHeadDim + 8 * hl) =
                make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4 *>(o_s + h * kHeadDim + 8 * hl + 4) =
                make_float4(o[4], o[5], o[6], o[7]);
            if (hl == 0) ml_s[h] = make_float2(M, L);
        }
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

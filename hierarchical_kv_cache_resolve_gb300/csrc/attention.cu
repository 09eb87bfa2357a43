// Sparse attention consumer over published slots (decode, MLA records).
//
// The attention backend reads the k records a resolve published for each
// request -- rows of the layer's [R*B][W] cache -- instead of the full
// context ("Inference Systems Infrastructure Notes (6): HiSparse", section 5
// "Why It Is Exact": only the placement of KV records changes; Pith review,
// "What carries the argument": page-table publication to the attention
// backend).  Records are MLA latent vectors of 576 bf16: keys are the whole
// record, values its first 512 elements; every request has `heads` query
// heads of 576 elements.
//
// Flash-decoding split: CTA (chunk, request, head group) gathers up to 128
// published rows into shared memory with cp.async (row by row: the rows are
// scattered over the cache), computes S = Q K^T for 16 heads with warp-level
// bf16 MMAs (fp32 accumulation), a softmax over its keys, O = P V, and writes
// the unnormalised O with its row maximum and sum.  A second kernel merges
// the chunks of every (request, head).  The work is bound by the gathered
// bytes (about 30 flops per byte at 16 heads), so the kernel is built around
// the gather; 16 heads fill exactly the 16 rows of an m16n8k16 MMA.
#include <cstdint>

#include "hs.h"
#include "hs_internal.cuh"

namespace hs {
namespace {

constexpr int kAttnThreads = 128;             // 4 warps
constexpr int kChunk = 128;                   // keys per CTA
constexpr int kGroup = 16;                    // heads per CTA
constexpr int kDimK = 576;                    // key (record) width, bf16
constexpr int kDimV = 512;                    // value width
constexpr int kRowBytes = kDimK * 2;          // 1152
constexpr int kPitch = kRowBytes + 16;        // 1168: eight rows of an ldmatrix
                                              // start on eight different banks
constexpr int kPPitch = kChunk * 2 + 16;      // 272
constexpr int kPart = kDimV + 4;              // O, max, sum, 2 pad: rows of 16n bytes

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kGroup * kPitch;
constexpr uint32_t kOffP = kOffKV + kChunk * kPitch;
constexpr uint32_t kOffRed = kOffP + kGroup * kPPitch;   // [2][4 warps][16] floats
constexpr uint32_t kOffRow = kOffRed + 2 * 4 * kGroup * 4;  // [128] int32 rows (-1 = masked)
constexpr uint32_t kAttnSmem = kOffRow + kChunk * 4;

__device__ __forceinline__ void cp_async16(void *smem, const void *g) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(g) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}

// D = A (16x16 bf16, row) * B (16x8 bf16, col) + D, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t l = __float_as_uint(lo), h = __float_as_uint(hi);
    // round to nearest even (finite inputs: probabilities in [0, 1])
    l = (l + 0x7FFFu + ((l >> 16) & 1u)) >> 16;
    h = (h + 0x7FFFu + ((h >> 16) & 1u)) >> 16;
    return l | (h << 16);
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_partial_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ cache,
                        int64_t cache_rows, const int32_t *__restrict__ idx, int k, int heads,
                        float scale_log2e, float *__restrict__ part) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *q_s = smem + kOffQ;
    uint8_t *kv_s = smem + kOffKV;
    uint8_t *p_s = smem + kOffP;
    float *red_max = reinterpret_cast<float *>(smem + kOffRed);
    float *red_sum = red_max + 4 * kGroup;
    int32_t *rows = reinterpret_cast<int32_t *>(smem + kOffRow);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = blockIdx.x, r = blockIdx.y, hg = blockIdx.z;
    const int nchunk = gridDim.x;
    const int e0 = chunk * kChunk;

    // ---- gather: the 16 query rows and up to 128 published records -------
    if (tid < kChunk) {
        const int e = e0 + tid;
        int32_t row = -1;
        if (e < k) {
            row = idx[(int64_t)r * k + e];
            if (row < 0 || (int64_t)row >= cache_rows) row = -1;  // masked key
        }
        rows[tid] = row;
    }
    const uint8_t *qg = q + ((int64_t)r * heads + (int64_t)hg * kGroup) * kRowBytes;
    for (int c = tid; c < kGroup * (kRowBytes / 16); c += kAttnThreads) {
        const int h = c / (kRowBytes / 16), part16 = c - h * (kRowBytes / 16);
        cp_async16(q_s + h * kPitch + part16 * 16, qg + (int64_t)h * kRowBytes + part16 * 16);
    }
    __syncthreads();
    for (int c = tid; c < kChunk * (kRowBytes / 16); c += kAttnThreads) {
        const int j = c / (kRowBytes / 16), part16 = c - j * (kRowBytes / 16);
        const int32_t row = rows[j];
        uint8_t *dst = kv_s + j * kPitch + part16 * 16;
        if (row >= 0)
            cp_async16(dst, cache + (int64_t)row * kRowBytes + part16 * 16);
        else
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();

    // ---- S = Q K^T: warp w takes keys [32w, 32w + 32), four 8-key tiles ----
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
    {
        const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int acol = (lane >> 4) * 8;
        const int bkey = (lane & 7) + (lane >> 4) * 8;
        const int bcol = ((lane >> 3) & 1) * 8;
#pragma unroll 4
        for (int ks = 0; ks < kDimK / 16; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, q_s + arow * kPitch + (ks * 16 + acol) * 2);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t b[4];
                const int key = warp * 32 + np * 16 + bkey;
                ldsm_x4(b, kv_s + key * kPitch + (ks * 16 + bcol) * 2);
                mma_bf16(s[2 * np], a, b[0], b[1]);
                mma_bf16(s[2 * np + 1], a, b[2], b[3]);
            }
        }
    }

    // ---- softmax over the CTA's keys, per head (base-2 exponent) ----------
    const int h0 = lane >> 2, h1 = h0 + 8;
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int key = warp * 32 + nt * 8 + (lane & 3) * 2;
        const bool v0 = rows[key] >= 0, v1 = rows[key + 1] >= 0;
        s[nt][0] = v0 ? s[nt][0] * scale_log2e : -INFINITY;
        s[nt][1] = v1 ? s[nt][1] * scale_log2e : -INFINITY;
        s[nt][2] = v0 ? s[nt][2] * scale_log2e : -INFINITY;
        s[nt][3] = v1 ? s[nt][3] * scale_log2e : -INFINITY;
        m0 = fmaxf(m0, fmaxf(s[nt][0], s[nt][1]));
        m1 = fmaxf(m1, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, o));
    }
    if ((lane & 3) == 0) {
        red_max[warp * kGroup + h0] = m0;
        red_max[warp * kGroup + h1] = m1;
    }
    __syncthreads();
    m0 = fmaxf(fmaxf(red_max[h0], red_max[kGroup + h0]),
               fmaxf(red_max[2 * kGroup + h0], red_max[3 * kGroup + h0]));
    m1 = fmaxf(fmaxf(red_max[h1], red_max[kGroup + h1]),
               fmaxf(red_max[2 * kGroup + h1], red_max[3 * kGroup + h1]));
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int key = warp * 32 + nt * 8 + (lane & 3) * 2;
        const float p00 = m0 == -INFINITY ? 0.f : exp2f(s[nt][0] - m0);
        const float p01 = m0 == -INFINITY ? 0.f : exp2f(s[nt][1] - m0);
        const float p10 = m1 == -INFINITY ? 0.f : exp2f(s[nt][2] - m1);
        const float p11 = m1 == -INFINITY ? 0.f : exp2f(s[nt][3] - m1);
        l0 += p00 + p01;
        l1 += p10 + p11;
        *reinterpret_cast<uint32_t *>(p_s + h0 * kPPitch + key * 2) = pack_bf16(p00, p01);
        *reinterpret_cast<uint32_t *>(p_s + h1 * kPPitch + key * 2) = pack_bf16(p10, p11);
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, o);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
    }
    if ((lane & 3) == 0) {
        red_sum[warp * kGroup + h0] = l0;
        red_sum[warp * kGroup + h1] = l1;
    }
    __syncthreads();

    // ---- O = P V: warp w takes value columns [128w, 128w + 128) -----------
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;
    {
        const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int acol = (lane >> 4) * 8;
        const int bkey = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int bcol = (lane >> 4) * 8;
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, p_s + arow * kPPitch + (ks * 16 + acol) * 2);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t b[4];
                const int d0 = warp * 128 + np * 16;
                ldsm_x4_t(b, kv_s + (ks * 16 + bkey) * kPitch + (d0 + bcol) * 2);
                mma_bf16(o[2 * np], a, b[0], b[1]);
                mma_bf16(o[2 * np + 1], a, b[2], b[3]);
            }
        }
    }

    // ---- partial results: O (unnormalised), max and sum per head ----------
    float *base = part + (((int64_t)r * nchunk + chunk) * heads + (int64_t)hg * kGroup) * kPart;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
        const int d = warp * 128 + nt * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2 *>(base + (int64_t)h0 * kPart + d) = make_float2(o[nt][0], o[nt][1]);
        *reinterpret_cast<float2 *>(base + (int64_t)h1 * kPart + d) = make_float2(o[nt][2], o[nt][3]);
    }
    if (tid < kGroup) {
        const float l = red_sum[tid] + red_sum[kGroup + tid] + red_sum[2 * kGroup + tid] +
                        red_sum[3 * kGroup + tid];
        const float m = fmaxf(fmaxf(red_max[tid], red_max[kGroup + tid]),
                              fmaxf(red_max[2 * kGroup + tid], red_max[3 * kGroup + tid]));
        base[(int64_t)tid * kPart + kDimV] = m;
        base[(int64_t)tid * kPart + kDimV + 1] = l;
    }
}

// Merges the chunks of one (request, head): O = sum_c O_c 2^(m_c - M) / L.
__global__ void __launch_bounds__(kAttnThreads)
    attn_combine_kernel(const float *__restrict__ part, int nchunk, int heads,
                        float *__restrict__ out) {
    const int rh = blockIdx.x;  // r * heads + h
    const int r = rh / heads, h = rh - r * heads;
    float M = -INFINITY;
    for (int c = 0; c < nchunk; ++c)
        M = fmaxf(M, part[(((int64_t)r * nchunk + c) * heads + h) * kPart + kDimV]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float L = 0.f;
    for (int c = 0; c < nchunk; ++c) {
        const float *pc = part + (((int64_t)r * nchunk + c) * heads + h) * kPart;
        const float mc = pc[kDimV];
        const float wgt = mc == -INFINITY ? 0.f : exp2f(mc - M);
        L += pc[kDimV + 1] * wgt;
        const float4 v = *reinterpret_cast<const float4 *>(pc + threadIdx.x * 4);
        acc[0] += v.x * wgt;
        acc[1] += v.y * wgt;
        acc[2] += v.z * wgt;
        acc[3] += v.w * wgt;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<float4 *>(out + (int64_t)rh * kDimV + threadIdx.x * 4) =
        make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
}

}  // namespace

size_t attention_workspace_bytes(int n_req, int k, int heads) {
    const int nchunk = (k + kChunk - 1) / kChunk;
    return (size_t)n_req * nchunk * heads * kPart * sizeof(float);
}

cudaError_t launch_attention(const void *q, const void *cache, int64_t cache_rows,
                             const int32_t *idx, int n_req, int k, int heads, float scale,
                             void *work, float *out, cudaStream_t st) {
    static_assert(kPart % 4 == 0, "partial rows stay 16-byte aligned (float4 reads)");
    static_assert(kDimV == 4 * kAttnThreads, "one float4 per combine thread");
    cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttnSmem);
    if (e != cudaSuccess) return e;
    const int nchunk = (k + kChunk - 1) / kChunk;
    const float scale_log2e = scale * 1.4426950408889634f;
    attn_partial_kernel<<<dim3(nchunk, n_req, heads / kGroup), kAttnThreads, kAttnSmem, st>>>(
        static_cast<const uint8_t *>(q), static_cast<const uint8_t *>(cache), cache_rows, idx, k,
        heads, scale_log2e, static_cast<float *>(work));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attn_combine_kernel<<<n_req * heads, kAttnThreads, 0, st>>>(static_cast<const float *>(work),
                                                                 nchunk, heads, out);
    return cudaGetLastError();
}

}  // namespace hs

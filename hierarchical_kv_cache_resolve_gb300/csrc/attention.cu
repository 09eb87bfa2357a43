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
// Flash-decoding split over a gather pipeline, merged inside a thread-block
// cluster: the C CTAs of a cluster share one request and 16 of its query
// heads, each owning a contiguous range of the request's k published rows.
//
// Gather.  In every CTA two producer warps move its rows 32 at a time into
// a two-stage shared-memory ring, 16 rows each, one bulk copy per row (the
// TMA engine; completion counted in bytes on the stage's mbarrier).  The
// rows are scattered over the cache, so there is no tile to describe.  The
// slot indices are read two stages ahead.  (A warp takes about a
// microsecond to have 32 row copies accepted, so two warps issue faster
// than one; 16-byte cp.async copies from a producer's lanes were measured
// slower, alone and beside the bulk copies.)
//
// Compute.  Four consumer warps form, per stage, S = Q K^T with warp-level
// bf16 MMAs (fp32 accumulation; each warp holds a quarter of the 576 query
// columns in registers and the four partial S tiles are summed through
// shared memory), an online softmax, and O += P V with P kept in registers.
//
// Merge.  The C partial results (unnormalised O, row maximum and sum) are
// merged through distributed shared memory, each CTA producing 512/C of
// the value columns, in a fixed order.
//
// The work is bound by the gathered bytes (about 30 flops per byte at 16
// heads), so the kernel is built around keeping the gather busy: two CTAs
// per SM, and a split count chosen so that the grid covers the GPU once.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include <cooperative_groups.h>

#include "hs.h"
#include "hs_internal.cuh"

namespace hs {
namespace {

namespace cg = cooperative_groups;

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarps = 2;               // each moves half of a stage's rows
constexpr int kAttnThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kStageKeys = 32;                // rows per pipeline stage
constexpr int kStages = 2;
constexpr int kMinSplitKeys = kStages * kStageKeys;
constexpr int kGroup = 16;                    // heads per CTA
constexpr int kDimK = 576;                    // key (record) width, bf16
constexpr int kDimV = 512;                    // value width
constexpr int kRowBytes = kDimK * 2;          // 1152
constexpr int kPitch = kRowBytes + 16;        // 1168: eight rows of an ldmatrix
                                              // start on eight different banks
constexpr int kKStepsPerWarp = kDimK / 16 / kConsumerWarps;  // 9
constexpr int kMaxCluster = 16;               // splits of one (request, head group)
constexpr int kOPitch = kDimV + 8;            // floats per row of a staged partial O
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: a bulk copy never takes that long

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kGroup * kPitch;
constexpr uint32_t kOffRed = kOffKV + kStages * kStageKeys * kPitch;
constexpr uint32_t kRedBytes = kConsumerWarps * 32 * 16 * 4;  // four partial S tiles
constexpr uint32_t kOffMask = kOffRed + 2 * kRedBytes;         // [2][kStages] half-stage masks
constexpr uint32_t kOffBar = kOffMask + 16;                    // full[2], empty[2], q
constexpr uint32_t kAttnSmem = kOffBar + 8 * (2 * kStages + 1);
static_assert(kStageKeys == 32, "one producer lane per row, one mask word per stage");
static_assert(kKStepsPerWarp * 16 * kConsumerWarps == kDimK, "query columns split evenly");
static_assert(kOffKV % 16 == 0 && kPitch % 16 == 0, "bulk copies land on 16-byte boundaries");
static_assert(kOffBar % 8 == 0, "mbarriers are 8-byte aligned");
static_assert(2 * (kAttnSmem + 1024) <= 233472, "two CTAs per SM");
// after the main loop: partial O [16][kOPitch] floats in the ring, max and
// sum per head, then the merge weights, in the S-reduction area
constexpr uint32_t kOffML = kOffRed;                              // [16] float2
constexpr uint32_t kOffAll = kOffML + kGroup * 8;                 // [kMaxCluster][16] float2
constexpr uint32_t kOffWts = kOffAll + kMaxCluster * kGroup * 8;  // [16][kMaxCluster]
constexpr uint32_t kOffLinv = kOffWts + kGroup * kMaxCluster * 4;  // [16]
static_assert(kGroup * kOPitch * 4 <= kStages * kStageKeys * kPitch, "partial O fits the ring");
static_assert(kOffLinv + kGroup * 4 <= kOffRed + 2 * kRedBytes, "merge scratch fits");

// Source of masked rows: finite zeros, so that P V never meets stale bytes.
__device__ __align__(128) uint8_t g_zero_row[kRowBytes];
// Bit 0: a pipeline wait ran out of time (the affected outputs are NaN).
__device__ uint32_t g_attn_status;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity; false after the limit.
// Inlined: a call would make the caller settle its loads in flight first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    return true;
}

// One row from global memory into this CTA's shared memory (TMA engine).
__device__ __forceinline__ void bulk_row(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Barrier 1 over the consumer warps with an AND of `v`: every consumer
// leaves with the same verdict, so none is left waiting at the next barrier.
__device__ __forceinline__ bool consumers_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kConsumerWarps * 32)
        : "memory");
    return r != 0;
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

// Cluster (request r, heads [16g, 16g + 16)); CTA `split` of it takes keys
// [split * split_keys, min(k, (split + 1) * split_keys)).
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ cache,
                int64_t cache_rows, const int32_t *__restrict__ idx, int k, int heads,
                int split_keys, float scale_log2e, float *__restrict__ out) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *q_s = smem + kOffQ;
    uint8_t *kv_s = smem + kOffKV;
    float4 *red = reinterpret_cast<float4 *>(smem + kOffRed);
    uint32_t *maskw = reinterpret_cast<uint32_t *>(smem + kOffMask);
    const uint32_t bar0 = smem_addr(smem + kOffBar);
    auto full_bar = [&](int b) { return bar0 + 8u * b; };
    auto empty_bar = [&](int b) { return bar0 + 8u * (kStages + b); };
    const uint32_t q_bar = bar0 + 8u * (2 * kStages);
    cg::cluster_group cluster = cg::this_cluster();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, nsplit = gridDim.x, r = blockIdx.y, g = blockIdx.z;
    const int key0 = split * split_keys;
    const int key1 = min(k, key0 + split_keys);
    // the last splits of a short request may be empty (they merge as zero)
    const int nstage = key1 > key0 ? (key1 - key0 + kStageKeys - 1) / kStageKeys : 0;

    if (tid == 0) {
        for (int b = 0; b < kStages; ++b) {
            mbar_init(full_bar(b), kProducerWarps);  // one arrival (with bytes) per producer
            mbar_init(empty_bar(b), kConsumerWarps);
        }
        mbar_init(q_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    bool ok = true;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;
    const int h0 = lane >> 2;  // C fragment rows h0 and h0 + 8

    if (warp >= kConsumerWarps) {
        // ---------------- producers: rows [16p, 16p + 16) of every stage ----
        const int p_id = warp - kConsumerWarps;
        constexpr int kHalf = kStageKeys / kProducerWarps;
        // the raw slot index of row `lane` of this warp's half of stage st
        // (-1 past the split); it is checked only when used, so the load
        // stays in flight
        auto load_row = [&](int st) {
            const int key = key0 + st * kStageKeys + p_id * kHalf + lane;
            int32_t row = -1;
            if (lane < kHalf && st < nstage && key < key1)
                row = __ldg(idx + (int64_t)r * k + key);
            return row;
        };
        // Slot indices are read kStages stages ahead, each into the register
        // its stage will use: the loop is unrolled by kStages so that no
        // register holding a load in flight is ever copied (a copy would wait
        // for the load).
        int32_t rows[kStages];
#pragma unroll
        for (int j = 0; j < kStages; ++j) rows[j] = load_row(j);
        if (p_id == 0) {
            if (lane == 0) mbar_arrive_expect_tx(q_bar, kGroup * kRowBytes);
            __syncwarp();
            if (lane < kGroup)
                bulk_row(smem_addr(q_s + lane * kPitch),
                         q + ((int64_t)r * heads + (int64_t)g * kGroup + lane) * kRowBytes,
                         kRowBytes, q_bar);
        }
        int issued = 0;
        for (int st0 = 0; st0 < nstage && ok; st0 += kStages) {
#pragma unroll
            for (int b = 0; b < kStages; ++b) {
                const int st = st0 + b;
                if (st >= nstage) break;
                if (st >= kStages) {
                    // the consumers released this buffer's previous stage
                    const bool free_ok = mbar_wait(empty_bar(b), ((st / kStages) - 1) & 1);
                    if (!__all_sync(0xFFFFFFFFu, free_ok)) {
                        ok = false;
                        break;
                    }
                }
                const int32_t raw = rows[b];
                rows[b] = load_row(st + kStages);  // in flight for kStages stages
                const bool use = raw >= 0 && (int64_t)raw < cache_rows;  // else a masked key
                const uint32_t valid = __ballot_sync(0xFFFFFFFFu, use);  // lanes >= 16: 0
                if (lane == 0) {
                    maskw[p_id * kStages + b] = valid;
                    mbar_arrive_expect_tx(full_bar(b), kHalf * kRowBytes);
                }
                __syncwarp();
                if (lane < kHalf) {
                    const void *src = use
                                          ? static_cast<const void *>(cache + (int64_t)raw * kRowBytes)
                                          : static_cast<const void *>(g_zero_row);
                    bulk_row(smem_addr(kv_s + (b * kStageKeys + p_id * kHalf + lane) * kPitch), src,
                             kRowBytes, full_bar(b));
                }
                issued = st + 1;
            }
        }
        // copies still in flight must land before the ring is reused or the
        // CTA exits: in a normal run the consumers have already waited for
        // them and this returns at once
        for (int st = max(0, issued - kStages); st < issued; ++st)
            if (!mbar_wait(full_bar(st % kStages), (st / kStages) & 1)) ok = false;
        if (p_id == 0 && !mbar_wait(q_bar, 0)) ok = false;
    } else {
        // ---------------- consumers ----------------
        ok = consumers_all(mbar_wait(q_bar, 0));
        // this warp's quarter of the query columns, as MMA A fragments
        uint32_t qa[kKStepsPerWarp][4];
        {
            const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int acol = (lane >> 4) * 8;
#pragma unroll
            for (int i = 0; i < kKStepsPerWarp; ++i)
                ldsm_x4(qa[i], q_s + arow * kPitch + ((warp * kKStepsPerWarp + i) * 16 + acol) * 2);
        }
        const int bkey = (lane & 7) + (lane >> 4) * 8;        // K rows (non-transposed loads)
        const int bcol = ((lane >> 3) & 1) * 8;
        const int vkey = (lane & 7) + ((lane >> 3) & 1) * 8;  // V rows (transposed loads)
        const int vcol = (lane >> 4) * 8;

        for (int st = 0; st < nstage && ok; ++st) {
            const int b = st % kStages;
            // on a timeout the stage is computed from whatever the buffer holds
            // (shared-memory reads only) and dropped at the barrier below
            const bool landed = mbar_wait(full_bar(b), (st / kStages) & 1);
            const uint8_t *kv = kv_s + b * kStageKeys * kPitch;

            // partial S over this warp's query columns: 16 heads x 32 keys
            float s[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
#pragma unroll
            for (int i = 0; i < kKStepsPerWarp; ++i) {
                const int col = (warp * kKStepsPerWarp + i) * 16 + bcol;
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bf[4];
                    ldsm_x4(bf, kv + (np * 16 + bkey) * kPitch + col * 2);
                    mma_bf16(s[2 * np], qa[i], bf[0], bf[1]);
                    mma_bf16(s[2 * np + 1], qa[i], bf[2], bf[3]);
                }
            }
            // sum the four warps' partial tiles (fixed order: every warp gets
            // the same S); buffers alternate by stage, so one barrier per
            // stage suffices
            float4 *rb = red + (st & 1) * (kRedBytes / 16);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                rb[(warp * 4 + nt) * 32 + lane] = make_float4(s[nt][0], s[nt][1], s[nt][2], s[nt][3]);
            if (!consumers_all(landed)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                float4 acc = rb[nt * 32 + lane];
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w) {
                    const float4 v = rb[(w * 4 + nt) * 32 + lane];
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                s[nt][0] = acc.x;
                s[nt][1] = acc.y;
                s[nt][2] = acc.z;
                s[nt][3] = acc.w;
            }

            // online softmax (base 2) over this stage's keys
            const uint32_t valid = maskw[b] | (maskw[kStages + b] << (kStageKeys / kProducerWarps));
            float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int key = nt * 8 + (lane & 3) * 2;
                const bool v0 = (valid >> key) & 1u, v1 = (valid >> (key + 1)) & 1u;
                s[nt][0] = v0 ? s[nt][0] * scale_log2e : -INFINITY;
                s[nt][1] = v1 ? s[nt][1] * scale_log2e : -INFINITY;
                s[nt][2] = v0 ? s[nt][2] * scale_log2e : -INFINITY;
                s[nt][3] = v1 ? s[nt][3] * scale_log2e : -INFINITY;
                x0 = fmaxf(x0, fmaxf(s[nt][0], s[nt][1]));
                x1 = fmaxf(x1, fmaxf(s[nt][2], s[nt][3]));
            }
#pragma unroll
            for (int d = 1; d <= 2; d <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(0xFFFFFFFFu, x0, d));
                x1 = fmaxf(x1, __shfl_xor_sync(0xFFFFFFFFu, x1, d));
            }
            const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
            const float a0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0);
            const float a1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
            m0 = n0;
            m1 = n1;
            uint32_t pa[2][4];
            float t0 = 0.f, t1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const float p00 = n0 == -INFINITY ? 0.f : exp2f(s[nt][0] - n0);
                const float p01 = n0 == -INFINITY ? 0.f : exp2f(s[nt][1] - n0);
                const float p10 = n1 == -INFINITY ? 0.f : exp2f(s[nt][2] - n1);
                const float p11 = n1 == -INFINITY ? 0.f : exp2f(s[nt][3] - n1);
                t0 += p00 + p01;
                t1 += p10 + p11;
                // the C fragment of keys [8nt, 8nt + 8) is half an A fragment of P
                pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p00, p01);
                pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p10, p11);
            }
            l0 = l0 * a0 + t0;
            l1 = l1 * a1 + t1;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                o[nt][0] *= a0;
                o[nt][1] *= a0;
                o[nt][2] *= a1;
                o[nt][3] *= a1;
            }

            // O += P V over this warp's 128 value columns
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t bf[4];
                    ldsm_x4_t(bf, kv + (kk * 16 + vkey) * kPitch + (warp * 128 + np * 16 + vcol) * 2);
                    mma_bf16(o[2 * np], pa[kk], bf[0], bf[1]);
                    mma_bf16(o[2 * np + 1], pa[kk], bf[2], bf[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(b));
        }
#pragma unroll
        for (int d = 1; d <= 2; d <<= 1) {
            l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, d);
            l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, d);
        }
    }
    if (!ok && lane == 0) atomicOr(&g_attn_status, 1u);

    // ---- stage this split's partial result in the (now idle) ring --------
    float *o_s = reinterpret_cast<float *>(kv_s);
    float2 *ml_s = reinterpret_cast<float2 *>(smem + kOffML);
    const int failed = __syncthreads_or(!ok);  // also: every warp is past the ring
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int d = warp * 128 + nt * 8 + (lane & 3) * 2;
            *reinterpret_cast<float2 *>(o_s + h0 * kOPitch + d) = make_float2(o[nt][0], o[nt][1]);
            *reinterpret_cast<float2 *>(o_s + (h0 + 8) * kOPitch + d) =
                make_float2(o[nt][2], o[nt][3]);
        }
        if (warp == 0 && (lane & 3) == 0) {
            const float nan = __int_as_float(0x7FC00000);  // NaN marks a failed split
            ml_s[h0] = make_float2(failed ? nan : m0, l0);
            ml_s[h0 + 8] = make_float2(failed ? nan : m1, l1);
        }
    }
    cluster.sync();  // every split's partial result is visible to the cluster

    // ---- merge: O = sum_c O_c 2^(m_c - M) / L, value columns of this CTA --
    float2 *ml_all = reinterpret_cast<float2 *>(smem + kOffAll);
    float *wts = reinterpret_cast<float *>(smem + kOffWts);
    float *linv = reinterpret_cast<float *>(smem + kOffLinv);
    // every split's (max, sum) per head, one remote load per thread
    for (int i = tid; i < nsplit * kGroup; i += kAttnThreads)
        ml_all[i] = cluster.map_shared_rank(ml_s, i / kGroup)[i % kGroup];
    __syncthreads();
    if (tid < kGroup) {
        const int h = tid;
        float M = -INFINITY;
        bool bad = false;
        for (int c = 0; c < nsplit; ++c) {
            const float mc = ml_all[c * kGroup + h].x;
            bad |= mc != mc;
            M = fmaxf(M, mc);
        }
        float L = 0.f;
        for (int c = 0; c < nsplit; ++c) {
            const float2 mlc = ml_all[c * kGroup + h];
            const float w = mlc.x == -INFINITY ? 0.f : exp2f(mlc.x - M);
            wts[h * kMaxCluster + c] = w;
            L += mlc.y * w;
        }
        linv[h] = bad ? __int_as_float(0x7FC00000) : L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    const int cols = kDimV / nsplit;  // nsplit is a power of two <= 16
    const int per_row = cols / 4;
    for (int it = tid; it < kGroup * per_row; it += kAttnThreads) {
        const int h = it / per_row;
        const int d = split * cols + (it - h * per_row) * 4;
        // all the splits' values first (remote loads in flight together), then
        // the sum in split order
        float4 v[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < nsplit)
                v[c] = *reinterpret_cast<const float4 *>(cluster.map_shared_rank(o_s, c) +
                                                         h * kOPitch + d);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < nsplit) {
                const float w = wts[h * kMaxCluster + c];
                acc.x += v[c].x * w;
                acc.y += v[c].y * w;
                acc.z += v[c].z * w;
                acc.w += v[c].w * w;
            }
        const float li = linv[h];
        *reinterpret_cast<float4 *>(out + ((int64_t)r * heads + (int64_t)g * kGroup + h) * kDimV + d) =
            make_float4(acc.x * li, acc.y * li, acc.z * li, acc.w * li);
    }
    cluster.sync();  // no CTA leaves while another still reads its shared memory
}

struct DeviceInfo {
    int dev = -1, sms = 0;
    int active[5] = {0, 0, 0, 0, 0};  // co-resident clusters of 1, 2, 4, 8, 16 CTAs
};

// Splits per (request, head group) -- the cluster size: a power of two, no
// more than ceil(k / 64), and the largest whose clusters for all the units
// are co-resident (one wave), never more CTAs than two per SM.
int nsplit_for(int n_req, int k, int heads, const DeviceInfo &di) {
    const int64_t units = (int64_t)n_req * (heads / kGroup);
    const int max_split = (k + kMinSplitKeys - 1) / kMinSplitKeys;
    int n = 1;
    for (int e = 1; e < 5; ++e) {
        const int c = 1 << e;
        if (c > max_split || units * c > 2 * (int64_t)di.sms || units > di.active[e]) break;
        n = c;
    }
    return n;
}

// Per-device set-up, once: shared-memory size and carve-out, and how many
// clusters of each size the device keeps co-resident (16-CTA clusters where
// non-portable sizes are allowed).
cudaError_t device_info(DeviceInfo *out) {
    static std::mutex mu;
    static DeviceInfo cached;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != cached.dev) {
        DeviceInfo d;
        d.dev = dev;
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kAttnSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        const bool big = cudaFuncSetAttribute(
                             attn_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                         cudaSuccess;
        for (int e = 0; e < 5; ++e) {
            const int c = 1 << e;
            if (c > 8 && !big) break;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(c, 1, 1);
            cfg.blockDim = dim3(kAttnThreads);
            cfg.dynamicSmemBytes = kAttnSmem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, attn_kernel, &cfg) != cudaSuccess) break;
            d.active[e] = clusters;
        }
        (void)cudaGetLastError();  // a refused query above leaves no sticky error
        cached = d;
    }
    *out = cached;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_attention(const void *q, const void *cache, int64_t cache_rows,
                             const int32_t *idx, int n_req, int k, int heads, float scale,
                             float *out, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int nsplit = nsplit_for(n_req, k, heads, di);
    const int stages = (k + kStageKeys - 1) / kStageKeys;
    const int split_keys = ((stages + nsplit - 1) / nsplit) * kStageKeys;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nsplit, n_req, heads / kGroup);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = kAttnSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel, static_cast<const uint8_t *>(q),
                              static_cast<const uint8_t *>(cache), cache_rows, idx, k, heads,
                              split_keys, scale * 1.4426950408889634f, out);
}

cudaError_t attention_status(uint32_t *status) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(v));
    if (e != cudaSuccess) return e;
    *status = v;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace hs

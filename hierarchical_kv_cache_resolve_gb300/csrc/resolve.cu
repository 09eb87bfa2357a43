// RESOLVE: one fused launch per sparse layer (HiSparse; "Inference Systems
// Infrastructure Notes (6): HiSparse", section 3 "RESOLVE: Five Stages in One
// Launch"; Pith review of arXiv 2608.07009, "What carries the argument").
//
// Grid: one thread-block cluster per request (n_req * C CTAs of kThreads).
//
// CTA 0 of a cluster (the leader) owns the request's metadata:
//   P0  cp.async the k selections, the slot map and the LRU order into shared
//       memory, zero the hash table and the position bitmap;
//   P1  reject positions outside [0, L), repeated positions and corrupt
//       metadata; insert every selection into a shared-memory open-addressing
//       table (32-bit key = position + 1, 16-bit selection index beside it,
//       at most a quarter full) and set its bit in the position bitmap;
//   P2  probe every slot's position: no bit means not selected, otherwise
//       the table gives the selection index the slot is a hit for;
//   P3  one warp-ballot scan over the selections (misses in selection order)
//       and one over the LRU order (non-hit slots in (stamp, slot) order):
//       the j-th miss gets the j-th non-hit slot as its victim;
//   P4  publish slots, update page table / slot map / stamps, and rebuild
//       the LRU order with a third ballot scan over the slots.
//
// CTAs 1..C-1 (the followers) move the data.  Follower f owns a contiguous
// share of the selection indices.  Before the leader has decided anything
// each warp predicts which of its selections miss from the page table (a
// position with no slot will miss) and stages those records from the mapped
// host pool into the CTA's staging pool (shared memory, slots taken with an
// atomic) with cp.async, so that the host-link transfer overlaps the
// leader's P0-P3.  After the cluster barrier it reads
// the leader's verdict through distributed shared memory: each staged record
// goes to its victim slot with one bulk (TMA) copy, or is dropped if the
// leader found a hit, and any miss of its share that was not staged is
// fetched with 16-byte non-coherent loads, so the leader's decision is
// always the one applied.  The leader commits the metadata (P4) while the
// followers store.  A cluster of one CTA does all of it in the leader, fetch
// after P3.  A resolve that consumes a prefetch plan uses the leader's fetch
// list instead of the prediction.
//
// Consecutive launches overlap: a plain resolve allows the next launch as
// soon as it starts, and does P0-P3 and the followers' staging before the
// previous grid has completed; it writes nothing to global memory before
// then and keeps its decision only if its inputs are unchanged once that
// grid has completed (the pair's resolve counter, written last by every
// commit, the request id and the selection), deciding again otherwise.
//
// Victim selection without sorting: the LRU order array is kept sorted by
// (stamp, slot).  A resolve at step t keeps the untouched slots in their old
// relative order and appends the victims (stamp 2t-1) and then the hits
// (stamp 2t), each group in slot order -- exactly the (stamp, slot) order of
// the new stamps -- so the victims are always the first m non-hit entries.
#include <mutex>

#include <cooperative_groups.h>

#include "hs.h"
#include "hs_internal.cuh"

namespace cg = cooperative_groups;

namespace hs {
namespace {

constexpr int kUnroll = 8;  // 16-byte loads in flight per thread in the fetch

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t r;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// Arrival that publishes nothing: it does not wait for this thread's
// outstanding memory operations (a follower's in-flight host loads).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16-byte read-only load that bypasses L1 allocation: used on the mapped
// host pool, which no kernel writes.
__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *g) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(g) : "memory");
}

__device__ __forceinline__ void cp_async4(void *smem, const void *g) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(g) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Issues an asynchronous global -> shared copy of nbytes (by the whole CTA):
// 16-byte pieces while both sides are 16-byte aligned, 4-byte pieces after
// that, plain 2-byte loads for what is left.  Completed by cp_async_wait_all
// and a barrier.
__device__ __forceinline__ void copy_to_smem(void *dst, const void *src, int nbytes) {
    uint8_t *d = static_cast<uint8_t *>(dst);
    const uint8_t *s = static_cast<const uint8_t *>(src);
    int done = 0;
    if (((reinterpret_cast<uintptr_t>(d) | reinterpret_cast<uintptr_t>(s)) & 15u) == 0) {
        const int n16 = nbytes >> 4;
        for (int i = threadIdx.x; i < n16; i += kThreads) cp_async16(d + 16 * i, s + 16 * i);
        done = n16 << 4;
    }
    if (((reinterpret_cast<uintptr_t>(d + done) | reinterpret_cast<uintptr_t>(s + done)) & 3u) == 0) {
        const int n4 = (nbytes - done) >> 2;
        for (int i = threadIdx.x; i < n4; i += kThreads)
            cp_async4(d + done + 4 * i, s + done + 4 * i);
        done += n4 << 2;
    }
    // what is left is made of 2-byte elements (u16 arrays of odd length)
    for (int i = done / 2 + threadIdx.x; i < nbytes / 2; i += kThreads)
        reinterpret_cast<uint16_t *>(d)[i] = reinterpret_cast<const uint16_t *>(s)[i];
}

// Orders this thread's generic-proxy writes to shared memory (cp.async
// included) before later async-proxy (bulk copy) reads of it.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk (TMA engine) copy of `bytes` (a multiple of 16, both ends 16-byte
// aligned) from shared memory to global memory, tracked by bulk groups.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, int bytes) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(ssrc);
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(s),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until the committed bulk copies have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Acquire load / release store of a u32 in global memory at GPU scope.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *a) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t *a, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// Programmatic dependent launch: wait for the grids this one depends on to
// complete (and their writes to be visible), then let the next grid in the
// stream start launching.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t r;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}

// A follower CTA's shared memory after the header, staging records into
// whatever the launch provides beyond its lists (see follower_lists_end).
__device__ __forceinline__ FollowerLayout follower_layout(int k, int W) {
    FollowerLayout f = follower_lists(k);
    const uint32_t total = dynamic_smem_bytes();
    const int cap = total > f.stage ? (int)((total - f.stage) / (uint32_t)W) : 0;
    f.cap = cap < kStageCap ? cap : kStageCap;
    return f;
}

// Multiplicative (Fibonacci) hashing: the top bits of pos * 2^32/phi.
__device__ __forceinline__ uint32_t hash_slot(int32_t pos, int shift) {
    return ((uint32_t)pos * 2654435761u) >> shift;
}

// Bit of `pos` in the membership bitmap: the position itself when the
// bitmap covers [0, L), otherwise a second multiplicative hash.
__device__ __forceinline__ uint32_t member_bit(int32_t pos, bool exact, int mshift) {
    return exact ? (uint32_t)pos : ((uint32_t)pos * 0x85EBCA77u) >> mshift;
}

// Copies F records: fetch-list entry j moves host_pair[fp[j]] to
// cache_pair[fs[j]] (entries with fs[j] < 0 are skipped).  The 16-byte
// chunks (entry, part) are spread over G threads; each thread keeps kUnroll
// loads in flight before storing.  `q_begin` skips chunks already done.
__device__ __forceinline__ void fetch_records(const uint8_t *__restrict__ host_pair,
                                              uint8_t *__restrict__ cache_pair,
                                              const int32_t *fp, const int32_t *fs, int F,
                                              int W, int g, int G, int q_begin = 0) {
    const int CW = W >> 4;
    const int Q = F * CW;
    for (int q0 = q_begin + g; q0 < Q; q0 += G * kUnroll) {
        uint4 v[kUnroll];
        int64_t doff[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int q = q0 + u * G;
            doff[u] = -1;
            if (q < Q) {
                const int j = q / CW;
                const int part = q - j * CW;
                const int32_t slot = fs[j];
                if (slot >= 0) {
                    v[u] = ld_nc_v4(host_pair + (int64_t)fp[j] * W + part * 16);
                    doff[u] = (int64_t)slot * W + part * 16;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (doff[u] >= 0) *reinterpret_cast<uint4 *>(cache_pair + doff[u]) = v[u];
    }
}

// Exclusive scan of one packed u32 per warp (two 16-bit counts side by side)
// across the CTA; returns this warp's base and leaves the total in *total.
__device__ __forceinline__ uint32_t warp_counts_exscan(uint32_t mine, uint32_t *sums,
                                                       uint32_t *total) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sums[w] = mine;
    __syncthreads();
    if (w == 0) {
        const uint32_t v = lane < kWarps ? sums[lane] : 0u;
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane < kWarps) sums[lane] = x - v;
        if (lane == kWarps - 1) sums[kWarps] = x;
    }
    __syncthreads();
    const uint32_t base = sums[w];
    *total = sums[kWarps];
    __syncthreads();
    return base;
}

// Stage timestamps (%globaltimer, ns) of the measurement variant: thread 0
// of every CTA writes times[(request * kMaxCluster + cta) * kStampSlots + s].
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// kMode: kModeResolve (hs_resolve), kModePlan (hs_prefetch_plan: read-only
// decision, plan written) or kModeNoFetch (the resolve without the miss
// fetch: every metadata step, no slot written; measurement only).
// kStamps: the same kernel with stage timestamps (measurement only).
template <int kMode, bool kStamps>
__global__ void __launch_bounds__(kThreads, 1)
    resolve_kernel(DevPool p, int layer, int n_req, const int32_t *__restrict__ req_ids,
                   const int32_t *__restrict__ sel_g, int k, int32_t *__restrict__ out_g,
                   const uint8_t *__restrict__ plan_in, uint8_t *__restrict__ plan_out,
                   unsigned long long *__restrict__ times, int plan_layer, int lead_k) {
    constexpr bool kPlanOnly = kMode == kModePlan;
    constexpr bool kNoFetch = kMode == kModeNoFetch;
    extern __shared__ __align__(16) uint8_t smem[];
    const bool with_plan = !kPlanOnly && plan_in != nullptr;
    const SmemLayout sl = smem_layout(p.B, k, with_plan, p.L);
    uint32_t *hdr = reinterpret_cast<uint32_t *>(smem + sl.hdr);
    uint32_t *sums = hdr + H_SUMS;
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + sl.keys);
    uint16_t *kidx = reinterpret_cast<uint16_t *>(smem + sl.kidx);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem + sl.bitmap);
    uint16_t *neworder = reinterpret_cast<uint16_t *>(smem + sl.keys);
    int32_t *sel_s = reinterpret_cast<int32_t *>(smem + sl.sel);
    int32_t *hit_s = reinterpret_cast<int32_t *>(smem + sl.hit);
    int32_t *spos_s = reinterpret_cast<int32_t *>(smem + sl.spos);
    uint16_t *order_s = reinterpret_cast<uint16_t *>(smem + sl.order);
    uint8_t *flags_s = smem + sl.flags;
    uint16_t *vrank_s = reinterpret_cast<uint16_t *>(smem + sl.vrank);
    int32_t *mpos = reinterpret_cast<int32_t *>(smem + sl.mpos);
    int32_t *mslot = reinterpret_cast<int32_t *>(smem + sl.mslot);
    int32_t *fpos = reinterpret_cast<int32_t *>(smem + sl.fpos);
    int32_t *fslot = reinterpret_cast<int32_t *>(smem + sl.fslot);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t crank = kPlanOnly ? 0u : cluster_ctarank();
    const uint32_t csize = kPlanOnly ? 1u : cluster_nctarank();
    const int ireq = (int)(blockIdx.x / csize);
    unsigned long long *stamp_row =
        kStamps ? times + ((size_t)ireq * kMaxCluster + crank) * kStampSlots : nullptr;
    auto stamp = [&](int slot) {
        if constexpr (kStamps) {
            if (tid == 0) stamp_row[slot] = globaltimer();
        }
    };
    stamp(S_ENTRY);
    const int B = p.B, H = sl.H, W = p.W;
    const int hshift = 33 - __ffs(H);          // 32 - log2(H)
    const int mshift = 33 - __ffs(sl.M);       // 32 - log2(M)
    const bool exact_bits = p.L <= (int64_t)sl.M;
    const int32_t *selr = sel_g + (int64_t)ireq * k;

    if (tid < H_SUMS) hdr[tid] = 0u;
    // Everything above touched only registers and shared memory.  Global
    // inputs may be written by the previous grid in the stream: a plan
    // waits for it here.  A resolve starts before it completes
    // (programmatic launch) and acts only on what it has checked after the
    // wait: the leader decides on the pair's metadata and keeps the
    // decision only if the pair's resolve counter (read before the
    // metadata, moved after every commit), the request id and the selection
    // are unchanged once the previous grid has completed, and decides again
    // otherwise; the followers of a plain resolve stage the records they
    // predict to miss and check each one against the leader's selection.
    // A consumed plan is read early too: it must come from a copy ordered
    // before this launch, and a copy is never launched before the plan it
    // replays has completed.  Nothing is written to global memory before
    // the wait, so a launch that overlaps the previous one stays exact.
    const bool early = !kPlanOnly;
    if (!early) grid_dependency_wait();
    allow_dependent_launch();
    if (crank == 0) copy_to_smem(sel_s, selr, 4 * k);  // independent of the request id

    int r = req_ids ? req_ids[ireq] : ireq;
    bool r_ok = r >= 0 && r < p.R;
    int64_t pair = (int64_t)layer * p.R + (r_ok ? r : 0);
    const uint8_t *host_pair = p.host + host_region(r_ok ? r : 0, layer, p.R, p.L, W);
    uint8_t *cache_pair = p.cache + pair * B * (int64_t)W;

    if (crank == 0) {
        bool took_busy = false;  // (thread 0)
        uint32_t t_seen = 0;     // (thread 0) the pair's resolve counter as read
        for (int attempt = 0;; ++attempt) {
            const bool speculative = early && attempt == 0;
            // ---------------- P0: load -------------------------------------
            uint32_t a0 = 0, t0 = 0;
            if (tid == 0) {
                hdr[H_ABORT] = 0u;
                hdr[H_NF] = 0u;
                hdr[H_PMISS] = 0u;
                hdr[H_PHIT] = 0u;
                hdr[H_PSTAT] = 0u;
                hdr[H_NL] = 0u;
                if (!r_ok) {
                    a0 |= HS_STATUS_REQ_RANGE;
                } else {
                    if (!kPlanOnly && !speculative && !took_busy) {
                        if (atomicCAS(&p.busy[pair], 0u, 1u) == 0u)
                            took_busy = true;
                        else
                            a0 |= HS_STATUS_REQ_BUSY;
                    }
                    // before the metadata copies below: a commit they might see
                    // in part moves the counter
                    t_seen = ld_acquire_gpu(&p.tcount[pair]);
                    t0 = t_seen + 1u;
                }
            }
            if (attempt > 0) copy_to_smem(sel_s, selr, 4 * k);
            __syncthreads();
            if (r_ok) {
                copy_to_smem(spos_s, p.slot_pos + pair * B, 4 * B);
                copy_to_smem(order_s, p.lru + pair * B, 2 * B);
            }
            {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                uint4 *kz = reinterpret_cast<uint4 *>(keys);
                for (int i = tid; i < H / 4; i += kThreads) kz[i] = z;
                uint4 *bz = reinterpret_cast<uint4 *>(bitmap);
                for (int i = tid; i < sl.M / 128; i += kThreads) bz[i] = z;
            }
            cp_async_wait_all();
            __syncthreads();  // header set, shared copies landed
            stamp(S_LOADED);

            // ---------------- P1: validate, hash build, membership bits ------
            {
                uint32_t bad = 0;
                if (tid == 0) {
                    bad = a0;
                    hdr[H_T] = t0;
                }
                if (r_ok) {
                    for (int i = tid; i < k; i += kThreads) {
                        const int32_t v = sel_s[i];
                        hit_s[i] = -1;
                        if (v < 0 || (int64_t)v >= p.L) {
                            bad |= HS_STATUS_POS_RANGE;
                            continue;
                        }
                        const uint32_t mb = member_bit(v, exact_bits, mshift);
                        atomicOr(&bitmap[mb >> 5], 1u << (mb & 31));
                        uint32_t h = hash_slot(v, hshift);
                        for (int probe = 0; probe < H; ++probe) {
                            const uint32_t old = atomicCAS(&keys[h], 0u, (uint32_t)v + 1u);
                            if (old == 0u) {
                                kidx[h] = (uint16_t)i;
                                break;
                            }
                            if (old == (uint32_t)v + 1u) {
                                bad |= HS_STATUS_POS_DUP;
                                break;
                            }
                            h = (h + 1) & (uint32_t)(H - 1);
                        }
                    }
                    for (int b = tid; b < B; b += kThreads) {
                        const int32_t v = spos_s[b];
                        flags_s[b] = 0;
                        if (v < -1 || (int64_t)v >= p.L || order_s[b] >= (uint16_t)B)
                            bad |= HS_STATUS_META;
                    }
                }
                if (bad) atomicOr(&hdr[H_ABORT], bad);
            }
            __syncthreads();
            stamp(S_HASHED);

            if (hdr[H_ABORT] == 0u) {
                // ------------- P2: probe the slots --------------------------
                // a slot whose position has no membership bit is not selected;
                // the others look their position up in the hash table
                for (int b0 = tid; b0 < B; b0 += kThreads * 4) {
                    int32_t pv[4];
                    uint32_t in[4];
    #pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int b = b0 + u * kThreads;
                        pv[u] = b < B ? spos_s[b] : -1;
                    }
    #pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        in[u] = 0u;
                        if (pv[u] >= 0) {
                            const uint32_t mb = member_bit(pv[u], exact_bits, mshift);
                            in[u] = (bitmap[mb >> 5] >> (mb & 31)) & 1u;
                        }
                    }
    #pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (!in[u]) continue;
                        const int32_t pos = pv[u];
                        uint32_t h = hash_slot(pos, hshift);
                        for (int probe = 0; probe < H; ++probe) {
                            const uint32_t key = keys[h];
                            if (key == 0u) break;
                            if (key == (uint32_t)pos + 1u) {
                                hit_s[kidx[h]] = b0 + u * kThreads;
                                flags_s[b0 + u * kThreads] = 1;
                                break;
                            }
                            h = (h + 1) & (uint32_t)(H - 1);
                        }
                    }
                }
                __syncthreads();
                stamp(S_PROBED);

                // ------------- P3: misses and victims (ballot scans) --------
                // warp w owns a contiguous block of 32*seg elements of each
                // array; element order = warp, then round, then lane.  Loads of
                // up to 8 rounds are issued before their ballots.
                const int segK = (k + kThreads - 1) / kThreads;
                const int segB = (B + kThreads - 1) / kThreads;
                const int baseK = warp * 32 * segK, baseB = warp * 32 * segB;
                const uint32_t lt = lanemask_lt();
                uint32_t cm = 0, cn = 0;
                for (int s0 = 0; s0 < segK; s0 += 8) {
                    bool pr[8];
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = baseK + (s0 + u) * 32 + lane;
                        pr[u] = s0 + u < segK && i < k && hit_s[i] < 0;
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (s0 + u < segK) cm += __popc(__ballot_sync(0xFFFFFFFFu, pr[u]));
                }
                for (int s0 = 0; s0 < segB; s0 += 8) {
                    int ob[8];
                    bool pr[8];
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int q = baseB + (s0 + u) * 32 + lane;
                        ob[u] = (s0 + u < segB && q < B) ? (int)order_s[q] : -1;
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u) pr[u] = ob[u] >= 0 && !(flags_s[ob[u]] & 1);
    #pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (s0 + u < segB) cn += __popc(__ballot_sync(0xFFFFFFFFu, pr[u]));
                }
                uint32_t total;
                const uint32_t base = warp_counts_exscan(cm | (cn << 16), sums, &total);
                const int m = (int)(total & 0xFFFFu);
                const int nh = (int)(total >> 16);
                uint32_t mr = base & 0xFFFFu, nr = base >> 16;
                for (int s0 = 0; s0 < segK; s0 += 8) {
                    bool pr[8];
                    int32_t sv[8];
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = baseK + (s0 + u) * 32 + lane;
                        pr[u] = s0 + u < segK && i < k && hit_s[i] < 0;
                        sv[u] = pr[u] ? sel_s[i] : 0;
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (s0 + u >= segK) break;
                        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pr[u]);
                        if (pr[u]) {
                            const uint32_t rank = mr + __popc(bal & lt);
                            mpos[rank] = sv[u];
                            hit_s[baseK + (s0 + u) * 32 + lane] = -2 - (int32_t)rank;
                        }
                        mr += __popc(bal);
                    }
                }
                for (int s0 = 0; s0 < segB; s0 += 8) {
                    int ob[8];
                    bool pr[8];
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int q = baseB + (s0 + u) * 32 + lane;
                        ob[u] = (s0 + u < segB && q < B) ? (int)order_s[q] : -1;
                    }
    #pragma unroll
                    for (int u = 0; u < 8; ++u) pr[u] = ob[u] >= 0 && !(flags_s[ob[u]] & 1);
    #pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (s0 + u >= segB) break;
                        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pr[u]);
                        if (pr[u]) {
                            const uint32_t rank = nr + __popc(bal & lt);
                            const int b = ob[u];
                            if ((int)rank < m) {
                                mslot[rank] = b;
                                flags_s[b] |= 2;
                                if (with_plan) vrank_s[b] = (uint16_t)rank;
                            } else {
                                neworder[rank - m] = (uint16_t)b;
                            }
                        }
                        nr += __popc(bal);
                    }
                }
                if (tid == 0) {
                    hdr[H_M] = (uint32_t)m;
                    hdr[H_NH] = (uint32_t)nh;
                    hdr[H_F] = (uint32_t)m;
                    hdr[H_FLIST] = 0u;
                }
                __syncthreads();

                // ------------- P3b: consume a plan --------------------------
                if (with_plan) {
                    const PlanHeader *ph = reinterpret_cast<const PlanHeader *>(plan_in);
                    const int32_t *eh =
                        reinterpret_cast<const int32_t *>(plan_in + 16 + (size_t)ireq * plan_entry_bytes(k));
                    const bool ok = ph->magic == kPlanMagic && ph->n_req == n_req && ph->k == k &&
                                    (ph->layer == layer || ph->layer == plan_layer) && eh[0] >= 0 &&
                                    eh[0] <= k && eh[1] == r;
                    const int mp = ok ? eh[0] : 0;
                    if (!ok && tid == 0) atomicOr(&hdr[H_PSTAT], HS_STATUS_PLAN);
                    const int32_t *ppos = eh + 4;
                    const int32_t *pslot = ppos + k;
                    const int n = m > mp ? m : mp;
                    for (int j = tid; j < n; j += kThreads) {
                        const int32_t pp = j < mp ? ppos[j] : -1;
                        const int32_t ps = j < mp ? pslot[j] : -1;
                        if (j < m && j < mp && pp == mpos[j] && ps == mslot[j]) {
                            atomicAdd(&hdr[H_PHIT], 1u);
                            continue;
                        }
                        atomicAdd(&hdr[H_PMISS], 1u);
                        if (j < m) {
                            const uint32_t f = atomicAdd(&hdr[H_NF], 1u);
                            fpos[f] = mpos[j];
                            fslot[f] = mslot[j];
                        }
                        if (j < mp) {
                            if (ps >= 0 && ps < B && pp >= 0 && (int64_t)pp < p.L) {
                                // the copy wrote slot ps: refill it with its owner
                                const int32_t owner = (flags_s[ps] & 2) ? mpos[vrank_s[ps]] : spos_s[ps];
                                if (owner >= 0) {
                                    const uint32_t f = atomicAdd(&hdr[H_NF], 1u);
                                    fpos[f] = owner;
                                    fslot[f] = ps;
                                }
                            } else {
                                atomicOr(&hdr[H_PSTAT], HS_STATUS_PLAN);
                            }
                        }
                    }
                    __syncthreads();
                    if (tid == 0) {
                        hdr[H_F] = hdr[H_NF];
                        hdr[H_FLIST] = 1u;
                    }
                    __syncthreads();
                }
            }
            stamp(S_DECIDED);
            if constexpr (kStamps) {
                if (tid == 0) stamp_row[S_ATTEMPTS] = (unsigned long long)(attempt + 1);
            }
            if (!speculative) {
                stamp(S_CHECKED);  // a decision taken after the wait stands as it is
                break;
            }

            // ---------------- the speculative decision stands only if its
            // inputs are unchanged now that the previous grid has completed
            grid_dependency_wait();
            const int r_now = req_ids ? req_ids[ireq] : ireq;
            int stale = r_now != r;
            for (int i = tid; i < k; i += kThreads) stale |= selr[i] != sel_s[i];
            if (tid == 0 && !stale && r_ok) {
                // claim the pair, then look at its counter: a resolve that held
                // it and has let it go has moved the counter before
                if (atomicCAS(&p.busy[pair], 0u, 1u) == 0u) {
                    took_busy = true;
                    stale = ld_acquire_gpu(&p.tcount[pair]) != t_seen;
                } else {
                    atomicOr(&hdr[H_ABORT], HS_STATUS_REQ_BUSY);
                }
            }
            if (!__syncthreads_or(stale)) {
                stamp(S_CHECKED);
                break;
            }
            // decide again on what the previous grid left
            r = r_now;
            r_ok = r >= 0 && r < p.R;
            pair = (int64_t)layer * p.R + (r_ok ? r : 0);
            host_pair = p.host + host_region(r_ok ? r : 0, layer, p.R, p.L, W);
            cache_pair = p.cache + pair * B * (int64_t)W;
        }  // attempts
        const uint32_t abort_bits = hdr[H_ABORT];
        if (abort_bits != 0u) {
            // rejected request: publish -1, leave metadata and slots alone
            if (!kPlanOnly) {
                int32_t *o = out_g + (int64_t)ireq * k;
                for (int i = tid; i < k; i += kThreads) o[i] = -1;
            }
            if (tid == 0) {
                atomicOr(p.status, abort_bits | (with_plan ? hdr[H_PSTAT] : 0u));
                hdr[H_F] = 0u;
                hdr[H_M] = 0u;
                if (took_busy) atomicExch(&p.busy[pair], 0u);
            }
            __syncthreads();
        }

        if (kPlanOnly) {
            int32_t *eh = reinterpret_cast<int32_t *>(plan_out + 16 + (size_t)ireq * plan_entry_bytes(k));
            const int m = abort_bits ? 0 : (int)hdr[H_M];
            if (tid == 0) {
                eh[0] = m;
                eh[1] = r;
                eh[2] = 0;
                eh[3] = 0;
                if (ireq == 0) {
                    PlanHeader *ph = reinterpret_cast<PlanHeader *>(plan_out);
                    ph->magic = kPlanMagic;
                    ph->n_req = n_req;
                    ph->k = k;
                    ph->layer = layer;
                }
            }
            for (int j = tid; j < m; j += kThreads) {
                eh[4 + j] = mpos[j];
                eh[4 + k + j] = mslot[j];
            }
            return;
        }
    } else if (kNoFetch) {
        // measurement variant without the fetch: the followers move nothing
        grid_dependency_wait();
    } else if (!with_plan) {
        // ---------------- follower F0: predict misses, stage their records --
        // Warp w takes blocks of 32 consecutive share entries (w, w + 16,
        // ...).  A lane reads its selection and the page-table entry of the
        // position; -1 predicts a miss.  For every predicted miss the warp
        // takes a slot of the CTA's staging pool (one atomic per block) and
        // issues cp.async copies of the record from the mapped host pool into
        // it, while the pool lasts; sbits[block] remembers which entries
        // were staged.
        const FollowerLayout fl = follower_layout(k, W);
        int32_t *stg = reinterpret_cast<int32_t *>(smem + fl.stg);
        int32_t *stgpos = reinterpret_cast<int32_t *>(smem + fl.stgpos);
        uint32_t *sbits = reinterpret_cast<uint32_t *>(smem + fl.sbits);
        uint8_t *stage = smem + fl.stage;
        const int nf = csize > 1 ? (int)csize - 1 : 1, f = (int)crank - 1;
        // the followers share [0, k - lead_k); the leader fetches the rest
        const int kf = k - lead_k;
        const int i0 = (int)((int64_t)f * kf / nf), i1 = (int)((int64_t)(f + 1) * kf / nf);
        const int ns = i1 - i0;
        const int nblk = (ns + 31) >> 5;
        const int32_t *pt = p.pt + pair * p.L;
        const int CW = W >> 4;
        for (int blk0 = warp; blk0 < nblk; blk0 += kWarps * 4) {
            int32_t pos[4], ptv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = (blk0 + u * kWarps) * 32 + lane;
                pos[u] = (blk0 + u * kWarps < nblk && e < ns) ? selr[i0 + e] : -1;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                ptv[u] = (r_ok && pos[u] >= 0 && (int64_t)pos[u] < p.L) ? pt[pos[u]] : 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int blk = blk0 + u * kWarps;
                if (blk >= nblk) break;
                uint32_t mask = __ballot_sync(0xFFFFFFFFu, ptv[u] == -1);
                uint32_t base = 0;
                if (lane == 0 && mask) base = atomicAdd(&hdr[H_NSTG], (uint32_t)__popc(mask));
                int slot = (int)__shfl_sync(0xFFFFFFFFu, base, 0);
                uint32_t staged = 0;
                if (kStamps && blk == 0) stamp(S_F_ISSUE);
                while (mask && slot < fl.cap) {
                    const int src = __ffs(mask) - 1;
                    mask &= mask - 1;
                    const int32_t q = __shfl_sync(0xFFFFFFFFu, pos[u], src);
                    uint8_t *dst = stage + (size_t)slot * W;
                    const uint8_t *from = host_pair + (int64_t)q * W;
                    for (int c = lane; c < CW; c += 32) cp_async16(dst + 16 * c, from + 16 * c);
                    if (lane == 0) {
                        stg[slot] = blk * 32 + src;
                        stgpos[slot] = q;
                    }
                    staged |= 1u << src;
                    ++slot;
                }
                if (lane == 0) sbits[blk] = staged;
            }
        }
        stamp(S_F_ISSUED);
        // the previous grid's writes are visible from here on; a request id
        // that changed under the early reads voids this CTA's staging
        grid_dependency_wait();
        stamp(S_F_WAITED);
        const int r_now = req_ids ? req_ids[ireq] : ireq;
        if (r_now != r) {
            r = r_now;
            r_ok = r >= 0 && r < p.R;
            pair = (int64_t)layer * p.R + (r_ok ? r : 0);
            host_pair = p.host + host_region(r_ok ? r : 0, layer, p.R, p.L, W);
            cache_pair = p.cache + pair * B * (int64_t)W;
            __syncthreads();  // every warp is done staging
            if (tid == 0) hdr[H_NSTG] = 0u;
            for (int blk = tid; blk < nblk; blk += kThreads) sbits[blk] = 0u;
        }
        __syncthreads();
    }

    if constexpr (!kPlanOnly) {
        // phase A: the leader publishes its decision (release); a follower
        // only says it is ready, without waiting for its loads in flight
        if (crank == 0)
            cluster_arrive();
        else
            cluster_arrive_relaxed();
        cluster_wait();
        stamp(S_VERDICT);

        if (crank == 0) {
            cluster_arrive_relaxed();  // phase B: the leader's shared memory stays valid until B
            if (plan_out != nullptr) {
                // an anchor's resolve also writes its miss plan -- the
                // (position, victim) pairs it commits -- for the layers that
                // share its selection to replay (after the previous grid)
                int32_t *eh =
                    reinterpret_cast<int32_t *>(plan_out + 16 + (size_t)ireq * plan_entry_bytes(k));
                const int m = hdr[H_ABORT] == 0u ? (int)hdr[H_M] : 0;
                if (tid == 0) {
                    eh[0] = m;
                    eh[1] = r;
                    eh[2] = 0;
                    eh[3] = 0;
                    if (ireq == 0) {
                        PlanHeader *ph = reinterpret_cast<PlanHeader *>(plan_out);
                        ph->magic = kPlanMagic;
                        ph->n_req = n_req;
                        ph->k = k;
                        ph->layer = layer;
                    }
                }
                for (int j = tid; j < m; j += kThreads) {
                    eh[4 + j] = mpos[j];
                    eh[4 + k + j] = mslot[j];
                }
            }
            if (hdr[H_ABORT] == 0u) {
                // ------------- P4: commit metadata, publish ------------------
                const uint32_t t = hdr[H_T];
                const int m = (int)hdr[H_M];
                const int nh = (int)hdr[H_NH];
                int32_t *o = out_g + (int64_t)ireq * k;
                const int32_t rowbase = r * B;
                for (int i = tid; i < k; i += kThreads) {
                    const int32_t hsl = hit_s[i];
                    o[i] = rowbase + (hsl >= 0 ? hsl : mslot[-2 - hsl]);
                }
                int32_t *pt = p.pt + pair * p.L;
                int32_t *sp = p.slot_pos + pair * B;
                uint32_t *st = p.stamp + pair * B;
                for (int j = tid; j < m; j += kThreads) {
                    const int32_t v = mslot[j];
                    const int32_t old = spos_s[v];
                    if (old >= 0) pt[old] = -1;
                    pt[mpos[j]] = v;
                    sp[v] = mpos[j];
                    st[v] = 2u * t - 1u;
                }
                // new LRU order: [untouched (placed by P3)] [victims] [hits]
                const int segB = (B + kThreads - 1) / kThreads;
                const int baseB = warp * 32 * segB;
                const uint32_t lt = lanemask_lt();
                uint32_t cv = 0, ch = 0;
                for (int s = 0; s < segB; ++s) {
                    const int b = baseB + s * 32 + lane;
                    const uint8_t fl = b < B ? flags_s[b] : 0;
                    cv += __popc(__ballot_sync(0xFFFFFFFFu, (fl & 2) != 0));
                    ch += __popc(__ballot_sync(0xFFFFFFFFu, (fl & 1) != 0));
                }
                uint32_t total;
                const uint32_t base = warp_counts_exscan(cv | (ch << 16), sums, &total);
                uint32_t vr = (uint32_t)(nh - m) + (base & 0xFFFFu);
                uint32_t hr = (uint32_t)nh + (base >> 16);
                for (int s = 0; s < segB; ++s) {
                    const int b = baseB + s * 32 + lane;
                    const uint8_t fl = b < B ? flags_s[b] : 0;
                    const uint32_t bv = __ballot_sync(0xFFFFFFFFu, (fl & 2) != 0);
                    const uint32_t bh = __ballot_sync(0xFFFFFFFFu, (fl & 1) != 0);
                    if (fl & 2) neworder[vr + __popc(bv & lt)] = (uint16_t)b;
                    if (fl & 1) {
                        neworder[hr + __popc(bh & lt)] = (uint16_t)b;
                        st[b] = 2u * t;
                    }
                    vr += __popc(bv);
                    hr += __popc(bh);
                }
                __syncthreads();
                uint16_t *lo = p.lru + pair * B;
                for (int b = tid; b < B; b += kThreads) lo[b] = neworder[b];
                const int F = (int)hdr[H_F];
                // the counter moves after every metadata write of the commit:
                // a later launch deciding early reads it before the metadata
                __syncthreads();
                if (tid == 0) {
                    __threadfence();
                    st_release_gpu(&p.tcount[pair], t);
                    unsigned long long *c = p.counters + (int64_t)layer * CTR_COUNT;
                    atomicAdd(&c[CTR_RESOLVES], 1ull);
                    atomicAdd(&c[CTR_HITS], (unsigned long long)(k - m));
                    atomicAdd(&c[CTR_MISSES], (unsigned long long)m);
                    if (!kNoFetch)
                    atomicAdd(&c[CTR_FETCHED], (unsigned long long)F * (unsigned long long)W);
                    if (with_plan) {
                        atomicAdd(&c[CTR_PLAN_HITS], (unsigned long long)hdr[H_PHIT]);
                        atomicAdd(&c[CTR_PLAN_MISMATCH], (unsigned long long)hdr[H_PMISS]);
                        if (hdr[H_PSTAT]) atomicOr(p.status, hdr[H_PSTAT]);
                    }
                }
                stamp(S_COMMITTED);
                if (!kNoFetch && csize == 1 && F > 0) {
                    const bool plist = hdr[H_FLIST] != 0u;
                    fetch_records(host_pair, cache_pair, plist ? fpos : mpos,
                                  plist ? fslot : mslot, F, W, tid, kThreads);
                } else if (!kNoFetch && csize > 1 && lead_k > 0 && !with_plan) {
                    // The leader's own share of the selection, [k - lead_k, k),
                    // fetched by this CTA once it has committed, while the
                    // followers store what they staged of theirs: one more SM
                    // on the request's records, with a single request's
                    // records on each SM.  Its misses are compacted into the
                    // hash table's index array (free since the probe, read by
                    // no follower).
                    int32_t *lp = reinterpret_cast<int32_t *>(smem + sl.kidx);
                    int32_t *ls = lp + lead_k;
                    for (int i = k - lead_k + tid; i < k; i += kThreads) {
                        const int32_t hsl = hit_s[i];
                        if (hsl <= -2) {
                            const uint32_t x = atomicAdd(&hdr[H_NL], 1u);
                            lp[x] = mpos[-2 - hsl];
                            ls[x] = mslot[-2 - hsl];
                        }
                    }
                    __syncthreads();
                    const int nl = (int)hdr[H_NL];
                    if (nl > 0) fetch_records(host_pair, cache_pair, lp, ls, nl, W, tid, kThreads);
                    stamp(S_LEAD_FETCHED);
                }
                if (tid == 0) {
                    __threadfence();
                    atomicExch(&p.busy[pair], 0u);
                }
            }
        } else if (kNoFetch) {
            cluster_arrive_relaxed();  // phase B: nothing to read from the leader
        } else if (with_plan) {
            // ------------- follower, plan consumed: the leader's fetch list ----
            grid_dependency_wait();  // (passed by the leader already)
            cg::cluster_group cl = cg::this_cluster();
            const uint32_t *lh = cl.map_shared_rank(hdr, 0);
            const int F = (int)lh[H_F];
            const bool plist = lh[H_FLIST] != 0u;
            int32_t *dp = plist ? fpos : mpos;
            int32_t *ds = plist ? fslot : mslot;
            const int32_t *lp = cl.map_shared_rank(dp, 0);
            const int32_t *ls = cl.map_shared_rank(ds, 0);
            for (int e = tid; e < F; e += kThreads) {
                dp[e] = lp[e];
                ds[e] = ls[e];
            }
            __syncthreads();
            cluster_arrive_relaxed();  // phase B: done reading the leader
            if (F > 0)
                fetch_records(host_pair, cache_pair, dp, ds, F, W, (int)(crank - 1) * kThreads + tid,
                              (int)(csize - 1) * kThreads);
        } else {
            // ------------- follower F1-F3: apply the leader's verdict ----------
            cg::cluster_group cl = cg::this_cluster();
            const uint32_t *lh = cl.map_shared_rank(hdr, 0);
            const int32_t *lhit = cl.map_shared_rank(hit_s, 0);
            const int32_t *lmslot = cl.map_shared_rank(mslot, 0);
            const bool abort = lh[H_ABORT] != 0u;
            const int32_t *lsel = cl.map_shared_rank(sel_s, 0);
            const FollowerLayout fl = follower_layout(k, W);
            int32_t *stg = reinterpret_cast<int32_t *>(smem + fl.stg);
            const int32_t *stgpos = reinterpret_cast<const int32_t *>(smem + fl.stgpos);
            uint32_t *sbits = reinterpret_cast<uint32_t *>(smem + fl.sbits);
            const uint8_t *stage = smem + fl.stage;
            const int nstaged = min((int)hdr[H_NSTG], fl.cap);
            int32_t *xp = reinterpret_cast<int32_t *>(smem + fl.xp);  // misses not staged
            int32_t *xs = reinterpret_cast<int32_t *>(smem + fl.xs);
            const int nf = csize > 1 ? (int)csize - 1 : 1, f = (int)crank - 1;
            const int kf = k - lead_k;
            const int i0 = (int)((int64_t)f * kf / nf), i1 = (int)((int64_t)(f + 1) * kf / nf);
            const int ns = i1 - i0;
            const int nblk = (ns + 31) >> 5;
            // F1: the victim slot of each staged record (-1: the leader found
            // a hit) replaces its share entry in stg, and the leader's misses
            // of this warp's blocks that were not staged go to the x list.
            // A staged record whose position is not the leader's selection
            // (read before the wait, changed since) is dropped and fetched
            // with the unstaged misses.
            if (!abort) {
                for (int s = tid; s < nstaged; s += kThreads) {
                    const int e = stg[s];
                    int32_t slot = -1;
                    if (lsel[i0 + e] == stgpos[s]) {
                        const int32_t hsl = lhit[i0 + e];
                        slot = hsl <= -2 ? lmslot[-2 - hsl] : -1;
                    } else {
                        atomicAnd(&sbits[e >> 5], ~(1u << (e & 31)));
                    }
                    stg[s] = slot;
                }
            }
            __syncthreads();
            if (!abort) {
                for (int blk = warp; blk < nblk; blk += kWarps) {
                    const int e = blk * 32 + lane;
                    const int32_t hsl = e < ns ? lhit[i0 + e] : -1;
                    if (hsl <= -2 && !((sbits[blk] >> lane) & 1u)) {
                        const uint32_t x = atomicAdd(&hdr[H_NX], 1u);
                        xp[x] = lsel[i0 + e];
                        xs[x] = lmslot[-2 - hsl];
                    }
                }
            }
            __syncthreads();
            cluster_arrive_relaxed();  // phase B: done reading the leader
            cp_async_wait_all();       // no copy into shared memory outlives the CTA
            __syncthreads();           // every thread's staged copies have landed
            stamp(S_F_LANDED);
            if (!abort) {
                // F2: one bulk copy per staged record from shared memory to
                // its victim slot, issued by the thread that owns the record
                fence_proxy_async_shared();
                bool stored = false;
                for (int s = tid; s < nstaged; s += kThreads) {
                    const int32_t slot = stg[s];
                    if (slot >= 0) {
                        bulk_store(cache_pair + (int64_t)slot * W, stage + (size_t)s * W, W);
                        stored = true;
                    }
                }
                if (stored) bulk_commit();
                // F3: misses that were not staged
                const int nx = (int)hdr[H_NX];
                if (nx > 0) fetch_records(host_pair, cache_pair, xp, xs, nx, W, tid, kThreads);
                if (stored) bulk_wait_read();  // shared memory is read before the CTA ends
            }
            if constexpr (kStamps) {
                __syncthreads();  // (measurement variant) every thread's copies issued
                stamp(S_F_STORED);
            }
        }
        cluster_wait();  // phase B: no CTA leaves while the leader is being read
        stamp(S_EXIT);
    }
}

}  // namespace

// Largest dynamic shared memory of a block on the current device (cached).
uint32_t device_smem_optin() {
    static std::mutex mu;
    static int cached_dev = -1;
    static uint32_t cached = 0;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev != cached_dev) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return 0;
        cached = (uint32_t)v;
        cached_dev = dev;
    }
    return cached;
}

cudaError_t prepare_kernels(size_t max_smem) {
    const void *fns[] = {
        reinterpret_cast<const void *>(resolve_kernel<kModeResolve, false>),
        reinterpret_cast<const void *>(resolve_kernel<kModePlan, false>),
        reinterpret_cast<const void *>(resolve_kernel<kModeResolve, true>),
        reinterpret_cast<const void *>(resolve_kernel<kModeNoFetch, false>),
        reinterpret_cast<const void *>(resolve_kernel<kModeNoFetch, true>),
    };
    for (const void *f : fns) {
        const cudaError_t e =
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
        if (e != cudaSuccess) return e;
    }
    return prepare_copy_kernel();
}

namespace {

// One resolve launch: a cluster of `cluster` CTAs per request, programmatic
// stream serialisation (the launch may overlap the previous grid in the
// stream: the kernel reads its inputs early and writes no global memory
// before that grid has completed).
template <int kMode, bool kStamps>
cudaError_t launch_variant(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                           const int32_t *sel, int k, int32_t *out, const void *plan,
                           unsigned long long *times, int cluster, cudaStream_t st,
                           int plan_layer = -1, void *plan_out = nullptr, bool overlap = true,
                           int lead_k = 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_req * cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    // A plain launch takes all the shared memory a CTA may have: the CTA is
    // alone on its SM anyway (512 threads x 96 registers), and the followers
    // stage more records before the leader decides.
    uint32_t smem = resolve_smem_bytes(p.B, k, plan != nullptr, p.L);
    if (!plan) {
        const uint32_t most = device_smem_optin();
        if (most > smem) smem = most;
    }
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // the leader fetches a share of the selection only beside followers,
    // and never from a plan (a consumed plan has its own fetch list)
    if (cluster < 2 || plan != nullptr || lead_k < 0 || lead_k >= k) lead_k = 0;
    return cudaLaunchKernelEx(&cfg, resolve_kernel<kMode, kStamps>, p, layer, n_req, req_ids, sel,
                              k, out, static_cast<const uint8_t *>(plan),
                              static_cast<uint8_t *>(plan_out), times, plan_layer, lead_k);
}

}  // namespace

cudaError_t launch_resolve(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                           const int32_t *sel, int k, int32_t *out, const void *plan,
                           int cluster, cudaStream_t st, int plan_layer, void *plan_out,
                           bool overlap, int lead_k) {
    return launch_variant<kModeResolve, false>(p, layer, n_req, req_ids, sel, k, out, plan,
                                               nullptr, cluster, st, plan_layer, plan_out, overlap,
                                               lead_k);
}

cudaError_t launch_resolve_measure(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                                   const int32_t *sel, int k, int32_t *out, bool no_fetch,
                                   unsigned long long *times, int cluster, cudaStream_t st,
                                   bool overlap, int lead_k) {
    if (no_fetch)
        return times ? launch_variant<kModeNoFetch, true>(p, layer, n_req, req_ids, sel, k, out,
                                                          nullptr, times, cluster, st, -1, nullptr,
                                                          overlap, 0)
                     : launch_variant<kModeNoFetch, false>(p, layer, n_req, req_ids, sel, k, out,
                                                           nullptr, nullptr, cluster, st, -1,
                                                           nullptr, overlap, 0);
    return times ? launch_variant<kModeResolve, true>(p, layer, n_req, req_ids, sel, k, out,
                                                      nullptr, times, cluster, st, -1, nullptr,
                                                      overlap, lead_k)
                 : launch_variant<kModeResolve, false>(p, layer, n_req, req_ids, sel, k, out,
                                                       nullptr, nullptr, cluster, st, -1, nullptr,
                                                       overlap, lead_k);
}

cudaError_t launch_plan(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                        const int32_t *sel, int k, void *plan, cudaStream_t st) {
    const SmemLayout sl = smem_layout(p.B, k, false, p.L);
    resolve_kernel<kModePlan, false><<<n_req, kThreads, sl.total, st>>>(
        p, layer, n_req, req_ids, sel, k, nullptr, nullptr, static_cast<uint8_t *>(plan),
        nullptr, -1, 0);
    return cudaGetLastError();
}

}  // namespace hs

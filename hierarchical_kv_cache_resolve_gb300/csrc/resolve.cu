// RESOLVE: one fused launch per sparse layer (HiSparse; "Inference Systems
// Infrastructure Notes (6): HiSparse", section 3 "RESOLVE: Five Stages in One
// Launch"; Pith review of arXiv 2608.07009, "What carries the argument").
//
// Grid: one thread-block cluster per request (n_req * C CTAs of kThreads).
// CTA 0 of a cluster (the leader) owns the request's metadata:
//   P0  load the k selections, the slot map and the LRU order into shared
//       memory; reject positions outside [0, L) and corrupt metadata;
//   P1  insert the selections into a shared-memory open-addressing hash
//       table (key = position, value = selection index); a repeated key is
//       a duplicate selection;
//   P2  probe every slot's position against the table: a found slot is a
//       hit for that selection index;
//   P3  one warp-ballot scan over the selections (misses in selection order)
//       fused with one over the LRU order (non-hit slots in (stamp, slot)
//       order): the j-th miss gets the j-th non-hit slot as its victim;
//   P4  publish slots, update page table / slot map / stamps, and rebuild
//       the LRU order with a second ballot scan over the slots.
// After P3 the fetch list (position, victim) is in the leader's shared
// memory; the other CTAs of the cluster copy it through distributed shared
// memory and fetch the records from the mapped host pool with 16-byte
// non-coherent loads, while the leader commits the metadata.  With a
// cluster of one CTA the leader fetches too.
//
// Victim selection without sorting: the LRU order array is kept sorted by
// (stamp, slot).  A resolve at step t keeps the untouched slots in their old
// relative order and appends the victims (stamp 2t-1) and then the hits
// (stamp 2t), each group in slot order -- exactly the (stamp, slot) order of
// the new stamps -- so the victims are always the first m non-hit entries.
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

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16-byte read-only load that bypasses L1 allocation: used on the mapped
// host pool, which no kernel writes.
__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t hash_pos(int32_t pos, int H) {
    return ((uint32_t)pos * 2654435761u) & (uint32_t)(H - 1);
}

// Copies F records: fetch-list entry j moves host_pair[fp[j]] to
// cache_pair[fs[j]].  The 16-byte chunks (entry, part) are spread over G
// threads; each thread keeps kUnroll loads in flight before storing.
__device__ __forceinline__ void fetch_records(const uint8_t *__restrict__ host_pair,
                                              uint8_t *__restrict__ cache_pair,
                                              const int32_t *fp, const int32_t *fs, int F,
                                              int W, int g, int G) {
    const int CW = W >> 4;
    const int Q = F * CW;
    for (int q0 = g; q0 < Q; q0 += G * kUnroll) {
        uint4 v[kUnroll];
        int64_t doff[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int q = q0 + u * G;
            doff[u] = -1;
            if (q < Q) {
                const int j = q / CW;
                const int part = q - j * CW;
                v[u] = ld_nc_v4(host_pair + (int64_t)fp[j] * W + part * 16);
                doff[u] = (int64_t)fs[j] * W + part * 16;
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

template <bool kPlanOnly>
__global__ void __launch_bounds__(kThreads)
    resolve_kernel(DevPool p, int layer, int n_req, const int32_t *__restrict__ req_ids,
                   const int32_t *__restrict__ sel_g, int k, int32_t *__restrict__ out_g,
                   const uint8_t *__restrict__ plan_in, uint8_t *__restrict__ plan_out) {
    extern __shared__ __align__(16) uint8_t smem[];
    const bool with_plan = !kPlanOnly && plan_in != nullptr;
    const SmemLayout sl = smem_layout(p.B, k, with_plan);
    uint32_t *hdr = reinterpret_cast<uint32_t *>(smem + sl.hdr);
    uint32_t *sums = hdr + H_SUMS;
    unsigned long long *tab = reinterpret_cast<unsigned long long *>(smem + sl.hash);
    uint16_t *neworder = reinterpret_cast<uint16_t *>(smem + sl.hash);
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
    const int B = p.B, H = sl.H;
    const int r = req_ids ? req_ids[ireq] : ireq;
    const bool r_ok = r >= 0 && r < p.R;
    const int64_t pair = (int64_t)layer * p.R + (r_ok ? r : 0);

    if (crank == 0) {
        // ---------------- P0: load -------------------------------------
        if (tid < H_SUMS) hdr[tid] = 0u;
        __syncthreads();
        bool took_busy = false;
        if (tid == 0) {
            uint32_t a = 0;
            if (!r_ok) {
                a |= HS_STATUS_REQ_RANGE;
            } else if (!kPlanOnly) {
                if (atomicCAS(&p.busy[pair], 0u, 1u) == 0u)
                    took_busy = true;
                else
                    a |= HS_STATUS_REQ_BUSY;
            }
            if (a) atomicOr(&hdr[H_ABORT], a);
            hdr[H_T] = r_ok ? p.tcount[pair] + 1u : 0u;
        }
        if (r_ok) {
            const int32_t *selr = sel_g + (int64_t)ireq * k;
            for (int i = tid; i < k; i += kThreads) {
                const int32_t v = selr[i];
                sel_s[i] = v;
                hit_s[i] = -1;
                if (v < 0 || (int64_t)v >= p.L) atomicOr(&hdr[H_ABORT], HS_STATUS_POS_RANGE);
            }
            const int32_t *sp = p.slot_pos + pair * B;
            const uint16_t *lo = p.lru + pair * B;
            for (int b = tid; b < B; b += kThreads) {
                const int32_t v = sp[b];
                const uint16_t o = lo[b];
                spos_s[b] = v;
                order_s[b] = o;
                flags_s[b] = 0;
                if (v < -1 || (int64_t)v >= p.L || o >= (uint16_t)B)
                    atomicOr(&hdr[H_ABORT], HS_STATUS_META);
            }
            for (int h = tid; h < H; h += kThreads) tab[h] = 0ull;
        }
        __syncthreads();

        // ---------------- P1: hash build --------------------------------
        if (hdr[H_ABORT] == 0u) {
            for (int i = tid; i < k; i += kThreads) {
                const int32_t key = sel_s[i];
                const unsigned long long e =
                    ((unsigned long long)(uint32_t)(key + 1) << 32) | (uint32_t)i;
                uint32_t h = hash_pos(key, H);
                for (int probe = 0; probe < H; ++probe) {
                    const unsigned long long old = atomicCAS(&tab[h], 0ull, e);
                    if (old == 0ull) break;
                    if ((uint32_t)(old >> 32) == (uint32_t)(key + 1)) {
                        atomicOr(&hdr[H_ABORT], HS_STATUS_POS_DUP);
                        break;
                    }
                    h = (h + 1) & (uint32_t)(H - 1);
                }
            }
        }
        __syncthreads();
        const uint32_t abort_bits = hdr[H_ABORT];

        if (abort_bits == 0u) {
            // ------------- P2: probe the slots --------------------------
            for (int b = tid; b < B; b += kThreads) {
                const int32_t pos = spos_s[b];
                if (pos < 0) continue;
                uint32_t h = hash_pos(pos, H);
                for (int probe = 0; probe < H; ++probe) {
                    const unsigned long long e = tab[h];
                    if (e == 0ull) break;
                    if ((uint32_t)(e >> 32) == (uint32_t)(pos + 1)) {
                        hit_s[(uint32_t)e] = b;
                        flags_s[b] = 1;
                        break;
                    }
                    h = (h + 1) & (uint32_t)(H - 1);
                }
            }
            __syncthreads();

            // ------------- P3: misses and victims (ballot scans) --------
            const int segK = (k + kThreads - 1) / kThreads;
            const int segB = (B + kThreads - 1) / kThreads;
            const int baseK = warp * 32 * segK, baseB = warp * 32 * segB;
            const uint32_t lt = lanemask_lt();
            uint32_t cm = 0, cn = 0;
            for (int s = 0; s < segK; ++s) {
                const int i = baseK + s * 32 + lane;
                cm += __popc(__ballot_sync(0xFFFFFFFFu, i < k && hit_s[i] < 0));
            }
            for (int s = 0; s < segB; ++s) {
                const int q = baseB + s * 32 + lane;
                cn += __popc(__ballot_sync(0xFFFFFFFFu, q < B && !(flags_s[order_s[q]] & 1)));
            }
            uint32_t total;
            const uint32_t base = warp_counts_exscan(cm | (cn << 16), sums, &total);
            const int m = (int)(total & 0xFFFFu);
            const int nh = (int)(total >> 16);
            uint32_t mr = base & 0xFFFFu, nr = base >> 16;
            for (int s = 0; s < segK; ++s) {
                const int i = baseK + s * 32 + lane;
                const bool pr = i < k && hit_s[i] < 0;
                const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pr);
                if (pr) {
                    const uint32_t rank = mr + __popc(bal & lt);
                    mpos[rank] = sel_s[i];
                    hit_s[i] = -2 - (int32_t)rank;
                }
                mr += __popc(bal);
            }
            for (int s = 0; s < segB; ++s) {
                const int q = baseB + s * 32 + lane;
                const int b = q < B ? (int)order_s[q] : 0;
                const bool pr = q < B && !(flags_s[b] & 1);
                const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pr);
                if (pr) {
                    const uint32_t rank = nr + __popc(bal & lt);
                    if ((int)rank < m) {
                        mslot[rank] = b;
                        flags_s[b] |= 2;
                        vrank_s[b] = (uint16_t)rank;
                    } else {
                        neworder[rank - m] = (uint16_t)b;
                    }
                }
                nr += __popc(bal);
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
                                ph->layer == layer && eh[0] >= 0 && eh[0] <= k && eh[1] == r;
                const int mp = ok ? eh[0] : 0;
                if (!ok && tid == 0) atomicOr(p.status, HS_STATUS_PLAN);
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
                            atomicOr(p.status, HS_STATUS_PLAN);
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
        } else {
            // rejected request: publish -1, leave metadata and slots alone
            if (!kPlanOnly) {
                int32_t *o = out_g + (int64_t)ireq * k;
                for (int i = tid; i < k; i += kThreads) o[i] = -1;
            }
            if (tid == 0) {
                atomicOr(p.status, abort_bits);
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
    }

    if constexpr (!kPlanOnly) {
        // ---------------- hand the fetch list to the cluster --------------
        cluster_arrive();  // phase A: leader has published
        cluster_wait();
        const int32_t *fp = mpos, *fs = mslot;
        int F = 0;
        if (crank == 0) {
            F = (int)hdr[H_F];
            if (hdr[H_FLIST]) { fp = fpos; fs = fslot; }
        } else {
            // copy the leader's list into the same place of this CTA's
            // shared memory (the layouts are identical)
            cg::cluster_group cl = cg::this_cluster();
            const uint32_t *lh = cl.map_shared_rank(hdr, 0);
            F = (int)lh[H_F];
            const bool plist = lh[H_FLIST] != 0u;
            int32_t *dp = plist ? fpos : mpos;
            int32_t *ds = plist ? fslot : mslot;
            const int32_t *lp = cl.map_shared_rank(dp, 0);
            const int32_t *ls = cl.map_shared_rank(ds, 0);
            for (int e = tid; e < F; e += kThreads) {
                dp[e] = lp[e];
                ds[e] = ls[e];
            }
            fp = dp;
            fs = ds;
            __syncthreads();
        }
        cluster_arrive();  // phase B: the leader's fetch list may be released

        const uint8_t *host_pair = p.host + ((int64_t)(r_ok ? r : 0) * p.NL + layer) * p.L * p.W;
        uint8_t *cache_pair = p.cache + pair * B * p.W;

        if (crank == 0 && hdr[H_ABORT] == 0u) {
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
            // new LRU order: [untouched (already placed by P3)] [victims] [hits]
            const int segB = (B + kThreads - 1) / kThreads;
            const int baseB = warp * 32 * segB;
            const uint32_t lt = lanemask_lt();
            uint32_t cv = 0, ch = 0;
            for (int s = 0; s < segB; ++s) {
                const int b = baseB + s * 32 + lane;
                const uint8_t f = b < B ? flags_s[b] : 0;
                cv += __popc(__ballot_sync(0xFFFFFFFFu, (f & 2) != 0));
                ch += __popc(__ballot_sync(0xFFFFFFFFu, (f & 1) != 0));
            }
            uint32_t total;
            const uint32_t base = warp_counts_exscan(cv | (ch << 16), sums, &total);
            uint32_t vr = (uint32_t)(nh - m) + (base & 0xFFFFu);
            uint32_t hr = (uint32_t)nh + (base >> 16);
            for (int s = 0; s < segB; ++s) {
                const int b = baseB + s * 32 + lane;
                const uint8_t f = b < B ? flags_s[b] : 0;
                const uint32_t bv = __ballot_sync(0xFFFFFFFFu, (f & 2) != 0);
                const uint32_t bh = __ballot_sync(0xFFFFFFFFu, (f & 1) != 0);
                if (f & 2) neworder[vr + __popc(bv & lt)] = (uint16_t)b;
                if (f & 1) {
                    neworder[hr + __popc(bh & lt)] = (uint16_t)b;
                    st[b] = 2u * t;
                }
                vr += __popc(bv);
                hr += __popc(bh);
            }
            __syncthreads();
            uint16_t *lo = p.lru + pair * B;
            for (int b = tid; b < B; b += kThreads) lo[b] = neworder[b];
            if (tid == 0) {
                p.tcount[pair] = t;
                unsigned long long *c = p.counters + (int64_t)layer * CTR_COUNT;
                atomicAdd(&c[CTR_RESOLVES], 1ull);
                atomicAdd(&c[CTR_HITS], (unsigned long long)(k - m));
                atomicAdd(&c[CTR_MISSES], (unsigned long long)m);
                atomicAdd(&c[CTR_FETCHED], (unsigned long long)F * (unsigned long long)p.W);
                if (with_plan) {
                    atomicAdd(&c[CTR_PLAN_HITS], (unsigned long long)hdr[H_PHIT]);
                    atomicAdd(&c[CTR_PLAN_MISMATCH], (unsigned long long)hdr[H_PMISS]);
                }
            }
        }

        // ---------------- P5: fetch the records -----------------------------
        if (F > 0) {
            if (csize == 1)
                fetch_records(host_pair, cache_pair, fp, fs, F, p.W, tid, kThreads);
            else if (crank > 0)
                fetch_records(host_pair, cache_pair, fp, fs, F, p.W,
                              (int)(crank - 1) * kThreads + tid, (int)(csize - 1) * kThreads);
        }
        if (crank == 0 && tid == 0 && hdr[H_ABORT] == 0u) {
            __threadfence();
            atomicExch(&p.busy[pair], 0u);
        }
        cluster_wait();  // phase B: no CTA leaves while the leader's list is read
    }
}

}  // namespace

cudaError_t prepare_kernels(size_t max_smem) {
    cudaError_t e = cudaFuncSetAttribute(resolve_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(resolve_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)max_smem);
}

cudaError_t launch_resolve(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                           const int32_t *sel, int k, int32_t *out, const void *plan,
                           int cluster, cudaStream_t st) {
    const SmemLayout sl = smem_layout(p.B, k, plan != nullptr);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_req * cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = sl.total;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, resolve_kernel<false>, p, layer, n_req, req_ids, sel, k, out,
                              static_cast<const uint8_t *>(plan), static_cast<uint8_t *>(nullptr));
}

cudaError_t launch_plan(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                        const int32_t *sel, int k, void *plan, cudaStream_t st) {
    const SmemLayout sl = smem_layout(p.B, k, false);
    resolve_kernel<true><<<n_req, kThreads, sl.total, st>>>(
        p, layer, n_req, req_ids, sel, k, nullptr, nullptr, static_cast<uint8_t *>(plan));
    return cudaGetLastError();
}

}  // namespace hs

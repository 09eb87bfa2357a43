// Internal declarations shared by the CUDA translation units of libhs.
//
// Data layout in HBM (one pool, L = L_ctx, R requests, N_l layers, B slots,
// W record bytes):
//   cache    [N_l][R][B][W]  u8     layer-major, so a layer's cache is one
//                                   [R*B][W] tensor and the published index
//                                   r*B + slot is a row of it
//   pt       [N_l][R][L]     i32    page table, -1 = host-only
//   slot_pos [N_l][R][B]     i32    position held by each slot, -1 = empty
//   stamp    [N_l][R][B]     u32    recency (0 empty, 2t-1 miss, 2t hit)
//   lru      [N_l][R][B]     u16    slots sorted by (stamp, slot)
//   tcount   [N_l][R]        u32    resolves done on the pair
//   busy     [N_l][R]        u32    1 while a resolve owns the pair
//   counters [N_l][8]        u64    see CTR_*
//   status   [1]             u32    HS_STATUS_* bits
// Host pool (pinned, device-mapped): host[N_l][R][L][W] (host_region).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace hs {

constexpr int kThreads = 512;          // threads per CTA of every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;         // portable cluster size limit
constexpr uint32_t kPlanMagic = 0x4C505348u;  // "HSPL"

enum Counter : int {
    CTR_RESOLVES = 0,
    CTR_HITS = 1,
    CTR_MISSES = 2,
    CTR_FETCHED = 3,
    CTR_PREFETCHED = 4,
    CTR_PLAN_HITS = 5,
    CTR_PLAN_MISMATCH = 6,
    CTR_COUNT = 8,
};

struct DevPool {
    const uint8_t *host;  // device address of the mapped host pool
    uint8_t *cache;
    int32_t *pt;
    int32_t *slot_pos;
    uint32_t *stamp;
    uint16_t *lru;
    uint32_t *tcount;
    uint32_t *busy;
    unsigned long long *counters;
    unsigned int *status;
    uint32_t *sink;  // a word only the touch kernel may write (never read)
    int32_t R, NL, B, W;
    int64_t L;
};

// Host records of (request r, layer l): the pool is layer-major,
// [N_l][R][L][W], so that one layer's launch reads one contiguous range.
__host__ __device__ inline int64_t host_region(int r, int l, int R, int64_t L, int W) {
    return ((int64_t)l * R + r) * L * W;
}

// Plan buffer: a 16-byte header {magic, n_req, k, layer}, then per request
// i an entry of 16 + 8k bytes: {m, req, 0, 0}, pos[k], slot[k].
struct PlanHeader {
    uint32_t magic;
    int32_t n_req, k, layer;
};

__host__ __device__ inline size_t plan_entry_bytes(int k) { return 16 + 8 * (size_t)k; }
__host__ __device__ inline size_t plan_bytes(int n_req, int k) {
    return 16 + (size_t)n_req * plan_entry_bytes(k);
}

// Hash table over the selected positions: 32-bit keys (position + 1, 0 =
// empty) and 16-bit selection indices, at most a quarter full.
__host__ __device__ inline int hash_capacity(int k) {
    int h = 64;
    while (h < 4 * k) h <<= 1;
    return h;
}

// Membership bitmap over positions: one bit per position while L <= 2^17
// (exact), otherwise 2^17 bits indexed by a hash of the position (a filter
// in front of the hash table).
constexpr int kMaxBitmapBits = 1 << 17;
__host__ __device__ inline int bitmap_bits(int64_t L) {
    int m = 1024;
    while (m < kMaxBitmapBits && (int64_t)m < L) m <<= 1;
    return m;
}

__host__ __device__ inline uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

// Shared-memory layout of the resolve / plan kernels for (B, k, L).
struct SmemLayout {
    uint32_t hdr;      // header words + per-warp scan sums
    uint32_t keys;     // u32[H]; after the probe it holds neworder u16[B]
    uint32_t kidx;     // u16[H] selection index of each key
    uint32_t bitmap;   // u32[M/32] membership bits
    uint32_t sel;      // i32[k]
    uint32_t hit;      // i32[k]: slot of a hit, -1 before ranking, -2-rank for misses
    uint32_t spos;     // i32[B]
    uint32_t order;    // u16[B]
    uint32_t flags;    // u8[B]: bit0 hit, bit1 victim
    uint32_t vrank;    // u16[B]: rank of a victim slot (plan consumption only)
    uint32_t mpos;     // i32[k]: miss positions by rank
    uint32_t mslot;    // i32[k]: victims by rank
    uint32_t fpos;     // i32[2k]: fetch list when a plan is consumed
    uint32_t fslot;    // i32[2k]
    uint32_t total;
    int H, M;
};

__host__ __device__ inline SmemLayout smem_layout(int B, int k, bool with_plan, int64_t L) {
    SmemLayout s;
    uint32_t o = 0;
    s.H = hash_capacity(k);
    s.M = bitmap_bits(L);
    s.hdr = o;    o += 256;
    s.keys = o;   { uint32_t a = 4u * s.H, b = 2u * B; o += align16(a > b ? a : b); }
    s.kidx = o;   o += align16(2u * s.H);
    s.bitmap = o; o += align16((uint32_t)s.M / 8u);
    s.sel = o;    o += align16(4u * k);
    s.hit = o;    o += align16(4u * k);
    s.spos = o;   o += align16(4u * B);
    s.order = o;  o += align16(2u * B);
    s.flags = o;  o += align16(1u * B);
    s.vrank = o;  o += with_plan ? align16(2u * B) : 0;
    s.mpos = o;   o += align16(4u * k);
    s.mslot = o;  o += align16(4u * k);
    s.fpos = o;   o += with_plan ? align16(8u * k) : 0;
    s.fslot = o;  o += with_plan ? align16(8u * k) : 0;
    s.total = o;
    return s;
}

// A follower CTA of a resolve cluster needs none of the leader's arrays.
// After the 256-byte header it keeps: for each record it staged, the share
// entry and the position (up to kStageCap records, a pool shared by its
// warps), one staged-bit word per block of 32 share entries,
// the list (positions, slots) of misses it did not stage, and then the
// staging area for whole records, `cap` records in all.
constexpr int kStageCap = 256;
struct FollowerLayout {
    uint32_t stg, stgpos, sbits, xp, xs, stage;
    int cap;
};

__host__ __device__ inline FollowerLayout follower_lists(int k) {
    FollowerLayout f;
    uint32_t o = 256;
    f.stg = o;   o += 4u * kStageCap;
    f.stgpos = o; o += 4u * kStageCap;
    f.sbits = o; o += align16(4u * (uint32_t)((k + 31) / 32));
    f.xp = o;    o += align16(4u * (uint32_t)k);
    f.xs = o;    o += align16(4u * (uint32_t)k);
    f.stage = (o + 127u) & ~127u;
    f.cap = 0;
    return f;
}

// Dynamic shared memory of a resolve launch: the leader's layout, and never
// less than what a follower's lists need.
__host__ __device__ inline uint32_t resolve_smem_bytes(int B, int k, bool with_plan, int64_t L) {
    const uint32_t a = smem_layout(B, k, with_plan, L).total;
    const uint32_t b = follower_lists(k).stage;
    return a > b ? a : b;
}

// Variants of the resolve kernel.
enum Mode : int {
    kModeResolve = 0,  // hs_resolve
    kModePlan = 1,     // hs_prefetch_plan
    kModeNoFetch = 2,  // hs_resolve_measure without the miss fetch
};

// Stage timestamps of hs_resolve_measure: slot indices of one CTA's row.
// Leader (CTA 0 of a cluster) and followers use the slots named for them.
constexpr int kStampSlots = 16;
enum Stamp : int {
    S_ENTRY = 0,      // both: first instruction
    S_LOADED = 1,     // leader: selection, slot map and LRU order in shared memory
    S_HASHED = 2,     // leader: validated, hash table and membership bits built
    S_PROBED = 3,     // leader: every slot probed (hits marked)
    S_DECIDED = 4,    // leader: misses ranked and victims chosen (decision)
    S_CHECKED = 5,    // leader: previous grid complete, early decision checked
    S_VERDICT = 6,    // both: past the cluster barrier that publishes the decision
    S_COMMITTED = 7,  // leader: page table, slot map, stamps, LRU order, counter written
    S_F_ISSUE = 8,    // follower: page-table predictions read, first staging copy issued
    S_F_ISSUED = 9,   // follower: every staging copy issued
    S_F_WAITED = 10,  // follower: previous grid complete
    S_F_LANDED = 11,  // follower: staged records in shared memory
    S_F_STORED = 12,  // follower: slot stores and unstaged fetches issued
    S_ATTEMPTS = 13,  // leader: decisions taken (a count, not a time)
    S_EXIT = 14,      // both: last instruction
    S_LEAD_FETCHED = 15,  // leader: its own share's misses fetched (launch overlap off)
};

// header word indices (u32 at smem + hdr)
enum Hdr : int {
    H_ABORT = 0,     // HS_STATUS_* bits that abort this request
    H_M = 1,         // misses
    H_NH = 2,        // non-hit slots
    H_F = 3,         // entries in the fetch list
    H_FLIST = 4,     // 0: fetch list = (mpos, mslot); 1: (fpos, fslot)
    H_T = 5,         // this resolve's t
    H_NF = 6,        // atomic fill counter of the plan-mode fetch list
    H_PMISS = 7,     // plan-mode mismatches
    H_PHIT = 8,      // plan-mode plan hits
    H_G = 9,         // follower: predicted misses in its share
    H_NX = 10,       // follower: leader misses it did not predict
    H_NSTG = 11,     // follower: staging slots handed out (may exceed the capacity)
    H_PSTAT = 12,    // plan-mode status bits, applied at the commit
    H_NL = 13,       // leader: misses of its own fetch share
    H_SUMS = 16,     // kWarps scan sums from here
};

// Host memory the GPU reads directly (hostmem.cu).  `dev` is the device
// address of `host` (the same address for VMM allocations).
struct HostBuffer {
    void *host;
    const void *dev;
    size_t bytes;               // requested
    size_t mapped;              // allocated (rounded up to the granularity)
    size_t granularity;         // VMM granularity or huge-page size, 0 for cudaHostAlloc
    size_t huge_bytes;          // bytes in transparent huge pages (huge-page kind)
    unsigned long long handle;  // VMM allocation handle, or the huge-page mapping's start
    int kind;                   // HS_HOST_ALLOC_*
    int numa;                   // node requested, -1 otherwise
};
int host_alloc(size_t bytes, int kind, int dev, HostBuffer *out);
int device_host_numa(int dev);
void host_free(HostBuffer *b);
int page_numa_node(const void *addr);

// launchers (resolve.cu, copy.cu, attention.cu, attention_heads.cu)
// plan_layer: a consumed plan may carry this layer id besides `layer` (the
// anchor whose resolve wrote it); plan_out: where an anchor's resolve
// writes its own miss plan (NULL: nowhere); overlap: the launch may start
// under the previous grid in the stream (programmatic stream
// serialisation); lead_k: the leader CTA fetches the misses among the last
// lead_k selections itself, the followers the rest (0: followers only).
cudaError_t launch_resolve(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                           const int32_t *sel, int k, int32_t *out, const void *plan,
                           int cluster, cudaStream_t st, int plan_layer = -1,
                           void *plan_out = nullptr, bool overlap = true, int lead_k = 0);
cudaError_t launch_plan(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                        const int32_t *sel, int k, void *plan, cudaStream_t st);
cudaError_t launch_resolve_measure(const DevPool &p, int layer, int n_req, const int32_t *req_ids,
                                   const int32_t *sel, int k, int32_t *out, bool no_fetch,
                                   unsigned long long *times, int cluster, cudaStream_t st,
                                   bool overlap, int lead_k);
// confined: every SM copies records of one request only (one CTA per SM,
// sm_count / n_req CTAs per request), for pools past the translation reach
cudaError_t launch_prefetch_copy(const DevPool &p, int layer, int n_req, int k,
                                 const void *plan, int sm_count, cudaStream_t st,
                                 int plan_layer, bool confined);
cudaError_t launch_init_lru(uint16_t *lru, int64_t pairs, int B, cudaStream_t st);
cudaError_t launch_touch(const void *p, size_t bytes, uint32_t *sink, int sm_count,
                         cudaStream_t st);
cudaError_t prepare_kernels(size_t max_smem);
cudaError_t prepare_copy_kernel();
cudaError_t launch_attention(const void *q, const void *cache, int64_t cache_rows,
                             const int32_t *idx, int n_req, int k, int heads, float scale,
                             float *out, cudaStream_t st);
cudaError_t attention_status(uint32_t *status);
cudaError_t launch_attention_heads(const void *q, const void *cache, int64_t cache_rows,
                                   const int32_t *idx, int n_req, int k, int heads, float scale,
                                   float *out, cudaStream_t st);
cudaError_t launch_gather_probe(const uint8_t *src, uint8_t *dst, const int32_t *idx,
                                int64_t n_rec, int W, int sm_count, cudaStream_t st);

}  // namespace hs

/*
 * hs.h -- C ABI of a GB300-native RESOLVE step for a two-level KV cache.
 *
 * The method (HiSparse, "Scaling Sparse-Attention Decoding with Hierarchical
 * KV Cache Management"; described in "Inference Systems Infrastructure Notes
 * (6): HiSparse" and in the Pith review of arXiv 2608.07009):
 *
 *  - every KV record lives in a pinned, device-mapped host pool, addressed
 *    contiguously by logical position; it is the only authoritative copy
 *    (notes, section 2 "Two-Level Hierarchy", items 1 and 2.1.2);
 *  - each (request, layer) pair owns B >= k GPU slots, a page table over the
 *    L_ctx positions (slot or host-only) and per-slot recency for LRU
 *    (notes, section 2, items 2 and 3);
 *  - one fused RESOLVE launch per sparse layer and decode step turns the k
 *    selected positions of every request into physical slot indices,
 *    fetching misses from host memory with GPU-thread loads (notes,
 *    section 3 "RESOLVE: Five Stages in One Launch"; Pith review, "What
 *    carries the argument");
 *  - for layers that share an anchor layer's selection, the misses are
 *    known before the layer runs: a plan is computed and replayed by a
 *    copy-only kernel on a side stream (notes, section 4 "Exact Layer-Wise
 *    Prefetching").
 *
 * Conventions
 *  - Every call returns an int: HS_OK (0) or a negative HS_ERR_* code.
 *  - hs_resolve, hs_prefetch_plan and hs_prefetch_copy only enqueue work on
 *    the given stream: they never synchronise, never allocate, and can be
 *    captured in a CUDA graph when their arguments stay fixed.
 *  - Errors in device-resident inputs (a position outside [0, L_ctx), a
 *    repeated position, a request id outside the pool, a request resolved
 *    twice at once, a malformed plan) never trap the GPU.  The kernel sets a
 *    bit in the pool's status word (HS_STATUS_*), publishes -1 for the whole
 *    request and leaves that request's metadata and slots untouched;
 *    hs_stats reports the bits and returns HS_ERR_DEVICE_INPUT.
 *  - Ownership: the pool owns the host pool and every device array it
 *    allocates; callers own selections, outputs, plans and streams.
 *  - Ordering: two operations on the same layer must not overlap on the GPU.
 *    A resolve that consumes a plan must be ordered after the
 *    hs_prefetch_copy of that plan (an event between the streams).
 *  - One device: the pool lives on the device current at hs_create_pool;
 *    every later call must run with that device current.
 */
#ifndef HS_H
#define HS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define HS_OK 0
#define HS_ERR_INVALID_ARG (-1)   /* bad descriptor, index, size or pointer */
#define HS_ERR_CUDA (-2)          /* a CUDA runtime call failed */
#define HS_ERR_NOMEM (-3)         /* allocation refused or over the limit */
#define HS_ERR_DEVICE_INPUT (-4)  /* a kernel flagged bad device input (hs_stats) */
#define HS_ERR_TIMEOUT (-5)       /* reserved: no call waits on the GPU with a limit */
#define HS_ERR_UNSUPPORTED (-6)   /* sizes beyond what this build's kernels handle */

/* ---- bits of the device status word (hs_stats_t.status) ---------------- */
#define HS_STATUS_POS_RANGE 0x1u  /* a selected position outside [0, L_ctx) */
#define HS_STATUS_POS_DUP 0x2u    /* a position selected twice in one request */
#define HS_STATUS_REQ_RANGE 0x4u  /* a request id outside [0, n_requests) */
#define HS_STATUS_REQ_BUSY 0x8u   /* a request resolved by two overlapping calls */
#define HS_STATUS_PLAN 0x10u      /* a plan that does not belong to this call */
#define HS_STATUS_META 0x20u      /* slot map or LRU order found corrupted */

/* Opaque pool: host records, GPU slots and metadata of every
 * (request, layer) pair.  Library-owned. */
typedef struct hs_pool hs_pool;

typedef struct {
    int32_t n_requests;   /* R: request rows in the pool (>= 1) */
    int32_t n_layers;     /* N_l: sparse layers (>= 1) */
    int64_t n_positions;  /* L_ctx: logical positions per request (1 .. 2^31-1) */
    int32_t record_bytes; /* W = W_KV * s: bytes per KV record, a multiple of 16 */
    int32_t slots;        /* B: GPU slots per (request, layer) (1 .. 32767) */
    int32_t max_k;        /* largest k passed to hs_resolve (1 .. slots) */
    /* layer_anchor[l]: the layer whose selection layer l shares (l itself for
       an anchor).  May be NULL (every layer its own anchor).  Copied. */
    const int32_t *layer_anchor;
    /* Refuse pools whose pinned host pool would exceed this many bytes
       (0: no limit beyond what the system grants).  HS_ERR_NOMEM. */
    uint64_t host_limit_bytes;
    /* How the host pool is allocated: HS_HOST_ALLOC_* (0: the library's
       choice, see HS_HOST_ALLOC_AUTO). */
    int32_t host_alloc;
    /* Whether consecutive resolves may overlap: HS_OVERLAP_* (0: the
       library's choice, see HS_OVERLAP_AUTO). */
    int32_t launch_overlap;
} hs_pool_desc;

/* ---- launch overlap (hs_pool_desc.launch_overlap) ---------------------- */
/* ON: a resolve may start under the kernel ahead of it in the stream
 * (programmatic dependent launch): it stages its predicted misses and
 * takes its decision while that kernel finishes, and keeps the decision
 * only if its inputs are unchanged once that kernel has completed.  Best
 * while every host record stays within the device's translation reach:
 * the reads of two or three layers' records then share it freely.
 * OFF: each resolve starts when the kernel ahead of it has completed, so
 * one layer's records are read at a time, and the leader CTA of each
 * request fetches a share of the misses beside its followers.  Best for
 * pools past the reach, where reads of several layers' records at once
 * thrash the device's translations.
 * AUTO: ON for pools of at most HS_OVERLAP_AUTO_MAX_HOST_BYTES of host
 * records, OFF above (measured on GB300: the 59 GB pool of 64 requests x 8
 * layers resolves 1.7x faster with OFF; 5 GB pools faster with ON). */
#define HS_OVERLAP_AUTO 0
#define HS_OVERLAP_ON 1
#define HS_OVERLAP_OFF 2
#define HS_OVERLAP_AUTO_MAX_HOST_BYTES (16ull << 30)

/* ---- host pool memory (hs_pool_desc.host_alloc, hs_link_probe) --------- */
/* The library's choice: for pools of at most HS_OVERLAP_AUTO_MAX_HOST_BYTES
 * of records, HS_HOST_ALLOC_PINNED; above, HS_HOST_ALLOC_THP_REGISTERED when
 * the kernel backs at least 90 % of the pool with huge pages, else
 * HS_HOST_ALLOC_PINNED.  (Measured on GB300: scattered 1152-byte GPU-thread
 * reads of cudaHostAlloc memory run at the full pinned-copy rate while the
 * pool stays within the device's translation reach, about 16 GiB, and
 * collapse past it, where huge-page memory reads twice as fast; VMM
 * host-NUMA memory reads at about a fifth of the rate at any size.) */
#define HS_HOST_ALLOC_AUTO 0
/* cudaHostAlloc(Mapped | Portable), made while the calling thread prefers
 * the host NUMA node closest to the device (set_mempolicy), so that the
 * pinned pages come from that node; the device reads them through its
 * mapping of the allocation. */
#define HS_HOST_ALLOC_PINNED 1
/* Virtual memory management API: one pinned host allocation on the NUMA
 * node closest to the device (cudaDevAttrHostNumaId), mapped at a 1 GiB
 * aligned virtual range readable and writable by the device and the host
 * at the same address. */
#define HS_HOST_ALLOC_VMM_NUMA 2
/* Anonymous host memory in transparent huge pages (madvise on the mapping,
 * aligned to the huge-page size), first touched by threads preferring the
 * device's host NUMA node, then pinned and mapped for the device with
 * cudaHostRegister(Mapped | Portable).  Warm, it reads scattered records
 * past the translation reach about twice as fast as cudaHostAlloc memory
 * (measured on GB300); the first resolves over freshly written records are
 * far slower (hs_touch_records, hs_warm_pool). */
#define HS_HOST_ALLOC_THP_REGISTERED 3

typedef struct {
    uint64_t resolves;          /* resolves committed (one per request per call) */
    uint64_t hits;              /* selected positions found resident */
    uint64_t misses;            /* selected positions fetched into a victim slot */
    uint64_t fetched_bytes;     /* bytes the resolve kernel copied from host */
    uint64_t prefetched_bytes;  /* bytes hs_prefetch_copy copied from host */
    uint64_t plan_hits;         /* misses whose copy a plan had already done */
    uint64_t plan_mismatches;   /* plan pairs or misses that did not match */
    uint32_t status;            /* HS_STATUS_* bits since the last hs_stats */
} hs_stats_t;

/* Device views of one layer, for the attention consumer and for checks.
 * Layout: the layer's cache is [n_requests * slots][record_bytes] bytes, so
 * a published index i addresses row i; the other arrays are
 * [n_requests][...] row-major. */
typedef struct {
    void *cache;          /* [R*B][W] slot contents (HBM) */
    int32_t *page_table;  /* [R][L_ctx] slot of each position, -1 = host-only */
    int32_t *slot_pos;    /* [R][B] position held by each slot, -1 = empty */
    uint32_t *stamps;     /* [R][B] recency: 0 empty, 2t-1 filled at the t-th
                             resolve of the pair, 2t hit at the t-th resolve */
    uint16_t *lru;        /* [R][B] slots in ascending (stamp, slot) order */
    uint32_t *resolves;   /* [R] resolves done on each pair (t) */
} hs_views;

/*
 * Creates a pool: allocates the pinned, device-mapped host pool
 * (R * N_l * L_ctx * W bytes, layer-major host[l][r][pos][W] -- one layer's
 * records one contiguous range -- left uninitialised) and
 * the device arrays: cache (N_l * R * B * W bytes), page tables
 * (N_l * R * L_ctx * 4 bytes), slot maps, stamps, LRU orders, counters.
 * All slots start empty, every page-table entry host-only, every stamp 0.
 * The device-side footprint of KV records per request is N_l * B * W
 * bytes whatever L_ctx is (notes, section 2, "HBM usage = N_l x B x W_KV x s").
 * Errors: HS_ERR_INVALID_ARG (desc fields out of range, out == NULL),
 * HS_ERR_NOMEM (over host_limit_bytes or an allocation failed),
 * HS_ERR_UNSUPPORTED (B or max_k needs more shared memory than a CTA has),
 * HS_ERR_CUDA.  On error *out is NULL and nothing stays allocated.
 */
int hs_create_pool(const hs_pool_desc *desc, hs_pool **out);

/* Synchronises the device, then frees everything the pool owns.
 * NULL is accepted and ignored. */
int hs_destroy_pool(hs_pool *pool);

/* Host address of the records of (req, layer): L_ctx * W bytes, record
 * `pos` at byte offset pos * W.  The caller (prefill, a generator) writes
 * them before the first resolve that can select them and must not change a
 * record while a kernel may read it. */
int hs_host_records(hs_pool *pool, int32_t req, int32_t layer, void **host_ptr);

/* Device views of `layer` (see hs_views). */
int hs_device_views(hs_pool *pool, int32_t layer, hs_views *out);

/* Where a pool's memory lives (for placement checks and reports). */
typedef struct {
    int32_t host_alloc;        /* HS_HOST_ALLOC_PINNED or HS_HOST_ALLOC_VMM_NUMA */
    int32_t device;            /* CUDA device of the pool */
    int32_t device_numa;       /* host NUMA node closest to that device, -1 unknown */
    int32_t host_numa_first;   /* NUMA node of the first page of the host pool, -1 unknown */
    int32_t host_numa_last;    /* NUMA node of its last page, -1 unknown */
    int32_t launch_overlap;    /* HS_OVERLAP_ON or HS_OVERLAP_OFF, as resolved */
    uint64_t host_bytes;       /* bytes of host records */
    uint64_t host_mapped_bytes;/* bytes allocated for them (granularity-rounded) */
    uint64_t host_granularity; /* VMM allocation granularity, 0 for cudaHostAlloc */
    uint64_t device_bytes;     /* bytes of device arrays the pool allocated */
    uint64_t host_huge_bytes;  /* bytes of the host pool in transparent huge pages */
    uint64_t warmup_us;        /* time the last hs_warm_pool took, µs (0: never called) */
} hs_pool_info_t;

/* Fills *out.  Errors: HS_ERR_INVALID_ARG (NULL pool or out). */
int hs_pool_info(hs_pool *pool, hs_pool_info_t *out);

/*
 * Reads every byte of the host records of (req, layer) once from the device
 * (16-byte loads; req and/or layer -1 for all), enqueued on `stream`.  Not
 * part of the method: on GB300 the device's first reads of host records the
 * CPU has just written are slow, so a caller that has just written records
 * (prefill) can pay that here, off the latency-critical path (measured:
 * 59 GB of a freshly written huge-page pool in 1.5-1.8 s).
 * Errors: HS_ERR_INVALID_ARG, HS_ERR_CUDA.
 */
int hs_touch_records(hs_pool *pool, int32_t req, int32_t layer, void *stream);

/*
 * Warms a pool after its records are written and before its first resolve:
 * every byte of the host records read once (hs_touch_records), sixteen
 * synthetic resolve steps through every (request, layer) pair (each step k
 * new distinct positions per request, so that every selection misses and
 * every slot is written), then the empty state of hs_create_pool again
 * (hs_reset).  Not part of the method: on GB300 the first resolve step over
 * a freshly written 59 GB huge-page pool took 1.3-3.1 s cold, 54-61 ms
 * after the synthetic steps alone and 7-98 ms after this call, depending on
 * the pool instance (2.0-2.9 s in all).  Synchronous; the time it took is hs_pool_info_t.warmup_us.  It
 * discards the pool's slot state, so it must not be called once real
 * resolves have run.  Errors: HS_ERR_INVALID_ARG, HS_ERR_NOMEM (its two
 * small selection buffers), HS_ERR_CUDA.
 */
int hs_warm_pool(hs_pool *pool);

/* Host NUMA node closest to CUDA device `device` (cudaDevAttrHostNumaId),
 * where a pool created on that device places its host records; -1 when
 * the system reports none or the device does not exist.  A process serving
 * several devices (one per rank) can bind each rank's threads to it. */
int hs_device_host_numa(int32_t device);

/*
 * RESOLVE for one sparse layer: for each of the n_req requests
 * r = d_req_ids[i] (or r = i when d_req_ids is NULL), given its k selected
 * positions d_sel[i][0..k), one fused launch
 *   1. builds a shared-memory hash table over the selected positions,
 *   2. probes every slot's position against it to mark hits,
 *   3. gives the j-th miss (selection order) the j-th victim, victims being
 *      the non-hit slots in ascending (stamp, slot) order,
 *   4. copies each missed record from the host pool into its victim slot
 *      with 16-byte non-coherent GPU-thread loads,
 *   5. updates page table, slot map, stamps (misses 2t-1, hits 2t) and LRU
 *      order, and writes d_out[i][j] = r * B + slot of d_sel[i][j].
 * (notes, section 3; Pith review, "What carries the argument".)
 * d_req_ids: device int32[n_req] or NULL; ids must be distinct.
 * d_sel: device int32[n_req][k]; d_out: device int32[n_req][k].  The three
 *   are 4-byte aligned (HS_ERR_INVALID_ARG otherwise).
 * d_plan: NULL, or a plan with the same n_req, request ids, selection and
 *   k, already copied by hs_prefetch_copy into this layer: one made by
 *   hs_prefetch_plan for this layer, or the miss plan hs_resolve_anchor
 *   wrote when it resolved this layer's anchor.  Misses the plan covered
 *   are not copied again; any plan pair that is not exactly this resolve's
 *   own is re-fetched (and a slot the copy wrote for such a pair is
 *   refilled with the record it must hold), so the result is the same with
 *   or without a plan.  16-byte aligned.
 * The launch may start before the kernel ahead of it in the stream has
 * completed (programmatic dependent launch; hs_resolve allows the next
 * launch as soon as it starts, so consecutive resolves overlap): it then
 * reads d_req_ids, d_sel, d_plan, the page table, the layer's metadata and
 * the host records early, stages predicted misses in shared memory (without
 * a plan) and takes its decision, but writes no global memory until that
 * kernel has completed, and keeps the decision only if the request id, all
 * k selections and the pair's resolve counter are unchanged by then (it
 * decides again otherwise).  The result is the one a launch started after
 * that kernel ended would give.  d_plan is not checked that way: the
 * ordering rule above (after the hs_prefetch_copy of the plan, which never
 * starts before the plan is complete) keeps it fixed.
 * n_req == 0 enqueues nothing.  Errors: HS_ERR_INVALID_ARG (layer, n_req > R,
 * k outside [1, max_k], NULL d_sel/d_out), HS_ERR_CUDA (launch failed).
 */
int hs_resolve(hs_pool *pool, int32_t layer, int32_t n_req, const int32_t *d_req_ids,
               const int32_t *d_sel, int32_t k, int32_t *d_out, const void *d_plan,
               void *stream);

/*
 * Measurement variant of hs_resolve (not for serving; it never feeds a
 * throughput figure of hs_resolve).  Same arguments, launch shape and
 * results as hs_resolve without a plan, with two options:
 *   flags & HS_MEASURE_NO_FETCH: the resolve without step 4 -- hash build,
 *     probe, victim choice, page-table / slot-map / stamp / LRU update and
 *     publication all run, no host record is read and no slot is written.
 *     It isolates the metadata cost, which the pages report as no
 *     measurable per-token cost against a no-IO baseline (Pith review,
 *     Fig. 7 "Miss-resolution breakdown" and the verdict's no-IO oracle).
 *     Afterwards the pool's slots no longer hold the records their slot
 *     map names: hs_reset before resolving for real.  fetched_bytes is not
 *     counted; resolves, hits and misses are.
 *   d_times (NULL: none): device u64[n_req][hs_measure_stamp_slots()],
 *     8-byte aligned; each CTA of request i's cluster (at most 8) writes
 *     %globaltimer nanosecond stamps of its stages into its row of 16
 *     (row i * 8 + cta; slot meanings in the HS_STAMP_* list below; slots
 *     a CTA does not reach are left as they were).
 * Errors as hs_resolve; HS_ERR_INVALID_ARG for unknown flags or a
 * misaligned d_times.
 */
#define HS_MEASURE_NO_FETCH 0x1
/* Stamp slots: leader = CTA 0 of a request's cluster, followers = the
 * others.  ENTRY, VERDICT (past the cluster barrier that publishes the
 * decision) and EXIT for every CTA; LOADED (selection and slot metadata in
 * shared memory), HASHED, PROBED, DECIDED (misses ranked, victims chosen),
 * CHECKED (previous grid complete, early decision confirmed), COMMITTED
 * (metadata written) for the leader; F_ISSUE (first staging copy issued),
 * F_ISSUED (all issued), F_WAITED (previous grid complete), F_LANDED
 * (staged records in shared memory), F_STORED (slot stores and unstaged
 * fetches issued) for followers; LEAD_FETCHED (the leader's own share of
 * misses fetched, when launch overlap is off) for the leader; ATTEMPTS
 * holds the leader's count of decisions, not a time. */
#define HS_STAMP_ENTRY 0
#define HS_STAMP_LOADED 1
#define HS_STAMP_HASHED 2
#define HS_STAMP_PROBED 3
#define HS_STAMP_DECIDED 4
#define HS_STAMP_CHECKED 5
#define HS_STAMP_VERDICT 6
#define HS_STAMP_COMMITTED 7
#define HS_STAMP_F_ISSUE 8
#define HS_STAMP_F_ISSUED 9
#define HS_STAMP_F_WAITED 10
#define HS_STAMP_F_LANDED 11
#define HS_STAMP_F_STORED 12
#define HS_STAMP_ATTEMPTS 13
#define HS_STAMP_EXIT 14
#define HS_STAMP_LEAD_FETCHED 15
int hs_resolve_measure(hs_pool *pool, int32_t layer, int32_t n_req, const int32_t *d_req_ids,
                       const int32_t *d_sel, int32_t k, int32_t *d_out, int32_t flags,
                       uint64_t *d_times, void *stream);

/* u64 entries per request in hs_resolve_measure's d_times (8 CTAs x 16). */
int32_t hs_measure_stamp_slots(void);

/*
 * hs_resolve of an anchor layer that also writes its miss plan: for every
 * request, the (position, victim slot) pairs it commits, in the format of
 * hs_prefetch_plan, into d_plan_out (hs_plan_bytes(n_req, k) bytes,
 * 16-byte aligned; a rejected request gets an empty entry).  The layers
 * that share the anchor's selection (desc.layer_anchor) and have seen the
 * same selections since the pool was created or reset hold the same slots
 * in the same recency order, so this is their miss plan too: the anchor's
 * miss plan that a copy-only kernel replays into them ahead of their own
 * resolves (notes, section 4 "Exact Layer-Wise Prefetching"; Pith review,
 * Fig. 8) -- hs_prefetch_copy(target, d_plan_out) on a side stream, then
 * hs_resolve(target, ..., d_plan_out), with no hs_prefetch_plan launch.
 * A layer whose history differs stays exact through the consuming
 * resolve's check of every pair.  The plan is written after the previous
 * grid in the stream has completed (like every global write of the
 * resolve); it must not be overwritten while a copy or resolve that
 * consumes it may run.  Errors as hs_resolve, and HS_ERR_INVALID_ARG for a
 * NULL or misaligned d_plan_out.
 */
int hs_resolve_anchor(hs_pool *pool, int32_t layer, int32_t n_req, const int32_t *d_req_ids,
                      const int32_t *d_sel, int32_t k, int32_t *d_out, void *d_plan_out,
                      void *stream);

/* Bytes of a plan buffer for n_req requests of k selections. */
size_t hs_plan_bytes(int32_t n_req, int32_t k);

/*
 * Exact layer-wise prefetch, plan half: runs steps 1-3 of hs_resolve for
 * target_layer against that layer's own current metadata, read-only, with
 * the anchor layer's selection d_sel, and writes the (position, victim)
 * pairs of every request into d_plan (hs_plan_bytes(n_req, k) bytes,
 * 16-byte aligned).  For a layer whose history matches its anchor's, the
 * plan is the anchor's miss plan (notes, section 4).  target_layer must
 * share anchor_layer's selection (desc.layer_anchor); the metadata of
 * target_layer must not change between this call and the resolve that
 * consumes the plan.  Errors as hs_resolve.
 */
int hs_prefetch_plan(hs_pool *pool, int32_t anchor_layer, int32_t target_layer,
                     int32_t n_req, const int32_t *d_req_ids, const int32_t *d_sel,
                     int32_t k, void *d_plan, void *stream);

/*
 * Exact layer-wise prefetch, copy half: a copy-only kernel that writes the
 * host record (r, target_layer, pos) into slot `slot` of request r for
 * every pair of d_plan (n_req, k as given to hs_prefetch_plan or
 * hs_resolve_anchor; a plan of target_layer or of its anchor layer).
 * Meant for a side stream so that the transfer overlaps other work (notes,
 * section 4).  It touches no metadata: the consuming hs_resolve commits it.
 */
int hs_prefetch_copy(hs_pool *pool, int32_t target_layer, int32_t n_req, int32_t k,
                     const void *d_plan, void *stream);

/*
 * Synchronises the device, then reports the counters of `layer` (-1: the
 * sum over all layers) and the status word, and clears the status word.
 * Returns HS_ERR_DEVICE_INPUT when a status bit was set (the counters are
 * still filled in).  Not callable during stream capture.
 */
int hs_stats(hs_pool *pool, int32_t layer, hs_stats_t *out);

/* Synchronises, then empties every slot of every pair (as after
 * hs_create_pool) and zeroes the counters; the host records are kept. */
int hs_reset(hs_pool *pool);

/*
 * Link ceiling probe (not part of the hot path).  Allocates `bytes` of host
 * memory the way host_alloc says (HS_HOST_ALLOC_*), and min(bytes, 1 GiB)
 * on the device, then reports the best of `reps` timed runs (CUDA events) of
 *   *h2d_gbs:    cudaMemcpyAsync host -> device of min(bytes, 1 GiB) from
 *                the start of the host buffer;
 *   *gather_gbs: a kernel that copies min(bytes, 1 GiB) worth of
 *                record_bytes-sized records, from record indices drawn
 *                uniformly over the WHOLE host buffer (a permutation when
 *                bytes <= 1 GiB), into device memory with 16-byte
 *                GPU-thread loads -- the miss fetch's access pattern over a
 *                pool of `bytes`.
 * Either output pointer may be NULL.  Frees what it allocated.
 * Errors: HS_ERR_INVALID_ARG, HS_ERR_NOMEM, HS_ERR_UNSUPPORTED (the
 * allocation kind is not available), HS_ERR_CUDA.
 */
int hs_link_probe(size_t bytes, int32_t reps, int32_t record_bytes, int32_t host_alloc,
                  double *h2d_gbs, double *gather_gbs);

/*
 * Sparse attention consumer over published slots (decode).  For each of
 * n_req requests and each of its `heads` query heads, attention of
 * q[i][h] (576 bf16) over the k records d_cache[d_idx[i][j]] -- the rows
 * hs_resolve published -- with keys = the whole 576-element bf16 record and
 * values = its first 512 elements (MLA latent records, 1152 bytes):
 *   out[i][h] = softmax_j(scale * q[i][h] . K_j) V_j     (fp32 out[n_req][heads][512]).
 * This is the attention backend reading the slots resolve publishes; the
 * model output is unchanged because only the placement of the records
 * changes (notes, section 5 "Why It Is Exact"; Pith review, "What carries
 * the argument").  Rows outside [0, cache_rows) are masked out (a request a
 * resolve rejected publishes -1); a head with no valid key gets zeros.
 * d_q: device bf16 [n_req][heads][576]; d_cache: a layer's cache,
 * cache_rows rows of 1152 bytes (hs_device_views); d_idx: device int32
 * [n_req][k]; d_out: device fp32.  d_q, d_cache and d_out 16-byte
 * aligned; n_req <= 65535; heads a positive multiple of 16.  One kernel is
 * enqueued on `stream` (a thread-block cluster per request and 16 heads,
 * whose CTAs split the keys and merge their partial results on chip);
 * nothing is allocated and no scratch memory is needed.  The split of the
 * keys depends on (n_req, k, heads) and the device only, so equal inputs
 * give bit-identical outputs.  A pipeline wait that runs out of time (one
 * second) makes the affected outputs NaN and sets HS_ATTN_STATUS_TIMEOUT
 * (see hs_attention_status).  Errors: HS_ERR_INVALID_ARG, HS_ERR_CUDA.
 */
int hs_sparse_attention(const void *d_q, const void *d_cache, int64_t cache_rows,
                        const int32_t *d_idx, int32_t n_req, int32_t k, int32_t heads,
                        float scale, float *d_out, void *stream);

#define HS_ATTN_STATUS_TIMEOUT 0x1u

/* Synchronises the device, then returns in *status and clears the
 * HS_ATTN_STATUS_* bits that hs_sparse_attention calls have set on the
 * current device since the last call (0: none).  Errors:
 * HS_ERR_INVALID_ARG (status == NULL), HS_ERR_CUDA. */
int hs_attention_status(uint32_t *status);

/*
 * Sparse attention consumer for token records of per-head blocks (the
 * Quest-style token records: for `heads` key-value heads of 128 dimensions,
 * the record holds the heads' bf16 keys, head after head, then their bf16
 * values, 512 bytes per head, so W = heads * 512).  For each of n_req
 * requests and each head h, attention of q[i][h] (128 bf16) over the k
 * records d_cache[d_idx[i][j]] -- the rows hs_resolve published:
 *   out[i][h] = softmax_j(scale * q[i][h] . K_jh) V_jh     (fp32 out[n_req][heads][128]),
 * with K_jh = elements [128h, 128h + 128) and V_jh = elements
 * [128(heads + h), 128(heads + h) + 128) of record j.  Like hs_sparse_attention
 * it is the consumer side of the exactness claim (notes, section 5 "Why It
 * Is Exact").  d_q: device bf16 [n_req][heads][128]; d_cache: device rows of
 * heads * 512 bytes, cache_rows of them; d_idx: device int32 [n_req][k]
 * (an index outside [0, cache_rows) masks its row; a request with every
 * row masked gets zeros); d_out: device fp32 [n_req][heads][128].  The
 * three buffers are 16-byte aligned.  Scores and sums are fp32 over the
 * bf16 inputs; one launch, no workspace, no waits that can time out; the
 * split of the rows depends on (n_req, k) and the device only, so equal
 * inputs give bit-identical outputs.  1 <= heads <= 8.  n_req == 0 enqueues
 * nothing.  Errors: HS_ERR_INVALID_ARG, HS_ERR_CUDA.
 */
int hs_sparse_attention_heads(const void *d_q, const void *d_cache, int64_t cache_rows,
                              const int32_t *d_idx, int32_t n_req, int32_t k, int32_t heads,
                              float scale, float *d_out, void *stream);

/* Kernels launched per call of hs_resolve / hs_prefetch_plan /
 * hs_prefetch_copy (for launch accounting; always 1 in this build). */
int32_t hs_kernels_per_call(void);

/* Static description of an error code. */
const char *hs_strerror(int code);

/* ---- resolve without allocating --------------------------------------- */

/* Largest request count hs_resolve_noalloc accepts. */
#define HS_NOALLOC_MAX_REQUESTS 4096

/* One layer's state, owned and allocated by the caller.  Initial (empty)
 * state: every page_table and slot_pos entry -1, stamps 0, lru[r][b] = b,
 * resolves 0 -- the state hs_create_pool gives its own arrays. */
typedef struct {
    int32_t n_requests;        /* R: request rows (1 .. HS_NOALLOC_MAX_REQUESTS) */
    int64_t n_positions;       /* L_ctx (1 .. 2^31-1) */
    int32_t record_bytes;      /* W: a multiple of 16 */
    int32_t slots;             /* B (1 .. 32767) */
    const void *host_records;  /* device-readable address of the records,
                                  [R][L_ctx][W]: record (r, pos) at byte
                                  (r * L_ctx + pos) * W, e.g. mapped pinned
                                  host memory */
    void *cache;               /* [R*B][W] slot contents */
    int32_t *page_table;       /* [R][L_ctx] */
    int32_t *slot_pos;         /* [R][B] */
    uint32_t *stamps;          /* [R][B] */
    uint16_t *lru;             /* [R][B] */
    uint32_t *resolves;        /* [R] */
} hs_layer_state;

/*
 * hs_resolve for one layer whose state the caller owns, without allocating
 * anything.  The pages have no counterpart to this call; it exists for
 * callers that cannot allocate device memory at the point where they
 * resolve: serving engines that hand all free device memory to their own
 * caching allocator at start-up (a cudaMalloc behind its back fails or
 * fragments that reserve), and latency-critical loops where cudaMalloc and
 * cudaFree would synchronise the device and stall every stream.
 *
 * Computation and output are those of hs_resolve (same kernel, same
 * d_req_ids / d_sel / k / d_out conventions, no plan).  The per-request
 * claim flags and counters that a pool keeps in its own device memory live
 * here in one fixed scratch array compiled into the library: room for
 * HS_NOALLOC_MAX_REQUESTS requests, held by every device that loads the
 * library until the process exits.  The first call on a device looks up
 * that array's device address (cudaGetSymbolAddress) and configures the
 * kernel; make that first call before any stream capture on the device.
 * The address is kept per device and per context: after a device reset the
 * next call (again outside a capture) looks it up anew in the new context.
 * Each call clears the part of the array it uses (an asynchronous memset on
 * `stream`) before launching, and every call shares the array: calls that
 * overlap on the GPU, on any streams, race.  Per-call counters are not
 * reported.
 *
 * d_status: NULL, or a device u32 into which the kernel ORs HS_STATUS_* bits
 *   for rejected requests (never cleared by the call).
 * Alignment: host_records and cache 16 bytes; page_table, slot_pos,
 * stamps, resolves, d_req_ids, d_sel, d_out and d_status 4 bytes; lru 2
 * bytes (the kernel's access widths).
 * Errors: HS_ERR_INVALID_ARG (NULL state/arrays/d_sel/d_out, fields out of
 * range, n_req > R, k outside [1, B], a misaligned pointer: refused before
 * anything is enqueued); HS_ERR_UNSUPPORTED (R above
 * HS_NOALLOC_MAX_REQUESTS, or B and k needing more shared memory than a CTA
 * has); HS_ERR_CUDA.  No cudaMalloc, cudaFree or allocating library routine
 * is called.
 */
int hs_resolve_noalloc(const hs_layer_state *state, int32_t n_req, const int32_t *d_req_ids,
                       const int32_t *d_sel, int32_t k, int32_t *d_out, uint32_t *d_status,
                       void *stream);

#ifdef __cplusplus
}
#endif
#endif /* HS_H */

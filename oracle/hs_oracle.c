/*
 * CPU oracle for the RESOLVE step of a two-level KV cache (HiSparse).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header or table with the CUDA path.
 *
 * What it computes, for one (request, layer) pair, follows the pages:
 *
 *  - State ("Inference Systems Infrastructure Notes (6): HiSparse", section 2,
 *    "Two-Level Hierarchy"): B hot-cache slots (B >= k), a page table over
 *    the L_ctx logical positions mapping each to a slot or to "host-only",
 *    and per-slot recency information for LRU.  The host pool (addressed by
 *    logical position, section 2.1) is the only authoritative copy.
 *  - One resolve per layer and step (same page, section 3 "RESOLVE"; Pith
 *    review, "What carries the argument"): detect hits among the selected
 *    positions, pick LRU victims with hits promoted above the misses fetched
 *    in this step, fetch the misses from host memory, update the page table
 *    and recency, publish one physical slot per selected entry.
 *
 * Readings where the pages are silent (each is restated in the design notes):
 *  - recency is a per-slot stamp: empty slots 0, a miss filled at the t-th
 *    resolve of this pair gets 2t-1, a hit gets 2t, so within one step hits
 *    rank above the step's misses and across steps it is plain LRU;
 *  - victims are the non-hit slots taken in ascending (stamp, slot) order,
 *    and the j-th miss in selection order receives the j-th victim;
 *  - published index of selected entry i is r*B + slot (a row of the
 *    layer's [R*B][W] cache);
 *  - a selection with a position outside [0, L), a repeated position, or
 *    k > B is rejected: outputs -1, state untouched.
 *
 * The "hit" test is the plain definition (page-table entry present), not the
 * hash-and-probe route of the GPU kernel; victim choice is a full sort of the
 * candidates.  Both are deliberately the slow, obvious form.
 *
 * Exact layer-wise prefetch (HiSparse notes, section 4 "Exact Layer-Wise
 * Prefetching"): a plan is the list of (position, victim slot) pairs that the
 * layer's next resolve will fill, computed read-only from the layer's own
 * state and the anchor's selection.  A copy step writes host[pos] into each
 * planned slot; the consuming resolve skips the copy of every miss whose pair
 * matches the plan exactly, fetches the others, and re-fetches the final
 * owner's record into any slot that a non-matching pair wrote, so that the
 * result never depends on the plan being right.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    ORA_OK = 0,
    ORA_ERR_ARG = 1,      /* k < 1, k > B, null pointers */
    ORA_ERR_RANGE = 2,    /* a selected position outside [0, L) */
    ORA_ERR_DUP = 3,      /* a position selected twice */
    ORA_ERR_STATE = 4,    /* internal inconsistency (page table vs slots) */
};

/* State of one (request, layer) pair.  All arrays are owned by the caller. */
typedef struct {
    int32_t B;            /* slots */
    int32_t W;            /* record bytes */
    int64_t L;            /* logical positions (L_ctx) */
    int32_t *slot_pos;    /* [B] position held by each slot, -1 = empty */
    uint32_t *stamp;      /* [B] recency stamps */
    int32_t *pt;          /* [L] page table: slot of each position, -1 = host-only */
    uint32_t *t;          /* number of resolves done on this pair */
    uint8_t *cache;       /* [B][W] mirror of the GPU slots, or NULL */
    const uint8_t *host;  /* [L][W] host records of this pair, or NULL */
    /* counters: 0 hits, 1 misses, 2 fetched bytes, 3 plan hits,
       4 plan mismatches, 5 prefetched bytes, 6 resolves */
    uint64_t *counters;
} ora_pair;

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

static int cmp_u64(const void *a, const void *b) {
    uint64_t x = *(const uint64_t *)a, y = *(const uint64_t *)b;
    return (x > y) - (x < y);
}

/* Selection must be k distinct positions in [0, L), 1 <= k <= B. */
int ora_validate(const ora_pair *s, const int32_t *sel, int32_t k) {
    if (!s || !sel || k < 1 || k > s->B) return ORA_ERR_ARG;
    for (int32_t i = 0; i < k; ++i)
        if (sel[i] < 0 || (int64_t)sel[i] >= s->L) return ORA_ERR_RANGE;
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    if (!tmp) return ORA_ERR_ARG;
    memcpy(tmp, sel, sizeof(int32_t) * (size_t)k);
    qsort(tmp, (size_t)k, sizeof(int32_t), cmp_i32);
    int rc = ORA_OK;
    for (int32_t i = 1; i < k; ++i)
        if (tmp[i] == tmp[i - 1]) { rc = ORA_ERR_DUP; break; }
    free(tmp);
    return rc;
}

/*
 * Hits, misses and victims, read-only.
 *   hit_slot[i]  slot holding sel[i], or -1 if sel[i] is a miss;
 *   miss_idx[j]  selection index of the j-th miss, in selection order;
 *   victim[j]    slot assigned to the j-th miss;
 *   *m_out       number of misses.
 */
int ora_plan(const ora_pair *s, const int32_t *sel, int32_t k, int32_t *hit_slot,
             int32_t *miss_idx, int32_t *victim, int32_t *m_out) {
    int rc = ora_validate(s, sel, k);
    if (rc) return rc;
    const int32_t B = s->B;
    uint8_t *held = (uint8_t *)calloc((size_t)B, 1);
    uint64_t *keys = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)B);
    if (!held || !keys) { free(held); free(keys); return ORA_ERR_ARG; }

    /* hits: the page table maps the position to a slot */
    int32_t m = 0;
    for (int32_t i = 0; i < k; ++i) {
        int32_t b = s->pt[sel[i]];
        if (b >= 0) {
            if (b >= B || s->slot_pos[b] != sel[i]) { rc = ORA_ERR_STATE; goto out; }
            hit_slot[i] = b;
            held[b] = 1;
        } else {
            hit_slot[i] = -1;
            miss_idx[m++] = i;
        }
    }
    /* victims: non-hit slots in ascending (stamp, slot) order */
    int32_t nc = 0;
    for (int32_t b = 0; b < B; ++b)
        if (!held[b]) keys[nc++] = ((uint64_t)s->stamp[b] << 32) | (uint32_t)b;
    qsort(keys, (size_t)nc, sizeof(uint64_t), cmp_u64);
    if (nc < m) { rc = ORA_ERR_STATE; goto out; }  /* impossible when k <= B */
    for (int32_t j = 0; j < m; ++j) victim[j] = (int32_t)(keys[j] & 0xFFFFFFFFu);
    *m_out = m;
out:
    free(held);
    free(keys);
    return rc;
}

/* Copy step of exact prefetch: cache[slot_j] = host[pos_j] for each pair. */
int ora_prefetch_copy(ora_pair *s, const int32_t *plan_pos, const int32_t *plan_slot,
                      int32_t plan_m) {
    for (int32_t j = 0; j < plan_m; ++j) {
        int32_t p = plan_pos[j], b = plan_slot[j];
        if (p < 0 || (int64_t)p >= s->L || b < 0 || b >= s->B) continue;
        if (s->cache && s->host)
            memcpy(s->cache + (size_t)b * s->W, s->host + (size_t)p * s->W, (size_t)s->W);
        s->counters[5] += (uint64_t)s->W;
    }
    return ORA_OK;
}

/*
 * One resolve.  out[i] = out_base + slot of sel[i] (out_base = r * B).
 * plan_m < 0 means "no plan"; otherwise plan_pos/plan_slot hold plan_m pairs
 * produced for this resolve and already copied by ora_prefetch_copy.
 * On a rejected selection every out[i] is -1 and the state is unchanged.
 */
int ora_resolve(ora_pair *s, const int32_t *sel, int32_t k, int32_t out_base, int32_t *out,
                int32_t *m_out, const int32_t *plan_pos, const int32_t *plan_slot,
                int32_t plan_m) {
    if (!s || !out) return ORA_ERR_ARG;
    const int32_t B = s->B;
    int32_t kk = k > 0 ? k : 0;
    int32_t *hit_slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)(kk + 1));
    int32_t *miss_idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(kk + 1));
    int32_t *victim = (int32_t *)malloc(sizeof(int32_t) * (size_t)(kk + 1));
    int32_t m = 0;
    int rc = (hit_slot && miss_idx && victim) ? ora_plan(s, sel, k, hit_slot, miss_idx, victim, &m)
                                              : ORA_ERR_ARG;
    if (rc) {
        for (int32_t i = 0; i < kk; ++i) out[i] = -1;
        if (m_out) *m_out = -1;
        free(hit_slot); free(miss_idx); free(victim);
        return rc;
    }
    const uint32_t t = ++*s->t;

    /* misses, in selection order, into their victims */
    for (int32_t j = 0; j < m; ++j) {
        int32_t i = miss_idx[j], v = victim[j], p = sel[i];
        int32_t old = s->slot_pos[v];
        if (old >= 0) s->pt[old] = -1;          /* evicted record becomes host-only */
        s->slot_pos[v] = p;
        s->pt[p] = v;
        s->stamp[v] = 2u * t - 1u;
        out[i] = out_base + v;
        int planned = plan_m >= 0 && j < plan_m && plan_pos[j] == p && plan_slot[j] == v;
        if (planned) {
            s->counters[3] += 1;
        } else {
            if (s->cache && s->host)
                memcpy(s->cache + (size_t)v * s->W, s->host + (size_t)p * s->W, (size_t)s->W);
            s->counters[2] += (uint64_t)s->W;
        }
    }
    /* hits: promoted above this step's misses */
    for (int32_t i = 0; i < k; ++i) {
        if (hit_slot[i] < 0) continue;
        s->stamp[hit_slot[i]] = 2u * t;
        out[i] = out_base + hit_slot[i];
    }
    /* plan pairs that were not this resolve's own (pos, victim): the copy
       step wrote their slot, so re-fetch whatever record owns it now */
    if (plan_m >= 0) {
        int32_t n = plan_m > m ? plan_m : m;
        for (int32_t j = 0; j < n; ++j) {
            int good = j < m && j < plan_m && plan_pos[j] == sel[miss_idx[j]] &&
                       plan_slot[j] == victim[j];
            if (good) continue;
            s->counters[4] += 1;
            if (j >= plan_m) continue;
            int32_t b = plan_slot[j], p = plan_pos[j];
            if (b < 0 || b >= B || p < 0 || (int64_t)p >= s->L) continue;
            int32_t owner = s->slot_pos[b];
            if (owner < 0) continue;
            if (s->cache && s->host)
                memcpy(s->cache + (size_t)b * s->W, s->host + (size_t)owner * s->W, (size_t)s->W);
            s->counters[2] += (uint64_t)s->W;
        }
    }
    s->counters[0] += (uint64_t)(k - m);
    s->counters[1] += (uint64_t)m;
    s->counters[6] += 1;
    if (m_out) *m_out = m;
    free(hit_slot); free(miss_idx); free(victim);
    return ORA_OK;
}

/*
 * Runs `steps` resolves of one pair back to back (no plan):
 * sel is [steps][sel_stride] (k entries used per step), out is [steps][k],
 * m is [steps].  Stops at the first rejected step and returns its code.
 */
int ora_run(ora_pair *s, const int32_t *sel, int32_t steps, int32_t sel_stride, int32_t k,
            int32_t out_base, int32_t *out, int32_t *m) {
    int32_t *scratch = 0;
    if (!out) {
        scratch = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
        if (!scratch) return ORA_ERR_ARG;
    }
    int rc = ORA_OK;
    for (int32_t t = 0; t < steps && rc == ORA_OK; ++t)
        rc = ora_resolve(s, sel + (size_t)t * sel_stride, k, out_base,
                         out ? out + (size_t)t * k : scratch, m ? m + t : 0, 0, 0, -1);
    free(scratch);
    return rc;
}

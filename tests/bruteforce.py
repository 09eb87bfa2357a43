"""Brute-force LRU replay, an independent route to the oracle's results.

No page table and no sorting: hits are found by scanning every slot for the
position, and each miss, in selection order, takes the slot with the
smallest (stamp, slot) among the slots neither hit nor already taken in this
step, found by a linear scan.  This is O(k*B) per step and only meant for tiny
inputs.  It follows the same reading of the pages as the oracle (stamps
2t-1 for misses, 2t for hits, ties to the lowest slot, misses filled in
selection order).
"""
from __future__ import annotations


class BrutePair:
    def __init__(self, B: int):
        self.B = B
        self.slot_pos = [-1] * B
        self.stamp = [0] * B
        self.t = 0
        self.hits = 0
        self.misses = 0

    def resolve(self, sel, out_base=0):
        """Returns (out, m) or raises ValueError on an invalid selection."""
        if len(sel) < 1 or len(sel) > self.B or len(set(sel)) != len(sel):
            raise ValueError("invalid selection")
        self.t += 1
        t = self.t
        hit_slot = []
        for p in sel:
            found = -1
            for b in range(self.B):
                if self.slot_pos[b] == p:
                    found = b
            hit_slot.append(found)
        taken = [False] * self.B
        for b in hit_slot:
            if b >= 0:
                taken[b] = True
        out = [0] * len(sel)
        m = 0
        new_stamp = list(self.stamp)
        for i, p in enumerate(sel):
            if hit_slot[i] >= 0:
                continue
            best = -1
            for b in range(self.B):
                if taken[b]:
                    continue
                if best < 0 or self.stamp[b] < self.stamp[best]:
                    best = b           # strict '<' keeps the lowest slot on ties
            taken[best] = True
            self.slot_pos[best] = p
            new_stamp[best] = 2 * t - 1
            out[i] = out_base + best
            m += 1
        for i, b in enumerate(hit_slot):
            if b >= 0:
                new_stamp[b] = 2 * t
                out[i] = out_base + b
        self.stamp = new_stamp
        self.hits += len(sel) - m
        self.misses += m
        return out, m

    def page_table(self, L):
        pt = [-1] * L
        for b, p in enumerate(self.slot_pos):
            if p >= 0:
                pt[p] = b
        return pt

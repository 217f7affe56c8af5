"""A plain Python statement of the expert tier's residency rules, for checking
the library's slot cache (moe_slot_cache_*) decision by decision.

"GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", "What
Colibri is actually doing":
- item 4: each layer owns a fixed number of slots; a hit advances a
  monotonic use clock; a miss is loaded and replaces the least recently used
  slot;
- item 5: a pinned hot store that is never evicted;
- item 6: at a safe point a few pins may be replaced by hotter experts, with
  a 25 % + 4 hysteresis;
- item 8: a call admits the union of its experts, each once.
The placement details the pages leave open are the library's documented
choices: a load takes the lowest free slot before evicting; the experts of
the set being admitted are never evicted by it; a prefetch counts no use and
leaves resident experts alone; repin first fills free hot-store capacity with
the most-used resident experts.
"""
from __future__ import annotations

HIT_PINNED, HIT_LRU, LOAD = 0, 1, 2


class TierModel:
    def __init__(self, n_experts: int, n_slots: int, n_pinned: int, call_slots: int):
        self.E, self.S, self.P, self.call_slots = n_experts, n_slots, n_pinned, call_slots
        self.expert = [None] * n_slots      # expert held by each slot
        self.stamp = [0] * n_slots          # use clock of the slot's last hit or load
        self.pinned = [False] * n_slots
        self.uses = [0] * n_experts
        self.clock = 0
        self.stats = dict(hits_pinned=0, hits_lru=0, misses=0, loads=0, evictions=0)

    def slot_of(self, e):
        return self.expert.index(e) if e in self.expert else None

    def _valid(self, ids):
        return all(0 <= e < self.E for e in ids) and len(set(ids)) == len(ids)

    def _place(self, ids, count_use: bool, pin: bool):
        """-> list of (slot, kind), or None (nothing changed) when it cannot."""
        if not self._valid(ids):
            return None
        present = {e: self.slot_of(e) for e in ids if self.slot_of(e) is not None}
        to_load = [e for e in ids if e not in present]
        held = set(present.values())
        evictable = [s for s in range(self.S)
                     if self.expert[s] is None or (not self.pinned[s] and s not in held)]
        if len(to_load) > len(evictable):
            return None
        if pin:
            after = sum(self.pinned) + sum(1 for e in ids
                                           if e not in present or not self.pinned[present[e]])
            if after > self.P or self.S - after < self.call_slots:
                return None
        out = []
        for e in ids:
            if e in present:
                s = present[e]
                kind = HIT_PINNED if self.pinned[s] else HIT_LRU
                if count_use:
                    self.clock += 1
                    self.stamp[s] = self.clock
                    self.stats["hits_pinned" if kind == HIT_PINNED else "hits_lru"] += 1
            else:
                free = [s for s in range(self.S) if self.expert[s] is None]
                if free:
                    s = free[0]
                else:
                    cands = [s for s in range(self.S)
                             if not self.pinned[s] and s not in held]
                    s = self._victim(cands)
                    self.stats["evictions"] += 1
                self.expert[s] = e
                self.clock += 1
                self.stamp[s] = self.clock
                held.add(s)
                kind = LOAD
                self.stats["loads"] += 1
                if count_use:
                    self.stats["misses"] += 1
            if pin:
                self.pinned[s] = True
            if count_use:
                self.uses[e] += 1
            out.append((s, kind))
        return out

    def _victim(self, cands):
        """The least recently used of the evictable slots."""
        return min(cands, key=lambda c: self.stamp[c])

    def admit(self, ids):
        return self._place(list(ids), True, False)

    def prefetch(self, ids):
        return self._place(list(ids), False, False)

    def pin(self, ids):
        return self._place(list(ids), False, True)

    def repin(self, max_swaps: int) -> int:
        def hot():
            c = [s for s in range(self.S) if self.expert[s] is not None and not self.pinned[s]]
            return min(c, key=lambda s: (-self.uses[self.expert[s]], self.expert[s])) if c else None

        def cold():
            c = [s for s in range(self.S) if self.expert[s] is not None and self.pinned[s]]
            return min(c, key=lambda s: (self.uses[self.expert[s]], -self.expert[s])) if c else None

        changes = 0
        while sum(self.pinned) < self.P and self.S - sum(self.pinned) - 1 >= self.call_slots:
            h = hot()
            if h is None:
                break
            self.pinned[h] = True
            changes += 1
        for _ in range(max_swaps):
            h, c = hot(), cold()
            if h is None or c is None:
                break
            if not self._swap_ok(self.uses[self.expert[h]], self.uses[self.expert[c]]):
                break
            self.pinned[c], self.pinned[h] = False, True
            changes += 1
        return changes

    @staticmethod
    def _swap_ok(hot_uses, cold_uses):
        """Item 6's hysteresis: the hot expert must be 25 % + 4 uses ahead."""
        return hot_uses > 1.25 * cold_uses + 4

    def slot_table(self):
        """slot_of per expert as the library reports it: slot, -(slot + 2)
        when pinned, -1 when absent."""
        t = [-1] * self.E
        for s, e in enumerate(self.expert):
            if e is not None:
                t[e] = -(s + 2) if self.pinned[s] else s
        return t

"""The expert tier's residency policy (moe_slot_cache_*), on the host.

Hand-worked sequences pin the rules of "GLM-5.2 on a 32 GB Mac", "What
Colibri is actually doing", items 4-6 and 8 (LRU with a use clock, a pinned
hot store, repinning with a 25 % + 4 hysteresis, one admission per expert of
a call's union); a randomised run then compares every decision with the plain
Python statement of the same rules in tier_model.py.  No GPU is needed.
"""
from __future__ import annotations

import numpy as np
import pytest

from tier_model import HIT_LRU, HIT_PINNED, LOAD, TierModel


@pytest.fixture(scope="module")
def m():
    from int4_routed_expert_gb300 import build as b
    b.build()
    import int4_routed_expert_gb300 as mod
    mod.load()
    return mod


def test_lru_sequence_by_hand(m):
    """E = 8, 4 slots.  Use clock: each hit or load takes the next tick.
    [3,5]: 3->s0 (t1), 5->s1 (t2).  [5,1]: 5 hit s1 (t3), 1->s2 (t4).
    [6,7]: 6->s3 (t5); no free slot, LRU is s0 (t1): 3 evicted, 7->s0 (t6).
    [5,3]: 5 hit s1 (t7); LRU of s0 (t6), s2 (t4), s3 (t5) is s2: 1 evicted."""
    c = m.SlotCache(8, 4, 1, 2)
    steps = [([3, 5], [0, 1], [LOAD, LOAD]),
             ([5, 1], [1, 2], [HIT_LRU, LOAD]),
             ([6, 7], [3, 0], [LOAD, LOAD]),
             ([5, 3], [1, 2], [HIT_LRU, LOAD])]
    for ids, slots, kinds in steps:
        s, k = c.admit(ids)
        assert list(s) == slots and list(k) == kinds, (ids, s, k)
    st, slot_of, uses = c.query()
    assert st == dict(hits_pinned=0, hits_lru=2, misses=6, loads=6, evictions=2,
                      n_resident=4, n_pinned=0)
    assert list(slot_of) == [-1, -1, -1, 2, -1, 1, 3, 0]
    assert list(uses) == [0, 1, 0, 2, 0, 3, 1, 1]


def test_pinned_expert_is_never_evicted(m):
    c = m.SlotCache(16, 4, 1, 3)
    s, k = c.pin([9])
    assert list(k) == [LOAD]
    pinned_slot = int(s[0])
    for i in range(40):
        ids = [(3 * i + j) % 16 for j in range(3) if (3 * i + j) % 16 != 9][:2]
        c.admit(ids)
        _, slot_of, _ = c.query()
        assert slot_of[9] == -(pinned_slot + 2)
    s, k = c.admit([9])
    assert list(k) == [HIT_PINNED] and int(s[0]) == pinned_slot
    st, _, _ = c.query()
    assert st["hits_pinned"] == 1 and st["n_pinned"] == 1


def test_prefetch_counts_no_use_and_keeps_resident_order(m):
    """After [0,1,2] (t1..t3) a prefetch of 1 must not refresh it: the next
    load still evicts 0 (t1), then 1 (t2), not 2."""
    c = m.SlotCache(8, 3, 0, 1)
    c.admit([0, 1, 2])
    s, k = c.prefetch([1])
    assert list(k) == [HIT_LRU]
    _, _, uses = c.query()
    assert list(uses[:3]) == [1, 1, 1]
    c.admit([5])
    c.admit([6])
    _, slot_of, _ = c.query()
    assert slot_of[0] == -1 and slot_of[1] == -1 and slot_of[2] >= 0
    # a prefetched load takes the current clock: it is not the next victim
    c.prefetch([7])          # evicts 2 (t3), the least recent
    c.admit([3])             # evicts 5 (t4), not 7
    _, slot_of, uses = c.query()
    assert slot_of[7] >= 0 and slot_of[5] == -1 and uses[7] == 0


def test_failed_operations_change_nothing(m):
    c = m.SlotCache(8, 4, 2, 2)
    c.pin([0, 1])
    c.admit([2, 3])
    before = c.query()
    for bad in ([2, 3, 4], [8], [-1], [4, 4]):
        with pytest.raises(m.MoeError):
            c.admit(bad)
        after = c.query()
        assert after[0] == before[0]
        assert after[1] == before[1] and after[2] == before[2]
    with pytest.raises(m.MoeError):
        c.pin([5])   # a third pin exceeds the hot store's 2 slots
    assert c.query()[0] == before[0]


@pytest.mark.parametrize("args", [(0, 1, 0, 1), (8, 0, 0, 1), (8, 9, 0, 1), (8, 4, 3, 2),
                                  (8, 4, -1, 1), (8, 4, 0, 0), (2048, 4, 0, 1)])
def test_create_rejects_bad_sizes(m, args):
    with pytest.raises(m.MoeError):
        m.SlotCache(*args)


def test_repin_hysteresis_boundary(m):
    """A pin with u uses is replaced only by an expert with more than
    1.25 u + 4 uses: u = 4 -> 9 uses do not swap, 10 do."""
    def setup(hot_uses):
        c = m.SlotCache(8, 4, 1, 2)
        c.pin([0])
        for _ in range(4):
            c.admit([0])
        for _ in range(hot_uses):
            c.admit([1])
        return c
    c = setup(9)
    assert c.repin(4) == 0
    assert c.query()[1][0] < -1 and c.query()[1][1] >= 0
    c = setup(10)
    assert c.repin(4) == 1
    _, slot_of, _ = c.query()
    assert slot_of[1] < -1 and slot_of[0] >= 0


def test_repin_fills_free_hot_store_capacity(m):
    c = m.SlotCache(8, 5, 2, 3)
    for ids, times in (([4], 3), ([2], 5), ([6], 1)):
        for _ in range(times):
            c.admit(ids)
    assert c.repin(0) == 2
    _, slot_of, _ = c.query()
    assert slot_of[2] < -1 and slot_of[4] < -1 and slot_of[6] >= 0


def _zipf_union(rng, E, k, T):
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    perm = rng.permutation(E)
    ids = set()
    for _ in range(T):
        ids.update(perm[rng.choice(E, size=k, replace=False, p=p)].tolist())
    out = sorted(ids)
    rng.shuffle(out)
    return out


@pytest.mark.parametrize("E,S,P,k,T", [(16, 8, 2, 3, 2), (64, 20, 4, 4, 3), (256, 40, 8, 8, 4)])
def test_random_sequence_matches_the_model(m, E, S, P, k, T):
    rng = np.random.default_rng(E + S)
    call = min(E, k * T)
    c = m.SlotCache(E, S, P, call)
    ref = TierModel(E, S, P, call)
    for step in range(600):
        op = rng.random()
        if op < 0.75:
            ids = _zipf_union(rng, E, k, int(rng.integers(1, T + 1)))
            name = "admit"
        elif op < 0.85:
            ids = rng.choice(E, size=int(rng.integers(1, call + 1)), replace=False).tolist()
            name = "prefetch"
        elif op < 0.92:
            ids = rng.choice(E, size=int(rng.integers(1, 3)), replace=False).tolist()
            name = "pin"
        else:
            n = int(rng.integers(0, 3))
            assert c.repin(n) == ref.repin(n), step
            ids = None
        if ids is not None:
            want = getattr(ref, name)(ids)
            if want is None:
                with pytest.raises(m.MoeError):
                    getattr(c, name)(ids)
            else:
                s, kk = getattr(c, name)(ids)
                assert [(int(a), int(b)) for a, b in zip(s, kk)] == want, (step, name, ids)
        st, slot_of, uses = c.query()
        for key, v in ref.stats.items():
            assert st[key] == v, (step, key)
        assert list(slot_of) == ref.slot_table(), step
        assert [int(u) for u in uses] == ref.uses, step


class _MruModel(TierModel):
    """Planted slip: evicts the most recently used slot."""

    def _victim(self, cands):
        return max(cands, key=lambda c: self.stamp[c])


class _NoClockOnHitModel(TierModel):
    """Planted slip: a hit does not refresh the use clock (FIFO, not LRU)."""

    def admit(self, ids):
        keep = list(self.stamp)
        out = self._place(list(ids), True, False)
        if out is not None:
            for (s, kind) in out:
                if kind != LOAD:
                    self.stamp[s] = keep[s]
        return out


class _NoHysteresisModel(TierModel):
    """Planted slip: a pin is replaced by any hotter expert."""

    @staticmethod
    def _swap_ok(hot_uses, cold_uses):
        return hot_uses > cold_uses


def _diverges(m, model_cls, E=64, S=20, P=4, k=4, T=3, steps=400, seed=5):
    rng = np.random.default_rng(seed)
    call = min(E, k * T)
    c = m.SlotCache(E, S, P, call)
    ref = model_cls(E, S, P, call)
    c.pin([1, 2])
    ref.pin([1, 2])
    for step in range(steps):
        if step % 25 == 24:
            if c.repin(2) != ref.repin(2):
                return True
            continue
        ids = _zipf_union(rng, E, k, int(rng.integers(1, T + 1)))
        s, kk = c.admit(ids)
        want = ref.admit(ids)
        if want is None or [(int(a), int(b)) for a, b in zip(s, kk)] != want:
            return True
        if list(c.query()[1]) != ref.slot_table():
            return True
    return False


@pytest.mark.parametrize("slip", [_MruModel, _NoClockOnHitModel, _NoHysteresisModel])
def test_the_comparison_catches_planted_slips(m, slip):
    """The randomised comparison has the power to see a wrong rule: each
    planted slip in the Python statement makes it disagree with the library,
    while the unmutated statement agrees (test_random_sequence_matches_the_model)."""
    assert not _diverges(m, TierModel)
    assert _diverges(m, slip)

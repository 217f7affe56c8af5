// Residency policy of the HBM expert tier (slot_cache.cuh) and its C ABI
// (include/moe.h, "Expert slot cache").  Host code only.
#include <stdio.h>

#include <new>

#include "moe_internal.cuh"
#include "slot_cache.cuh"

namespace moe {

SlotCache::SlotCache(int n_experts, int n_slots, int n_pinned)
    : E_(n_experts),
      pin_max_(n_pinned),
      slot_expert_(n_slots, -1),
      expert_slot_(n_experts, -1),
      last_use_(n_slots, 0),
      pinned_(n_slots, 0),
      uses_(n_experts, 0) {}

const char* SlotCache::check_ids(const int32_t* ids, int n) const {
  static thread_local char msg[160];
  if (n < 0) return "the number of experts is negative";
  if (n > 0 && !ids) return "the expert ids are NULL";
  std::vector<uint8_t> seen(E_, 0);
  for (int i = 0; i < n; ++i) {
    const int e = ids[i];
    if (e < 0 || e >= E_) {
      snprintf(msg, sizeof(msg), "expert id %d at index %d is outside [0, %d)", e, i, E_);
      return msg;
    }
    if (seen[e]) {
      snprintf(msg, sizeof(msg), "expert id %d appears twice", e);
      return msg;
    }
    seen[e] = 1;
  }
  return nullptr;
}

int SlotCache::n_resident() const {
  int n = 0;
  for (int32_t e : slot_expert_) n += e >= 0 ? 1 : 0;
  return n;
}

int SlotCache::n_pinned() const {
  int n = 0;
  for (uint8_t p : pinned_) n += p;
  return n;
}

// Least recently used slot that is occupied, unpinned and not kept; -1 if none.
int SlotCache::victim(const std::vector<uint8_t>& keep) const {
  int best = -1;
  for (int s = 0; s < n_slots(); ++s) {
    if (slot_expert_[s] < 0 || pinned_[s] || keep[s]) continue;
    if (best < 0 || last_use_[s] < last_use_[best]) best = s;
  }
  return best;
}

const char* SlotCache::place(const int32_t* ids, int n, int32_t* slot, int32_t* kind, bool use,
                             bool pin_them) {
  static thread_local char msg[200];
  if (const char* m = check_ids(ids, n)) return m;
  if (n > 0 && (!slot || !kind)) return "the slot or kind output is NULL";
  const int S = n_slots();
  std::vector<uint8_t> keep(S, 0);
  int loads = 0, new_pins = 0;
  for (int i = 0; i < n; ++i) {
    const int s = expert_slot_[ids[i]];
    if (s >= 0) {
      keep[s] = 1;
      new_pins += pinned_[s] ? 0 : 1;
    } else {
      ++loads;
      ++new_pins;
    }
  }
  int avail = 0;
  for (int s = 0; s < S; ++s)
    avail += (slot_expert_[s] < 0 || (!pinned_[s] && !keep[s])) ? 1 : 0;
  if (loads > avail) {
    snprintf(msg, sizeof(msg), "%d experts to load but only %d slots are free or evictable",
             loads, avail);
    return msg;
  }
  if (pin_them) {
    const int pins = n_pinned() + new_pins;
    if (pins > pin_max_) {
      snprintf(msg, sizeof(msg), "%d pinned experts would exceed the hot store's %d slots",
               pins, pin_max_);
      return msg;
    }
    if (S - pins < call_slots_) {
      snprintf(msg, sizeof(msg), "pinning would leave %d unpinned slots; a call needs %d",
               S - pins, call_slots_);
      return msg;
    }
  }
  for (int i = 0; i < n; ++i) {
    const int e = ids[i];
    int s = expert_slot_[e];
    if (s >= 0) {
      kind[i] = pinned_[s] ? kSlotHitPinned : kSlotHitLru;
      if (use) {
        last_use_[s] = ++clock_;
        if (pinned_[s])
          ++st_.hits_pinned;
        else
          ++st_.hits_lru;
      }
    } else {
      for (int f = 0; f < S && s < 0; ++f)
        if (slot_expert_[f] < 0) s = f;
      if (s < 0) {
        s = victim(keep);
        expert_slot_[slot_expert_[s]] = -1;
        ++st_.evictions;
      }
      slot_expert_[s] = e;
      expert_slot_[e] = s;
      last_use_[s] = ++clock_;
      keep[s] = 1;
      kind[i] = kSlotLoad;
      ++st_.loads;
      if (use) ++st_.misses;
    }
    if (pin_them) pinned_[s] = 1;
    if (use) ++uses_[e];
    slot[i] = s;
  }
  return nullptr;
}

const char* SlotCache::admit(const int32_t* ids, int n, int32_t* slot, int32_t* kind) {
  return place(ids, n, slot, kind, true, false);
}

const char* SlotCache::prefetch(const int32_t* ids, int n, int32_t* slot, int32_t* kind) {
  return place(ids, n, slot, kind, false, false);
}

const char* SlotCache::pin(const int32_t* ids, int n, int32_t* slot, int32_t* kind) {
  return place(ids, n, slot, kind, false, true);
}

int SlotCache::repin(int max_swaps) {
  const int S = n_slots();
  // hottest resident unpinned slot (most uses, then the lower expert id)
  auto hottest = [&]() {
    int best = -1;
    for (int s = 0; s < S; ++s) {
      const int e = slot_expert_[s];
      if (e < 0 || pinned_[s]) continue;
      if (best < 0) {
        best = s;
        continue;
      }
      const int b = slot_expert_[best];
      if (uses_[e] > uses_[b] || (uses_[e] == uses_[b] && e < b)) best = s;
    }
    return best;
  };
  // coldest pinned slot (fewest uses, then the higher expert id)
  auto coldest = [&]() {
    int best = -1;
    for (int s = 0; s < S; ++s) {
      const int e = slot_expert_[s];
      if (e < 0 || !pinned_[s]) continue;
      if (best < 0) {
        best = s;
        continue;
      }
      const int b = slot_expert_[best];
      if (uses_[e] < uses_[b] || (uses_[e] == uses_[b] && e > b)) best = s;
    }
    return best;
  };
  int changes = 0;
  while (n_pinned() < pin_max_ && S - n_pinned() - 1 >= call_slots_) {
    const int h = hottest();
    if (h < 0) break;
    pinned_[h] = 1;
    ++changes;
  }
  for (int i = 0; i < max_swaps; ++i) {
    const int h = hottest(), c = coldest();
    if (h < 0 || c < 0) break;
    // uses(hot) > 1.25 * uses(cold) + 4, in integers
    if (!(4 * uses_[slot_expert_[h]] > 5 * uses_[slot_expert_[c]] + 16)) break;
    pinned_[c] = 0;
    pinned_[h] = 1;
    ++changes;
  }
  return changes;
}

}  // namespace moe

struct moe_slot_cache {
  moe::SlotCache c;
  moe_slot_cache(int e, int s, int p) : c(e, s, p) {}
};

extern "C" {

moe_status_t moe_slot_cache_create(int n_experts, int n_slots, int n_pinned, int call_slots,
                                   moe_slot_cache_t** out) {
  if (!out) {
    moe::set_thread_error("moe_slot_cache_create: out is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (n_experts < 1 || n_experts > 1024 || n_slots < 1 || n_slots > n_experts || n_pinned < 0 ||
      call_slots < 1 || n_slots - n_pinned < call_slots) {
    moe::set_thread_error(
        "moe_slot_cache_create: need 1 <= n_slots <= n_experts <= 1024, n_pinned >= 0, "
        "call_slots >= 1 and n_slots - n_pinned >= call_slots (got %d, %d, %d, %d)",
        n_experts, n_slots, n_pinned, call_slots);
    return MOE_ERR_INVALID_ARG;
  }
  moe_slot_cache* c = new (std::nothrow) moe_slot_cache(n_experts, n_slots, n_pinned);
  if (!c) {
    moe::set_thread_error("moe_slot_cache_create: host allocation failed");
    return MOE_ERR_OOM;
  }
  c->c.set_min_call_slots(call_slots);
  *out = c;
  return MOE_OK;
}

static moe_status_t cache_op(moe_slot_cache_t* c, const int32_t* ids, int n, int32_t* slot,
                             int32_t* kind, int op, const char* name) {
  if (!c) {
    moe::set_thread_error("%s: cache is NULL", name);
    return MOE_ERR_INVALID_ARG;
  }
  const char* m = op == 0   ? c->c.admit(ids, n, slot, kind)
                  : op == 1 ? c->c.prefetch(ids, n, slot, kind)
                            : c->c.pin(ids, n, slot, kind);
  if (m) {
    moe::set_thread_error("%s: %s", name, m);
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe_status_t moe_slot_cache_admit(moe_slot_cache_t* c, const int32_t* ids, int n, int32_t* slot,
                                  int32_t* kind) {
  return cache_op(c, ids, n, slot, kind, 0, "moe_slot_cache_admit");
}

moe_status_t moe_slot_cache_prefetch(moe_slot_cache_t* c, const int32_t* ids, int n,
                                     int32_t* slot, int32_t* kind) {
  return cache_op(c, ids, n, slot, kind, 1, "moe_slot_cache_prefetch");
}

moe_status_t moe_slot_cache_pin(moe_slot_cache_t* c, const int32_t* ids, int n, int32_t* slot,
                                int32_t* kind) {
  return cache_op(c, ids, n, slot, kind, 2, "moe_slot_cache_pin");
}

int moe_slot_cache_repin(moe_slot_cache_t* c, int max_swaps) {
  if (!c || max_swaps < 0) return -1;
  return c->c.repin(max_swaps);
}

moe_status_t moe_slot_cache_query(const moe_slot_cache_t* c, moe_slot_cache_stats_t* st,
                                  int32_t* slot_of, uint64_t* uses) {
  if (!c) {
    moe::set_thread_error("moe_slot_cache_query: cache is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (st) {
    const moe::SlotCacheStats& s = c->c.stats();
    st->hits_pinned = s.hits_pinned;
    st->hits_lru = s.hits_lru;
    st->misses = s.misses;
    st->loads = s.loads;
    st->evictions = s.evictions;
    st->n_resident = c->c.n_resident();
    st->n_pinned = c->c.n_pinned();
  }
  for (int e = 0; e < c->c.n_experts(); ++e) {
    if (slot_of) {
      const int s = c->c.slot_of(e);
      // a pinned slot is reported as -(slot + 2), so that -1 stays "absent"
      slot_of[e] = s < 0 ? -1 : (c->c.is_pinned(s) ? -(s + 2) : s);
    }
    if (uses) uses[e] = c->c.uses(e);
  }
  return MOE_OK;
}

void moe_slot_cache_destroy(moe_slot_cache_t* c) { delete c; }

}  // extern "C"

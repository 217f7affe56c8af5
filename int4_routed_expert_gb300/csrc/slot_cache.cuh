// Residency policy of the HBM expert tier (host code, no device work).
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", "What
// Colibri is actually doing": the routed experts live in a larger, slower
// tier and a bounded set of slots holds the ones in use.
//   item 4 (per-layer bounded LRU): a layer owns a fixed number of slots; a
//          hit advances a monotonic use clock; a miss is loaded and takes the
//          place of the least recently used slot;
//   item 5 (pinned hot store): a separate set of slots that is never evicted;
//   item 6 (live LFRU): at a safe point a few pins may be replaced by hotter
//          experts, with a 25 % + 4 hysteresis against oscillation;
//   item 8 (batch union): a call admits the distinct experts its tokens
//          selected, each once.
// Here the slower tier is pinned host memory and the slots are HBM; the tier
// (tier.cu) copies the loads and runs the kernels.  Every decision is a pure
// function of the call sequence, so the policy can be checked on the host.
#pragma once

#include <stdint.h>

#include <vector>

namespace moe {

// How an expert of an admitted set was found.
enum SlotKind : int32_t {
  kSlotHitPinned = 0,  // resident in the hot store
  kSlotHitLru = 1,     // resident in an LRU slot
  kSlotLoad = 2,       // not resident: assigned a slot that must be filled
};

struct SlotCacheStats {
  uint64_t hits_pinned = 0;  // admitted experts found in the hot store
  uint64_t hits_lru = 0;     // admitted experts found in an LRU slot
  uint64_t misses = 0;       // admitted experts that had to be loaded
  uint64_t loads = 0;        // slots filled (misses, prefetches and pins)
  uint64_t evictions = 0;    // resident experts displaced by a load
};

class SlotCache {
 public:
  // n_pinned: how many of the n_slots the hot store may hold.
  SlotCache(int n_experts, int n_slots, int n_pinned);

  int n_experts() const { return E_; }
  int n_slots() const { return static_cast<int>(slot_expert_.size()); }
  int n_pinned_max() const { return pin_max_; }

  // Checks a set of expert ids: each in [0, E) and none twice.  Returns an
  // error message or nullptr.
  const char* check_ids(const int32_t* ids, int n) const;

  // One call's union of distinct experts.  Hits advance the use clock (in
  // the order given); misses take a free slot, else the least recently used
  // unpinned slot whose expert is not in the set, evicting that expert.
  // Every expert counts one use.  slot[i] / kind[i] receive the slot and
  // SlotKind of ids[i].  Returns nullptr, or an error message with nothing
  // changed (bad ids, or more misses than evictable slots).
  const char* admit(const int32_t* ids, int n, int32_t* slot, int32_t* kind);

  // Prefetch: the same placement with no use counted; an expert already
  // resident is left as it is (no clock update).  Loaded slots take the
  // current clock, so that a prefetch is not the next eviction.
  const char* prefetch(const int32_t* ids, int n, int32_t* slot, int32_t* kind);

  // Hot store: makes each expert resident (loading it when needed) and pins
  // its slot.  Fails with nothing changed when the pins would exceed
  // n_pinned, or when the unpinned slots left could no longer hold one call.
  const char* pin(const int32_t* ids, int n, int32_t* slot, int32_t* kind);

  // Live repinning at a safe point: first the hottest resident unpinned
  // experts fill free hot-store capacity; then, up to max_swaps times, the
  // hottest resident unpinned expert replaces the coldest pinned one when
  // uses(hot) > 1.25 * uses(cold) + 4.  Only flags change (no loads).
  // Returns the number of pins added or replaced.
  int repin(int max_swaps);

  // Unpinned slots that one call's union must fit in.
  int min_call_slots() const { return call_slots_; }
  void set_min_call_slots(int n) { call_slots_ = n; }

  int slot_of(int e) const { return expert_slot_[e]; }
  int expert_in(int s) const { return slot_expert_[s]; }
  bool is_pinned(int s) const { return pinned_[s] != 0; }
  uint64_t uses(int e) const { return uses_[e]; }
  int n_resident() const;
  int n_pinned() const;
  const SlotCacheStats& stats() const { return st_; }

 private:
  const char* place(const int32_t* ids, int n, int32_t* slot, int32_t* kind, bool use,
                    bool pin_them);
  int victim(const std::vector<uint8_t>& keep) const;

  int E_;
  int pin_max_;
  int call_slots_ = 1;
  uint64_t clock_ = 0;
  std::vector<int32_t> slot_expert_;  // [n_slots] expert or -1
  std::vector<int32_t> expert_slot_;  // [E] slot or -1
  std::vector<uint64_t> last_use_;    // [n_slots] use clock of the last hit or load
  std::vector<uint8_t> pinned_;       // [n_slots]
  std::vector<uint64_t> uses_;        // [E] admissions counted per expert
  SlotCacheStats st_;
};

}  // namespace moe

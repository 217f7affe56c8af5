// Expert tier (include/moe.h, "Expert tier"): the routed experts of a layer
// in pinned host memory, a bounded set of them in HBM slots.
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", "What
// Colibri is actually doing", the runtime hierarchy (router output -> batch
// union -> hot-store / LRU hit or miss -> expert compute) and items 4-10.
// The GPU edition keeps the pages' decisions (slot_cache.cuh) and maps their
// mechanisms onto CUDA:
//   - the slower tier is page-locked host memory; a miss is a set of
//     cudaMemcpyAsync copies (one per matrix) on the tier's copy stream;
//   - resident-first submission (item 9): the experts already in HBM, and
//     the shared expert, are launched first; the loaded ones are launched
//     after a stream wait on their copies' event;
//   - no partially filled slot is ever read (item 10): a slot filled by an
//     earlier prefetch whose copies may still run joins the second phase;
//   - a slot is refilled only after the last call that may read it: the
//     copy stream waits on the event recorded after the tier's last call
//     (the pages' working slots serve the same purpose on the host).
// The experts run on the SIMT batch kernels (gemv.cu) with a slot table.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>
#include <vector>

#include "moe_internal.cuh"
#include "slot_cache.cuh"
#include "tier_internal.cuh"

namespace {

constexpr int kRing = 64;  // copy batches that may be in flight at once
constexpr int kMats = 6;   // gate_q, gate_s, up_q, up_s, down_q, down_s

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

struct moe_tier {
  moe_config_t cfg{};
  moe_layer_t* L = nullptr;          // layer whose routed arrays are the slots
  moe::SlotCache* cache = nullptr;
  const uint8_t* host_base[kMats] = {};  // routed arrays in host memory
  uint8_t* slot_base[kMats] = {};        // the same arrays over the slots (HBM)
  size_t mat_bytes[kMats] = {};          // bytes of one expert's matrix
  void* pool = nullptr;
  cudaStream_t copy_s = nullptr;
  cudaEvent_t gu_ev[kRing] = {};     // a batch's gate/up copies have landed
  cudaEvent_t batch_ev[kRing] = {};  // all of a batch's copies have landed
  cudaEvent_t call_done = nullptr;  // recorded after the last call's kernels
  bool any_call = false;
  long long n_batches = 0;     // copy batches issued
  long long done_batches = 0;  // batches known to have completed
  std::vector<long long> fill_batch;  // [n_slots] batch that last filled the slot, -1: none
  int32_t* h_union = nullptr;  // pinned host [1 + E]: n_active, active ids
  int32_t* h_tab = nullptr;    // pinned host [E]: slot table staging
  int32_t* d_tab = nullptr;    // device [E]: slot table of the current call
  uint64_t h2d = 0;            // expert bytes copied into HBM
  // set by a failed CUDA call after the slot cache had taken its decisions:
  // the slots may no longer hold what the cache says, so every later call
  // is refused
  bool broken = false;
  char err[512] = {};
};

namespace {

void terr(moe_tier* t, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  if (t)
    vsnprintf(t->err, sizeof(t->err), fmt, ap);
  else {
    char buf[512];
    vsnprintf(buf, sizeof(buf), fmt, ap);
    moe::set_thread_error("%s", buf);
  }
  va_end(ap);
}

moe_status_t tcuda(moe_tier* t, cudaError_t e, const char* what) {
  terr(t, "%s: %s", what, cudaGetErrorString(e));
  if (t) t->broken = true;
  return MOE_ERR_CUDA;
}

// Refuses calls on a tier that a failed CUDA call left inconsistent.
bool refuse_broken(moe_tier* t, const char* what) {
  if (!t->broken) return false;
  terr(t, "%s: the tier is unusable after an earlier CUDA error", what);
  return true;
}

void free_tier(moe_tier* t) {
  if (!t) return;
  if (t->copy_s) cudaStreamSynchronize(t->copy_s);
  if (t->L) moe_destroy(t->L);  // waits for the device
  for (cudaEvent_t& e : t->batch_ev)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t& e : t->gu_ev)
    if (e) cudaEventDestroy(e);
  if (t->call_done) cudaEventDestroy(t->call_done);
  if (t->copy_s) cudaStreamDestroy(t->copy_s);
  cudaFree(t->pool);
  cudaFree(t->d_tab);
  cudaFreeHost(t->h_union);
  cudaFreeHost(t->h_tab);
  delete t->cache;
  delete t;
}

// Advances the watermark of completed copy batches (in issue order).
void refresh_done(moe_tier* t) {
  while (t->done_batches < t->n_batches) {
    const cudaError_t e = cudaEventQuery(t->batch_ev[t->done_batches % kRing]);
    if (e != cudaSuccess) {
      if (e == cudaErrorNotReady) cudaGetLastError();
      break;
    }
    ++t->done_batches;
  }
}

// Copies the experts placed with kind kSlotLoad into their slots as one
// batch on the copy stream, gate/up matrices of every load first (event
// gu_ev), then the down matrices (event batch_ev), so that the gate/up
// kernels of the loaded experts can start while their down matrices are
// still on the way; returns the batch number in *batch (-1 when nothing was
// loaded).
cudaError_t load(moe_tier* t, const int32_t* ids, const int32_t* slot, const int32_t* kind, int n,
                 long long* batch) {
  *batch = -1;
  int nl = 0;
  for (int i = 0; i < n; ++i) nl += kind[i] == moe::kSlotLoad ? 1 : 0;
  if (nl == 0) return cudaSuccess;
  // at most kRing batches in flight, so that every batch keeps its event
  if (t->n_batches - t->done_batches >= kRing) {
    const cudaError_t e = cudaEventSynchronize(t->batch_ev[t->n_batches % kRing]);
    if (e != cudaSuccess) return e;
    refresh_done(t);
  }
  cudaError_t e = cudaSuccess;
  // the slots being refilled may be read by the tier's last call
  if (t->any_call) e = cudaStreamWaitEvent(t->copy_s, t->call_done, 0);
  const long long b = t->n_batches;
  // matrices 0-3: gate and up weights and scales; 4-5: down
  for (int part = 0; part < 2 && e == cudaSuccess; ++part) {
    for (int i = 0; i < n && e == cudaSuccess; ++i) {
      if (kind[i] != moe::kSlotLoad) continue;
      const size_t e_id = static_cast<size_t>(ids[i]), s = static_cast<size_t>(slot[i]);
      for (int m = part * 4; m < (part ? kMats : 4) && e == cudaSuccess; ++m) {
        e = cudaMemcpyAsync(t->slot_base[m] + s * t->mat_bytes[m],
                            t->host_base[m] + e_id * t->mat_bytes[m], t->mat_bytes[m],
                            cudaMemcpyHostToDevice, t->copy_s);
        t->h2d += t->mat_bytes[m];
      }
    }
    if (e == cudaSuccess)
      e = cudaEventRecord(part ? t->batch_ev[b % kRing] : t->gu_ev[b % kRing], t->copy_s);
  }
  if (e != cudaSuccess) return e;
  ++t->n_batches;
  for (int i = 0; i < n; ++i)
    if (kind[i] == moe::kSlotLoad) t->fill_batch[slot[i]] = b;
  *batch = b;
  return cudaSuccess;
}

// Routes x on s and reads the union of the selected experts to the host.
moe_status_t route_union(moe_tier* t, const void* x, moe_dtype_t dt, int T, const float* gamma,
                         float eps, cudaStream_t s, int* n_union) {
  const moe::Workspace& ws = t->L->ws;
  cudaError_t e = moe::layer_route(t->L, x, dt, T, gamma, eps, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(t->h_union, ws.n_active, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(t->h_union + 1, ws.active, static_cast<size_t>(t->cfg.n_experts) * 4,
                        cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return tcuda(t, e, "expert tier (routing)");
  const int n = t->h_union[0];
  if (n < 0 || n > t->cfg.n_experts) {
    terr(t, "expert tier: the routing produced %d active experts", n);
    return MOE_ERR_CUDA;
  }
  *n_union = n;
  return MOE_OK;
}

moe_status_t place_and_load(moe_tier* t, const int32_t* ids, int n, int op, const char* what) {
  std::vector<int32_t> slot(n > 0 ? n : 1), kind(n > 0 ? n : 1);
  const char* m = op == 1 ? t->cache->prefetch(ids, n, slot.data(), kind.data())
                          : t->cache->pin(ids, n, slot.data(), kind.data());
  if (m) {
    terr(t, "%s: %s", what, m);
    return MOE_ERR_INVALID_ARG;
  }
  long long b;
  const cudaError_t e = load(t, ids, slot.data(), kind.data(), n, &b);
  if (e != cudaSuccess) return tcuda(t, e, what);
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_tier_create(const moe_config_t* cfg, const moe_weights_t* w,
                             const moe_tier_config_t* tcfg, moe_tier_t** out) {
  if (!out) {
    moe::set_thread_error("moe_tier_create: out is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (!cfg || !w || !tcfg) {
    moe::set_thread_error("moe_tier_create: cfg, w and tcfg must not be NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (const char* m = moe::config_error(cfg)) {
    moe::set_thread_error("moe_tier_create: %s", m);
    return MOE_ERR_UNSUPPORTED;
  }
  const int E = cfg->n_experts;
  const long long tk = static_cast<long long>(cfg->max_tokens) * cfg->top_k;
  const int call_slots = tk < E ? static_cast<int>(tk) : E;
  if (tcfg->n_slots < 1 || tcfg->n_slots > E || tcfg->n_pinned < 0 ||
      tcfg->n_slots - tcfg->n_pinned < call_slots) {
    moe::set_thread_error(
        "moe_tier_create: need 1 <= n_slots <= n_experts and n_slots - n_pinned >= "
        "min(n_experts, max_tokens * top_k) = %d (got n_slots %d, n_pinned %d)",
        call_slots, tcfg->n_slots, tcfg->n_pinned);
    return MOE_ERR_INVALID_ARG;
  }
  const void* host[kMats] = {w->gate_q, w->gate_s, w->up_q, w->up_s, w->down_q, w->down_s};
  for (int m = 0; m < kMats; ++m) {
    cudaPointerAttributes a;
    if (!host[m] || (reinterpret_cast<uintptr_t>(host[m]) & 15u) != 0 ||
        cudaPointerGetAttributes(&a, host[m]) != cudaSuccess || a.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      moe::set_thread_error(
          "moe_tier_create: the routed arrays must be 16-byte aligned page-locked host memory "
          "(cudaHostAlloc or cudaHostRegister)");
      return MOE_ERR_INVALID_ARG;
    }
  }
  moe_tier* t = new (std::nothrow) moe_tier();
  if (!t) {
    moe::set_thread_error("moe_tier_create: host allocation failed");
    return MOE_ERR_OOM;
  }
  t->cfg = *cfg;
  const size_t H = cfg->hidden, I = cfg->inter;
  const size_t qbH = cfg->weight_format == MOE_W_INT8 ? H : H / 2;
  const size_t qbI = cfg->weight_format == MOE_W_INT8 ? I : I / 2;
  const size_t sbH = (cfg->group_size == 0 ? 1 : H / 32) * 2;
  const size_t sbI = (cfg->group_size == 0 ? 1 : I / 32) * 2;
  const size_t mb[kMats] = {I * qbH, I * sbH, I * qbH, I * sbH, H * qbI, H * sbI};
  size_t off[kMats], total = 0;
  for (int m = 0; m < kMats; ++m) {
    t->mat_bytes[m] = mb[m];
    t->host_base[m] = static_cast<const uint8_t*>(host[m]);
    off[m] = total;
    total += up256(mb[m] * tcfg->n_slots);
  }
  cudaError_t e = cudaMalloc(&t->pool, total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    moe::set_thread_error("moe_tier_create: %zu bytes of HBM slots: %s", total,
                          cudaGetErrorString(e));
    free_tier(t);
    return MOE_ERR_OOM;
  }
  for (int m = 0; m < kMats; ++m) t->slot_base[m] = static_cast<uint8_t*>(t->pool) + off[m];
  moe_weights_t wl = *w;
  wl.gate_q = t->slot_base[0];
  wl.gate_s = reinterpret_cast<const uint16_t*>(t->slot_base[1]);
  wl.up_q = t->slot_base[2];
  wl.up_s = reinterpret_cast<const uint16_t*>(t->slot_base[3]);
  wl.down_q = t->slot_base[4];
  wl.down_s = reinterpret_cast<const uint16_t*>(t->slot_base[5]);
  const moe_status_t st = moe::layer_create_slots(cfg, &wl, tcfg->n_slots, &t->L);
  if (st != MOE_OK) {
    free_tier(t);  // the message of layer_create_slots stays
    return st;
  }
  e = cudaStreamCreateWithFlags(&t->copy_s, cudaStreamNonBlocking);
  for (int i = 0; i < kRing && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&t->batch_ev[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t->gu_ev[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t->call_done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMalloc(&t->d_tab, static_cast<size_t>(E) * 4);
  if (e == cudaSuccess) e = cudaMallocHost(&t->h_union, static_cast<size_t>(E + 1) * 4);
  if (e == cudaSuccess) e = cudaMallocHost(&t->h_tab, static_cast<size_t>(E) * 4);
  if (e == cudaSuccess) e = cudaMemset(t->d_tab, 0, static_cast<size_t>(E) * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaGetLastError();
    moe::set_thread_error("moe_tier_create: %s", cudaGetErrorString(e));
    free_tier(t);
    return MOE_ERR_CUDA;
  }
  t->cache = new (std::nothrow) moe::SlotCache(E, tcfg->n_slots, tcfg->n_pinned);
  if (!t->cache) {
    moe::set_thread_error("moe_tier_create: host allocation failed");
    free_tier(t);
    return MOE_ERR_OOM;
  }
  t->cache->set_min_call_slots(call_slots);
  t->fill_batch.assign(tcfg->n_slots, -1);
  *out = t;
  return MOE_OK;
}

moe_status_t moe_tier_forward(moe_tier_t* t, const void* x, moe_dtype_t dtype, int T, float* y,
                              const float* rms_gamma, float rms_eps, int accumulate,
                              moe_plan_t* plan_out, void* stream) {
  if (!t) {
    moe::set_thread_error("moe_tier_forward: tier is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (refuse_broken(t, "moe_tier_forward")) return MOE_ERR_CUDA;
  moe_status_t st =
      moe::layer_check_call(t->L, &x, dtype, T, &y, rms_gamma, accumulate, plan_out, false);
  if (st != MOE_OK) {
    terr(t, "%s", moe_last_error(t->L));
    return st;
  }
  if (T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // 1. route, read the union (every earlier call on s has completed after this)
  int n = 0;
  if ((st = route_union(t, x, dtype, T, rms_gamma, rms_eps, s, &n)) != MOE_OK) return st;
  const int32_t* ids = t->h_union + 1;
  // 2. admit; copy the loads
  std::vector<int32_t> slot(n > 0 ? n : 1), kind(n > 0 ? n : 1);
  if (const char* m = t->cache->admit(ids, n, slot.data(), kind.data())) {
    terr(t, "moe_tier_forward: %s", m);
    return MOE_ERR_CAPACITY;
  }
  refresh_done(t);
  long long batch;
  cudaError_t e = load(t, ids, slot.data(), kind.data(), n, &batch);
  if (e != cudaSuccess) return tcuda(t, e, "moe_tier_forward (expert copies)");
  // 3. slot table: phase 0 = resident with its copies complete, 1 = the rest
  long long wait = -1;
  int n0 = 0;
  for (int i = 0; i < n; ++i) {
    const long long fb = t->fill_batch[slot[i]];
    const bool late = kind[i] == moe::kSlotLoad || fb >= t->done_batches;
    if (late && fb > wait) wait = fb;
    n0 += late ? 0 : 1;
    t->h_tab[ids[i]] = ((late ? 1 : 0) << moe::kSlotPhaseShift) | slot[i];
  }
  const moe::Workspace& ws = t->L->ws;
  const moe::Shape& sh = t->L->sh;
  const moe_weights_t& w = t->L->w;
  e = cudaMemcpyAsync(t->d_tab, t->h_tab, static_cast<size_t>(t->cfg.n_experts) * 4,
                      cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && (n0 > 0 || sh.n_shared)) {
    e = moe::launch_gate_up_slots(w, sh, T, ws, t->d_tab, 0, s);
    if (e == cudaSuccess) e = moe::launch_down_slots(w, sh, T, ws, t->d_tab, 0, s);
  }
  if (e == cudaSuccess && wait >= 0) {
    // batches land in order: the newest one the late experts need covers the
    // older ones, its gate/up part before its down part
    e = cudaStreamWaitEvent(s, t->gu_ev[wait % kRing], 0);
    if (e == cudaSuccess) e = moe::launch_gate_up_slots(w, sh, T, ws, t->d_tab, 1, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, t->batch_ev[wait % kRing], 0);
    if (e == cudaSuccess) e = moe::launch_down_slots(w, sh, T, ws, t->d_tab, 1, s);
  }
  if (e == cudaSuccess) e = moe::launch_combine(sh, T, ws, y, accumulate, s);
  if (e == cudaSuccess) e = cudaEventRecord(t->call_done, s);
  if (e == cudaSuccess) e = moe::layer_copy_plan(t->L, T, plan_out, s);
  if (e != cudaSuccess) return tcuda(t, e, "moe_tier_forward");
  t->any_call = true;
  return MOE_OK;
}

moe_status_t moe_tier_prefetch(moe_tier_t* t, const int32_t* ids, int n) {
  if (!t) {
    moe::set_thread_error("moe_tier_prefetch: tier is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (refuse_broken(t, "moe_tier_prefetch")) return MOE_ERR_CUDA;
  refresh_done(t);
  return place_and_load(t, ids, n, 1, "moe_tier_prefetch");
}

moe_status_t moe_tier_prefetch_routed(moe_tier_t* t, const void* x, moe_dtype_t dtype, int T,
                                      const float* rms_gamma, float rms_eps, void* stream) {
  if (!t) {
    moe::set_thread_error("moe_tier_prefetch_routed: tier is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (refuse_broken(t, "moe_tier_prefetch_routed")) return MOE_ERR_CUDA;
  moe_status_t st =
      moe::layer_check_call(t->L, &x, dtype, T, nullptr, rms_gamma, 0, nullptr, true);
  if (st != MOE_OK) {
    terr(t, "%s", moe_last_error(t->L));
    return st;
  }
  if (T == 0) return MOE_OK;
  int n = 0;
  st = route_union(t, x, dtype, T, rms_gamma, rms_eps, static_cast<cudaStream_t>(stream), &n);
  if (st != MOE_OK) return st;
  refresh_done(t);
  return place_and_load(t, t->h_union + 1, n, 1, "moe_tier_prefetch_routed");
}

moe_status_t moe_tier_pin(moe_tier_t* t, const int32_t* ids, int n) {
  if (!t) {
    moe::set_thread_error("moe_tier_pin: tier is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (refuse_broken(t, "moe_tier_pin")) return MOE_ERR_CUDA;
  refresh_done(t);
  return place_and_load(t, ids, n, 2, "moe_tier_pin");
}

moe_status_t moe_tier_repin(moe_tier_t* t, int max_swaps, int* changed) {
  if (!t || max_swaps < 0) {
    if (t)
      terr(t, "moe_tier_repin: max_swaps must be >= 0");
    else
      moe::set_thread_error("moe_tier_repin: tier is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  const int c = t->cache->repin(max_swaps);
  if (changed) *changed = c;
  return MOE_OK;
}

moe_status_t moe_tier_query(moe_tier_t* t, moe_slot_cache_stats_t* stats, int32_t* slot_of,
                            uint64_t* uses, uint64_t* h2d_bytes) {
  if (!t) {
    moe::set_thread_error("moe_tier_query: tier is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  const moe::SlotCache& c = *t->cache;
  if (stats) {
    const moe::SlotCacheStats& s = c.stats();
    stats->hits_pinned = s.hits_pinned;
    stats->hits_lru = s.hits_lru;
    stats->misses = s.misses;
    stats->loads = s.loads;
    stats->evictions = s.evictions;
    stats->n_resident = c.n_resident();
    stats->n_pinned = c.n_pinned();
  }
  for (int e = 0; e < c.n_experts(); ++e) {
    if (slot_of) {
      const int s = c.slot_of(e);
      slot_of[e] = s < 0 ? -1 : (c.is_pinned(s) ? -(s + 2) : s);
    }
    if (uses) uses[e] = c.uses(e);
  }
  if (h2d_bytes) *h2d_bytes = t->h2d;
  return MOE_OK;
}

const char* moe_tier_last_error(const moe_tier_t* t) {
  return t ? t->err : moe_last_error(nullptr);
}

void moe_tier_destroy(moe_tier_t* t) { free_tier(t); }

}  // extern "C"

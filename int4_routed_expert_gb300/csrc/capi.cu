// C ABI of the MoE layer (include/moe.h): validation, workspace, dispatch
// between the fused single-token kernel, the tensor-core grouped GEMM and
// the SIMT general path, phase tracing.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cuda.h>

#include <new>

#include "moe_internal.cuh"
#include "tier_internal.cuh"

using moe::Shape;
using moe::Workspace;

namespace {

thread_local char g_err[512];

void set_err(moe_layer* h, const char* fmt, ...) {
  char* dst = h ? h->err : g_err;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(dst, 512, fmt, ap);
  va_end(ap);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

const char* check_config(const moe_config_t* c) {
  if (!c) return "cfg is NULL";
  if (c->hidden % 256 != 0 || c->hidden < 256 || c->hidden > 12288)
    return "hidden must be a multiple of 256 in [256, 12288]";
  if (c->inter % 32 != 0 || c->inter < 32 || c->inter > 8192)
    return "inter must be a multiple of 32 in [32, 8192]";
  if (c->n_shared != 0 && c->n_shared != 1) return "n_shared must be 0 or 1";
  if (c->n_shared &&
      (c->shared_inter % 32 != 0 || c->shared_inter < 32 || c->shared_inter > 8192))
    return "shared_inter must be a multiple of 32 in [32, 8192]";
  if (c->n_experts < 1 || c->n_experts > 1024) return "n_experts must be in [1, 1024]";
  if (c->n_group < 1 || c->n_experts % c->n_group != 0)
    return "n_experts must be a multiple of n_group";
  if (c->topk_group < 1 || c->topk_group > c->n_group) return "topk_group must be in [1, n_group]";
  if (c->top_k < 1 || c->top_k > 32) return "top_k must be in [1, 32]";
  if (c->top_k > c->topk_group * (c->n_experts / c->n_group))
    return "top_k exceeds the experts of the kept groups";
  if (c->group_size != 32 && c->group_size != 0)
    return "group_size must be 32 (grouped scales) or 0 (one scale a row)";
  if (c->weight_format != MOE_W_INT4 && c->weight_format != MOE_W_INT8)
    return "weight_format must be MOE_W_INT4 or MOE_W_INT8";
  if (c->max_tokens < 1 || c->max_tokens > 65536) return "max_tokens must be in [1, 65536]";
  if (!(c->routed_scaling_factor == c->routed_scaling_factor) ||
      c->routed_scaling_factor > 3.0e38f || c->routed_scaling_factor < -3.0e38f)
    return "routed_scaling_factor must be finite";
  return nullptr;
}

const char* check_weights(const moe_config_t* c, const moe_weights_t* w) {
  if (!w) return "weights is NULL";
  const void* req[] = {w->router_w, w->router_bias, w->gate_q, w->gate_s, w->up_q,
                       w->up_s,     w->down_q,      w->down_s};
  for (const void* p : req) {
    if (!p) return "a routed-expert or router pointer is NULL";
    if (!aligned16(p)) return "weight pointers must be 16-byte aligned";
  }
  if (c->n_shared) {
    const void* sp[] = {w->sh_gate_q, w->sh_gate_s, w->sh_up_q,
                        w->sh_up_s,   w->sh_down_q, w->sh_down_s};
    for (const void* p : sp) {
      if (!p) return "a shared-expert pointer is NULL";
      if (!aligned16(p)) return "weight pointers must be 16-byte aligned";
    }
  }
  return nullptr;
}

// cuMemGetAddressRange of the driver API: base and size of the allocation
// holding a device address.
using AddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

AddressRangeFn address_range_fn() {
  static AddressRangeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<AddressRangeFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// The kernels and the TMA tensor maps read every byte of a weight array that
// the shape implies, so an array must lie in device (or managed) memory of the
// handle's device and inside allocations that hold all of it; anything else
// would surface as an out-of-bounds access inside a kernel.  Adjacent
// allocations are followed, since a virtual range mapped in pieces reports
// one piece at a time.
const char* check_extent(const void* p, size_t bytes, int device) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return "is not a CUDA pointer";
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return "is not device memory";
  if (a.type == cudaMemoryTypeDevice && a.device != device)
    return "is on another device than the current one";
  const AddressRangeFn fn = address_range_fn();
  if (!fn) return "cannot be checked (no cuMemGetAddressRange in the driver)";
  CUdeviceptr cur = reinterpret_cast<CUdeviceptr>(p);
  const CUdeviceptr end = cur + bytes;
  while (cur < end) {
    CUdeviceptr base = 0;
    size_t size = 0;
    if (fn(&base, &size, cur) != CUDA_SUCCESS || base > cur || base + size <= cur)
      return "extends past the end of its allocation";
    cur = base + size;
  }
  return nullptr;
}

// E_routed: experts the routed arrays hold (n_experts, or the expert tier's
// slots); the router arrays always hold n_experts.
const char* check_weight_memory(const moe_config_t* c, const moe_weights_t* w, size_t E_routed,
                                int device, const char** which) {
  const size_t E = c->n_experts, H = c->hidden, I = c->inter, Er = E_routed;
  // bytes of a K-long row's weights and of its scales, in the format
  auto qb = [&](size_t K) { return c->weight_format == MOE_W_INT8 ? K : K / 2; };
  auto sb = [&](size_t K) { return (c->group_size == 0 ? 1 : K / 32) * 2; };
  struct A {
    const char* name;
    const void* p;
    size_t bytes;
  };
  const A routed[] = {{"router_w", w->router_w, E * H * 4},
                      {"router_bias", w->router_bias, E * 4},
                      {"gate_q", w->gate_q, Er * I * qb(H)},
                      {"gate_s", w->gate_s, Er * I * sb(H)},
                      {"up_q", w->up_q, Er * I * qb(H)},
                      {"up_s", w->up_s, Er * I * sb(H)},
                      {"down_q", w->down_q, Er * H * qb(I)},
                      {"down_s", w->down_s, Er * H * sb(I)}};
  for (const A& x : routed)
    if (const char* m = check_extent(x.p, x.bytes, device)) {
      *which = x.name;
      return m;
    }
  if (!c->n_shared) return nullptr;
  const size_t Is = c->shared_inter;
  const A shared[] = {{"sh_gate_q", w->sh_gate_q, Is * qb(H)},
                      {"sh_gate_s", w->sh_gate_s, Is * sb(H)},
                      {"sh_up_q", w->sh_up_q, Is * qb(H)},
                      {"sh_up_s", w->sh_up_s, Is * sb(H)},
                      {"sh_down_q", w->sh_down_q, H * qb(Is)},
                      {"sh_down_s", w->sh_down_s, H * sb(Is)}};
  for (const A& x : shared)
    if (const char* m = check_extent(x.p, x.bytes, device)) {
      *which = x.name;
      return m;
    }
  return nullptr;
}

// Workspace layout: each buffer 256-byte aligned, in this order.
struct Layout {
  size_t off[23];
  size_t total;
  int hstride;
  size_t dm_cpart;  // float offset of dm_cpart inside dm_part
};

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

Layout layout_for(const moe_config_t* c) {
  Layout L{};
  const size_t Tm = c->max_tokens, H = c->hidden, E = c->n_experts, k = c->top_k;
  const int Imax = c->n_shared ? (c->inter > c->shared_inter ? c->inter : c->shared_inter)
                               : c->inter;
  // row stride of the activation buffer: Imax floats padded to the
  // swizzled layout of the single-token kernel (multiple of 1024)
  L.hstride = ((Imax / 32 + 31) / 32) * 1024;
  const size_t N = Tm * k, R = N + Tm;
  const size_t Ts = Tm < 4 ? Tm : 4;  // tokens of the in-kernel routers
  // f16 rows and chunk list of the tensor-core path (shapes it takes only)
  const bool tc = c->hidden % 256 == 0 && c->inter % 256 == 0 &&
                  (!c->n_shared || c->shared_inter % 256 == 0);
  // single-token tensor-core kernel (shapes it takes only)
  const bool dm = c->hidden % 1024 == 0 && c->inter % 1024 == 0 &&
                  (!c->n_shared || c->shared_inter == c->inter);
  const int Is = c->n_shared ? c->shared_inter : 0;
  const size_t dm_f = dm ? moe::dm_part_floats(c->hidden, c->inter, Is, c->top_k, c->n_shared) : 0;
  const size_t dm_c = dm ? moe::dm_cnt_words(c->hidden, c->inter, Is, c->top_k, c->n_shared) : 0;
  L.dm_cpart = dm_f - (dm ? static_cast<size_t>(c->top_k + c->n_shared) * (c->inter / 8) : 0);
  const size_t sz[23] = {
      Tm * H * 4,            // xf
      Tm * E * 4,            // logits
      N * 4,                 // ids
      N * 4,                 // topw
      E * 4,                 // counts
      (E + 1) * 4,           // offsets
      N * 4,                 // perm
      N * 4,                 // inv
      E * 4,                 // active
      4,                     // n_active
      R * L.hstride * 4,     // hbuf
      R * H * 4,             // obuf
      Ts * E * 4,            // sval
      Ts * E * 4,            // skey
      256,                   // dev_err
      3 * 32 * 4,            // dslot
      256,                   // gbar
      tc ? R * H * 2 : 0,    // x16
      tc ? R * Imax * 2 : 0, // h16
      tc ? moe::tc_max_chunks(c->max_tokens, c->top_k, c->n_experts) * 16 : 0,  // chunks
      4,                     // n_rchunks
      dm_f * 4,              // dm_part (+ dm_cpart)
      512 + dm_c * 4,        // dm_pub (generation, ids, weights; both single-token kernels), dm_cnt
  };
  size_t o = 0;
  for (int i = 0; i < 23; ++i) {
    L.off[i] = o;
    o += up256(sz[i]);
  }
  L.total = o;
  return L;
}

Workspace carve(char* base, const Layout& L) {
  Workspace w{};
  w.xf = reinterpret_cast<float*>(base + L.off[0]);
  w.logits = reinterpret_cast<float*>(base + L.off[1]);
  w.ids = reinterpret_cast<int32_t*>(base + L.off[2]);
  w.topw = reinterpret_cast<float*>(base + L.off[3]);
  w.counts = reinterpret_cast<int32_t*>(base + L.off[4]);
  w.offsets = reinterpret_cast<int32_t*>(base + L.off[5]);
  w.perm = reinterpret_cast<int32_t*>(base + L.off[6]);
  w.inv = reinterpret_cast<int32_t*>(base + L.off[7]);
  w.active = reinterpret_cast<int32_t*>(base + L.off[8]);
  w.n_active = reinterpret_cast<int32_t*>(base + L.off[9]);
  w.hbuf = reinterpret_cast<float*>(base + L.off[10]);
  w.obuf = reinterpret_cast<float*>(base + L.off[11]);
  w.sval = reinterpret_cast<float*>(base + L.off[12]);
  w.skey = reinterpret_cast<float*>(base + L.off[13]);
  w.dev_err = reinterpret_cast<int32_t*>(base + L.off[14]);
  w.dslot = reinterpret_cast<int32_t*>(base + L.off[15]);
  w.gbar = reinterpret_cast<unsigned long long*>(base + L.off[16]);
  w.x16 = reinterpret_cast<__half*>(base + L.off[17]);
  w.h16 = reinterpret_cast<__half*>(base + L.off[18]);
  w.chunks = reinterpret_cast<int4*>(base + L.off[19]);
  w.n_rchunks = reinterpret_cast<int32_t*>(base + L.off[20]);
  w.dm_part = reinterpret_cast<float*>(base + L.off[21]);
  w.dm_cpart = w.dm_part + L.dm_cpart;
  w.dm_pub_gen = reinterpret_cast<unsigned long long*>(base + L.off[22]);
  w.dm_pub_id = reinterpret_cast<int32_t*>(base + L.off[22] + 128);
  w.dm_pub_w = reinterpret_cast<float*>(base + L.off[22] + 256);
  w.dm_cnt = reinterpret_cast<unsigned*>(base + L.off[22] + 512);
  w.hstride = L.hstride;
  return w;
}

moe_status_t cuda_fail(moe_layer* h, cudaError_t e, const char* what) {
  set_err(h, "%s: %s", what, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

// Records one event before the first kernel and one after each phase of a
// traced call.
struct Tracer {
  moe_layer* h = nullptr;
  cudaStream_t s = nullptr;
  int call = -1;
  int n = 0;
  void start(moe_layer* hh, cudaStream_t ss) {
    if (!hh->trace_ev || hh->trace_used >= hh->trace_cap) return;
    h = hh;
    s = ss;
    call = h->trace_used++;
    h->trace_nrec[call] = 0;
    cudaEventRecord(h->trace_ev[call * (MOE_N_PHASES + 1)], s);
  }
  bool on() const { return call >= 0; }
  void mark(int phase) {
    if (call < 0 || n >= MOE_N_PHASES) return;
    h->trace_phase[call * MOE_N_PHASES + n] = phase;
    ++n;
    h->trace_nrec[call] = n;
    cudaEventRecord(h->trace_ev[call * (MOE_N_PHASES + 1) + n], s);
  }
  static void mark_cb(void* ctx, int phase) { static_cast<Tracer*>(ctx)->mark(phase); }
};

moe_status_t check_call(moe_layer* h, const void* x, moe_dtype_t dt, int T, const float* gamma) {
  if (T < 0) {
    set_err(h, "T must be >= 0 (got %d)", T);
    return MOE_ERR_INVALID_ARG;
  }
  if (T > h->cfg.max_tokens) {
    set_err(h, "T = %d exceeds max_tokens = %d of the handle", T, h->cfg.max_tokens);
    return MOE_ERR_CAPACITY;
  }
  if (T == 0) return MOE_OK;
  if (dt != MOE_F32 && dt != MOE_BF16) {
    set_err(h, "unknown dtype %d", static_cast<int>(dt));
    return MOE_ERR_INVALID_ARG;
  }
  if (!x || !aligned16(x)) {
    set_err(h, "x must be a non-NULL 16-byte aligned device pointer");
    return MOE_ERR_INVALID_ARG;
  }
  if (gamma && !aligned16(gamma)) {
    set_err(h, "rms_gamma must be 16-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

moe_status_t check_plan(moe_layer* h, const moe_plan_t* p) {
  if (!p) return MOE_OK;
  const void* m[] = {p->topk_ids, p->topk_w, p->counts, p->offsets,
                     p->perm,     p->active, p->n_active};
  for (const void* q : m)
    if (q && !aligned4(q)) {
      set_err(h, "plan buffers must be 4-byte aligned");
      return MOE_ERR_INVALID_ARG;
    }
  return MOE_OK;
}

cudaError_t copy_plan(moe_layer* h, int T, const moe_plan_t* p, cudaStream_t s) {
  if (!p) return cudaSuccess;
  const Workspace& ws = h->ws;
  const int E = h->cfg.n_experts;
  const size_t N = static_cast<size_t>(T) * h->cfg.top_k;
  struct C {
    void* dst;
    const void* src;
    size_t bytes;
  } cs[] = {{p->topk_ids, ws.ids, N * 4},        {p->topk_w, ws.topw, N * 4},
            {p->counts, ws.counts, E * 4ul},     {p->offsets, ws.offsets, (E + 1) * 4ul},
            {p->perm, ws.perm, N * 4},           {p->active, ws.active, E * 4ul},
            {p->n_active, ws.n_active, 4}};
  for (const C& c : cs) {
    if (!c.dst) continue;
    const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t run_route(moe_layer* h, const void* x, moe_dtype_t dt, int T, const float* gamma,
                      float eps, cudaStream_t s, Tracer& tr) {
  const Shape& sh = h->sh;
  const Workspace& ws = h->ws;
  cudaError_t e = moe::launch_prep(x, dt, T, sh.H, gamma, eps, ws.xf, s);
  if (e != cudaSuccess) return e;
  tr.mark(0);
  e = moe::launch_router_logits(ws.xf, T, sh.H, h->w.router_w, sh.E, ws.logits, s);
  if (e != cudaSuccess) return e;
  tr.mark(1);
  e = moe::launch_select(ws.logits, h->w.router_bias, T, sh, ws.ids, ws.topw, s);
  if (e != cudaSuccess) return e;
  tr.mark(2);
  e = moe::launch_plan(ws.ids, T, sh.k, sh.E, ws.counts, ws.offsets, ws.perm, ws.inv,
                       ws.active, ws.n_active, s);
  if (e != cudaSuccess) return e;
  tr.mark(3);
  return cudaSuccess;
}

const char* kPhaseNames[MOE_N_PHASES] = {
    "prep",    "router_logits", "select",  "plan",       "gate_up", "down",
    "combine", "decode_fused",  "tc_prep", "tc_gate_up", "tc_down", "tc_front"};

void free_trace(moe_layer* h) {
  if (h->trace_ev) {
    for (int i = 0; i < h->trace_cap * (MOE_N_PHASES + 1); ++i) cudaEventDestroy(h->trace_ev[i]);
    delete[] h->trace_ev;
  }
  delete[] h->trace_phase;
  delete[] h->trace_nrec;
  h->trace_ev = nullptr;
  h->trace_phase = nullptr;
  h->trace_nrec = nullptr;
  h->trace_cap = 0;
  h->trace_used = 0;
}

}  // namespace

namespace moe {
// Message for moe_last_error(NULL) on this thread (entry points without a handle).
void set_thread_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

const char* config_error(const moe_config_t* c) { return check_config(c); }

const char* device_extent_error(const void* p, size_t bytes, int device) {
  return check_extent(p, bytes, device);
}
}  // namespace moe

extern "C" {

size_t moe_workspace_bytes(const moe_config_t* cfg) {
  if (check_config(cfg)) return 0;
  return layout_for(cfg).total;
}

moe_status_t moe_layer_create(const moe_config_t* cfg, const moe_weights_t* w,
                              moe_layer_t** out) {
  if (!cfg || check_config(cfg)) return moe::layer_create_slots(cfg, w, 0, out);
  return moe::layer_create_slots(cfg, w, cfg->n_experts, out);
}

}  // extern "C"

moe_status_t moe::layer_create_slots(const moe_config_t* cfg, const moe_weights_t* w,
                                     int routed_experts, moe_layer_t** out) {
  if (!out) {
    set_err(nullptr, "out is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (const char* m = check_config(cfg)) {
    set_err(nullptr, "%s", m);
    return MOE_ERR_UNSUPPORTED;
  }
  if (const char* m = check_weights(cfg, w)) {
    set_err(nullptr, "%s", m);
    return MOE_ERR_INVALID_ARG;
  }
  moe_layer* h = new (std::nothrow) moe_layer();
  if (!h) {
    set_err(nullptr, "host allocation failed");
    return MOE_ERR_OOM;
  }
  h->cfg = *cfg;
  h->w = *w;
  h->sh = Shape{cfg->hidden, cfg->inter, cfg->n_shared ? cfg->shared_inter : 0,
                cfg->n_experts, cfg->top_k, cfg->n_group, cfg->topk_group, cfg->n_shared,
                cfg->routed_scaling_factor, cfg->weight_format, cfg->group_size};
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount,
                                                   h->device);
  if (e != cudaSuccess) {
    set_err(nullptr, "no usable CUDA device: %s", cudaGetErrorString(e));
    delete h;
    return MOE_ERR_CUDA;
  }
  const Layout L = layout_for(cfg);
  e = cudaMalloc(&h->ws_base, L.total);
  if (e != cudaSuccess) {
    set_err(nullptr, "workspace allocation of %zu bytes failed: %s", L.total,
            cudaGetErrorString(e));
    cudaGetLastError();
    delete h;
    return MOE_ERR_OOM;
  }
  // (after the workspace allocation, which has made the device's context
  // current on this thread for the driver query)
  const char* which = "";
  if (const char* m = check_weight_memory(cfg, w, static_cast<size_t>(routed_experts),
                                          h->device, &which)) {
    set_err(nullptr, "weight array %s %s", which, m);
    cudaFree(h->ws_base);
    delete h;
    return MOE_ERR_INVALID_ARG;
  }
  h->ws_bytes = L.total;
  h->ws = carve(static_cast<char*>(h->ws_base), L);
  e = cudaMemset(h->ws_base, 0, L.total);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    set_err(nullptr, "workspace initialisation failed: %s", cudaGetErrorString(e));
    cudaFree(h->ws_base);
    delete h;
    return MOE_ERR_CUDA;
  }
  // tensor-core path: TMA tensor maps over the weights and the f16 rows;
  // single-token tensor-core kernel: TMA tensor maps over the weights (not
  // for the expert tier's slots, which only the SIMT batch kernels read)
  const bool all = routed_experts == cfg->n_experts;
  h->tc = all && moe::tc_path_ok(h->sh)
              ? moe::tc_create_maps(h->w, h->sh, h->ws, cfg->max_tokens)
              : nullptr;
  h->dm = all && moe::dm_shape_ok(h->sh) ? moe::dm_create_maps(h->w, h->sh) : nullptr;
  *out = h;
  return MOE_OK;
}

extern "C" {

// x or y of a call as the kernels address it: device (or managed) memory as
// it is, pinned host memory through its device mapping (the kernels then read
// and write it across the host link, with no staging copy).  Other host
// memory is refused before any launch.
static moe_status_t resolve_io(moe_layer_t* h, const void* p, const void** out, const char* what) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    set_err(h, "%s: the CUDA driver does not know this pointer", what);
    return MOE_ERR_INVALID_ARG;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *out = p;
    return MOE_OK;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) {
    *out = at.devicePointer;
    return MOE_OK;
  }
  set_err(h, "%s must be device memory or pinned host memory mapped into the device's "
             "address space", what);
  return MOE_ERR_INVALID_ARG;
}

}  // extern "C"

moe_status_t moe::layer_check_call(moe_layer* h, const void** x, moe_dtype_t dtype, int T,
                                   float** y, const float* rms_gamma, int accumulate,
                                   const moe_plan_t* plan_out, bool route_only) {
  moe_status_t st = check_call(h, *x, dtype, T, rms_gamma);
  if (st != MOE_OK || T == 0) return st;
  if ((st = check_plan(h, plan_out)) != MOE_OK) return st;
  if (route_only) return resolve_io(h, *x, x, "x");
  if (!*y || !aligned16(*y)) {
    set_err(h, "y must be a non-NULL 16-byte aligned device pointer");
    return MOE_ERR_INVALID_ARG;
  }
  const size_t H = h->cfg.hidden;
  const uintptr_t xb = reinterpret_cast<uintptr_t>(*x);
  const uintptr_t xe = xb + static_cast<size_t>(T) * H * (dtype == MOE_BF16 ? 2 : 4);
  const uintptr_t yb = reinterpret_cast<uintptr_t>(*y);
  const uintptr_t ye = yb + static_cast<size_t>(T) * H * 4;
  if (xb < ye && yb < xe) {
    const bool residual_form =
        dtype == MOE_F32 && accumulate && rms_gamma != nullptr && xb == yb;
    if (!residual_form) {
      set_err(h, "x and y overlap; only the in-place residual form (f32, accumulate, "
                 "rms_gamma, y == x) is allowed");
      return MOE_ERR_INVALID_ARG;
    }
  }
  if ((st = resolve_io(h, *x, x, "x")) != MOE_OK) return st;
  const void* yd = nullptr;
  if ((st = resolve_io(h, *y, &yd, "y")) != MOE_OK) return st;
  *y = static_cast<float*>(const_cast<void*>(yd));
  return MOE_OK;
}

cudaError_t moe::layer_route(moe_layer* h, const void* x, moe_dtype_t dt, int T,
                             const float* gamma, float eps, cudaStream_t s) {
  Tracer none;
  return run_route(h, x, dt, T, gamma, eps, s, none);
}

cudaError_t moe::layer_copy_plan(moe_layer* h, int T, const moe_plan_t* p, cudaStream_t s) {
  return copy_plan(h, T, p, s);
}

extern "C" {

moe_status_t moe_route(moe_layer_t* h, const void* x, moe_dtype_t dtype, int T,
                       const float* rms_gamma, float rms_eps, moe_plan_t* plan_out,
                       void* stream) {
  if (!h) {
    set_err(nullptr, "handle is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  moe_status_t st = check_call(h, x, dtype, T, rms_gamma);
  if (st != MOE_OK || T == 0) return st;
  if ((st = resolve_io(h, x, &x, "x")) != MOE_OK) return st;
  if ((st = check_plan(h, plan_out)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Tracer none;
  cudaError_t e = run_route(h, x, dtype, T, rms_gamma, rms_eps, s, none);
  if (e == cudaSuccess) e = copy_plan(h, T, plan_out, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "moe_route");
  return MOE_OK;
}

moe_status_t moe_forward(moe_layer_t* h, const void* x, moe_dtype_t dtype, int T, float* y,
                         const float* rms_gamma, float rms_eps, int accumulate,
                         moe_plan_t* plan_out, void* stream) {
  if (!h) {
    set_err(nullptr, "handle is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  moe_status_t st =
      moe::layer_check_call(h, &x, dtype, T, &y, rms_gamma, accumulate, plan_out, false);
  if (st != MOE_OK || T == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Tracer tr;
  tr.start(h, s);
  const Shape& sh = h->sh;
  const Workspace& ws = h->ws;
  cudaError_t e;
  // one token: a single-kernel path when the shape fits one (the SIMT
  // kernel, measured faster where both fit; else the tensor-core one); else
  // the tensor-core grouped GEMM when the shape fits that, else the SIMT path
  const bool fused = moe::decode_path_ok(sh, T, h->n_sm);
  if (!fused && moe::dm_path_ok(sh, T, h->n_sm, h->dm)) {
    moe::PhaseMarker pm{tr.on() ? &Tracer::mark_cb : nullptr, &tr};
    e = moe::launch_dm(*h->dm, h->w, sh, x, dtype, rms_gamma, rms_eps, ws, y, accumulate,
                       h->n_sm, &h->decode_calls, pm, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (single-token tensor-core path)");
  } else if (fused) {
    moe::PhaseMarker pm{tr.on() ? &Tracer::mark_cb : nullptr, &tr};
    // the plan reaches the workspace only when the caller asked for it
    e = moe::launch_decode(h->w, sh, T, x, dtype, rms_gamma, rms_eps, ws, y, accumulate,
                           plan_out != nullptr ? 1 : 0, h->n_sm, &h->decode_calls, pm, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (single-token path)");
  } else if (h->tc) {
    if (moe::front_path_ok(sh, T, h->n_sm)) {
      // small batch: routing, plan and f16 rows in one cooperative kernel
      e = moe::launch_front(h->w, sh, T, x, dtype, rms_gamma, rms_eps, ws, h->n_sm,
                            &h->decode_calls, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (routing front end)");
      tr.mark(11);
    } else {
      e = run_route(h, x, dtype, T, rms_gamma, rms_eps, s, tr);
      if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (routing)");
      e = moe::launch_tc_prep(sh, T, ws, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (grouped GEMM rows)");
      tr.mark(8);
    }
    e = moe::launch_tc_gemm(*h->tc, sh, T, ws, 0, h->n_sm, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (grouped GEMM gate/up)");
    tr.mark(9);
    e = moe::launch_tc_gemm(*h->tc, sh, T, ws, 1, h->n_sm, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (grouped GEMM down)");
    tr.mark(10);
    e = moe::launch_combine(sh, T, ws, y, accumulate, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (combine)");
    tr.mark(6);
  } else {
    e = run_route(h, x, dtype, T, rms_gamma, rms_eps, s, tr);
    if (e == cudaSuccess) {
      e = moe::launch_gate_up(h->w, sh, T, ws, s);
      tr.mark(4);
    }
    if (e == cudaSuccess) {
      e = moe::launch_down(h->w, sh, T, ws, s);
      tr.mark(5);
    }
    if (e == cudaSuccess) {
      e = moe::launch_combine(sh, T, ws, y, accumulate, s);
      tr.mark(6);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward");
  }
  e = copy_plan(h, T, plan_out, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "moe_forward (plan copy)");
  return MOE_OK;
}

void moe_destroy(moe_layer_t* h) {
  if (!h) return;
  int cur = -1;
  cudaGetDevice(&cur);
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_trace(h);
  moe::tc_destroy_maps(h->tc);
  moe::dm_destroy_maps(h->dm);
  cudaFree(h->ws_base);
  if (cur >= 0) cudaSetDevice(cur);
  delete h;
}

const char* moe_last_error(const moe_layer_t* h) { return h ? h->err : g_err; }

moe_status_t moe_trace_enable(moe_layer_t* h, int n_calls) {
  if (!h) {
    set_err(nullptr, "handle is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (n_calls < 0 || n_calls > 65536) {
    set_err(h, "n_calls must be in [0, 65536]");
    return MOE_ERR_INVALID_ARG;
  }
  cudaDeviceSynchronize();
  free_trace(h);
  if (n_calls == 0) return MOE_OK;
  const int ne = n_calls * (MOE_N_PHASES + 1);
  h->trace_ev = new (std::nothrow) cudaEvent_t[ne];
  h->trace_phase = new (std::nothrow) int[n_calls * MOE_N_PHASES];
  h->trace_nrec = new (std::nothrow) int[n_calls];
  if (!h->trace_ev || !h->trace_phase || !h->trace_nrec) {
    delete[] h->trace_ev;
    delete[] h->trace_phase;
    delete[] h->trace_nrec;
    h->trace_ev = nullptr;
    h->trace_phase = nullptr;
    h->trace_nrec = nullptr;
    set_err(h, "host allocation failed");
    return MOE_ERR_OOM;
  }
  for (int i = 0; i < ne; ++i) {
    const cudaError_t e = cudaEventCreate(&h->trace_ev[i]);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(h->trace_ev[j]);
      delete[] h->trace_ev;
      h->trace_ev = nullptr;
      delete[] h->trace_phase;
      delete[] h->trace_nrec;
      h->trace_phase = nullptr;
      h->trace_nrec = nullptr;
      return cuda_fail(h, e, "cudaEventCreate");
    }
  }
  h->trace_cap = n_calls;
  h->trace_used = 0;
  return MOE_OK;
}

moe_status_t moe_trace_read(moe_layer_t* h, float* ms, int cap, int* n_calls, int* n_phases) {
  if (!h || !ms || !n_calls || !n_phases || cap < 0) {
    set_err(h, "moe_trace_read: NULL argument or negative cap");
    return MOE_ERR_INVALID_ARG;
  }
  *n_phases = MOE_N_PHASES;
  const int n = h->trace_used < cap ? h->trace_used : cap;
  *n_calls = n;
  for (int c = 0; c < n; ++c) {
    for (int p = 0; p < MOE_N_PHASES; ++p) ms[c * MOE_N_PHASES + p] = 0.0f;
    const int nr = h->trace_nrec[c];
    cudaEvent_t* ev = h->trace_ev + c * (MOE_N_PHASES + 1);
    if (nr > 0) {
      const cudaError_t e = cudaEventSynchronize(ev[nr]);
      if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventSynchronize");
    }
    for (int r = 0; r < nr; ++r) {
      float t = 0.0f;
      const cudaError_t e = cudaEventElapsedTime(&t, ev[r], ev[r + 1]);
      if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventElapsedTime");
      ms[c * MOE_N_PHASES + h->trace_phase[c * MOE_N_PHASES + r]] += t;
    }
  }
  h->trace_used = 0;
  return MOE_OK;
}

const char* moe_trace_phase_name(int phase) {
  if (phase < 0 || phase >= MOE_N_PHASES) return nullptr;
  return kPhaseNames[phase];
}

moe_status_t moe_device_status(moe_layer_t* h, int32_t* flags) {
  if (!h || !flags) {
    set_err(h, "moe_device_status: NULL argument");
    return MOE_ERR_INVALID_ARG;
  }
  int32_t v = 0;
  cudaError_t e = cudaMemcpy(&v, h->ws.dev_err, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "moe_device_status");
  *flags = v;
  if (v != 0) {
    // A call that gave up left the grid-barrier counter and the two-part
    // counters out of step with the handle's count of barrier rounds; every
    // later single-token or small-batch call would wait for targets it cannot
    // reach.  Start them all again from zero.
    const Layout L = layout_for(&h->cfg);
    e = cudaMemset(h->ws.dev_err, 0, sizeof(v));
    if (e == cudaSuccess) e = cudaMemset(h->ws.gbar, 0, sizeof(unsigned long long));
    if (e == cudaSuccess && L.off[22] < L.total)
      e = cudaMemset(static_cast<char*>(h->ws_base) + L.off[22], 0, L.total - L.off[22]);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(h, e, "moe_device_status (clear)");
    h->decode_calls = 0;
    set_err(h, "a bounded wait inside a kernel gave up (flags 0x%x); the outputs of the "
               "affected call are not valid",
            static_cast<unsigned>(v));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t moe_selftest_desync(moe_layer_t* h) {
  if (!h) {
    set_err(nullptr, "moe_selftest_desync: handle is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  // the state a call that gave up leaves: the next call's grid-barrier
  // targets lie beyond what its CTAs' arrivals reach
  h->decode_calls += 1;
  return MOE_OK;
}

}  // extern "C"

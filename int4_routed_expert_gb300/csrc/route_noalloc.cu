// moe_route_noalloc: the routing step (optional RMSNorm, router logits,
// noaux_tc selection, routing plan) for callers that must not allocate
// device memory, with its intermediate buffers in a fixed block of static
// device memory instead of a handle's workspace.  See include/moe.h.
#include <mutex>

#include "moe_internal.cuh"

namespace {

// Scratch of the routing step.  Nothing in it needs to start at zero: every
// buffer a kernel reads has been written in full by the kernel before it.
constexpr size_t kNoAllocScratchBytes = 2u << 20;  // 2 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mu;
void* g_addr[kMaxDevices] = {};

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Address of this device's scratch, with that device current.  Looked up
// once per device and cached for calls made while their stream is being
// captured (a capture allows no module loading); every other call looks it
// up again, so that a device reset, after which the module loads anew and
// the array can move, leaves no stale address behind.
cudaError_t scratch_address(cudaStream_t s, unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    cs = cudaStreamCaptureStatusActive;  // unknown: do not touch the module
  }
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (g_addr[dev] == nullptr || cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_addr[dev]);
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" moe_status_t moe_route_noalloc(const moe_config_t* cfg, const float* router_w,
                                          const float* router_bias, const void* x,
                                          moe_dtype_t dtype, int T, const float* rms_gamma,
                                          float rms_eps, moe_plan_t* plan_out, void* stream) {
  if (!cfg) {
    moe::set_thread_error("moe_route_noalloc: cfg is NULL");
    return MOE_ERR_UNSUPPORTED;
  }
  {
    // validated like moe_layer_create, except max_tokens, which this call
    // does not use (T is limited by the scratch instead)
    moe_config_t c = *cfg;
    c.max_tokens = 1;
    if (const char* m = moe::config_error(&c)) {
      moe::set_thread_error("moe_route_noalloc: %s", m);
      return MOE_ERR_UNSUPPORTED;
    }
  }
  if (T < 0) {
    moe::set_thread_error("moe_route_noalloc: T must be >= 0");
    return MOE_ERR_INVALID_ARG;
  }
  if (T == 0) return MOE_OK;
  if (!router_w || !router_bias || !x || !aligned(router_w, 16) || !aligned(router_bias, 16) ||
      !aligned(x, 16) || (rms_gamma && !aligned(rms_gamma, 16)) ||
      (dtype != MOE_F32 && dtype != MOE_BF16)) {
    moe::set_thread_error(
        "moe_route_noalloc: router_w, router_bias and x must be non-NULL and 16-byte "
        "aligned (rms_gamma too when given), dtype MOE_F32 or MOE_BF16");
    return MOE_ERR_INVALID_ARG;
  }
  if (plan_out) {
    const void* m[] = {plan_out->topk_ids, plan_out->topk_w, plan_out->counts,
                       plan_out->offsets,  plan_out->perm,   plan_out->active,
                       plan_out->n_active};
    for (const void* p : m)
      if (p && !aligned(p, 4)) {
        moe::set_thread_error("moe_route_noalloc: plan buffers must be 4-byte aligned");
        return MOE_ERR_INVALID_ARG;
      }
  }
  const size_t H = cfg->hidden, E = cfg->n_experts, k = cfg->top_k;
  const size_t N = static_cast<size_t>(T) * k;
  const size_t sz[10] = {static_cast<size_t>(T) * H * 4, static_cast<size_t>(T) * E * 4,
                         N * 4, N * 4, E * 4, (E + 1) * 4, N * 4, N * 4, E * 4, 4};
  size_t off[10], total = 0;
  for (int i = 0; i < 10; ++i) {
    off[i] = total;
    total += up256(sz[i]);
  }
  if (total > kNoAllocScratchBytes) {
    moe::set_thread_error(
        "moe_route_noalloc: T = %d needs %zu bytes of scratch, above the fixed %zu "
        "(T * (hidden + n_experts) * 4 + 16 * T * top_k + 12 * n_experts plus alignment "
        "must fit in 2 MiB)",
        T, total, kNoAllocScratchBytes);
    return MOE_ERR_CAPACITY;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    // the router arrays are read in full by the logits and selection
    // kernels: a host pointer or a short buffer must not reach them
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
      moe::set_thread_error("moe_route_noalloc: no usable CUDA device: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    const char* which = "router_w";
    const char* m = moe::device_extent_error(router_w, E * H * 4, dev);
    if (!m) {
      which = "router_bias";
      m = moe::device_extent_error(router_bias, E * 4, dev);
    }
    if (m) {
      moe::set_thread_error("moe_route_noalloc: %s %s", which, m);
      return MOE_ERR_INVALID_ARG;
    }
  }
  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(s, &base);
  if (e != cudaSuccess) {
    moe::set_thread_error("moe_route_noalloc: scratch address lookup failed: %s",
                          cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  float* xf = reinterpret_cast<float*>(base + off[0]);
  float* logits = reinterpret_cast<float*>(base + off[1]);
  int32_t* ids = plan_out && plan_out->topk_ids ? plan_out->topk_ids
                                                : reinterpret_cast<int32_t*>(base + off[2]);
  float* topw = plan_out && plan_out->topk_w ? plan_out->topk_w
                                             : reinterpret_cast<float*>(base + off[3]);
  int32_t* counts = plan_out && plan_out->counts ? plan_out->counts
                                                 : reinterpret_cast<int32_t*>(base + off[4]);
  int32_t* offsets = plan_out && plan_out->offsets ? plan_out->offsets
                                                   : reinterpret_cast<int32_t*>(base + off[5]);
  int32_t* perm = plan_out && plan_out->perm ? plan_out->perm
                                             : reinterpret_cast<int32_t*>(base + off[6]);
  int32_t* inv = reinterpret_cast<int32_t*>(base + off[7]);
  int32_t* active = plan_out && plan_out->active ? plan_out->active
                                                 : reinterpret_cast<int32_t*>(base + off[8]);
  int32_t* n_active = plan_out && plan_out->n_active
                          ? plan_out->n_active
                          : reinterpret_cast<int32_t*>(base + off[9]);
  const moe::Shape sh{cfg->hidden, cfg->inter, cfg->n_shared ? cfg->shared_inter : 0,
                      cfg->n_experts, cfg->top_k, cfg->n_group, cfg->topk_group,
                      cfg->n_shared, cfg->routed_scaling_factor};
  e = moe::launch_prep(x, dtype, T, sh.H, rms_gamma, rms_eps, xf, s);
  if (e == cudaSuccess) e = moe::launch_router_logits(xf, T, sh.H, router_w, sh.E, logits, s);
  if (e == cudaSuccess) e = moe::launch_select(logits, router_bias, T, sh, ids, topw, s);
  if (e == cudaSuccess)
    e = moe::launch_plan(ids, T, sh.k, sh.E, counts, offsets, perm, inv, active, n_active, s);
  if (e != cudaSuccess) {
    moe::set_thread_error("moe_route_noalloc: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Shared definitions of the fused single-token kernel (decode_fused.cuh):
// arguments, the RMSNorm and activation staging helpers, the grid barrier,
// the in-kernel router (logits in the fixed order, register selection) and
// the launch helpers.
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", N1
// (MoE bullet), N2 (packed int4 gate/up/down with grouped scales), N4 (route
// first, stream the selected experts once); "colibri-strix/README.md",
// "What's implemented" (noaux_tc router, shared expert).
#pragma once

#include "moe_internal.cuh"
#include "router_math.cuh"
#include "stream_common.cuh"

namespace moe {
namespace dec {

constexpr int kMaxEntries = 32;       // T * k
constexpr int kRowsC = 4;             // down-projection rows per item
constexpr int kMaxLocalExperts = 8;   // router experts per CTA
constexpr int kRouterWarps = 8;       // one warp per logit segment

struct DecArgs {
  moe_weights_t w;
  Shape sh;
  int T;
  const void* x;
  int dt;
  const float* gamma;
  float eps;
  Workspace ws;
  float* y;
  int accumulate;
  int write_plan = 1;  // the single-token kernels write the call's plan to the workspace
  unsigned long long gtarget;   // grid-barrier count that completes this call's first barrier
  unsigned long long gtarget2;  // ... and its second (fused single-token kernel)
};

// Balanced split of n items over B parts: [begin, end) of part b.
__host__ __device__ __forceinline__ void split_range(int n, int b, int B, int& begin,
                                                     int& end) {
  const int base = n / B, rem = n % B;
  begin = b * base + (b < rem ? b : rem);
  end = begin + base + (b < rem ? 1 : 0);
}

// Chunks of 32 groups per lane for a K-long row: K < 1024 -> 1 (lanes past
// K/32 idle); else K / 1024 when that is an instantiated count; 0 otherwise.
__host__ __device__ inline int chunks_per_lane(int K) {
  if (K % 32 != 0) return 0;
  if (K < 1024) return 1;
  if (K % 1024 != 0) return 0;
  const int c = K / 1024;
  return (c == 1 || c == 2 || c == 4 || c == 6 || c == 8) ? c : 0;
}

// fp32 reciprocal root of one token's RMSNorm, reduced by the first 8 warps
// of the CTA (warp = segment) in the fixed fp64 order; valid in rf after the
// caller's __syncthreads.  dseg: 8 doubles of shared memory.
__device__ inline void rms_partial(const DecArgs& a, int t, double* dseg) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kRouterWarps) return;
  const int H = a.sh.H, L = H / kSeg, chunks = L / 4;
  const size_t base = static_cast<size_t>(t) * H + static_cast<size_t>(warp) * L;
  double acc = 0.0;
  for (int c = lane; c < chunks; c += 32) {
    const float4 v = load_x4(a.x, a.dt, base + 4 * c);
    acc = __fma_rn(static_cast<double>(v.x), static_cast<double>(v.x), acc);
    acc = __fma_rn(static_cast<double>(v.y), static_cast<double>(v.y), acc);
    acc = __fma_rn(static_cast<double>(v.z), static_cast<double>(v.z), acc);
    acc = __fma_rn(static_cast<double>(v.w), static_cast<double>(v.w), acc);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) acc = __dadd_rn(acc, __shfl_down_sync(0xffffffffu, acc, d));
  if (lane == 0) dseg[warp] = acc;
}

__device__ inline float rms_finish(const DecArgs& a, const double* dseg) {
  double a0 = __dadd_rn(dseg[0], dseg[4]), a1 = __dadd_rn(dseg[1], dseg[5]);
  double a2 = __dadd_rn(dseg[2], dseg[6]), a3 = __dadd_rn(dseg[3], dseg[7]);
  a0 = __dadd_rn(a0, a2);
  a1 = __dadd_rn(a1, a3);
  const double mean = __ddiv_rn(__dadd_rn(a0, a1), static_cast<double>(a.sh.H));
  return __double2float_rn(
      __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(mean, static_cast<double>(a.eps)))));
}

// x_hat for elements idx..idx+3 of token t (x row offset included in idx).
__device__ __forceinline__ float4 xhat4(const DecArgs& a, size_t idx, int k, float rf) {
  float4 v = load_x4(a.x, a.dt, idx);
  if (a.gamma != nullptr) {
    const float4 g = __ldg(reinterpret_cast<const float4*>(a.gamma + k));
    v.x = __fmul_rn(__fmul_rn(v.x, rf), g.x);
    v.y = __fmul_rn(__fmul_rn(v.y, rf), g.y);
    v.z = __fmul_rn(__fmul_rn(v.z, rf), g.z);
    v.w = __fmul_rn(__fmul_rn(v.w, rf), g.w);
  }
  return v;
}

// Stores x_hat[k..k+3] (k % 4 == 0) pre-scaled into the swizzled layout.
__device__ __forceinline__ void swz_store4(float* dst, int k, float4 v) {
  const int g = k >> 5, i = k & 31;
  v.x *= swz_prescale(i);
  v.y *= swz_prescale(i + 1);
  v.z *= swz_prescale(i + 2);
  v.w *= swz_prescale(i + 3);
  *reinterpret_cast<float4*>(dst + swz_index(g, i)) = v;
}

// ---- grid barrier: a monotonic 64-bit counter in the workspace ---------
//
// Every CTA adds one per barrier round; round r of the handle completes when
// the counter reaches r * gridDim.x.  Waits are bounded.
__device__ __forceinline__ void gbar_arrive(unsigned long long* p) {
  asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}

__device__ __forceinline__ unsigned long long gbar_load(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Lane 0 polls the grid-barrier counter (bounded); returns false on timeout.
__device__ inline bool gbar_wait(unsigned long long* p, unsigned long long target, int* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    if (gbar_load(p) < target) {
      const long long t0 = clock64();
      while (gbar_load(p) < target) {
        if (clock64() - t0 > kWaitClocks) {
          atomicOr(err, kErrWaitTimeout);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  __threadfence();
  return ok != 0;
}

// 4- and 8-byte global -> shared copies (cp.async, through L1) and the
// arrive-on of an mbarrier once this thread's copies so far have landed
// (the pending count is raised first, so the phase waits for them).
__device__ __forceinline__ void cp_async_ca4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_ca8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ const void* align_down4(const void* p) {
  return reinterpret_cast<const void*>(reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(3));
}

// Release store of a monotonic generation word (read with gbar_wait).
__device__ __forceinline__ void publish_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

template <int EPL>
__device__ __forceinline__ void select_token(const DecArgs& a, int t, int& id, float& w) {
  const size_t o = static_cast<size_t>(t) * a.sh.E;
  warp_select_regs<EPL>(a.ws.skey + o, a.ws.sval + o, a.sh, id, w);
}

// Router logits from shared memory: xn = x_hat in natural order [H], wr =
// the CTA's router rows [L][H] (expert blockIdx.x + l * gridDim.x).  Same
// fixed order and roundings as router_cta; warp 0 writes the results.
__device__ __forceinline__ void router_cta_smem(const DecArgs& a, const float* xn, const float* wr,
                                                float* lseg) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kRouterWarps) return;
  const int H = a.sh.H, E = a.sh.E;
  const int L = (E + gridDim.x - 1) / gridDim.x;
  const int Lseg = H / kSeg, chunks = Lseg / 4;
  for (int l = 0; l < L; ++l) {
    const int e = blockIdx.x + l * gridDim.x;
    if (e >= E) break;
    const float* w = wr + static_cast<size_t>(l) * H;
    float acc = 0.0f;
    for (int c = lane; c < chunks; c += 32) {
      const int kk = warp * Lseg + 4 * c;
      const float4 xv = *reinterpret_cast<const float4*>(xn + kk);
      const float4 w4 = *reinterpret_cast<const float4*>(w + kk);
      acc = __fmaf_rn(xv.x, w4.x, acc);
      acc = __fmaf_rn(xv.y, w4.y, acc);
      acc = __fmaf_rn(xv.z, w4.z, acc);
      acc = __fmaf_rn(xv.w, w4.w, acc);
    }
    const float p = segment_tree(acc);
    if (lane == 0) lseg[l * kRouterWarps + warp] = p;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kRouterWarps * 32) : "memory");
  if (warp == 0) {
    const int e = blockIdx.x + lane * gridDim.x;
    if (lane < L && e < E) {
      float sg[kSeg];
#pragma unroll
      for (int s = 0; s < kSeg; ++s) sg[s] = lseg[lane * kRouterWarps + s];
      const float logit = segments_sum(sg);
      const float sv = router_sigmoid(logit);
      a.ws.logits[e] = logit;
      a.ws.sval[e] = sv;
      a.ws.skey[e] = __fadd_rn(sv, __ldg(a.w.router_bias + e));
    }
  }
}

// Router logits of this CTA's experts (blockIdx.x + l * gridDim.x) by warps
// 0..7, one logit segment each, in the fixed order; warp 0 then writes the
// logits, scores and keys of those experts.  Called by every warp; only
// warps 0..7 take part (they meet on named barrier 1).  rfs: the tokens'
// RMSNorm scales (read when gamma is given).  The caller publishes.
// RC: upper bound of the chunks a lane handles (H / 1024, at least 1); the
// loop is unrolled so that all of a lane's loads are in flight together.
template <int NT, int RC>
__device__ __forceinline__ void router_cta(const DecArgs& a, float* lseg, const float* rfs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kRouterWarps) return;
  const int H = a.sh.H, E = a.sh.E, T = a.T;
  const int L = (E + gridDim.x - 1) / gridDim.x;
  const int Lseg = H / kSeg, chunks = Lseg / 4;
  float acc[kMaxLocalExperts][NT];
#pragma unroll
  for (int l = 0; l < kMaxLocalExperts; ++l)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[l][t] = 0.0f;
#pragma unroll
  for (int ci = 0; ci < RC; ++ci) {
    const int c = lane + 32 * ci;
    if (c >= chunks) break;
    const int kk = warp * Lseg + 4 * c;
    float4 xv[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
      xv[t] = t < T ? xhat4(a, static_cast<size_t>(t) * H + kk, kk,
                            a.gamma != nullptr ? rfs[t] : 1.0f)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int l = 0; l < kMaxLocalExperts; ++l) {
      const int e = blockIdx.x + l * gridDim.x;
      if (l < L && e < E) {
        const float4 w4 =
            __ldg(reinterpret_cast<const float4*>(a.w.router_w + static_cast<size_t>(e) * H + kk));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          float s = acc[l][t];
          s = __fmaf_rn(xv[t].x, w4.x, s);
          s = __fmaf_rn(xv[t].y, w4.y, s);
          s = __fmaf_rn(xv[t].z, w4.z, s);
          s = __fmaf_rn(xv[t].w, w4.w, s);
          acc[l][t] = s;
        }
      }
    }
  }
#pragma unroll
  for (int l = 0; l < kMaxLocalExperts; ++l) {
    if (l >= L) break;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float p = segment_tree(acc[l][t]);
      if (lane == 0) lseg[(l * kRouterWarps + warp) * NT + t] = p;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kRouterWarps * 32) : "memory");
  if (warp == 0) {
    const int l = lane / NT, t = lane % NT;
    const int e = blockIdx.x + l * gridDim.x;
    if (l < L && t < T && e < E) {
      float sg[kSeg];
#pragma unroll
      for (int s = 0; s < kSeg; ++s) sg[s] = lseg[(l * kRouterWarps + s) * NT + t];
      const float logit = segments_sum(sg);
      const float sv = router_sigmoid(logit);
      const size_t o = static_cast<size_t>(t) * E + e;
      a.ws.logits[o] = logit;
      a.ws.sval[o] = sv;
      a.ws.skey[o] = __fadd_rn(sv, __ldg(a.w.router_bias + e));
    }
  }
}

// ---- host side ------------------------------------------------------------

// Launch with cudaLaunchKernelEx: optional programmatic stream serialisation
// (the kernel may start while the previous one finishes; it waits with
// griddepcontrol.wait) and optional cooperative launch (all CTAs resident).
template <typename K>
cudaError_t launch_k(K kernel, int grid, int threads, size_t smem, cudaStream_t s,
                     const DecArgs& a, bool pdl, bool coop) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (coop) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace dec
}  // namespace moe

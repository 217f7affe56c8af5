// Routing front end of the grouped GEMM for small batches (T <= 4, T*k <= 32)
// in one cooperative kernel, instead of the prep / logits / select / plan /
// chunk-list kernels of larger batches.  Same results as those kernels,
// bit for bit.
//
//   1. every CTA: RMSNorm scales of the T tokens (when gamma is given) and the
//      router logits of its own experts (blockIdx.x + l * gridDim.x) in the
//      fixed order; scores and keys to the workspace; grid barrier.
//   2. every CTA, redundantly: warp t selects token t (register selection),
//      warp 0 builds the plan of the T*k entries in registers (stable: expert
//      ascending, entry index ascending inside an expert).
//   3. CTA 0 writes the plan, the active list and the chunk list (one chunk
//      per active expert: at most 32 rows); CTA b writes f16 activation rows
//      b, b + G, ... (plan positions, then the shared expert's token rows).
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy": N1
// (MoE bullet: sigmoid router, group-limited top-k, renormalised gates), N4
// and "G3 implementation status" (route the whole batch first; stable
// row/rank batch union).
#include "decode_common.cuh"
#include "smem_opt_in.cuh"

namespace moe {
namespace dec {
namespace {

constexpr int kFrontThreads = kRouterWarps * 32;  // 256
constexpr int kFrontNT = 4;

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// x[idx..idx+3] as f32 from the shared-memory copy of x (f32 or bf16).
__device__ __forceinline__ float4 load_x4_smem(const void* xb, int dt, size_t idx) {
  if (dt == MOE_BF16) {
    const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(xb) + idx);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(xb) + idx);
}

// x_hat[idx..idx+3] from the shared-memory copy of x; k = column.
__device__ __forceinline__ float4 xhat4_at(const void* xb, int dt, size_t idx, int k, float rf,
                                           const float* gamma) {
  float4 v = load_x4_smem(xb, dt, idx);
  if (gamma != nullptr) {
    const float4 g = __ldg(reinterpret_cast<const float4*>(gamma + k));
    v.x = __fmul_rn(__fmul_rn(v.x, rf), g.x);
    v.y = __fmul_rn(__fmul_rn(v.y, rf), g.y);
    v.z = __fmul_rn(__fmul_rn(v.z, rf), g.z);
    v.w = __fmul_rn(__fmul_rn(v.w, rf), g.w);
  }
  return v;
}

// Sum of squares of token t (fixed order of the router, fp64) from the copy
// of x in shared memory; warps 0..7 write one partial each to dseg.
__device__ __forceinline__ void rms_partial_at(const void* xb, int dt, int H, int t, double* dseg) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = H / kSeg, chunks = L / 4;
  const size_t base = static_cast<size_t>(t) * H + static_cast<size_t>(warp) * L;
  double acc = 0.0;
  for (int c = lane; c < chunks; c += 32) {
    const float4 v = load_x4_smem(xb, dt, base + 4 * c);
    acc = __fma_rn(static_cast<double>(v.x), static_cast<double>(v.x), acc);
    acc = __fma_rn(static_cast<double>(v.y), static_cast<double>(v.y), acc);
    acc = __fma_rn(static_cast<double>(v.z), static_cast<double>(v.z), acc);
    acc = __fma_rn(static_cast<double>(v.w), static_cast<double>(v.w), acc);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) acc = __dadd_rn(acc, __shfl_down_sync(0xffffffffu, acc, d));
  if (lane == 0) dseg[warp] = acc;
}

// Router logits of this CTA's experts for NT tokens, read from shared
// memory (xb: the tokens' x rows, wr: the CTA's router rows), in the same
// fixed order and roundings as router_cta.
template <int NT, int RC>
__device__ __forceinline__ void router_cta_at(const DecArgs& a, const void* xb, const float* wr,
                                              float* lseg, const float* rfs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
      xv[t] = t < T ? xhat4_at(xb, a.dt, static_cast<size_t>(t) * H + kk, kk,
                               a.gamma != nullptr ? rfs[t] : 1.0f, a.gamma)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int l = 0; l < kMaxLocalExperts; ++l) {
      const int e = blockIdx.x + l * gridDim.x;
      if (l < L && e < E) {
        const float4 w4 = *reinterpret_cast<const float4*>(wr + static_cast<size_t>(l) * H + kk);
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
  __syncthreads();
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

template <int RC>
__global__ void __launch_bounds__(kFrontThreads, 1) front_kernel(const __grid_constant__ DecArgs a) {
  extern __shared__ __align__(16) unsigned char fsm[];  // x rows, then the CTA's router rows
  __shared__ __align__(8) uint64_t ldbar;
  __shared__ float lseg[kMaxLocalExperts * kRouterWarps * kFrontNT];
  __shared__ double dseg[8];
  __shared__ float rfs[kFrontNT];
  __shared__ int s_id[kMaxEntries], s_perm[kMaxEntries];
  __shared__ int s_ok;
  const Shape& sh = a.sh;
  const Workspace& ws = a.ws;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, k = sh.k, E = sh.E, H = sh.H, N = T * k;

  // 1. x rows and this CTA's router rows into shared memory by TMA (one
  //    round trip instead of one per loop step), RMSNorm scales, logits of
  //    this CTA's experts, grid barrier
  const int esz = a.dt == static_cast<int>(MOE_BF16) ? 2 : 4;
  const uint32_t xbytes = static_cast<uint32_t>(T) * H * esz;
  const int G = gridDim.x, Lx = (E + G - 1) / G;
  int nl = 0;
  for (int l = 0; l < Lx; ++l) nl += (blockIdx.x + l * G < E) ? 1 : 0;
  const float* wr = reinterpret_cast<const float*>(fsm + ((xbytes + 15) & ~15u));
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ldbar), 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(smem_u32(&ldbar), xbytes + static_cast<uint32_t>(nl) * H * 4);
    bulk_g2s(smem_u32(fsm), a.x, xbytes, smem_u32(&ldbar));
    for (int l = 0; l < nl; ++l)
      bulk_g2s(smem_u32(wr + static_cast<size_t>(l) * H),
               a.w.router_w + static_cast<size_t>(blockIdx.x + l * G) * H, H * 4,
               smem_u32(&ldbar));
  }
  __syncthreads();
  const int landed = mbar_wait(smem_u32(&ldbar), 0, ws.dev_err) ? 1 : 0;
  if (!__syncthreads_and(landed)) return;
  if (a.gamma != nullptr) {
    for (int t = 0; t < T; ++t) {
      rms_partial_at(fsm, a.dt, H, t, dseg);
      __syncthreads();
      if (threadIdx.x == 0) rfs[t] = rms_finish(a, dseg);
      __syncthreads();
    }
  }
  router_cta_at<kFrontNT, RC>(a, fsm, wr, lseg, rfs);
  __syncthreads();
  if (warp == 0) {
    __threadfence();
    __syncwarp();
    if (lane == 0) gbar_arrive(ws.gbar);
    const bool ok = gbar_wait(ws.gbar, a.gtarget, ws.dev_err);
    if (lane == 0) s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  if (!s_ok) return;

  // 2. selection of token t by warp t, then the plan by warp 0
  if (warp < T) {
    int id = 0;
    float w = 0.0f;
    switch (fast_select_epl(sh)) {
      case 1: select_token<1>(a, warp, id, w); break;
      case 2: select_token<2>(a, warp, id, w); break;
      case 4: select_token<4>(a, warp, id, w); break;
      default: select_token<8>(a, warp, id, w); break;
    }
    if (lane < k) {
      s_id[warp * k + lane] = id;
      if (blockIdx.x == 0) {
        ws.ids[warp * k + lane] = id;
        ws.topw[warp * k + lane] = w;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int e = lane < N ? s_id[lane] : 0x7fffffff;
    int less = 0, before = 0, first_less = 0;
    for (int j = 0; j < N; ++j) {
      const int o = s_id[j];
      less += o < e ? 1 : 0;
      before += (o == e && j < lane) ? 1 : 0;
    }
    const bool first = lane < N && before == 0;
    const unsigned firsts = __ballot_sync(0xffffffffu, first);
    for (int j = 0; j < N; ++j)
      first_less += (((firsts >> j) & 1u) && s_id[j] < e) ? 1 : 0;
    const int pos = less + before;  // plan position of entry `lane`
    if (lane < N) s_perm[pos] = lane;
    if (blockIdx.x == 0) {
      if (lane < N) {
        ws.perm[pos] = lane;
        ws.inv[lane] = pos;
      }
      if (first) {
        int cnt = 0;
        for (int j = 0; j < N; ++j) cnt += s_id[j] == e ? 1 : 0;
        ws.active[first_less] = e;
        ws.chunks[first_less] = make_int4(less, cnt, e, 0);
      }
      if (lane == 0) {
        *ws.n_active = __popc(firsts);
        *ws.n_rchunks = __popc(firsts);
        ws.offsets[E] = N;
      }
    }
  }
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int cnt = 0, off = 0;
      for (int j = 0; j < N; ++j) {
        const int o = s_id[j];
        cnt += o == e ? 1 : 0;
        off += o < e ? 1 : 0;
      }
      ws.counts[e] = cnt;
      ws.offsets[e] = off;
    }
  }
  __syncthreads();

  // 3. f16 activation rows (8-element order of the grouped GEMM's
  //    dequantised weights: 0,4,1,5,2,6,3,7)
  const int rows = N + (sh.n_shared ? T : 0);
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int t = r < N ? s_perm[r] / k : r - N;
    const float rf = a.gamma != nullptr ? rfs[t] : 1.0f;
    uint4* dst = reinterpret_cast<uint4*>(ws.x16 + static_cast<size_t>(r) * H);
    for (int o = threadIdx.x; o < H / 8; o += blockDim.x) {
      const size_t idx = static_cast<size_t>(t) * H + 8 * o;
      const float4 lo = xhat4(a, idx, 8 * o, rf), hi = xhat4(a, idx + 4, 8 * o + 4, rf);
      dst[o] = make_uint4(pack_h2(lo.x, hi.x), pack_h2(lo.y, hi.y), pack_h2(lo.z, hi.z),
                          pack_h2(lo.w, hi.w));
    }
  }
}

}  // namespace
}  // namespace dec

size_t front_smem_bytes(const Shape& sh, int T, int n_sm) {
  using namespace dec;
  const size_t L = (sh.E + n_sm - 1) / n_sm;
  return ((static_cast<size_t>(T) * sh.H * 4 + 15) & ~static_cast<size_t>(15)) + L * sh.H * 4;
}

namespace dec {
namespace {
// Opts the kernel in to `smem` bytes of dynamic shared memory (static shared
// memory comes on top, so the 48 KB default is not enough at 48 KB).
template <int RC>
cudaError_t front_attr(size_t smem) {
  static std::atomic<size_t> set[kMaxDevices];  // per instantiation
  return opt_in_smem(reinterpret_cast<const void*>(front_kernel<RC>), set, smem);
}
}  // namespace
}  // namespace dec

bool front_path_ok(const Shape& sh, int T, int n_sm) {
  using namespace dec;
  if (T < 1 || T > kFrontNT || T * sh.k > kMaxEntries) return false;
  if (front_smem_bytes(sh, T, n_sm) > 200 * 1024) return false;
  const int epl = fast_select_epl(sh);
  if (epl != 1 && epl != 2 && epl != 4 && epl != 8) return false;
  if (n_sm < 1 || (sh.E + n_sm - 1) / n_sm > kMaxLocalExperts) return false;
  return chunks_per_lane(sh.H) != 0 && sh.H % 8 == 0;
}

cudaError_t launch_front(const moe_weights_t& w, const Shape& sh, int T, const void* x,
                         moe_dtype_t dt, const float* gamma, float eps, const Workspace& ws,
                         int n_sm, unsigned long long* calls, cudaStream_t s) {
  using namespace dec;
  DecArgs a = {};
  a.w = w;
  a.sh = sh;
  a.T = T;
  a.x = x;
  a.dt = static_cast<int>(dt);
  a.gamma = gamma;
  a.eps = eps;
  a.ws = ws;
  a.gtarget = (*calls + 1) * static_cast<unsigned long long>(n_sm);
  const size_t smem = front_smem_bytes(sh, T, n_sm);  // f32 bound on the x copy
  cudaError_t e;
  switch (chunks_per_lane(sh.H)) {
#define MOE_FRONT_CASE(RC)                                                      \
  case RC:                                                                      \
    e = front_attr<RC>(smem);                                                   \
    if (e == cudaSuccess)                                                       \
      e = launch_k(front_kernel<RC>, n_sm, kFrontThreads, smem, s, a, false, true); \
    break;
    MOE_FRONT_CASE(1)
    MOE_FRONT_CASE(2)
    MOE_FRONT_CASE(4)
    MOE_FRONT_CASE(6)
    MOE_FRONT_CASE(8)
#undef MOE_FRONT_CASE
    default:
      return cudaErrorInvalidValue;
  }
  if (e == cudaSuccess) *calls += 1;
  return e;
}

}  // namespace moe

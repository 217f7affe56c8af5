// General router: input preparation (optional RMSNorm), router logits and
// the noaux_tc selection, one stage per kernel.  Compiled with -fmad=false:
// every product and sum of the router is rounded where the definition says.
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", N1
// "GLM-5.2 graph" (MoE bullet); "colibri-strix/README.md", "What's
// implemented"; RMSNorm: "Model support - run anything mlx-lm runs", 6.4
// "GLM-5.2" (multiplicative weight, double-accumulated reduction) and the
// first page's "G4 - serial native MTP" (float64 squared sums).
#include "moe_internal.cuh"
#include "router_math.cuh"

namespace moe {
namespace {

constexpr int kPrepThreads = 256;  // 8 warps = the 8 segments

// One CTA per token.  Without gamma: xf = fp32(x).  With gamma:
//   ss = sum of squares in fp64, in the segment order of the router logits
//   r  = 1 / sqrt(ss / H + eps)             (fp64, each step rounded)
//   xf = (x * fp32(r)) * gamma              (two fp32 products)
__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(const void* __restrict__ x, int dt, int H, const float* __restrict__ gamma,
            float eps, float* __restrict__ xf) {
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t base = static_cast<size_t>(t) * H;
  __shared__ double seg[kSeg];
  __shared__ float rr;
  if (gamma != nullptr) {
    const int L = H / kSeg, chunks = L / 4;
    double acc = 0.0;
    for (int c = lane; c < chunks; c += 32) {
      const float4 v = load_x4(x, dt, base + warp * L + 4 * c);
      acc = __fma_rn(static_cast<double>(v.x), static_cast<double>(v.x), acc);
      acc = __fma_rn(static_cast<double>(v.y), static_cast<double>(v.y), acc);
      acc = __fma_rn(static_cast<double>(v.z), static_cast<double>(v.z), acc);
      acc = __fma_rn(static_cast<double>(v.w), static_cast<double>(v.w), acc);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc = __dadd_rn(acc, __shfl_down_sync(0xffffffffu, acc, d));
    if (lane == 0) seg[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      double a0 = __dadd_rn(seg[0], seg[4]), a1 = __dadd_rn(seg[1], seg[5]);
      double a2 = __dadd_rn(seg[2], seg[6]), a3 = __dadd_rn(seg[3], seg[7]);
      a0 = __dadd_rn(a0, a2);
      a1 = __dadd_rn(a1, a3);
      const double ss = __dadd_rn(a0, a1);
      const double mean = __ddiv_rn(ss, static_cast<double>(H));
      rr = __double2float_rn(
          __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(mean, static_cast<double>(eps)))));
    }
    __syncthreads();
    const float r = rr;
    for (int i = threadIdx.x * 4; i < H; i += kPrepThreads * 4) {
      const float4 v = load_x4(x, dt, base + i);
      const float4 g = __ldg(reinterpret_cast<const float4*>(gamma + i));
      float4 o;
      o.x = __fmul_rn(__fmul_rn(v.x, r), g.x);
      o.y = __fmul_rn(__fmul_rn(v.y, r), g.y);
      o.z = __fmul_rn(__fmul_rn(v.z, r), g.z);
      o.w = __fmul_rn(__fmul_rn(v.w, r), g.w);
      *reinterpret_cast<float4*>(xf + base + i) = o;
    }
  } else {
    for (int i = threadIdx.x * 4; i < H; i += kPrepThreads * 4)
      *reinterpret_cast<float4*>(xf + base + i) = load_x4(x, dt, base + i);
  }
}

// Router logits for a tile of kTE experts x kTT tokens per CTA; warp s owns
// segment s, lane j the chunks j, j+32, ... of it (the fixed order above).
constexpr int kTE = 4, kTT = 8;

__global__ void __launch_bounds__(256)
logits_kernel(const float* __restrict__ xf, int T, int H, const float* __restrict__ Wr,
              int E, float* __restrict__ logits) {
  const int e0 = blockIdx.x * kTE, t0 = blockIdx.y * kTT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = H / kSeg, chunks = L / 4;
  __shared__ float segsum[kSeg][kTE * kTT];
  float acc[kTE][kTT];
#pragma unroll
  for (int a = 0; a < kTE; ++a)
#pragma unroll
    for (int b = 0; b < kTT; ++b) acc[a][b] = 0.0f;
  for (int c = lane; c < chunks; c += 32) {
    const size_t off = static_cast<size_t>(warp) * L + 4 * c;
    float4 w[kTE];
#pragma unroll
    for (int a = 0; a < kTE; ++a) {
      const int e = min(e0 + a, E - 1);
      w[a] = __ldg(reinterpret_cast<const float4*>(Wr + static_cast<size_t>(e) * H + off));
    }
#pragma unroll
    for (int b = 0; b < kTT; ++b) {
      const int t = min(t0 + b, T - 1);
      const float4 v = *reinterpret_cast<const float4*>(xf + static_cast<size_t>(t) * H + off);
#pragma unroll
      for (int a = 0; a < kTE; ++a) {
        float s = acc[a][b];
        s = __fmaf_rn(v.x, w[a].x, s);
        s = __fmaf_rn(v.y, w[a].y, s);
        s = __fmaf_rn(v.z, w[a].z, s);
        s = __fmaf_rn(v.w, w[a].w, s);
        acc[a][b] = s;
      }
    }
  }
  // the 32 segment trees at once: lane L ends with value L = (a, b)
  static_assert(kTE * kTT == 32, "one value per lane");
  float v[32];
#pragma unroll
  for (int a = 0; a < kTE; ++a)
#pragma unroll
    for (int b = 0; b < kTT; ++b) v[a * kTT + b] = acc[a][b];
  segsum[warp][lane] = segment_tree32(v);
  __syncthreads();
  if (threadIdx.x < kTE * kTT) {
    const int a = threadIdx.x / kTT, b = threadIdx.x % kTT;
    const int e = e0 + a, t = t0 + b;
    if (e < E && t < T) {
      float sg[kSeg];
#pragma unroll
      for (int s = 0; s < kSeg; ++s) sg[s] = segsum[s][threadIdx.x];
      logits[static_cast<size_t>(t) * E + e] = segments_sum(sg);
    }
  }
}

constexpr int kSelWarps = 4;

// One warp per token; scores, keys and flags staged in shared memory.
__global__ void __launch_bounds__(kSelWarps * 32)
select_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T,
              Shape sh, int32_t* __restrict__ ids, float* __restrict__ topw) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + warp;
  const int E = sh.E;
  float* s = sm + static_cast<size_t>(warp) * (2 * E + sh.n_group + (2 * E + 3) / 4 + 1);
  float* key = s + E;
  float* gsc = key + E;
  uint8_t* taken = reinterpret_cast<uint8_t*>(gsc + sh.n_group);
  uint8_t* gkept = taken + E;
  if (t >= T) return;
  for (int e = lane; e < E; e += 32) {
    const float v = router_sigmoid(logits[static_cast<size_t>(t) * E + e]);
    s[e] = v;
    key[e] = __fadd_rn(v, bias[e]);
  }
  __syncwarp();
  warp_select(s, key, gsc, gkept, taken, sh, ids + static_cast<size_t>(t) * sh.k,
              topw + static_cast<size_t>(t) * sh.k);
}

// One warp per token, everything in registers (shapes accepted by
// fast_select_epl): same ids and weights as select_kernel.
template <int EPL>
__global__ void __launch_bounds__(kSelWarps * 32)
select_regs_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T,
                   Shape sh, int32_t* __restrict__ ids, float* __restrict__ topw) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + warp;
  if (t >= T) return;
  int id;
  float w;
  warp_select_logits<EPL>(logits + static_cast<size_t>(t) * sh.E, bias, sh, id, w);
  if (lane < sh.k) {
    ids[static_cast<size_t>(t) * sh.k + lane] = id;
    topw[static_cast<size_t>(t) * sh.k + lane] = w;
  }
}

size_t select_smem(const Shape& sh) {
  const int E = sh.E;
  return static_cast<size_t>(kSelWarps) * (2 * E + sh.n_group + (2 * E + 3) / 4 + 1) * 4;
}

}  // namespace

cudaError_t launch_prep(const void* x, moe_dtype_t dtype, int T, int H, const float* gamma,
                        float eps, float* xf, cudaStream_t s) {
  prep_kernel<<<T, kPrepThreads, 0, s>>>(x, static_cast<int>(dtype), H, gamma, eps, xf);
  return cudaGetLastError();
}

cudaError_t launch_router_logits(const float* xf, int T, int H, const float* Wr, int E,
                                 float* logits, cudaStream_t s) {
  const dim3 grid((E + kTE - 1) / kTE, (T + kTT - 1) / kTT);
  logits_kernel<<<grid, 256, 0, s>>>(xf, T, H, Wr, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* logits, const float* bias, int T, const Shape& sh,
                          int32_t* ids, float* topw, cudaStream_t s) {
  const int grid = (T + kSelWarps - 1) / kSelWarps;
  switch (fast_select_epl(sh)) {
#define MOE_SEL_CASE(EPL)                                                                     \
  case EPL:                                                                                   \
    select_regs_kernel<EPL><<<grid, kSelWarps * 32, 0, s>>>(logits, bias, T, sh, ids, topw); \
    return cudaGetLastError();
    MOE_SEL_CASE(1)
    MOE_SEL_CASE(2)
    MOE_SEL_CASE(4)
    MOE_SEL_CASE(8)
    MOE_SEL_CASE(16)
#undef MOE_SEL_CASE
    default:
      break;
  }
  const size_t smem = select_smem(sh);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  select_kernel<<<(T + kSelWarps - 1) / kSelWarps, kSelWarps * 32, smem, s>>>(logits, bias, T,
                                                                           sh, ids, topw);
  return cudaGetLastError();
}

}  // namespace moe

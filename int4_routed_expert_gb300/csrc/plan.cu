// Routing plan: per-expert counts, offsets, the stable permutation of the
// T*k (token, slot) entries grouped by expert, its inverse, and the list of
// active experts.
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", N4
// "Scheduling and prediction" (route the whole batch first, build the
// unique expert union, run each expert once over every row that chose it)
// and "G3 implementation status" (stable row/rank batch union).  Order:
// experts ascending; inside an expert, entries i = t*k + j ascending.
//
// One CTA of 1024 threads.  Warp w owns the contiguous entry block
// [w*B, (w+1)*B), B = ceil(N/32), so entries of lower warps precede those of
// higher warps and each warp walks its block in order; that makes the
// permutation stable without any sort.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;

__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += o;
    }
    wsum[lane] = wi - w;  // exclusive
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  const int r = wsum[warp] + inc - v;
  total = wsum[32];
  __syncthreads();
  return r;
}

// smem: cnt[32][E] ints (per-warp, per-expert running bases), base[E].
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ ids, int N, int E, int32_t* __restrict__ counts,
            int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
            int32_t* __restrict__ inv, int32_t* __restrict__ active,
            int32_t* __restrict__ n_active) {
  extern __shared__ int psm[];
  int* cnt = psm;                 // [32][E]
  int* ebase = psm + 32 * E;      // [E] offsets
  __shared__ int wsum[33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * E; i += kPlanThreads) cnt[i] = 0;
  __syncthreads();
  const int B = (N + kPlanWarps - 1) / kPlanWarps;
  const int b0 = min(N, warp * B), b1 = min(N, b0 + B);
  const unsigned lt = (1u << lane) - 1u;
  // pass 1: per-warp counts
  for (int i0 = b0; i0 < b1; i0 += 32) {
    const int i = i0 + lane;
    const bool ok = i < b1;
    const int e = ok ? ids[i] : -1 - lane;  // distinct dummies never match a real id
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    if (ok && (grp & lt) == 0) cnt[warp * E + e] += __popc(grp);
  }
  __syncthreads();
  // pass 2 (E <= 1024 == threads, checked at create time): per-expert
  // exclusive bases over warps, then offsets and the active list
  {
    const int e = threadIdx.x;
    int c = 0;
    if (e < E) {
      for (int w = 0; w < kPlanWarps; ++w) {
        const int v = cnt[w * E + e];
        cnt[w * E + e] = c;
        c += v;
      }
    }
    int tot, n_act;
    const int off = block_exclusive_scan(c, wsum, tot);
    const int apos = block_exclusive_scan(c > 0 ? 1 : 0, wsum, n_act);
    if (e < E) {
      counts[e] = c;
      offsets[e] = off;
      ebase[e] = off;
      if (c > 0) active[apos] = e;
    }
    if (threadIdx.x == 0) {
      offsets[E] = N;
      *n_active = n_act;
    }
  }
  __syncthreads();
  // pass 3: positions in entry order
  for (int i0 = b0; i0 < b1; i0 += 32) {
    const int i = i0 + lane;
    const bool ok = i < b1;
    const int e = ok ? ids[i] : -1 - lane;
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    if (ok) {
      const int p = ebase[e] + cnt[warp * E + e] + __popc(grp & lt);
      perm[p] = i;
      inv[i] = p;
    }
    __syncwarp();
    if (ok && (grp & lt) == 0) cnt[warp * E + e] += __popc(grp);
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* ids, int T, int k, int E, int32_t* counts,
                        int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active,
                        int32_t* n_active, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(33) * E * sizeof(int);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  plan_kernel<<<1, kPlanThreads, smem, s>>>(ids, T * k, E, counts, offsets, perm, inv, active,
                                           n_active);
  return cudaGetLastError();
}

}  // namespace moe

// Router arithmetic shared by the general and the small-batch kernels.
//
// Every operation here is pinned to one IEEE rounding (explicit _rn
// intrinsics), so that the selected expert ids are bit-exact whatever the
// compiler's contraction settings.
//
// Definitions (page title, then section):
//  - "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy",
//    N1 "GLM-5.2 graph" MoE bullet and "G2 implementation status": sigmoid
//    scores, selection by score + correction bias, un-biased gate weights,
//    lower expert id wins an exact tie, routed scaling.
//  - "colibri-strix/README.md", "What's implemented": DeepSeek-V3-style
//    noaux_tc router with group-limited top-k and routed_scaling_factor.
// Readings where the pages are silent:
//  - logit summation order: 8 equal segments of H; in segment s, lane j
//    owns the 4-element chunks j, j+32, ... and accumulates them in
//    ascending order with fused multiply-adds from 0; the 32 lane partials
//    are summed pairwise by halving (16, 8, 4, 2, 1), then the 8 segment
//    sums the same way (4, 2, 1);
//  - sigmoid(z) = 1 / (1 + exp(-z)) with an own exp: Cody-Waite reduction
//    against a two-part ln 2, degree-7 Taylor polynomial, scaling by 2^n;
//    exp's argument is limited to [-32, 88] (outside, the sigmoid is exactly
//    1 or 0);
//  - group score = sum of the two largest keys of the group (the key itself
//    when a group holds one expert); groups ranked by score, lower index on
//    a tie; experts of dropped groups are excluded;
//  - w_j = (s_j / sum_j s_j) * routed_scaling_factor, sum in slot order.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.cuh"

namespace moe {

constexpr int kSeg = 8;               // segments of the logit reduction
constexpr int kNoIndex = 0x7fffffff;  // "no candidate" in an arg-max

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) {
  return __uint_as_float(b << 16);
}

// Four consecutive activations x[idx .. idx+3] as fp32 (idx % 4 == 0).
__device__ __forceinline__ float4 load_x4(const void* x, int dt, size_t idx) {
  if (dt == MOE_BF16) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + idx));
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
  }
  return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx));
}

// exp(t) for t in [-32, 88] (Cody & Waite reduction, Taylor degree 7).
// Constants: fp32 roundings of log2(e), of ln 2 cut to 16 significant bits,
// of the remainder ln 2 - ln2_hi, and of 1/i! for i = 3..7.
__device__ __forceinline__ float router_exp(float t) {
  const float kLog2e = __uint_as_float(0x3fb8aa3bu);
  const float kLn2Hi = __uint_as_float(0x3f317200u);
  const float kLn2Lo = __uint_as_float(0x35bfbe8eu);
  const float n = rintf(__fmul_rn(t, kLog2e));
  float r = __fmaf_rn(-n, kLn2Hi, t);
  r = __fmaf_rn(-n, kLn2Lo, r);
  float p = __uint_as_float(0x39500d01u);          // 1/7!
  p = __fmaf_rn(p, r, __uint_as_float(0x3ab60b61u));  // 1/6!
  p = __fmaf_rn(p, r, __uint_as_float(0x3c088889u));  // 1/5!
  p = __fmaf_rn(p, r, __uint_as_float(0x3d2aaaabu));  // 1/4!
  p = __fmaf_rn(p, r, __uint_as_float(0x3e2aaaabu));  // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int ni = static_cast<int>(n);
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

__device__ __forceinline__ float router_sigmoid(float z) {
  const float t = -z;
  if (t > 88.0f) return 0.0f;
  if (t < -32.0f) return 1.0f;
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, router_exp(t)));
}

// (va, ia) ranks before (vb, ib): larger value first, lower index on a tie.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Arg-max over the warp under ranks_before.  Lanes without a candidate pass
// idx = kNoIndex; every lane returns the winner (kNoIndex if none).
__device__ __forceinline__ void warp_argmax(float& v, int& idx) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, d);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, d);
    if (oi != kNoIndex && (idx == kNoIndex || ranks_before(ov, oi, v, idx))) {
      v = ov;
      idx = oi;
    }
  }
  v = __shfl_sync(0xffffffffu, v, 0);
  idx = __shfl_sync(0xffffffffu, idx, 0);
}

// Sum of the 32 lane partials of one segment, pairwise by halving; the
// result is valid in lane 0.
__device__ __forceinline__ float segment_tree(float p) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) p = __fadd_rn(p, __shfl_down_sync(0xffffffffu, p, d));
  return p;
}

// segment_tree of 32 values at once: v[i] holds lane L's partial of value i;
// on return lane L holds the full sum of value L.  Each step adds the halves
// of the lanes L and L ^ d that lane L keeps (the lower half when bit d of L
// is clear), so value i is summed over the same lane pairs in the same order
// (d = 16, 8, 4, 2, 1) as segment_tree, bit for bit, with 31 shuffles
// instead of 160.
__device__ __forceinline__ float segment_tree32(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int d = 16 >> s, n = 16 >> s;  // partner distance, values kept
    const bool hi = (lane & d) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = hi ? v[n + i] : v[i];
      const float send = hi ? v[i] : v[n + i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, d));
    }
  }
  return v[0];
}

// Sum of the 8 segment sums (d = 4, 2, 1).
__device__ __forceinline__ float segments_sum(const float* seg) {
  float a0 = __fadd_rn(seg[0], seg[4]), a1 = __fadd_rn(seg[1], seg[5]);
  float a2 = __fadd_rn(seg[2], seg[6]), a3 = __fadd_rn(seg[3], seg[7]);
  a0 = __fadd_rn(a0, a2);
  a1 = __fadd_rn(a1, a3);
  return __fadd_rn(a0, a1);
}

// General selection of one token by one warp.
//   s, key : [E] un-biased scores and keys (s + bias), any memory space
//   gsc    : [n_group] scratch, flags: [E] scratch bytes (shared memory)
// Writes ids[0..k) and w[0..k).
__device__ inline void warp_select(const float* s, const float* key, float* gsc,
                                   uint8_t* gkept, uint8_t* taken, const Shape& sh,
                                   int32_t* ids, float* w) {
  const int lane = threadIdx.x & 31;
  const int E = sh.E, G = E / sh.n_group;
  for (int g = lane; g < sh.n_group; g += 32) {
    float a = -INFINITY, b = -INFINITY;
    for (int e = g * G; e < (g + 1) * G; ++e) {
      const float v = key[e];
      if (v > a) {
        b = a;
        a = v;
      } else if (v > b) {
        b = v;
      }
    }
    gsc[g] = (G >= 2) ? __fadd_rn(a, b) : a;
    gkept[g] = 0;
  }
  for (int e = lane; e < E; e += 32) taken[e] = 0;
  __syncwarp();
  for (int r = 0; r < sh.topk_group; ++r) {
    float bv = 0.0f;
    int bi = kNoIndex;
    for (int g = lane; g < sh.n_group; g += 32) {
      if (gkept[g]) continue;
      if (bi == kNoIndex || ranks_before(gsc[g], g, bv, bi)) {
        bv = gsc[g];
        bi = g;
      }
    }
    warp_argmax(bv, bi);
    if (lane == 0) gkept[bi] = 1;
    __syncwarp();
  }
  float my_s = 0.0f, sum = 0.0f;
  int my_id = 0;
  for (int j = 0; j < sh.k; ++j) {
    float bv = 0.0f;
    int bi = kNoIndex;
    for (int e = lane; e < E; e += 32) {
      if (taken[e] || !gkept[e / G]) continue;
      const float v = key[e];
      if (bi == kNoIndex || ranks_before(v, e, bv, bi)) {
        bv = v;
        bi = e;
      }
    }
    warp_argmax(bv, bi);
    const float sj = s[bi];
    if (lane == 0) taken[bi] = 1;
    if (lane == j) {
      my_s = sj;
      my_id = bi;
    }
    sum = __fadd_rn(sum, sj);
    __syncwarp();
  }
  if (lane < sh.k) {
    ids[lane] = my_id;
    w[lane] = __fmul_rn(__fdiv_rn(my_s, sum), sh.rsf);
  }
}

// Shapes served by the register-resident selection: E = 32 * EPL experts,
// lane L holding experts L*EPL .. L*EPL+EPL-1, and a group spanning a
// power-of-two number of whole lanes.  Returns EPL, or 0.
__host__ __device__ inline int fast_select_epl(const Shape& sh) {
  if (sh.E % 32 != 0) return 0;
  const int epl = sh.E / 32;
  if (epl != 1 && epl != 2 && epl != 4 && epl != 8 && epl != 16 && epl != 32) return 0;
  const int G = sh.E / sh.n_group;
  if (G % epl != 0) return 0;
  const int lpg = G / epl;
  if (lpg < 1 || lpg > 32 || (lpg & (lpg - 1)) != 0) return 0;
  return epl;
}

// Order-preserving code of a float key: a > b  <=>  code(a) > code(b) for
// non-NaN keys other than -0 (a key s + b with s > 0 is never -0).  Code 0
// is left for "no candidate".
__device__ __forceinline__ uint32_t key_code(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Register-resident selection of one token by one warp (shapes accepted by
// fast_select_epl).  gkey / gs: the token's [E] keys and scores in global
// memory (read through L2).  Same result as warp_select: groups are ranked
// in one step (each group leader counts the groups that rank before it);
// each of the k rounds takes the maximum key code over the warp with one
// redux.sync, and the lowest lane holding it wins, which is the lower
// expert id on a tie because lane L holds experts L*EPL .. L*EPL+EPL-1.
// Lanes < k receive (id, w) of slot `lane` in out_id / out_w.
template <int EPL>
__device__ __forceinline__ void warp_select_core(const float (&kv)[EPL], const float (&sv)[EPL],
                                                 const Shape& sh, int& out_id, float& out_w);

template <int EPL>
__device__ __forceinline__ void warp_select_regs(const float* gkey, const float* gs,
                                                 const Shape& sh, int& out_id, float& out_w) {
  const int lane = threadIdx.x & 31;
  float kv[EPL], sv[EPL];
#pragma unroll
  for (int q = 0; q < EPL; q += (EPL >= 4 ? 4 : EPL)) {
    if constexpr (EPL >= 4) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(gkey + lane * EPL + q));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(gs + lane * EPL + q));
      kv[q] = a.x; kv[q + 1] = a.y; kv[q + 2] = a.z; kv[q + 3] = a.w;
      sv[q] = b.x; sv[q + 1] = b.y; sv[q + 2] = b.z; sv[q + 3] = b.w;
    } else {
#pragma unroll
      for (int u = 0; u < EPL; ++u) {
        kv[q + u] = __ldcg(gkey + lane * EPL + q + u);
        sv[q + u] = __ldcg(gs + lane * EPL + q + u);
      }
    }
  }
  warp_select_core<EPL>(kv, sv, sh, out_id, out_w);
}

// Same selection from a token's [E] router logits: lane L scores experts
// L*EPL .. L*EPL+EPL-1 itself (s = sigmoid(logit), key = s + bias).
template <int EPL>
__device__ __forceinline__ void warp_select_logits(const float* glog, const float* bias,
                                                   const Shape& sh, int& out_id, float& out_w) {
  const int lane = threadIdx.x & 31;
  float kv[EPL], sv[EPL];
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = lane * EPL + q;
    sv[q] = router_sigmoid(glog[e]);
    kv[q] = __fadd_rn(sv[q], bias[e]);
  }
  warp_select_core<EPL>(kv, sv, sh, out_id, out_w);
}

template <int EPL>
__device__ __forceinline__ void warp_select_core(const float (&kv)[EPL], const float (&sv)[EPL],
                                                 const Shape& sh, int& out_id, float& out_w) {
  const int lane = threadIdx.x & 31;
  const int G = sh.E / sh.n_group;
  const int lpg = G / EPL;
  // group score: top two keys of the lane, merged over the lpg lanes
  float a = -INFINITY, b = -INFINITY;
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const float v = kv[q];
    if (v > a) {
      b = a;
      a = v;
    } else if (v > b) {
      b = v;
    }
  }
  for (int d = 1; d < lpg; d <<= 1) {
    const float oa = __shfl_xor_sync(0xffffffffu, a, d);
    const float ob = __shfl_xor_sync(0xffffffffu, b, d);
    const float hi = fmaxf(a, oa), lo = fminf(a, oa);
    b = fmaxf(lo, fmaxf(b, ob));
    a = hi;
  }
  const float gscore = (G >= 2) ? __fadd_rn(a, b) : a;
  const int my_group = lane / lpg;
  // a group is kept when fewer than topk_group groups rank before it
  int before = 0;
  for (int g2 = 0; g2 < sh.n_group; ++g2) {
    const float o = __shfl_sync(0xffffffffu, gscore, g2 * lpg);
    before += (o > gscore || (o == gscore && g2 < my_group)) ? 1 : 0;
  }
  const bool in_kept = before < sh.topk_group;
  // candidate codes (0 = not a candidate)
  uint32_t code[EPL];
#pragma unroll
  for (int q = 0; q < EPL; ++q) code[q] = in_kept ? key_code(kv[q]) : 0u;
  float my_s = 0.0f, sum = 0.0f;
  int my_id = 0;
  for (int j = 0; j < sh.k; ++j) {
    uint32_t best = 0;
#pragma unroll
    for (int q = 0; q < EPL; ++q) best = max(best, code[q]);
    const uint32_t m = __reduce_max_sync(0xffffffffu, best);
    const unsigned holders = __ballot_sync(0xffffffffu, best == m && m != 0u);
    const int owner = __ffs(holders) - 1;
    // the owner's lowest slot holding the maximum
    int slot = EPL;
#pragma unroll
    for (int q = EPL - 1; q >= 0; --q) slot = (code[q] == m) ? q : slot;
    float sl = 0.0f;
#pragma unroll
    for (int q = 0; q < EPL; ++q) sl = (q == slot) ? sv[q] : sl;
    const float sj = __shfl_sync(0xffffffffu, sl, owner);
    const int oslot = __shfl_sync(0xffffffffu, slot, owner);
    if (lane == owner) {
#pragma unroll
      for (int q = 0; q < EPL; ++q) code[q] = (q == slot) ? 0u : code[q];
    }
    if (lane == j) {
      my_s = sj;
      my_id = owner * EPL + oslot;
    }
    sum = __fadd_rn(sum, sj);
  }
  out_id = my_id;
  out_w = __fmul_rn(__fdiv_rn(my_s, sum), sh.rsf);
}

}  // namespace moe

// dec_ab: router + gate/up projections of the small-batch path (see
// decode_common.cuh).  One cooperative CTA per SM, WARPS warps, each warp
// streaming its own rows through a STAGES-deep ring of TMA bulk copies.
//
// Per CTA:
//   1. RMSNorm scale (if gamma) and x_hat of the NT tokens, pre-scaled and
//      swizzled into shared memory (zeros for tokens >= T).
//   2. Every warp starts the copies of its shared-expert rows: they need no
//      routing.
//   3. Warps 0..7 compute the router logits of the CTA's experts
//      (blockIdx.x + l * gridDim.x) in the fixed segment order; warp 0 turns
//      them into scores and keys, publishes them and arrives on the grid
//      barrier.
//   4. Each warp consumes its shared rows; then it waits for the grid
//      barrier (all experts scored), derives the selection and the plan
//      itself, and streams its share of the selected experts' rows.
//   5. Per row pair (gate, up): h = SiLU(g) * u for the tokens of the row's
//      expert, stored at its plan position, pre-scaled for dec_c.
#pragma once

#include "decode_common.cuh"

namespace moe {
namespace dec {

__device__ __forceinline__ uint32_t word_of(const uint4& q, int wi) {
  return wi == 0 ? q.x : wi == 1 ? q.y : wi == 2 ? q.z : q.w;
}

template <int NT, int STAGES, int WARPS, int CPL>
__global__ void __launch_bounds__(WARPS * 32, 1) dec_ab_kernel(const __grid_constant__ DecArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const Shape& sh = a.sh;
  const Workspace& ws = a.ws;
  const int H = sh.H, I = sh.I, E = sh.E, T = a.T, k = sh.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int xpad = swz_pad(H);
  const int stage_bytes = H + H / 8;
  const int GK = H / 32;  // groups per row
  const int L = (E + gridDim.x - 1) / gridDim.x;

  float* xs = reinterpret_cast<float*>(smem);
  unsigned char* ring = smem + static_cast<size_t>(NT) * xpad * 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(WARPS) * STAGES * stage_bytes);
  float* lseg = reinterpret_cast<float*>(bars + WARPS * STAGES);
  double* dseg = reinterpret_cast<double*>(lseg + L * kRouterWarps * NT);
  float* rfs = reinterpret_cast<float*>(dseg + 8);

  // 1. RMSNorm scales and the staged activations
  if (a.gamma != nullptr) {
    for (int t = 0; t < T; ++t) {
      rms_partial(a, t, dseg);
      __syncthreads();
      if (threadIdx.x == 0) rfs[t] = rms_finish(a, dseg);
      __syncthreads();
    }
  }
  for (int t = 0; t < NT; ++t) {
    float* dst = xs + static_cast<size_t>(t) * xpad;
    if (t < T) {
      const float rf = a.gamma != nullptr ? rfs[t] : 1.0f;
      for (int k4 = threadIdx.x * 4; k4 < H; k4 += WARPS * 128)
        swz_store4(dst, k4, xhat4(a, static_cast<size_t>(t) * H + k4, k4, rf));
    } else {
      for (int i = threadIdx.x * 4; i < xpad; i += WARPS * 128)
        *reinterpret_cast<float4*>(dst + i) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const uint32_t bar0 = smem_u32(bars + warp * STAGES);
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
  }
  __syncthreads();

  // this warp's shared-expert rows
  int cb, ce, wb, we;
  split_range(sh.n_shared ? sh.Is : 0, blockIdx.x, gridDim.x, cb, ce);
  split_range(ce - cb, warp, WARPS, wb, we);
  const int sh0 = cb + wb, n_sh = we - wb;

  LanePlan lp;
  lp.n_act = 0;
  lp.e = lp.p0 = lp.n = 0;
  lp.tmask = 0;
  int q0 = 0, n_rt = 0;
  bool planned = false, failed = false;
  int issued = 0, consumed = 0;
  const uint32_t ring_w = smem_u32(ring + static_cast<size_t>(warp) * STAGES * stage_bytes);

  // source rows of item j (warp-uniform)
  auto issue = [&](int j) {
    const uint8_t *gq, *uq;
    const uint16_t *gs, *us;
    if (j < n_sh) {
      const size_t r = sh0 + j;
      gq = a.w.sh_gate_q + r * (H / 2);
      uq = a.w.sh_up_q + r * (H / 2);
      gs = a.w.sh_gate_s + r * (H / 32);
      us = a.w.sh_up_s + r * (H / 32);
    } else {
      const int q = q0 + (j - n_sh);
      const int slot = q / I, r = q - slot * I;
      const int e = __shfl_sync(0xffffffffu, lp.e, slot);
      const size_t row = static_cast<size_t>(e) * I + r;
      gq = a.w.gate_q + row * (H / 2);
      uq = a.w.up_q + row * (H / 2);
      gs = a.w.gate_s + row * (H / 32);
      us = a.w.up_s + row * (H / 32);
    }
    if (lane == 0) {
      const int st = j % STAGES;
      const uint32_t dst = ring_w + st * stage_bytes;
      const uint32_t bar = bar0 + 8 * st;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, stage_bytes);
      bulk_g2s(dst, gq, H / 2, bar);
      bulk_g2s(dst + H / 2, uq, H / 2, bar);
      bulk_g2s(dst + H, gs, H / 16, bar);
      bulk_g2s(dst + H + H / 16, us, H / 16, bar);
    }
  };
  auto refill = [&]() {
    const int limit = planned ? n_sh + n_rt : n_sh;
    while (issued < limit && issued < consumed + STAGES) issue(issued++);
  };

  // 2. shared-expert copies go out before the router work
  refill();

  // 3. router logits of this CTA's experts
  router_cta<NT, CPL>(a, lseg, rfs);
  if (warp == 0) {
    __threadfence();
    __syncwarp();
    if (lane == 0) gbar_arrive(ws.gbar);
  }
  pdl_launch_dependents();

  const int epl = fast_select_epl(sh);
  const uint32_t magic = kMagic;
  const float4* xs4 = reinterpret_cast<const float4*>(xs);

  // 4./5. consume
  for (;;) {
    if (!planned && consumed == n_sh) {
      if (!gbar_wait(ws.gbar, a.gtarget, ws.dev_err)) {
        failed = true;
        break;
      }
      warp_route_plan(a, epl, blockIdx.x == 0 && warp == 0, lp);
      int rb, re, b2, e2;
      split_range(lp.n_act * I, blockIdx.x, gridDim.x, rb, re);
      split_range(re - rb, warp, WARPS, b2, e2);
      q0 = rb + b2;
      n_rt = e2 - b2;
      planned = true;
      refill();
    }
    if (planned && consumed >= n_sh + n_rt) break;
    const int st = consumed % STAGES;
    if (!mbar_wait(bar0 + 8 * st, (consumed / STAGES) & 1, ws.dev_err)) {
      failed = true;
      break;
    }
    const unsigned char* sb = ring + (static_cast<size_t>(warp) * STAGES + st) * stage_bytes;
    const uint4* gq4 = reinterpret_cast<const uint4*>(sb);
    const uint4* uq4 = reinterpret_cast<const uint4*>(sb + H / 2);
    const uint16_t* gsc = reinterpret_cast<const uint16_t*>(sb + H);
    const uint16_t* usc = reinterpret_cast<const uint16_t*>(sb + H + H / 16);
    float2 ga[NT], ua[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) ga[t] = ua[t] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int g = c * 32 + lane;
      if (CPL == 1 && g >= GK) break;
      const uint4 qa = gq4[g], qb = uq4[g];
      const float sa = half_bits_to_f32(gsc[g]), sbv = half_bits_to_f32(usc[g]);
      float2 da[NT], db[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) da[t] = db[t] = make_float2(0.f, 0.f);
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        const DqWord dg = dq_word(word_of(qa, wi), magic);
        const DqWord du = dq_word(word_of(qb, wi), magic);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float4* xt = xs4 + static_cast<size_t>(t) * (xpad / 4) + (c * 8 + 2 * wi) * 32 + lane;
          const float4 x0 = xt[0], x1 = xt[32];
          da[t] = dq_fma(dg, x0, x1, da[t]);
          db[t] = dq_fma(du, x0, x1, db[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        ga[t] = __ffma2_rn(da[t], make_float2(sa, sa), ga[t]);
        ua[t] = __ffma2_rn(db[t], make_float2(sbv, sbv), ua[t]);
      }
    }
    // the item's destination rows (warp-uniform)
    const int j = consumed;
    int row, slot = -1;
    if (j < n_sh) {
      row = sh0 + j;
    } else {
      const int q = q0 + (j - n_sh);
      slot = q / I;
      row = q - slot * I;
    }
    const int sp0 = __shfl_sync(0xffffffffu, lp.p0, slot < 0 ? 0 : slot);
    const unsigned stm = __shfl_sync(0xffffffffu, lp.tmask, slot < 0 ? 0 : slot);
    float my_h = 0.0f;
    int my_row = -1;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float gsum = warp_sum(ga[t].x + ga[t].y);
      const float usum = warp_sum(ua[t].x + ua[t].y);
      if (lane == t) {
        const float silu = gsum / (1.0f + expf(-gsum));
        my_h = silu * usum;
        if (t < T) {
          if (slot < 0)
            my_row = T * k + t;
          else if ((stm >> t) & 1u)
            my_row = sp0 + __popc(stm & ((1u << t) - 1u));
        }
      }
    }
    if (my_row >= 0)
      ws.hbuf[static_cast<size_t>(my_row) * ws.hstride + swz_index(row >> 5, row & 31)] =
          my_h * swz_prescale(row & 31);
    ++consumed;
    __syncwarp();
    refill();
  }
  if (failed) {
    // let this warp's copies in flight land before the CTA exits
    for (int j = consumed; j < issued; ++j)
      mbar_wait(bar0 + 8 * (j % STAGES), (j / STAGES) & 1, ws.dev_err);
  }
}

template <int NT, int STAGES, int WARPS>
cudaError_t launch_ab_cpl(const DecArgs& a, int cpl, size_t smem, int n_sm, cudaStream_t s) {
  switch (cpl) {
#define MOE_AB_CASE(C)                                                            \
  case C: {                                                                       \
    auto kern = dec_ab_kernel<NT, STAGES, WARPS, C>;                              \
    static bool smem_set = false;                                                 \
    static size_t smem_max = 0;                                                   \
    if (!smem_set || smem > smem_max) {                                           \
      const cudaError_t e = set_smem_once(kern, smem);                            \
      if (e != cudaSuccess) return e;                                             \
      smem_set = true;                                                            \
      smem_max = smem;                                                            \
    }                                                                             \
    return launch_k(kern, n_sm, WARPS * 32, smem, s, a, /*pdl=*/false, /*coop=*/true); \
  }
    MOE_AB_CASE(1)
    MOE_AB_CASE(2)
    MOE_AB_CASE(4)
    MOE_AB_CASE(6)
    MOE_AB_CASE(8)
#undef MOE_AB_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dec
}  // namespace moe

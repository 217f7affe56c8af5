// dec_c: down projections + weighted combine of the small-batch path (see
// decode_common.cuh).  One CTA per SM, launched with programmatic
// dependent launch behind dec_ab and waiting on it with
// griddepcontrol.wait before touching its outputs.
//
// Slots: the selected experts of the call (ascending, from the plan dec_ab
// published), then the shared expert.  CTA b owns a balanced range of
// 4-row blocks of y; its (row block, slot) items, slots fastest, are split
// evenly over the warps, each warp streaming the 4 down rows of an item
// (one TMA bulk copy for the packed rows, one for their scales) through its
// ring.  A warp accumulates the gate-weighted dot products of consecutive
// items of one row block in registers; row blocks split between warps are
// finished from shared memory in warp order, so y is deterministic.
//
//   y_t[r] = (accumulate ? y_t[r] : 0) + sum over slots of w_slot,t * o_slot,t[r]
// with w = the token's gate weight for a selected expert (0 if the token did
// not select it) and 1 for the shared expert.
#pragma once

#include "decode_common.cuh"

namespace moe {
namespace dec {

struct CSlot {
  int e;               // expert, -1 for the shared expert
  int p0, n;           // plan positions of the slot's entries
  int hrow[kMaxNT];    // row of the activation buffer per token
  float wt[kMaxNT];    // gate weight per token (0: token did not pick it)
};

__device__ __forceinline__ uint32_t cword(const uint4& q, int wi) {
  return wi == 0 ? q.x : wi == 1 ? q.y : wi == 2 ? q.z : q.w;
}

template <int NT, int STAGES, int WARPS, bool H_SMEM, int CPL>
__global__ void __launch_bounds__(WARPS * 32, 1) dec_c_kernel(const __grid_constant__ DecArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ CSlot slots[kMaxEntries + 1];
  __shared__ int s_nslots, s_nact;
  const Shape& sh = a.sh;
  const Workspace& ws = a.ws;
  const int H = sh.H, I = sh.I, E = sh.E, T = a.T, k = sh.k, N = T * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stage_bytes = kRowsC * (I / 2 + I / 16);
  const int GK = I / 32;
  const int hstride = ws.hstride;

  unsigned char* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(WARPS) * STAGES * stage_bytes);
  uint64_t* hbar = bars + WARPS * STAGES;
  float* part = reinterpret_cast<float*>(hbar + 2);          // [WARPS][2][kRowsC][NT]
  float* hs = part + WARPS * 2 * kRowsC * NT;                // (N + T) rows x hstride

  // everything below reads dec_ab's outputs
  pdl_wait();

  if (warp == 0) {
    int n_act = __ldcg(ws.n_active);
    n_act = n_act < 0 ? 0 : (n_act > N ? N : n_act);
    if (lane < n_act) {
      CSlot& s = slots[lane];
      int e = __ldcg(ws.dslot + lane), p0 = __ldcg(ws.dslot + 32 + lane),
          n = __ldcg(ws.dslot + 64 + lane);
      e = e < 0 ? 0 : (e >= E ? E - 1 : e);
      p0 = p0 < 0 ? 0 : (p0 > N ? N : p0);
      n = n < 0 ? 0 : (p0 + n > N ? N - p0 : n);
      s.e = e;
      s.p0 = p0;
      s.n = n;
#pragma unroll
      for (int t = 0; t < kMaxNT; ++t) {
        s.hrow[t] = 0;
        s.wt[t] = 0.0f;
      }
      for (int m = 0; m < n; ++m) {
        int i = __ldcg(ws.perm + p0 + m);
        i = i < 0 ? 0 : (i >= N ? N - 1 : i);
        const int t = i / k;
        if (t < NT) {
          s.hrow[t] = p0 + m;
          s.wt[t] = __ldcg(ws.topw + i);
        }
      }
    }
    if (lane == 0) {
      if (sh.n_shared) {
        CSlot& s = slots[n_act];
        s.e = -1;
        s.p0 = N;
        s.n = T;
#pragma unroll
        for (int t = 0; t < kMaxNT; ++t) {
          s.hrow[t] = t < T ? N + t : 0;
          s.wt[t] = t < T ? 1.0f : 0.0f;
        }
      }
      s_nact = n_act;
      s_nslots = n_act + sh.n_shared;
    }
  }
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(smem_u32(bars + warp * STAGES + s), 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(hbar), 1);
    fence_barrier_init();
  }
  __syncthreads();

  // the plan's counts and offsets for callers that asked for the plan
  if (blockIdx.x == 0) {
    const int n_act = s_nact;
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      int c = 0, off = 0;
      for (int q = 0; q < n_act; ++q) {
        if (slots[q].e == e) c = slots[q].n;
        if (slots[q].e < e) off += slots[q].n;
      }
      if (e < E) ws.counts[e] = c;
      ws.offsets[e] = e < E ? off : N;
    }
  }

  bool failed = false;
  if (H_SMEM) {
    const uint32_t hb = smem_u32(hbar);
    if (threadIdx.x == 0) {
      const uint32_t bytes = static_cast<uint32_t>(static_cast<size_t>(N + T) * hstride * 4);
      mbar_arrive_expect_tx(hb, bytes);
      bulk_g2s(smem_u32(hs), ws.hbuf, bytes, hb);
    }
  }

  const int S = s_nslots;
  int rb0, rb1;
  split_range(H / kRowsC, blockIdx.x, gridDim.x, rb0, rb1);
  const int n_items = (rb1 - rb0) * S;
  int i0, i1;
  split_range(n_items, warp, WARPS, i0, i1);
  const int n_my = i1 - i0;
  const uint32_t bar0 = smem_u32(bars + warp * STAGES);
  const uint32_t ring_w = smem_u32(ring + static_cast<size_t>(warp) * STAGES * stage_bytes);

  auto issue = [&](int j) {
    if (lane == 0) {
      const int item = i0 + j;
      const int lr = item / S, sl = item - lr * S;
      const int r0 = (rb0 + lr) * kRowsC;
      const int e = slots[sl].e;
      const uint8_t* q;
      const uint16_t* sc;
      if (e >= 0) {
        const size_t row = static_cast<size_t>(e) * H + r0;
        q = a.w.down_q + row * (I / 2);
        sc = a.w.down_s + row * (I / 32);
      } else {
        q = a.w.sh_down_q + static_cast<size_t>(r0) * (I / 2);
        sc = a.w.sh_down_s + static_cast<size_t>(r0) * (I / 32);
      }
      const int st = j % STAGES;
      const uint32_t dst = ring_w + st * stage_bytes;
      const uint32_t bar = bar0 + 8 * st;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, stage_bytes);
      bulk_g2s(dst, q, kRowsC * (I / 2), bar);
      bulk_g2s(dst + kRowsC * (I / 2), sc, kRowsC * (I / 16), bar);
    }
  };
  int issued = 0;
  while (issued < n_my && issued < STAGES) issue(issued++);

  if (H_SMEM) {
    if (!mbar_wait(smem_u32(hbar), 0, ws.dev_err)) failed = true;
  }
  const float* hsrc = H_SMEM ? hs : ws.hbuf;
  const uint32_t magic = kMagic;

  float tot[kRowsC][NT];
#pragma unroll
  for (int r = 0; r < kRowsC; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) tot[r][t] = 0.0f;

  const int lr_first = n_my > 0 ? i0 / S : 0;
  auto flush = [&](int lr) {
    const bool owned = lr * S >= i0 && (lr + 1) * S <= i1;
    float mine = 0.0f;
#pragma unroll
    for (int r = 0; r < kRowsC; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = warp_sum(tot[r][t]);
        if (lane == r * NT + t) mine = v;
        tot[r][t] = 0.0f;
      }
    if (lane < kRowsC * NT) {
      const int r = lane / NT, t = lane % NT;
      if (owned) {
        if (t < T) {
          float* yp = a.y + static_cast<size_t>(t) * H + (rb0 + lr) * kRowsC + r;
          *yp = a.accumulate ? *yp + mine : mine;
        }
      } else {
        part[((warp * 2 + (lr == lr_first ? 0 : 1)) * kRowsC + r) * NT + t] = mine;
      }
    }
  };

  int consumed = 0;
  int cur_lr = lr_first;
  while (!failed && consumed < n_my) {
    const int st = consumed % STAGES;
    if (!mbar_wait(bar0 + 8 * st, (consumed / STAGES) & 1, ws.dev_err)) {
      failed = true;
      break;
    }
    const int item = i0 + consumed;
    const int lr = item / S, sl = item - lr * S;
    if (lr != cur_lr) {
      flush(cur_lr);
      cur_lr = lr;
    }
    const unsigned char* sb = ring + (static_cast<size_t>(warp) * STAGES + st) * stage_bytes;
    const CSlot& slot = slots[sl];
    const float4* hp[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
      hp[t] = reinterpret_cast<const float4*>(hsrc + static_cast<size_t>(slot.hrow[t]) * hstride);
    float2 acc[kRowsC][NT];
#pragma unroll
    for (int r = 0; r < kRowsC; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[r][t] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int g = c * 32 + lane;
      if (CPL == 1 && g >= GK) break;
      uint4 q[kRowsC];
      float s[kRowsC];
#pragma unroll
      for (int r = 0; r < kRowsC; ++r) {
        q[r] = reinterpret_cast<const uint4*>(sb + r * (I / 2))[g];
        s[r] = half_bits_to_f32(
            reinterpret_cast<const uint16_t*>(sb + kRowsC * (I / 2) + r * (I / 16))[g]);
      }
      float2 d[kRowsC][NT];
#pragma unroll
      for (int r = 0; r < kRowsC; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) d[r][t] = make_float2(0.f, 0.f);
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        float4 h0[NT], h1[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float4* p = hp[t] + (c * 8 + 2 * wi) * 32 + lane;
          if (H_SMEM) {
            h0[t] = p[0];
            h1[t] = p[32];
          } else {
            h0[t] = __ldcg(p);
            h1[t] = __ldcg(p + 32);
          }
        }
#pragma unroll
        for (int r = 0; r < kRowsC; ++r) {
          const DqWord dw = dq_word(cword(q[r], wi), magic);
#pragma unroll
          for (int t = 0; t < NT; ++t) d[r][t] = dq_fma(dw, h0[t], h1[t], d[r][t]);
        }
      }
#pragma unroll
      for (int r = 0; r < kRowsC; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
          acc[r][t] = __ffma2_rn(d[r][t], make_float2(s[r], s[r]), acc[r][t]);
    }
#pragma unroll
    for (int r = 0; r < kRowsC; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) tot[r][t] = fmaf(slot.wt[t], acc[r][t].x + acc[r][t].y, tot[r][t]);
    ++consumed;
    __syncwarp();
    while (issued < n_my && issued < consumed + STAGES) issue(issued++);
  }
  if (!failed && n_my > 0) flush(cur_lr);
  if (failed) {
    for (int j = consumed; j < issued; ++j)
      mbar_wait(bar0 + 8 * (j % STAGES), (j / STAGES) & 1, ws.dev_err);
    if (H_SMEM) mbar_wait(smem_u32(hbar), 0, ws.dev_err);
  }
  __syncthreads();

  // row blocks shared by several warps: sum their parts in warp order
  const int nlr = rb1 - rb0;
  for (int idx = threadIdx.x; idx < nlr * kRowsC * NT; idx += blockDim.x) {
    const int lr = idx / (kRowsC * NT), r = (idx / NT) % kRowsC, t = idx % NT;
    if (t >= T) continue;
    bool direct = false;
    float v = 0.0f;
    for (int w = 0; w < WARPS; ++w) {
      int w0, w1;
      split_range(n_items, w, WARPS, w0, w1);
      if (w0 == w1) continue;
      const int f = w0 / S, l = (w1 - 1) / S;
      if (lr < f || lr > l) continue;
      if (lr * S >= w0 && (lr + 1) * S <= w1) {
        direct = true;
        break;
      }
      v += part[((w * 2 + (lr == f ? 0 : 1)) * kRowsC + r) * NT + t];
    }
    if (!direct) {
      float* yp = a.y + static_cast<size_t>(t) * H + (rb0 + lr) * kRowsC + r;
      *yp = a.accumulate ? *yp + v : v;
    }
  }
}

template <int NT, bool H_SMEM>
cudaError_t launch_c_cpl(const DecArgs& a, int cpl, size_t smem, int n_sm, bool pdl,
                         cudaStream_t s) {
  switch (cpl) {
#define MOE_C_CASE(C)                                                            \
  case C: {                                                              \
    auto kern = dec_c_kernel<NT, kStagesC, kWarpsC, H_SMEM, C>;          \
    static size_t smem_max = 0;                                          \
    if (smem > smem_max) {                                               \
      const cudaError_t e = set_smem_once(kern, smem);                   \
      if (e != cudaSuccess) return e;                                    \
      smem_max = smem;                                                   \
    }                                                                    \
    return launch_k(kern, n_sm, kWarpsC * 32, smem, s, a, pdl, false);   \
  }
    MOE_C_CASE(1)
    MOE_C_CASE(2)
    MOE_C_CASE(4)
    MOE_C_CASE(6)
    MOE_C_CASE(8)
#undef MOE_C_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace dec
}  // namespace moe

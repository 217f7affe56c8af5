// dec_fused: the whole layer for one token in one cooperative kernel (one
// CTA per SM, WARPS warps).  Each warp streams a sequence of items through
// its own ring of TMA bulk copies:
//
//   [shared gate/up rows] [shared down row blocks] [routed gate/up rows]
//   [routed down row blocks]
//
// A copy is issued as soon as its source is known (shared items at once,
// routed items once the plan is known), up to STAGES items ahead; the
// compute of an item waits only for what it reads:
//   shared gate/up  x_hat (staged in shared memory by the prologue)
//   shared down     barrier 1: every CTA has scored its router experts and
//                   written its shared-expert h rows
//   routed gate/up  the plan (after barrier 1, warp 0 of CTA 0 selects the
//                   experts and publishes them; warp 0 of every CTA reads
//                   them, derives the plan and hands it to the other warps
//                   in shared memory; they stream shared down rows meanwhile)
//   routed down     barrier 2: every routed h row is written
// Down-projection results of the CTA's rows go to a (row, slot) table in
// shared memory; at the end the CTA sums each row over the slots in a fixed
// order (selected experts ascending, then the shared expert) into y, so y
// is deterministic.  Weight rows are never re-read and x, h and partial
// sums stay on chip or in L2.
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", N1
// (MoE bullet), N2 and "G2 - native GLM-5.2 correctness spine" (int4 gate/
// up/down, dequant -> f32 MAC), N4 (route first, stream each selected
// expert once); "colibri-strix/README.md", "What's implemented".
#pragma once

#include "decode_common.cuh"
#include "smem_opt_in.cuh"

namespace moe {
namespace dec {

constexpr int kSlotsP = kMaxEntries + 1;  // columns of the partial table
constexpr int kSharedCol = kMaxEntries;   // column of the shared expert
constexpr int kWarpsF = 12, kStagesF = 2;

__host__ __device__ inline int fused_stage_bytes(const Shape& sh) {
  const int gu = sh.H + sh.H / 8;                   // gate row + up row + their scales
  const int dn = kRowsC * (sh.I / 2 + sh.I / 16);   // 4 down rows + their scales
  return ((gu > dn ? gu : dn) + 15) & ~15;
}

__host__ __device__ inline int fused_rows_max(const Shape& sh, int grid) {
  return ((sh.H / kRowsC + grid - 1) / grid) * kRowsC;
}

__host__ __device__ inline size_t fused_smem_bytes(const Shape& sh, int grid) {
  const int L = (sh.E + grid - 1) / grid;
  size_t b = static_cast<size_t>(swz_pad(sh.H)) * 4;                          // x_hat
  b += static_cast<size_t>(kWarpsF) * kStagesF * fused_stage_bytes(sh);     // rings
  b += static_cast<size_t>(kWarpsF) * kStagesF * 8 + 4 * 8;                 // mbarriers
  b += static_cast<size_t>(fused_rows_max(sh, grid)) * kSlotsP * 4;         // partials
  b += static_cast<size_t>(L) * kRouterWarps * 4;                           // logit segments
  b += 8 * 8 + 16;                                                          // fp64 partials, rf
  return b;
}

__device__ __forceinline__ uint32_t fword(const uint4& q, int wi) {
  return wi == 0 ? q.x : wi == 1 ? q.y : wi == 2 ? q.z : q.w;
}

// Sums of v0..v3 over the warp: lane L receives the sum of v_r with
// r = 2 * bit4(L) + bit3(L) (lanes 0, 8, 16, 24 hold rows 0..3).
__device__ __forceinline__ float warp_sum4(float v0, float v1, float v2, float v3) {
  const int lane = threadIdx.x & 31;
  const bool hi = lane & 16;
  float a0 = hi ? v2 : v0, a1 = hi ? v3 : v1;
  const float b0 = hi ? v0 : v2, b1 = hi ? v1 : v3;
  a0 += __shfl_xor_sync(0xffffffffu, b0, 16);
  a1 += __shfl_xor_sync(0xffffffffu, b1, 16);
  const bool h8 = lane & 8;
  float c = h8 ? a1 : a0;
  const float d = h8 ? a0 : a1;
  c += __shfl_xor_sync(0xffffffffu, d, 8);
  c += __shfl_xor_sync(0xffffffffu, c, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

// Sums of g and u over the warp: lanes 0..15 receive g, lanes 16..31 u.
__device__ __forceinline__ float warp_sum2(float g, float u) {
  const bool hi = threadIdx.x & 16;
  float a = hi ? u : g;
  const float b = hi ? g : u;
  a += __shfl_xor_sync(0xffffffffu, b, 16);
  a += __shfl_xor_sync(0xffffffffu, a, 8);
  a += __shfl_xor_sync(0xffffffffu, a, 4);
  a += __shfl_xor_sync(0xffffffffu, a, 2);
  a += __shfl_xor_sync(0xffffffffu, a, 1);
  return a;
}

template <int CPLH, int CPLI, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32, 1)
dec_fused_kernel(const __grid_constant__ DecArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_cnt2, s_nact;
  __shared__ int s_pe[kMaxEntries], s_pp0[kMaxEntries];
  __shared__ float s_pw[kMaxEntries];
  const Shape& sh = a.sh;
  const Workspace& ws = a.ws;
  const int H = sh.H, I = sh.I, E = sh.E, k = sh.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int xpad = swz_pad(H);
  const int SB = fused_stage_bytes(sh);
  const int GKH = H / 32, GKI = I / 32;
  const int L = (E + G - 1) / G;
  const int rows_max = fused_rows_max(sh, G);
  const size_t hstride = ws.hstride;
  int rb0, rb1;
  split_range(H / kRowsC, b, G, rb0, rb1);
  const int nrb = rb1 - rb0;

  float* xs = reinterpret_cast<float*>(smem);
  unsigned char* ring = smem + static_cast<size_t>(xpad) * 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(WARPS) * STAGES * SB);
  // [0] barrier 1 passed, [1] plan ready, [2] barrier 2 passed, [3] router rows landed
  uint64_t* sync_bars = bars + WARPS * STAGES;
  float* part = reinterpret_cast<float*>(sync_bars + 4);
  float* lseg = part + static_cast<size_t>(rows_max) * kSlotsP;
  double* dseg = reinterpret_cast<double*>(lseg + L * kRouterWarps);
  float* rfs = reinterpret_cast<float*>(dseg + 8);
  const uint32_t g1bar = smem_u32(sync_bars), planbar = smem_u32(sync_bars + 1),
                 g2bar = smem_u32(sync_bars + 2), rbar = smem_u32(sync_bars + 3);

  // ---- prologue: router rows by TMA, RMSNorm scale, x_hat, barriers --------
  // Before the weight stream starts, the ring area holds x_hat in natural
  // order and this CTA's router rows (when they fit), so that the router
  // reads shared memory only.
  bool failed = false;
  float* xn = reinterpret_cast<float*>(ring);
  float* wr = xn + H;
  const bool router_in_smem =
      static_cast<size_t>(L + 1) * H * 4 <= static_cast<size_t>(WARPS) * STAGES * SB;
  const uint32_t bar0 = smem_u32(bars + warp * STAGES);
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
  }
  if (threadIdx.x == 0) {
    mbar_init(g1bar, 1);
    mbar_init(planbar, 1);
    mbar_init(g2bar, 1);
    mbar_init(rbar, 1);
    fence_barrier_init();
    s_cnt2 = 0;
    s_nact = 0;
    if (router_in_smem) {
      int nl = 0;
      for (int l = 0; l < L; ++l) nl += (b + l * G < E) ? 1 : 0;
      mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(nl) * H * 4);
      for (int l = 0; l < nl; ++l)
        bulk_g2s(smem_u32(wr + static_cast<size_t>(l) * H),
                 a.w.router_w + static_cast<size_t>(b + l * G) * H, H * 4, rbar);
    }
  }
  float rf = 1.0f;
  if (a.gamma != nullptr) {
    rms_partial(a, 0, dseg);
    __syncthreads();
    if (threadIdx.x == 0) rfs[0] = rms_finish(a, dseg);
    __syncthreads();
    rf = rfs[0];
  }
  for (int k4 = threadIdx.x * 4; k4 < H; k4 += WARPS * 128) {
    const float4 v = xhat4(a, k4, k4, rf);
    swz_store4(xs, k4, v);
    if (router_in_smem) *reinterpret_cast<float4*>(xn + k4) = v;
  }
  __syncthreads();

  // ---- this warp's items -------------------------------------------------
  // sequence: shared gate/up rows | routed gate/up rows | down row blocks of
  // the routed slots and the shared expert (routed parts once the plan is
  // known).  Warp 0 finishes the router, waits for barrier 1 and derives the
  // plan; the shared gate/up rows go to the warps whose ring stages lie past
  // the router's staging area, so their copies can start at once.
  int wfree = router_in_smem
                  ? static_cast<int>((static_cast<size_t>(L + 1) * H * 4 + STAGES * SB - 1) /
                                     (static_cast<size_t>(STAGES) * SB))
                  : 1;
  if (wfree < 1) wfree = 1;
  if (wfree > WARPS - 1) wfree = WARPS - 1;
  int c0, c1, w0 = 0, w1 = 0;
  split_range(sh.n_shared ? sh.Is : 0, b, G, c0, c1);
  if (warp >= wfree) split_range(c1 - c0, warp - wfree, WARPS - wfree, w0, w1);
  const int sgu0 = c0 + w0, n_sgu = w1 - w0;
  int n_rgu = 0, n_dn = 0;
  int rgu_s = 0, rgu_r = 0;  // first routed gate/up item: slot, row
  int dn_s = 0, dn_l = 0;    // first down item: slot index, local row block
  int n_slots = 0;           // routed slots + shared expert
  bool planned = false;
  int issued = 0, consumed = 0;
  const uint32_t ring_w = smem_u32(ring + static_cast<size_t>(warp) * STAGES * SB);
  // scales: one per 32 values, or one per row (group size 0)
  const bool row_scaled = sh.gsz == 0;
  const size_t ssh = row_scaled ? 1 : H / 32, ssi = row_scaled ? 1 : I / 32;
  const uint32_t magic = kMagic;

  auto rgu_at = [&](int o, int& slot, int& row) {
    slot = rgu_s;
    row = rgu_r + o;
    while (row >= I) {
      row -= I;
      ++slot;
    }
  };
  auto dn_at = [&](int o, int& si, int& lr) {
    si = dn_s;
    lr = dn_l + o;
    while (lr >= nrb) {
      lr -= nrb;
      ++si;
    }
  };
  const int n_act_k = k;  // one token: k distinct experts
  auto issue = [&](int j) {
    const uint8_t *q0p, *q1p = nullptr;
    const uint16_t *s0p, *s1p = nullptr;
    bool gu;
    if (j < n_sgu) {
      const size_t r = sgu0 + j;
      gu = true;
      q0p = a.w.sh_gate_q + r * (H / 2);
      q1p = a.w.sh_up_q + r * (H / 2);
      s0p = a.w.sh_gate_s + r * ssh;
      s1p = a.w.sh_up_s + r * ssh;
    } else if (j < n_sgu + n_rgu) {
      int slot, r;
      rgu_at(j - n_sgu, slot, r);
      const size_t row = static_cast<size_t>(s_pe[slot]) * I + r;
      gu = true;
      q0p = a.w.gate_q + row * (H / 2);
      q1p = a.w.up_q + row * (H / 2);
      s0p = a.w.gate_s + row * ssh;
      s1p = a.w.up_s + row * ssh;
    } else {
      int si, lr;
      dn_at(j - n_sgu - n_rgu, si, lr);
      const size_t r0 = static_cast<size_t>(rb0 + lr) * kRowsC;
      gu = false;
      if (si < n_act_k) {
        const size_t row = static_cast<size_t>(s_pe[si]) * H + r0;
        q0p = a.w.down_q + row * (I / 2);
        s0p = a.w.down_s + row * ssi;
      } else {
        q0p = a.w.sh_down_q + r0 * (I / 2);
        s0p = a.w.sh_down_s + r0 * ssi;
      }
    }
    if (lane == 0) {
      const int st = j % STAGES;
      const uint32_t dst = ring_w + st * SB;
      const uint32_t bar = bar0 + 8 * st;
      fence_proxy_async_smem();
      if (row_scaled) {
        // one scale a row: too small for a bulk copy, so the 4-byte word
        // holding it (gate/up rows) or the 4 rows' 8 bytes (down) come by
        // cp.async, whose arrival the stage's phase also waits for (the
        // arrive comes first, so the phase cannot complete without it)
        if (gu) {
          cp_async_ca4(dst + H, align_down4(s0p));
          cp_async_ca4(dst + H + 4, align_down4(s1p));
        } else {
          cp_async_ca8(dst + kRowsC * (I / 2), s0p);
        }
        cp_async_mbar_arrive(bar);
        mbar_arrive_expect_tx(bar, gu ? H : kRowsC * (I / 2));
        if (gu) {
          bulk_g2s(dst, q0p, H / 2, bar);
          bulk_g2s(dst + H / 2, q1p, H / 2, bar);
        } else {
          bulk_g2s(dst, q0p, kRowsC * (I / 2), bar);
        }
      } else if (gu) {
        mbar_arrive_expect_tx(bar, H + H / 8);
        bulk_g2s(dst, q0p, H / 2, bar);
        bulk_g2s(dst + H / 2, q1p, H / 2, bar);
        bulk_g2s(dst + H, s0p, H / 16, bar);
        bulk_g2s(dst + H + H / 16, s1p, H / 16, bar);
      } else {
        mbar_arrive_expect_tx(bar, kRowsC * (I / 2 + I / 16));
        bulk_g2s(dst, q0p, kRowsC * (I / 2), bar);
        bulk_g2s(dst + kRowsC * (I / 2), s0p, kRowsC * (I / 16), bar);
      }
    }
  };
  auto known = [&]() { return planned ? n_sgu + n_rgu + n_dn : n_sgu; };
  auto refill = [&]() {
    const int lim = known();
    while (issued < lim && issued < consumed + STAGES) issue(issued++);
  };
  auto take_plan = [&]() {
    int r0, r1, x0, x1;
    split_range(n_act_k * I, b, G, r0, r1);
    split_range(r1 - r0, warp, WARPS, x0, x1);
    n_rgu = x1 - x0;
    rgu_s = (r0 + x0) / I;
    rgu_r = (r0 + x0) - rgu_s * I;
    n_slots = n_act_k + (sh.n_shared ? 1 : 0);
    split_range(n_slots * nrb, warp, WARPS, x0, x1);
    n_dn = x1 - x0;
    dn_s = nrb > 0 ? x0 / nrb : 0;
    dn_l = x0 - dn_s * nrb;
    planned = true;
  };

  // warps clear of the router's staging area start their copies now
  if (warp >= wfree) refill();

  // ---- router logits of this CTA's experts --------------------------------
  if (router_in_smem) {
    // every thread waits for the rows, so that the ring area is quiet before
    // the weight stream reuses it
    if (!mbar_wait(rbar, 0, ws.dev_err)) failed = true;
    router_cta_smem(a, xn, wr, lseg);
  } else {
    router_cta<1, CPLH>(a, lseg, rfs);
  }
  __syncthreads();
  refill();

  if (warp == 0 && !failed) {
    // barrier 1: every expert of the grid is scored
    __threadfence();
    __syncwarp();
    if (lane == 0) gbar_arrive(ws.gbar);
    bool ok = gbar_wait(ws.gbar, a.gtarget, ws.dev_err);
    // CTA 0 selects the experts and publishes them; the other CTAs wait for
    // the publication instead of selecting themselves (the same result), so
    // that every CTA starts the routed rows at about the same time
    int id = 0;
    float w = 0.0f;
    if (ok && b == 0) {
      switch (fast_select_epl(sh)) {
        case 1: select_token<1>(a, 0, id, w); break;
        case 2: select_token<2>(a, 0, id, w); break;
        case 4: select_token<4>(a, 0, id, w); break;
        default: select_token<8>(a, 0, id, w); break;
      }
      if (lane < k) {
        ws.dm_pub_id[lane] = id;
        ws.dm_pub_w[lane] = w;
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) publish_u64(ws.dm_pub_gen, a.gtarget);
    } else if (ok) {
      ok = gbar_wait(ws.dm_pub_gen, a.gtarget, ws.dev_err);
      if (ok && lane < k) {
        id = __ldcg(ws.dm_pub_id + lane);
        w = __ldcg(ws.dm_pub_w + lane);
      }
    }
    if (!ok) {
      failed = true;
    } else {
      // the plan: for one token the k selected experts are distinct, so the
      // expert slot is the rank of its id
      int rank = 0;
      for (int j = 0; j < k; ++j) {
        const int o = __shfl_sync(0xffffffffu, id, j);
        rank += (o < id) ? 1 : 0;
      }
      if (lane < k) {
        s_pe[rank] = id;
        s_pp0[rank] = rank;
        s_pw[rank] = w;
      }
      if (lane == 0) s_nact = k;
      __syncwarp();
      if (lane == 0) mbar_arrive(planbar);
      if (b == 0 && a.write_plan) {
        // the plan of the call for moe_forward's plan output (under load
        // these stores hold warp 0 for several microseconds, so they are
        // made only when the caller asked for the plan)
        if (lane < k) {
          ws.ids[lane] = id;
          ws.topw[lane] = w;
          ws.perm[rank] = lane;
          ws.inv[lane] = rank;
          ws.active[rank] = id;
          ws.dslot[rank] = id;
          ws.dslot[32 + rank] = rank;
          ws.dslot[64 + rank] = 1;
        }
        if (lane == 0) *ws.n_active = k;
        for (int e0 = 0; e0 < E; e0 += 32) {
          const int ex = e0 + lane;
          int cnt = 0, off = 0;
          for (int j = 0; j < k; ++j) {
            const int o = __shfl_sync(0xffffffffu, id, j);
            cnt += (o == ex) ? 1 : 0;
            off += (o < ex) ? 1 : 0;
          }
          if (ex < E) {
            ws.counts[ex] = cnt;
            ws.offsets[ex] = off;
          }
        }
        if (lane == 0) ws.offsets[E] = k;
      }
      __syncwarp();
      take_plan();
      refill();
    }
  }

  // Arrival of this warp on the CTA's gate/up counter; the last warp of the
  // CTA arrives on grid barrier 2, waits for it (lane 0 polls) and releases
  // the CTA's down-projection items.  Returns false if the barrier timed out.
  auto arrive2 = [&]() -> bool {
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&s_cnt2, 1) == WARPS - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return true;
    if (lane == 0) {
      __threadfence();
      gbar_arrive(ws.gbar);
    }
    const bool ok = gbar_wait(ws.gbar, a.gtarget2, ws.dev_err);
    if (ok && lane == 0) mbar_arrive(g2bar);
    return ok;
  };

  // ---- item loop ---------------------------------------------------------
  const float4* xs4 = reinterpret_cast<const float4*>(xs);
  float4 hreg[CPLI][8];
  int h_slot = -1;
  bool arrived2 = false, g2 = false;
  while (!failed) {
    if (!planned && issued == n_sgu && (consumed == n_sgu || issued < consumed + STAGES)) {
      // pick up warp 0's plan: blocking once nothing else is left
      bool ready;
      if (consumed == n_sgu) {
        ready = mbar_wait(planbar, 0, ws.dev_err);
        if (!ready) {
          failed = true;
          break;
        }
      } else {
        int r = lane == 0 ? static_cast<int>(mbar_try_wait(planbar, 0)) : 0;
        ready = __shfl_sync(0xffffffffu, r, 0) != 0;
      }
      if (ready) {
        __syncwarp();
        take_plan();
        refill();
        continue;
      }
    }
    if (planned && !arrived2 && consumed == n_sgu + n_rgu) {
      arrived2 = true;
      if (!arrive2()) {
        failed = true;
        break;
      }
    }
    if (consumed >= known()) break;
    const int st = consumed % STAGES;
    if (!mbar_wait(bar0 + 8 * st, (consumed / STAGES) & 1, ws.dev_err)) {
      failed = true;
      break;
    }
    const unsigned char* sb = ring + (static_cast<size_t>(warp) * STAGES + st) * SB;
    const int j = consumed;
    if (j < n_sgu + n_rgu) {
      // gate/up row pair: h = SiLU(g) * u
      int row, hrow;
      if (j < n_sgu) {
        row = sgu0 + j;
        hrow = k;  // the shared expert's row of the single token
      } else {
        int slot;
        rgu_at(j - n_sgu, slot, row);
        hrow = s_pp0[slot];
      }
      const uint4* gq4 = reinterpret_cast<const uint4*>(sb);
      const uint4* uq4 = reinterpret_cast<const uint4*>(sb + H / 2);
      // grouped: scale g of the row; one a row: the half of the 4-byte word
      // that holds this row's scale (rows 2m, 2m + 1 share a word)
      const uint16_t* gsc = reinterpret_cast<const uint16_t*>(sb + H);
      const uint16_t* usc = row_scaled ? gsc + 2 : reinterpret_cast<const uint16_t*>(sb + H + H / 16);
      const int smask = row_scaled ? 0 : -1, soff = row_scaled ? (row & 1) : 0;
      float2 ga = make_float2(0.f, 0.f), ua = ga;
      // kept rolled: the body is what a cold instruction cache has to fetch
#pragma unroll 1
      for (int c = 0; c < CPLH; ++c) {
        const int g = c * 32 + lane;
        if (CPLH == 1 && g >= GKH) break;
        const uint4 qa = gq4[g], qb = uq4[g];
        const float sa = half_bits_to_f32(gsc[(g & smask) + soff]);
        const float sbv = half_bits_to_f32(usc[(g & smask) + soff]);
        const float4* xg = xs4 + (c * 8) * 32 + lane;
        float2 da0 = make_float2(0.f, 0.f), da1 = da0, db0 = da0, db1 = da0;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
          const float4 x0 = xg[(2 * wi) * 32], x1 = xg[(2 * wi + 1) * 32];
          const DqWord dg = dq_word(fword(qa, wi), magic);
          const DqWord du = dq_word(fword(qb, wi), magic);
          if (wi & 1) {
            da1 = dq_fma(dg, x0, x1, da1);
            db1 = dq_fma(du, x0, x1, db1);
          } else {
            da0 = dq_fma(dg, x0, x1, da0);
            db0 = dq_fma(du, x0, x1, db0);
          }
        }
        ga = __ffma2_rn(__fadd2_rn(da0, da1), make_float2(sa, sa), ga);
        ua = __ffma2_rn(__fadd2_rn(db0, db1), make_float2(sbv, sbv), ua);
      }
      const float s2 = warp_sum2(ga.x + ga.y, ua.x + ua.y);
      const float usum = __shfl_sync(0xffffffffu, s2, 16);
      if (lane == 0) {
        const float silu = s2 / (1.0f + expf(-s2));
        ws.hbuf[static_cast<size_t>(hrow) * hstride + swz_index(row >> 5, row & 31)] =
            silu * usum * swz_prescale(row & 31);
      }
    } else {
      // four down rows of one slot, weighted into the partial table
      if (!g2) {
        if (!mbar_wait(g2bar, 0, ws.dev_err)) {
          failed = true;
          break;
        }
        g2 = true;
      }
      int si, lr;
      dn_at(j - n_sgu - n_rgu, si, lr);
      const bool shared = si >= n_act_k;
      const int col = shared ? kSharedCol : si;
      const float wt = shared ? 1.0f : s_pw[si];
      if (col != h_slot) {
        const int hrow = shared ? k : s_pp0[si];
        const float4* hp = reinterpret_cast<const float4*>(ws.hbuf + hrow * hstride);
#pragma unroll
        for (int c = 0; c < CPLI; ++c)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            hreg[c][q] = (CPLI > 1 || lane < GKI) ? __ldcg(hp + (c * 8 + q) * 32 + lane)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        h_slot = col;
      }
      float2 acc[kRowsC];
#pragma unroll
      for (int r = 0; r < kRowsC; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < CPLI; ++c) {
        const int g = c * 32 + lane;
        if (CPLI == 1 && g >= GKI) break;
        uint4 q[kRowsC];
        float sc[kRowsC];
#pragma unroll
        for (int r = 0; r < kRowsC; ++r) {
          q[r] = reinterpret_cast<const uint4*>(sb + r * (I / 2))[g];
          sc[r] = half_bits_to_f32(reinterpret_cast<const uint16_t*>(sb + kRowsC * (I / 2))
                                       [row_scaled ? r : r * (I / 32) + g]);
        }
        float2 d0[kRowsC], d1[kRowsC];
#pragma unroll
        for (int r = 0; r < kRowsC; ++r) d0[r] = d1[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
          for (int r = 0; r < kRowsC; ++r) {
            const DqWord dw = dq_word(fword(q[r], wi), magic);
            if (wi & 1)
              d1[r] = dq_fma(dw, hreg[c][2 * wi], hreg[c][2 * wi + 1], d1[r]);
            else
              d0[r] = dq_fma(dw, hreg[c][2 * wi], hreg[c][2 * wi + 1], d0[r]);
          }
        }
#pragma unroll
        for (int r = 0; r < kRowsC; ++r)
          acc[r] = __ffma2_rn(__fadd2_rn(d0[r], d1[r]), make_float2(sc[r], sc[r]), acc[r]);
      }
      const float v = warp_sum4(acc[0].x + acc[0].y, acc[1].x + acc[1].y, acc[2].x + acc[2].y,
                                acc[3].x + acc[3].y);
      if ((lane & 7) == 0) {
        const int r = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
        part[(lr * kRowsC + r) * kSlotsP + col] = wt * v;
      }
    }
    ++consumed;
    __syncwarp();
    refill();
  }
  if (failed) {
    for (int jj = consumed; jj < issued; ++jj)
      mbar_wait(bar0 + 8 * (jj % STAGES), (jj / STAGES) & 1, ws.dev_err);
  }
  __syncthreads();

  // ---- y rows of this CTA: routed slots in expert order, then shared ------
  const int n_act = s_nact;
  for (int i = threadIdx.x; i < nrb * kRowsC; i += blockDim.x) {
    const float* pr = part + static_cast<size_t>(i) * kSlotsP;
    float v = 0.0f;
    for (int q = 0; q < n_act; ++q) v += pr[q];
    if (sh.n_shared) v += pr[kSharedCol];
    float* yp = a.y + static_cast<size_t>(rb0) * kRowsC + i;
    *yp = a.accumulate ? *yp + v : v;
  }
}

template <int CPLH, int CPLI>
cudaError_t launch_fused(const DecArgs& a, size_t smem, int n_sm, cudaStream_t s) {
  auto kern = dec_fused_kernel<CPLH, CPLI, kWarpsF, kStagesF>;
  // the opt-in is an attribute of the kernel on one device: kept per device
  static std::atomic<size_t> smem_set[kMaxDevices];
  const cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), smem_set, smem);
  if (e != cudaSuccess) return e;
  return launch_k(kern, n_sm, kWarpsF * 32, smem, s, a, /*pdl=*/false, /*coop=*/true);
}

}  // namespace dec
}  // namespace moe

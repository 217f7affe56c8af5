// dm_kernel: the whole layer for one token in one cooperative kernel (one
// CTA per SM), with every expert projection on the tensor cores
// (mma.sync m16n8k16, f16 operands, f32 accumulation).
//
// Work items.  An item is a weight tile of 16 rows x 1024 K: 8 KB of int4
// brought by one TMA tensor copy and 1 KB of scales brought by cp.async
// (16 bytes per lane), into a two-stage ring owned by one consumer warp.
// (The SM's TMA unit pays per copy and per row of a box whatever the row's
// width, so the 64-byte scale rows go through the load/store path.)
//
//   gate/up item  16 gate rows, or the same 16 up rows, of one expert (a
//                 "block" of the intermediate dimension), one K chunk;
//   down item     16 rows of one expert's down matrix (a "tile" of y), one
//                 chunk of the intermediate dimension.
// The units of each phase are split evenly over the CTAs (contiguous
// ranges) and, inside a CTA, over the warps (contiguous blocks):
//   shared gate/up  (block, gate|up, chunk)
//   routed gate/up  (slot, block, gate|up, chunk)
//   down            (tile, slot, chunk)            computed after grid barrier 2
// where the slots are the selected experts in id order, then the shared
// expert.  No weight copy is issued before the plan is known: streaming
// during the router -> barrier 1 -> selection path measured slower.  A warp keeps a running sum over its consecutive units of one
// block matrix (of one tile, each unit weighted by its slot's gate weight)
// and writes one partial per block matrix (tile) to shared memory; the CTA
// then adds each one's partials in warp order.  A block or tile cut by a CTA
// range boundary has exactly two parts: each part is published in the
// workspace and the CTA that counts second on an atomic counter adds them.
// Every sum has a fixed order, so the outputs do not depend on timing.
//
// Tensor-core dequantisation.  For a packed word w with nibbles u_0..u_7 of
// one weight row, lop3((w & 0x000F000F) | 0x64006400) is the f16 pair
// (1024 + u_0, 1024 + u_4) and the mask 0x00F000F0 gives (1024 + 16 u_1,
// 1024 + 16 u_5), both exact; w >> 8 yields nibbles 2, 6 and 3, 7 the same
// way.  These pairs are the A fragments of the MMA as they are: the K order
// inside each 32-group is permuted the same way in A and in B.  B holds the
// activation in f16, divided by 16 where the A value carries 16 u.  Then
//   A.B = sum_i (u_i - 8) x_i + corr,   corr = sum_i (1024 + 8 * 2^p_i) b_i,
// so the two MMAs of a 32-group start from C = -corr (a per-group constant
// of the activation) and give sum_i (u_i - 8) x_i, which the group's f16
// scale multiplies into the row's fp32 sum.
//
// Roles: every warp consumes items and issues its own copies; warp 0 also
// takes the control steps (grid barriers, the selection and the plan,
// staging the h fragments after barrier 2) at points where the other warps
// wait for them anyway.
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", N1
// (MoE bullet), N2 and "G2 - native GLM-5.2 correctness spine" (int4 gate/
// up/down, group-32 scales, SwiGLU), N4 (route first, stream each selected
// expert once); "colibri-strix/README.md", "What's implemented" (noaux_tc
// router, shared expert).
#include <cuda_fp16.h>

#include <new>

#include "decode_common.cuh"
#include "smem_opt_in.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace dm {

using dec::DecArgs;
using dec::kMaxEntries;
using dec::split_range;
using dec::gbar_arrive;
using dec::gbar_wait;
using dec::publish_u64;

constexpr int kNW = 8;                    // warps (8: 255 registers a thread)
constexpr int kThreads = kNW * 32;
// the prologue's RMSNorm and router use warps 0..7 (one per logit segment)
// and meet on a named barrier of those 256 threads
static_assert(kThreads / 32 >= dec::kRouterWarps, "the router needs 8 warps in the CTA");
constexpr int kStages = 2;                // ring stages per consumer warp
constexpr int kKc = 1024;                 // K per item
constexpr int kNCH = kKc / 256;           // 128-byte chunks of a row per item
constexpr int kGPI = kKc / 32;            // scale groups per item
constexpr int kQB = 16 * kKc / 2;         // packed weight bytes per item
constexpr int kSB = 16 * kGPI * 2;        // scale bytes per item
constexpr int kBarC = 2;                  // named barrier of the consumer warps
constexpr int kXIt = (12288 / 8 + kThreads - 1) / kThreads;  // x fragments per thread (H <= 12288)
constexpr size_t kSmemLimit = 227 * 1024 - 1024;

struct Maps {
  CUtensorMap gq[2][2];  // [routed, shared][gate, up]: {128 B, rows, H/256}, box {128, 16, kNCH}
  CUtensorMap dq[2];     // [routed, shared]: {128 B, rows, I/256}, box {128, 16, kNCH}
};

struct Args {
  DecArgs a;
  Maps m;
  int seg_sg, seg_rg, seg_d;  // partial-table rows per warp for each phase
};

// Unit counts of the phases (whole layer).
struct Geo {
  int NKH, NKI;    // K chunks of a gate/up row (H / kKc), of a down row (I / kKc)
  int BI, BS;      // 16-row blocks of a routed / the shared expert
  int UB;          // gate/up units per block (gate and up, every chunk)
  int nslot, UT;   // down slots (selected experts + shared), down units per tile
  int n_sg, n_rg, n_d;
};

__host__ __device__ inline Geo geo_of(const Shape& sh) {
  Geo g;
  g.NKH = sh.H / kKc;
  g.NKI = sh.I / kKc;
  g.BI = sh.I / 16;
  g.BS = sh.n_shared ? sh.Is / 16 : 0;
  g.UB = 2 * g.NKH;
  g.nslot = sh.k + (sh.n_shared ? 1 : 0);
  g.UT = g.nslot * g.NKI;
  g.n_sg = g.BS * g.UB;
  g.n_rg = sh.k * g.BI * g.UB;
  g.n_d = (sh.H / 16) * g.UT;
  return g;
}

// Dynamic shared memory (offsets from a 1024-byte aligned base).
struct Smem {
  size_t ringq, rings, bfr, corr, part, bars, total;
};

__host__ __device__ inline Smem smem_of(const Shape& sh, const Geo& g, int seg_total) {
  Smem s;
  const size_t nx = sh.H / 32, nh = static_cast<size_t>(g.nslot) * (sh.I / 32);
  const size_t ng = nx > nh ? nx : nh;  // 32-groups of the B fragments (x, then h)
  s.ringq = 0;
  s.rings = s.ringq + static_cast<size_t>(kNW) * kStages * kQB;
  s.bfr = s.rings + static_cast<size_t>(kNW) * kStages * kSB;
  s.corr = s.bfr + ng * 64;
  s.part = s.corr + ng * 4;
  s.bars = s.part + static_cast<size_t>(kNW) * seg_total * 64;
  s.total = s.bars + 8 * (kNW * kStages + 8);
  return s;
}

// CTA b's range of a phase of n units in spans of `span` (blocks, tiles):
// split over min(G, n / span) CTAs, so that every part holds at least one
// span and a span is cut at most once; the other CTAs get none.
__host__ __device__ inline void phase_range(int n, int span, int b, int G, int& lo, int& hi) {
  const int Gp = n / span < G ? n / span : G;
  if (b < Gp) {
    split_range(n, b, Gp, lo, hi);
  } else {
    lo = hi = 0;
  }
}

__device__ __forceinline__ uint32_t lop_f16(uint32_t a, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(0x64006400u));
  return r;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                      uint32_t& d) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr));
}

// 16-byte global -> shared copy through L2 (cp.async); its mbarrier
// arrive-on is dec::cp_async_mbar_arrive.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
using dec::cp_async_mbar_arrive;

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ float half_lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

// Correction weight of B-fragment register `reg` (A carries 16 u in the odd
// registers): 1024 + 8 * 2^p.
__device__ __forceinline__ float corr_weight(int reg) { return (reg & 1) ? 1152.0f : 1032.0f; }

// One item: rows r and r + 8 of the 16-row tile in (x, y), every lane (the
// 8 columns of the MMA carry the same activation).  The tile sits in shared
// memory as [chunk][row][128 B], 128-byte swizzled; q_lane: the lane's
// ldmatrix row address in chunk 0; sw[gp]: swizzled offsets of the pairs.
// Called from one place: the gate/up and the down items run the same
// instructions, which are then already in the instruction cache when the
// down phase starts.
__device__ __forceinline__ float2 item_dot(uint32_t q_lane, const unsigned char* sp,
                                           const uint4* bfr, const float* cor,
                                           const uint32_t (&sw)[4], int r, int t) {
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < kNCH; ++h) {
    // scales of the chunk's 8 groups for rows r and r + 8, and their corrs
    const uint4 s4 = *reinterpret_cast<const uint4*>(sp + r * (kGPI * 2) + h * 16);
    const uint4 s48 = *reinterpret_cast<const uint4*>(sp + (r + 8) * (kGPI * 2) + h * 16);
    const float4 ca = *reinterpret_cast<const float4*>(cor + h * 8);
    const float4 cb = *reinterpret_cast<const float4*>(cor + h * 8 + 4);
#pragma unroll
    for (int gp = 0; gp < 4; ++gp) {
      uint32_t w0, w1, w2, w3;
      ldsm4(q_lane + h * 2048 + sw[gp], w0, w1, w2, w3);
      const int gc = h * 8 + 2 * gp;  // group of the pair inside the item
      const uint32_t sr = gp == 0 ? s4.x : gp == 1 ? s4.y : gp == 2 ? s4.z : s4.w;
      const uint32_t sr8 = gp == 0 ? s48.x : gp == 1 ? s48.y : gp == 2 ? s48.z : s48.w;
      const float2 cr = gp == 0 ? make_float2(ca.x, ca.y)
                        : gp == 1 ? make_float2(ca.z, ca.w)
                        : gp == 2 ? make_float2(cb.x, cb.y)
                                  : make_float2(cb.z, cb.w);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 bq = bfr[(gc + q) * 4 + t];
        const float nc = -(q ? cr.y : cr.x);
        const uint32_t wa = q ? w2 : w0, wb = q ? w3 : w1;
        float d[4] = {nc, nc, nc, nc};
        mma16816(d, lop_f16(wa, 0x000F000Fu), lop_f16(wb, 0x000F000Fu),
                 lop_f16(wa, 0x00F000F0u), lop_f16(wb, 0x00F000F0u), bq.x, bq.y);
        const uint32_t wa2 = wa >> 8, wb2 = wb >> 8;
        mma16816(d, lop_f16(wa2, 0x000F000Fu), lop_f16(wb2, 0x000F000Fu),
                 lop_f16(wa2, 0x00F000F0u), lop_f16(wb2, 0x00F000F0u), bq.z, bq.w);
        const float s0 = q ? half_hi(sr) : half_lo(sr);
        const float s1 = q ? half_hi(sr8) : half_lo(sr8);
        acc = __ffma2_rn(make_float2(s0, s1), make_float2(d[0], d[2]), acc);
      }
    }
  }
  return acc;
}

// Two-part combine of a block or tile cut by a CTA range boundary: lane l
// of the half-warp holds the two values of row l; part 0 is the lower
// range; gp: [2 parts][2][16] floats.  Returns true in the half-warp that
// finishes the unit (v then holds part 0 + part 1).  Called by all 32 lanes;
// `active` per half-warp.
__device__ __forceinline__ bool two_part(bool active, float2& v, float* gp, unsigned* cnt,
                                         int part) {
  const int hl = threadIdx.x & 15;
  if (active) {
    __stcg(gp + part * 32 + hl, v.x);
    __stcg(gp + part * 32 + 16 + hl, v.y);
    __threadfence();
  }
  __syncwarp();
  unsigned old = 0;
  if (active && hl == 0) old = atomicAdd(cnt, 1u);
  old = __shfl_sync(0xffffffffu, old, 0, 16);
  const bool second = active && (old & 1u);
  if (second) {
    __threadfence();
    const float ox = __ldcg(gp + (1 - part) * 32 + hl);
    const float oy = __ldcg(gp + (1 - part) * 32 + 16 + hl);
    v.x = part == 0 ? v.x + ox : ox + v.x;
    v.y = part == 0 ? v.y + oy : oy + v.y;
  }
  return second;
}

__global__ void __launch_bounds__(kThreads, 1) dm_kernel(const __grid_constant__ Args p) {
  const DecArgs& a = p.a;
  const Shape& sh = a.sh;
  const Workspace& ws = a.ws;
  const Geo g = geo_of(sh);
  const int H = sh.H, I = sh.I, k = sh.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int SEG = p.seg_sg + p.seg_rg + p.seg_d;
  const Smem L = smem_of(sh, g, SEG);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ int s_pe[kMaxEntries];
  __shared__ float s_pw[kMaxEntries];
  __shared__ float lseg[dec::kMaxLocalExperts * dec::kRouterWarps];
  __shared__ double dseg[8];
  __shared__ float rfs[1];

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L.bars);
  const uint32_t cb = smem_u32(bars + kNW * kStages);
  // control barriers: plan ready, barrier 2 passed, h fragments landed,
  // router rows landed
  const uint32_t planbar = cb, b2pass = cb + 8, hbar = cb + 16, rbar = cb + 24;
  int sg0, sg1, rg0, rg1, d0, d1;
  phase_range(g.n_sg, g.UB, b, G, sg0, sg1);
  phase_range(g.n_rg, g.UB, b, G, rg0, rg1);
  phase_range(g.n_d, g.UT, b, G, d0, d1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNW * kStages; ++i) mbar_init(smem_u32(bars + i), 1);
    for (int i = 0; i < 4; ++i) mbar_init(cb + 8 * i, 1);
    fence_barrier_init();
    // this CTA's router rows into the (still idle) ring area: the router
    // reads shared memory only, and no weight copy competes with the path
    // router -> barrier 1 -> selection -> plan
    const int Lr = (sh.E + G - 1) / G;
    int nl = 0;
    for (int l = 0; l < Lr; ++l) nl += (b + l * G < sh.E) ? 1 : 0;
    mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(nl) * H * 4);
    for (int l = 0; l < nl; ++l)
      bulk_g2s(smem_u32(sm + L.ringq + static_cast<size_t>(l) * H * 4),
               a.w.router_w + static_cast<size_t>(b + l * G) * H, H * 4, rbar);
  }
  if (threadIdx.x < kMaxEntries) {
    s_pe[threadIdx.x] = 0;
    s_pw[threadIdx.x] = 0.0f;
  }
  __syncthreads();

  // ---- RMSNorm scale, x fragments, router logits (all warps) ------------
  const int Lr = (sh.E + G - 1) / G;  // router rows of this CTA (at most)
  bool pro_ok = true;
  {
  const int pthr = kThreads;
  float rf = 1.0f;
  if (a.gamma != nullptr) {
    dec::rms_partial(a, 0, dseg);  // warps 0..7
    __syncthreads();
    if (threadIdx.x == 0) rfs[0] = dec::rms_finish(a, dseg);
    __syncthreads();
    rf = rfs[0];
  }
  {
    // x_hat[g*32 + 8t .. +8] -> fragment (g, t): register reg holds the
    // elements reg (low half) and reg + 4 (high half), divided by 16 in the
    // odd registers; corr of group g summed over its 4 fragments.  All of a
    // thread's loads first.
    uint4* xbf = reinterpret_cast<uint4*>(sm + L.bfr);
    float* xcorr = reinterpret_cast<float*>(sm + L.corr);
    float* xn = reinterpret_cast<float*>(sm + L.ringq) + static_cast<size_t>(Lr) * H;
    float4 va[kXIt], vb[kXIt];
#pragma unroll
    for (int it = 0; it < kXIt; ++it) {
      const int idx = threadIdx.x + it * pthr;
      if (idx < H / 8) {
        va[it] = dec::xhat4(a, idx * 8, idx * 8, rf);
        vb[it] = dec::xhat4(a, idx * 8 + 4, idx * 8 + 4, rf);
      }
    }
#pragma unroll
    for (int it = 0; it < kXIt; ++it) {
      const int idx = threadIdx.x + it * pthr;
      if (idx >= H / 8) break;
      const float4 v0 = va[it], v1 = vb[it];
      reinterpret_cast<float4*>(xn)[idx * 2] = v0;
      reinterpret_cast<float4*>(xn)[idx * 2 + 1] = v1;
      const float xv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t word[4];
      float cs = 0.0f;
#pragma unroll
      for (int reg = 0; reg < 4; ++reg) {
        const float scl = (reg & 1) ? 0.0625f : 1.0f;
        const __half lo = __float2half_rn(xv[reg] * scl), hi = __float2half_rn(xv[reg + 4] * scl);
        word[reg] = static_cast<uint32_t>(__half_as_ushort(lo)) |
                    (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
        cs = __fmaf_rn(corr_weight(reg), __half2float(lo), cs);
        cs = __fmaf_rn(corr_weight(reg), __half2float(hi), cs);
      }
      xbf[idx] = make_uint4(word[0], word[1], word[2], word[3]);
      cs += __shfl_xor_sync(0xffffffffu, cs, 1);
      cs += __shfl_xor_sync(0xffffffffu, cs, 2);
      if ((idx & 3) == 0) xcorr[idx >> 2] = cs;
    }
  }
  __syncthreads();
  if (!__all_sync(0xffffffffu, mbar_wait(rbar, 0, ws.dev_err))) pro_ok = false;
  // warps 0..7, one logit segment each (named barrier 1 of 256 threads)
  dec::router_cta_smem(a, reinterpret_cast<const float*>(sm + L.ringq) + static_cast<size_t>(Lr) * H,
                       reinterpret_cast<const float*>(sm + L.ringq), lseg);
  __syncthreads();
  }


  // ================= consumer warps =================
  const int nthr = kNW * 32;  // threads of the consumers' named barrier
  int x0, x1;
  split_range(sg1 - sg0, warp, kNW, x0, x1);
  const int wsg0 = sg0 + x0, nsg = x1 - x0;
  split_range(rg1 - rg0, warp, kNW, x0, x1);
  const int wrg0 = rg0 + x0, nrg = x1 - x0;
  split_range(d1 - d0, warp, kNW, x0, x1);
  const int wd0 = d0 + x0, nd = x1 - x0;
  const int ngu = nsg + nrg, n_items = ngu + nd;
  unsigned char* rq = sm + L.ringq + static_cast<size_t>(warp) * kStages * kQB;
  unsigned char* rs = sm + L.rings + static_cast<size_t>(warp) * kStages * kSB;
  const uint32_t fb0 = smem_u32(bars + warp * kStages);
  bool planned = false, failed = !pro_ok;

  // Item j of the warp as a position in its phase's unit space, advanced
  // item by item without divisions (they are taken at phase starts only).
  //   gate/up: key = block * 2 + matrix, c = K chunk, and for routed units
  //            slot / be = the block's expert slot and block in the expert
  //   down:    key = tile, slot, c = chunk of the intermediate dimension
  struct Cursor {
    int j, c, key, slot, be;
  };
  auto cursor_at = [&](Cursor& cu, int jj) {
    cu.j = jj;
    cu.be = 0;
    if (jj < nsg) {
      const int u = wsg0 + jj;
      cu.key = u / g.NKH;
      cu.c = u % g.NKH;
      cu.slot = k;
    } else if (jj < ngu) {
      const int u = wrg0 + (jj - nsg);
      cu.key = u / g.NKH;
      cu.c = u % g.NKH;
      cu.slot = (cu.key >> 1) / g.BI;
      cu.be = (cu.key >> 1) % g.BI;
    } else {
      const int u = wd0 + (jj - ngu), rem = u % g.UT;
      cu.key = u / g.UT;
      cu.slot = rem / g.NKI;
      cu.c = rem % g.NKI;
    }
  };
  auto cursor_next = [&](Cursor& cu) {
    ++cu.j;
    if (cu.j == nsg || cu.j == ngu) {
      cursor_at(cu, cu.j);
    } else if (cu.j < ngu) {
      if (++cu.c == g.NKH) {
        cu.c = 0;
        ++cu.key;
        if (cu.j > nsg && (cu.key & 1) == 0 && ++cu.be == g.BI) {
          cu.be = 0;
          ++cu.slot;
        }
      }
    } else if (++cu.c == g.NKI) {
      cu.c = 0;
      if (++cu.slot == g.nslot) {
        cu.slot = 0;
        ++cu.key;
      }
    }
  };
  Cursor ic;  // next item to issue
  cursor_at(ic, 0);
  auto issue = [&]() {
    const int st = ic.j % kStages;
    const uint32_t q = smem_u32(rq + st * kQB), sc = smem_u32(rs + st * kSB), fb = fb0 + 8 * st;
    int row;
    size_t srow;  // scales per weight row
    const uint16_t* sbase;
    const CUtensorMap* qm;
    if (ic.j < ngu) {
      const int e = ic.j < nsg ? 1 : 0, mat = ic.key & 1;
      row = e ? (ic.key >> 1) * 16 : s_pe[ic.slot] * I + ic.be * 16;
      sbase = e ? (mat ? a.w.sh_up_s : a.w.sh_gate_s) : (mat ? a.w.up_s : a.w.gate_s);
      srow = H / 32;
      qm = &p.m.gq[e][mat];
    } else {
      const int e = ic.slot >= k ? 1 : 0;
      row = e ? ic.key * 16 : s_pe[ic.slot] * H + ic.key * 16;
      sbase = e ? a.w.sh_down_s : a.w.down_s;
      srow = I / 32;
      qm = &p.m.dq[e];
    }
    // scales [16 rows][kGPI]: lane -> rows lane/4 and lane/4 + 8, 16-byte part lane % 4
    const int i0 = lane >> 2, part = lane & 3;
    const uint16_t* s0 = sbase + static_cast<size_t>(row + i0) * srow + ic.c * kGPI + part * 8;
    cp_async16(sc + i0 * (kGPI * 2) + part * 16, s0);
    cp_async16(sc + (i0 + 8) * (kGPI * 2) + part * 16, s0 + 8 * srow);
    cp_async_mbar_arrive(fb);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(fb, kQB);
      tc::tma_load_3d(q, qm, 0, row, ic.c * kNCH, fb);
    }
    cursor_next(ic);
  };
  // The ring's stages are read by ldmatrix and shared loads whose results
  // feed the item's MMAs before the stage is refilled, so a refill needs no
  // proxy fence; the one generic write to the ring area (x_hat for the
  // router) is fenced once, before the first copy.
  auto refill = [&](int consumed) {
    const int lim = planned ? n_items : 0;
    while (ic.j < lim && ic.j < consumed + kStages) issue();
  };
  auto wait_item = [&](int j) -> bool {
    const bool ok = mbar_wait(fb0 + 8 * (j % kStages), (j / kStages) & 1, ws.dev_err);
    return __all_sync(0xffffffffu, ok);
  };
  auto get_plan = [&]() {
    if (planned) return;
    if (lane == 0) fence_proxy_async_smem();
    const bool ok = __all_sync(0xffffffffu, mbar_wait(planbar, 0, ws.dev_err));
    planned = true;  // after a failed wait the slots read as expert 0
    if (!ok) failed = true;
  };
  // Control steps, taken by consumer warp 0 while the other warps would
  // wait anyway: barrier 1 and the plan (before any routed item), barrier 2
  // and the h fragments (between the gate/up and the down items).
  // CTA 0 selects the experts and publishes them; the other CTAs wait for
  // the publication instead of selecting themselves (the same result), so
  // that every CTA starts streaming at the same time.
  bool ctl_ok = false;
  auto control_plan = [&]() {
    bool ok = __all_sync(0xffffffffu, pro_ok);
    if (ok) {
      // barrier 1: every router expert of the grid is scored
      __threadfence();
      __syncwarp();
      if (lane == 0) gbar_arrive(ws.gbar);
      ok = gbar_wait(ws.gbar, a.gtarget, ws.dev_err);
    }
    int id = 0, rank = 0;
    float w = 0.0f;
    if (ok && b == 0) {
      switch (fast_select_epl(sh)) {
        case 1: dec::select_token<1>(a, 0, id, w); break;
        case 2: dec::select_token<2>(a, 0, id, w); break;
        case 4: dec::select_token<4>(a, 0, id, w); break;
        default: dec::select_token<8>(a, 0, id, w); break;
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
    if (ok) {
      // one token: the k experts are distinct; slot = rank of the id
      for (int j = 0; j < k; ++j) {
        const int o = __shfl_sync(0xffffffffu, id, j);
        rank += (o < id) ? 1 : 0;
      }
      if (lane < k) {
        s_pe[rank] = id;
        s_pw[rank] = w;
      }
    }
    // published even after a failed wait (the error word is set; the
    // consumers then stream expert 0 instead of waiting)
    __syncwarp();
    if (lane == 0) mbar_arrive(planbar);
    if (ok && b == 0) {
      // the plan of the call (moe_forward's plan output), after the plan is
      // published: not on the consumers' path
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
      for (int e0 = 0; e0 < sh.E; e0 += 32) {
        const int ex = e0 + lane;
        int cnt = 0, off = 0;
        for (int j = 0; j < k; ++j) {
          const int o = __shfl_sync(0xffffffffu, id, j);
          cnt += (o == ex) ? 1 : 0;
          off += (o < ex) ? 1 : 0;
        }
        if (ex < sh.E) {
          ws.counts[ex] = cnt;
          ws.offsets[ex] = off;
        }
      }
      if (lane == 0) ws.offsets[sh.E] = k;
    }
    ctl_ok = ok;
  };
  auto control_barrier2 = [&]() {
    if (ctl_ok) {
      // barrier 2: every h row of the layer is written
      __threadfence();
      __syncwarp();
      if (lane == 0) gbar_arrive(ws.gbar);
      gbar_wait(ws.gbar, a.gtarget2, ws.dev_err);
    }
    if (lane == 0) {
      mbar_arrive(b2pass);
      // the h fragments of all slots, written by the generic proxy in other
      // CTAs, read here by the async proxy
      fence_proxy_async_global();
      fence_proxy_async_smem();
      const uint32_t bytes = static_cast<uint32_t>(I / 32) * 64;
      mbar_arrive_expect_tx(hbar, bytes * g.nslot);
      const unsigned char* src = reinterpret_cast<const unsigned char*>(ws.h16);
      for (int s = 0; s < g.nslot; ++s)
        bulk_g2s(smem_u32(sm + L.bfr + static_cast<size_t>(s) * bytes),
                 src + static_cast<size_t>(s) * bytes, bytes, hbar);
    }
  };

  // no weight copy before the plan: streaming during the router -> barrier
  // 1 -> selection path (even of the shared expert) measured slower
  if (warp == 0) control_plan();
  if (b == 0 && warp == 1) {
    // idle until the plan: fetch the selection code into the SM's
    // instruction cache for warp 0 (keys not final; result unused)
    int id = 0;
    float w = 0.0f;
    switch (fast_select_epl(sh)) {
      case 1: dec::select_token<1>(a, 0, id, w); break;
      case 2: dec::select_token<2>(a, 0, id, w); break;
      case 4: dec::select_token<4>(a, 0, id, w); break;
      default: dec::select_token<8>(a, 0, id, w); break;
    }
    if (id == -12345) s_pw[0] = w;  // keeps the call
  }
  // the weight copies start with the plan (the ring held the router rows)
  get_plan();
  refill(0);

  // ---- items --------------------------------------------------------------
  const int rr = lane & 7, m4 = lane >> 3, r = lane >> 2, t = lane & 3;
  uint32_t sw[4];
#pragma unroll
  for (int gp = 0; gp < 4; ++gp) sw[gp] = static_cast<uint32_t>(((2 * gp + (m4 >> 1)) ^ rr) << 4);
  const uint32_t lane_q = (m4 & 1) * 1024 + rr * 128;
  float* P = reinterpret_cast<float*>(sm + L.part);
  float* Pw = P + static_cast<size_t>(warp) * SEG * 16;
  float2 sacc = make_float2(0.f, 0.f);
  int skey = -1, seg = 0, sbase = 0;
  auto flush = [&]() {
    if (skey >= 0) {
      if (t == 0) {
        Pw[(sbase + seg) * 16 + r] = sacc.x;
        Pw[(sbase + seg) * 16 + r + 8] = sacc.y;
      }
      ++seg;
    }
    sacc = make_float2(0.f, 0.f);
    skey = -1;
  };

  // gate/up blocks -> h fragments (once every gate/up item of the CTA is in)
  auto finish_gate_up = [&]() {
    tc::named_sync(kBarC, nthr);
    {
      const int bs0 = sg0 / g.UB, bs1 = sg1 > sg0 ? (sg1 - 1) / g.UB + 1 : bs0;
      const int br0 = rg0 / g.UB, br1 = rg1 > rg0 ? (rg1 - 1) / g.UB + 1 : br0;
      const int nbs = bs1 - bs0, n_blk = nbs + (br1 - br0);
      const int hw = threadIdx.x >> 4, hl = lane & 15;
      uint4* hb = reinterpret_cast<uint4*>(ws.h16);
      for (int base = 0; base < n_blk; base += kNW * 2) {
        const int i = base + hw;
        const bool valid = i < n_blk;
        const bool shd = i < nbs;
        const int blk = shd ? bs0 + i : br0 + (i - nbs);  // block index inside its phase
        const int c0 = shd ? sg0 : rg0, c1 = shd ? sg1 : rg1;
        const int pb = shd ? 0 : p.seg_sg;
        const int u_lo = blk * g.UB, u_hi = u_lo + g.UB;
        float2 v = make_float2(0.f, 0.f);  // (gate, up) of row hl
        if (valid) {
          for (int w = 0; w < kNW; ++w) {
            int y0, y1;
            split_range(c1 - c0, w, kNW, y0, y1);
            const int wb0 = c0 + y0, wb1 = c0 + y1;
            const int k0 = wb0 / g.NKH;  // first key of the warp's block
            for (int mat = 0; mat < 2; ++mat) {
              const int lo = u_lo + mat * g.NKH, hi = lo + g.NKH;
              if (wb0 < wb1 && wb0 < hi && wb1 > lo) {
                const float pv = P[(static_cast<size_t>(w) * SEG + pb + (blk * 2 + mat - k0)) * 16 + hl];
                if (mat == 0) v.x += pv; else v.y += pv;
              }
            }
          }
        }
        const bool cut = valid && (u_lo < c0 || u_hi > c1);
        const int gi = shd ? blk : g.BS + blk;
        bool done = valid && !cut;
        if (__any_sync(0xffffffffu, cut))
          done = two_part(cut, v, ws.dm_part + static_cast<size_t>(gi) * 64, ws.dm_cnt + gi,
                          u_lo < c0 ? 1 : 0) || done;
        // h = SiLU(g) * u of row hl; rows 8t'..8t'+7 of the block form one
        // fragment (group blk / 2, t = 2 (blk & 1) + hl / 8)
        const float hv = v.x / (1.0f + expf(-v.x)) * v.y;
        const int reg = hl & 3;
        const __half hf = __float2half_rn(reg & 1 ? hv * 0.0625f : hv);
        uint32_t bits = __half_as_ushort(hf);
        float cp = corr_weight(reg) * __half2float(hf);
        bits |= __shfl_down_sync(0xffffffffu, bits, 4, 8) << 16;
        cp += __shfl_down_sync(0xffffffffu, cp, 4, 8);
        cp += __shfl_down_sync(0xffffffffu, cp, 2, 8);
        cp += __shfl_down_sync(0xffffffffu, cp, 1, 8);
        const uint32_t w1 = __shfl_down_sync(0xffffffffu, bits, 1, 8);
        const uint32_t w2 = __shfl_down_sync(0xffffffffu, bits, 2, 8);
        const uint32_t w3 = __shfl_down_sync(0xffffffffu, bits, 3, 8);
        if (done && (hl & 7) == 0) {
          const int slot = shd ? k : blk / g.BI, be = shd ? blk : blk % g.BI;
          const int oct = be * 2 + (hl >> 3);  // octet of rows inside the expert
          hb[(static_cast<size_t>(slot) * (I / 32) + oct / 4) * 4 + (oct & 3)] =
              make_uint4(bits, w1, w2, w3);
          ws.dm_cpart[static_cast<size_t>(slot) * (I / 8) + oct] = cp;
        }
      }
    }
    tc::named_sync(kBarC, nthr);
  };
  // h fragments and their corrections, after grid barrier 2
  auto start_down = [&]() {
    // corr of every h group: the four octet parts in order
    if (!__all_sync(0xffffffffu, mbar_wait(b2pass, 0, ws.dev_err))) failed = true;
    __threadfence();
    float* hcorr = reinterpret_cast<float*>(sm + L.corr);
    const float4* cp4 = reinterpret_cast<const float4*>(ws.dm_cpart);
    for (int q = threadIdx.x; q < g.nslot * (I / 32); q += nthr) {
      const float4 c4 = __ldcg(cp4 + q);
      hcorr[q] = ((c4.x + c4.y) + c4.z) + c4.w;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(hbar, 0, ws.dev_err))) failed = true;
    tc::named_sync(kBarC, nthr);
  };

  // One loop over the warp's items (one copy of the item code, so that it
  // is already in the instruction cache when the down items start):
  // shared gate/up, routed gate/up, [h fragments], down.
  const uint4* bfr = reinterpret_cast<const uint4*>(sm + L.bfr);
  const float* cor = reinterpret_cast<const float*>(sm + L.corr);
  int j = 0;
  bool down = false;
  Cursor cc;  // next item to consume
  cursor_at(cc, 0);
  for (;;) {
    if (j == nsg && !down) {  // shared -> routed: new partial region
      flush();
      seg = 0;
      sbase = p.seg_sg;
    }
    if (j == ngu && !down) {
      flush();
      finish_gate_up();
      if (warp == 0) control_barrier2();
      start_down();
      down = true;
      seg = 0;
      sbase = p.seg_sg + p.seg_rg;
    }
    if (j >= n_items) break;
    if (failed) {
      if (down) break;
      j = ngu;  // skip to the gate/up -> down step, which every warp takes
      cursor_at(cc, j);
      continue;
    }
    if (!wait_item(j)) {
      failed = true;
      continue;
    }
    const int st = j % kStages;
    size_t gb;  // first B-fragment group of the item
    float wt;
    if (!down) {
      gb = static_cast<size_t>(cc.c) * kGPI;
      wt = 1.0f;
    } else {
      gb = static_cast<size_t>(cc.slot) * (I / 32) + cc.c * kGPI;
      wt = cc.slot < k ? s_pw[cc.slot] : 1.0f;
    }
    const int key = cc.key;
    cursor_next(cc);
    const float2 acc = item_dot(smem_u32(rq + st * kQB) + lane_q, rs + st * kSB, bfr + gb * 4,
                                cor + gb, sw, r, t);
    if (key != skey) {
      flush();
      skey = key;
    }
    sacc.x = __fmaf_rn(wt, acc.x, sacc.x);
    sacc.y = __fmaf_rn(wt, acc.y, sacc.y);
    __syncwarp();
    refill(j + 1);
    ++j;
  }
  flush();
  // copies still in flight land before the CTA exits
  for (int jj = j; jj < ic.j; ++jj) wait_item(jj);

  // ---- y tiles -------------------------------------------------------------
  tc::named_sync(kBarC, nthr);
  {
    const int t0 = d0 / g.UT, t1 = d1 > d0 ? (d1 - 1) / g.UT + 1 : t0;
    const int n_t = t1 - t0;
    const int hw = threadIdx.x >> 4, hl = lane & 15;
    const int pb = p.seg_sg + p.seg_rg;
    for (int base = 0; base < n_t; base += kNW * 2) {
      const int i = base + hw;
      const bool valid = i < n_t;
      const int tile = t0 + i;
      const int u_lo = tile * g.UT, u_hi = u_lo + g.UT;
      float2 v = make_float2(0.f, 0.f);
      if (valid) {
        for (int w = 0; w < kNW; ++w) {
          int y0, y1;
          split_range(d1 - d0, w, kNW, y0, y1);
          const int wb0 = d0 + y0, wb1 = d0 + y1;
          if (wb0 < wb1 && wb0 < u_hi && wb1 > u_lo)
            v.x += P[(static_cast<size_t>(w) * SEG + pb + (tile - wb0 / g.UT)) * 16 + hl];
        }
      }
      const bool cut = valid && (u_lo < d0 || u_hi > d1);
      const int gi = g.BS + k * g.BI + tile;
      bool done = valid && !cut;
      if (__any_sync(0xffffffffu, cut))
        done = two_part(cut, v, ws.dm_part + static_cast<size_t>(gi) * 64, ws.dm_cnt + gi,
                        u_lo < d0 ? 1 : 0) || done;
      if (done) {
        float* yp = a.y + static_cast<size_t>(tile) * 16 + hl;
        *yp = a.accumulate ? *yp + v.x : v.x;
      }
    }
  }
}

// ---- host side ----------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  }
  return fn;
}

// rows x (K/2) packed bytes, viewed as {128 B, rows, K/256}: a box of `box_rows`
// rows x 4 chunks of 128 B lands as [chunk][row][128 B], 128-byte swizzled.
bool encode_q3(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {128, rows, K / 256};
  const cuuint64_t strides[2] = {K / 2, 128};
  const cuuint32_t box[3] = {128, box_rows, static_cast<cuuint32_t>(kNCH)};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Partial-table rows a warp can need in one phase: its block of at most
// ceil(ceil(N / Gp) / kNW) units touches at most that / run + 2 runs of
// `run` units with one key (block matrix, tile); Gp as in phase_range.
int seg_rows(int n_units, int span, int G, int run) {
  const int Gp = n_units / span < G ? n_units / span : G;
  if (Gp < 1) return 0;
  const int per_cta = (n_units + Gp - 1) / Gp;
  const int per_warp = (per_cta + kNW - 1) / kNW;
  return per_warp == 0 ? 0 : (per_warp + run - 1) / run + 1;
}

struct Plan {
  int seg_sg, seg_rg, seg_d;
  size_t smem;
};

Plan plan_of(const Shape& sh, int G) {
  const Geo g = geo_of(sh);
  Plan pl;
  // gate/up segments are (block, matrix) runs of NKH units inside spans of UB
  pl.seg_sg = seg_rows(g.n_sg, g.UB, G, g.NKH);
  pl.seg_rg = seg_rows(g.n_rg, g.UB, G, g.NKH);
  pl.seg_d = seg_rows(g.n_d, g.UT, G, g.UT);
  pl.smem = smem_of(sh, g, pl.seg_sg + pl.seg_rg + pl.seg_d).total + 1024;
  return pl;
}

}  // namespace dm

bool dm_shape_ok(const Shape& sh) {
  if (!grouped_int4(sh)) return false;
  if (sh.H % dm::kKc != 0 || sh.H > 12288) return false;
  if (sh.I % dm::kKc != 0) return false;
  if (sh.n_shared && sh.Is != sh.I) return false;
  if (sh.k > dec::kMaxEntries) return false;
  const int epl = fast_select_epl(sh);
  return epl >= 1 && epl <= 8;
}

dm::Maps* dm_create_maps(const moe_weights_t& w, const Shape& sh) {
  using namespace dm;
  if (!dm_shape_ok(sh)) return nullptr;
  Maps* m = new (std::nothrow) Maps;
  if (!m) return nullptr;
  const uint64_t H = sh.H, I = sh.I, E = sh.E;
  bool ok = encode_q3(&m->gq[0][0], w.gate_q, H, E * I, 16) &&
            encode_q3(&m->gq[0][1], w.up_q, H, E * I, 16) &&
            encode_q3(&m->dq[0], w.down_q, I, E * H, 16);
  if (sh.n_shared) {
    ok = ok && encode_q3(&m->gq[1][0], w.sh_gate_q, H, I, 16) &&
         encode_q3(&m->gq[1][1], w.sh_up_q, H, I, 16) &&
         encode_q3(&m->dq[1], w.sh_down_q, I, H, 16);
  } else {
    // never read: copies of the routed maps keep every entry valid
    m->gq[1][0] = m->gq[0][0];
    m->gq[1][1] = m->gq[0][1];
    m->dq[1] = m->dq[0];
  }
  if (!ok) {
    delete m;
    return nullptr;
  }
  return m;
}

void dm_destroy_maps(dm::Maps* m) { delete m; }

bool dm_path_ok(const Shape& sh, int T, int n_sm, const dm::Maps* maps) {
  if (T != 1 || maps == nullptr || n_sm < 1) return false;
  if (!dm_shape_ok(sh)) return false;
  const int Lr = (sh.E + n_sm - 1) / n_sm;
  if (Lr > dec::kMaxLocalExperts) return false;
  // router rows and x_hat fit the ring area, where they sit until the plan
  if (static_cast<size_t>(Lr + 1) * sh.H * 4 > static_cast<size_t>(dm::kNW) * dm::kStages * dm::kQB)
    return false;
  return dm::plan_of(sh, n_sm).smem <= dm::kSmemLimit;
}

size_t dm_part_floats(int H, int I, int Is, int k, int n_shared) {
  const size_t BS = n_shared ? Is / 16 : 0, BI = I / 16;
  return (BS + static_cast<size_t>(k) * BI + H / 16) * 64 +
         static_cast<size_t>(k + (n_shared ? 1 : 0)) * (I / 8);
}

size_t dm_cnt_words(int H, int I, int Is, int k, int n_shared) {
  const size_t BS = n_shared ? Is / 16 : 0, BI = I / 16;
  return BS + static_cast<size_t>(k) * BI + H / 16;
}

cudaError_t launch_dm(const dm::Maps& maps, const moe_weights_t& w, const Shape& sh, const void* x,
                      moe_dtype_t dt, const float* gamma, float eps, const Workspace& ws, float* y,
                      int accumulate, int n_sm, unsigned long long* calls, const PhaseMarker& pm,
                      cudaStream_t s) {
  using namespace dm;
  Args p;
  p.a.w = w;
  p.a.sh = sh;
  p.a.T = 1;
  p.a.x = x;
  p.a.dt = static_cast<int>(dt);
  p.a.gamma = gamma;
  p.a.eps = eps;
  p.a.ws = ws;
  p.a.y = y;
  p.a.accumulate = accumulate;
  p.a.gtarget = (*calls + 1) * static_cast<unsigned long long>(n_sm);
  p.a.gtarget2 = (*calls + 2) * static_cast<unsigned long long>(n_sm);
  p.m = maps;
  const Plan pl = plan_of(sh, n_sm);
  p.seg_sg = pl.seg_sg;
  p.seg_rg = pl.seg_rg;
  p.seg_d = pl.seg_d;
  static std::atomic<size_t> smem_set[kMaxDevices];
  {
    const cudaError_t e =
        opt_in_smem(reinterpret_cast<const void*>(dm_kernel), smem_set, pl.smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dm_kernel, p);
  if (e != cudaSuccess) return e;
  *calls += 2;
  pm.mark(7);
  return cudaSuccess;
}

}  // namespace moe

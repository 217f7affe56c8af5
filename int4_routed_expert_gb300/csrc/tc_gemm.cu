// Tensor-core grouped GEMM of the routed experts for multi-token batches
// (prefill, and any batch the small-batch kernels do not take).
//
// What it computes ("GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri
// hierarchy": N2 per-expert gate/up/down int4 tensors with grouped scales,
// N4 each expert runs once over the rows routed to it; "G2 - native GLM-5.2
// correctness spine": dequantise, multiply, accumulate in f32):
//   gate/up pass: for every expert e and its plan rows P_e,
//       h[p][r] = SiLU(sum_k Wg[e][r][k] x[p][k]) * (sum_k Wu[e][r][k] x[p][k])
//   down pass:   o[p][m] = sum_r Wd[e][m][r] h[p][r]
// the shared expert runs the same way over all T tokens (rows T*k + t).
//
// Precision: the tensor cores multiply f16 operands.  The dequantised weight
// (u - 8) * s is rounded once to f16 (relative error <= 2^-11); the
// activations are rounded to f16 (bf16 inputs are exact); products are
// accumulated in f32 in tensor memory.
//
// Structure (one persistent CTA per SM, 23 warps):
//   warp 20      TMA producer of the weights: per 256-wide K stage, the int4
//                tile of 128 weight rows (128-byte swizzled) and its f16
//                scales, into a 7-deep shared-memory ring.  With one scale
//                a row ("G2 implementation status": Colibri's whole-row
//                group) only the tile is copied: the dequantisers emit the
//                exact u - 8 and the epilogue multiplies each row's f32
//                accumulator by the row's scale (constant along K).
//   warp 21      TMA producer of the activations: per stage up to 64 f16
//                rows (four 64-wide K slabs, 128-byte swizzled), 3-deep ring.
//   warps 0..15  dequantisers: each thread owns one weight row (TMEM lane)
//                and one 64-wide K slab of every stage (two scale groups),
//                turns the 64 nibbles into f16 (u - 8) * s with LOP3 +
//                HSUB2/HFMA2 + HMUL2 and stores them to a TMEM A buffer
//                (3 buffers of one stage).
//   warp 22      MMA issuer: tcgen05.mma kind::f16, M = 128, N = tokens
//                rounded to 16, A from TMEM, B from shared memory, D (f32)
//                in one of two TMEM accumulators.
//   warps 16..19 epilogue: TMEM -> registers; gate/up: SwiGLU and the f16
//                activation row for the down pass; down: f32 output rows.
// Weights and scales are loaded with the L2 evict-first policy (read once),
// activation rows with evict-last (every M tile of a chunk re-reads them).
// Every wait is bounded; a wait that gives up sets the device error word and
// the role stops.
//
// Weight rows of one gate/up item: 64 gate rows r0..r0+63 and the matching
// 64 up rows; TMEM lane 32q + l holds gate row r0 + 16q + l for l < 16 and
// up row r0 + 16q + l - 16 for l >= 16, so SiLU(g) * u pairs lanes l and
// l + 16 of one warp.  K order: the dequantiser emits the nibbles of a 32-bit word
// as the f16 pairs (0,4) (1,5) (2,6) (3,7); the activation rows are stored
// with the same order inside every 8 elements so that the contraction pairs
// matching elements (an order inside the dot product only).
#include <string.h>

#include <new>

#include "moe_internal.cuh"
#include "smem_opt_in.cuh"
#include "tc_ptx.cuh"

namespace moe {

struct TcMaps {
  CUtensorMap gu_q[2][2];  // [routed, shared][gate, up] int4 rows, box 128 B x 64 rows
  CUtensorMap gu_s[2][2];  // scales, box 8 x 64
  CUtensorMap dn_q[2];     // [routed, shared] down int4 rows, box 128 B x 128 rows
  CUtensorMap dn_s[2];     // scales, box 8 x 128
  CUtensorMap x16;         // [R][H] f16 activations, box 64 x 16
  CUtensorMap h16;         // [R][Imax] f16 SwiGLU rows, box 64 x 16
  // one scale a row: [routed, shared][gate, up, down] scale arrays (the
  // scale maps above are then unused)
  const uint16_t* rs[2][3];
  int row_scaled;
};

namespace tc {

constexpr int kKS = 256;                     // K per stage
constexpr int kAQBytes = 128 * 128;          // int4 tile: 128 rows x 256 nibbles
constexpr int kASBytes = 128 * 16;           // 8 f16 scales per row
constexpr int kWBytes = kAQBytes + kASBytes; // 18432, multiple of 1024
constexpr int kDqWarps = 16, kEpWarps = 4;
constexpr int kWarpWProd = kDqWarps + kEpWarps, kWarpBProd = kWarpWProd + 1,
              kWarpMma = kWarpBProd + 1;
constexpr int kThreads = (kWarpMma + 1) * 32;  // 736
constexpr uint32_t kTmemCols = 512;

// Two instantiations by the rows of a chunk (the MMA's N):
//   NMAX = 64:  7-deep weight ring, 3 activation slots of 32 KB, 3 TMEM A
//               buffers, two 64-column accumulators (batches of a few rows
//               per expert: the weight stream is the bound)
//   NMAX = 128: 5-deep weight ring, 2 activation slots of 64 KB, 2 A buffers,
//               two 128-column accumulators (many rows per expert: an
//               M = 128, N = 128 MMA runs the tensor core at full rate)
// TMEM columns: accumulator d at NMAX * d, A buffer b at 2 * NMAX + 128 * b.
template <int NMAX>
struct Cfg {
  static constexpr int kNMax = NMAX;
  static constexpr int kBStages = NMAX == 64 ? 3 : 2;
  static constexpr int kABufs = kBStages;  // A buffers and B slots advance together
  static constexpr int kWStages = NMAX == 64 ? 7 : 5;
  static constexpr int kSlabBytes = NMAX * 128;  // NMAX rows x 64 f16
  static constexpr int kBBytes = 4 * kSlabBytes;
  static constexpr int kSmemBytes = 1024 + kBStages * kBBytes + kWStages * kWBytes + 512;
  static_assert(2 * NMAX + 128 * kABufs <= static_cast<int>(kTmemCols), "TMEM columns");
};

struct Args {
  CUtensorMap aq[2][2];  // [routed, shared][gate, up] (down: [..][0])
  CUtensorMap as[2][2];
  CUtensorMap b;
  const uint16_t* rs[2][2];  // one scale a row: [routed, shared][gate, up] (down: [..][0])
  int row_scaled;
  Workspace ws;
  int T, N, H, I, Is, Imax;
  int mt_r, mt_s;    // M tiles per chunk (routed, shared)
  int ks_r, ks_s;    // K stages per item
  int n_sh_chunks;
  int chunk;         // rows per chunk (the instantiation's NMAX)
};

struct Item {
  int row0, n, e, mt;
};

__device__ __forceinline__ Item decode_item(const Args& a, int i) {
  Item t;
  const int n_sh_items = a.n_sh_chunks * a.mt_s;
  if (i < n_sh_items) {
    const int c = i / a.mt_s;
    t.mt = i - c * a.mt_s;
    t.row0 = a.N + a.chunk * c;
    t.n = min(a.chunk, a.T - a.chunk * c);
    t.e = -1;
  } else {
    const int j = i - n_sh_items;
    const int c = j / a.mt_r;
    t.mt = j - c * a.mt_r;
    const int4 ch = a.ws.chunks[c];
    t.row0 = ch.x;
    t.n = ch.y;
    t.e = ch.z;
  }
  return t;
}

// Item i, or an empty item past the end.  The roles decode the next item one
// item ahead, so that the chunk-list load is off the item boundary.
__device__ __forceinline__ Item item_or_empty(const Args& a, int i, int total) {
  if (i < total) return decode_item(a, i);
  Item t;
  t.row0 = t.n = t.e = t.mt = 0;
  return t;
}

__device__ __forceinline__ uint32_t lop(uint32_t v, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(0x64006400u));
  return r;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) {
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}
__device__ __forceinline__ __half2 u2h(uint32_t u) {
  __half2 h;
  memcpy(&h, &u, 4);
  return h;
}

// One 32-bit word of 8 nibbles -> four f16 pairs (u-8)*s, order (0,4) (1,5)
// (2,6) (3,7).  1024 + u and 1024 + 16u are exact in f16; subtracting 1032,
// or scaling by 1/16 and subtracting 72, leaves u - 8 exactly; the multiply
// by the scale rounds once.
__device__ __forceinline__ void dq_word_f16(uint32_t v, __half2 s2, uint32_t* out) {
  const __half2 k1032 = u2h(0x64086408u), k16 = u2h(0x2C002C00u), km72 = u2h(0xD480D480u);
  const uint32_t v8 = v >> 8;
  const __half2 a = __hsub2(u2h(lop(v, 0x000F000Fu)), k1032);
  const __half2 b = __hfma2(u2h(lop(v, 0x00F000F0u)), k16, km72);
  const __half2 c = __hsub2(u2h(lop(v8, 0x000F000Fu)), k1032);
  const __half2 d = __hfma2(u2h(lop(v8, 0x00F000F0u)), k16, km72);
  out[0] = h2u(__hmul2(a, s2));
  out[1] = h2u(__hmul2(b, s2));
  out[2] = h2u(__hmul2(c, s2));
  out[3] = h2u(__hmul2(d, s2));
}

// The same without the scale: four f16 pairs u - 8, exact (one scale a row:
// the row's scale multiplies the f32 accumulator in the epilogue instead).
__device__ __forceinline__ void dq_word_f16_raw(uint32_t v, uint32_t* out) {
  const __half2 k1032 = u2h(0x64086408u), k16 = u2h(0x2C002C00u), km72 = u2h(0xD480D480u);
  const uint32_t v8 = v >> 8;
  out[0] = h2u(__hsub2(u2h(lop(v, 0x000F000Fu)), k1032));
  out[1] = h2u(__hfma2(u2h(lop(v, 0x00F000F0u)), k16, km72));
  out[2] = h2u(__hsub2(u2h(lop(v8, 0x000F000Fu)), k1032));
  out[3] = h2u(__hfma2(u2h(lop(v8, 0x00F000F0u)), k16, km72));
}

// One lane of a converged warp (the lowest active lane).
__device__ __forceinline__ bool elect_one() {
  uint32_t p;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(p));
  return p != 0;
}

// Bounded wait whose outcome every lane of the warp shares, so that a warp
// never splits before a warp-collective tcgen05 operation.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
}

// position of element e (0..7) inside its group of 8 in the f16 rows
__device__ __forceinline__ int kpos8(int r) { return (r & ~7) | ((r & 3) << 1) | ((r >> 2) & 1); }

// Shared-memory row of the weight tile that TMEM lane L holds.  Gate/up: the
// tile's rows 0..63 are gate rows, 64..127 the matching up rows; lane 32q + l
// takes gate row 16q + l (l < 16) or up row 16q + l - 16 (l >= 16), so one
// warp holds both halves of its 16 SwiGLU rows.  Down: the identity.
template <int MODE>
__device__ __forceinline__ int tile_row(int L) {
  if (MODE == 1) return L;
  const int q = L >> 5, l = L & 31;
  return l < 16 ? 16 * q + l : 48 + 16 * q + l;
}

// MODE 0: gate/up, 1: down; RS: one scale a row (else grouped scales)
template <int MODE, int NMAX, bool RS>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ Args a) {
  using C = Cfg<NMAX>;
  constexpr int kWStages = C::kWStages, kBStages = C::kBStages, kABufs = C::kABufs;
  constexpr int kSlabBytes = C::kSlabBytes, kBBytes = C::kBBytes;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* bring = smem;                                  // kBStages x kBBytes
  unsigned char* wring = smem + kBStages * kBBytes;             // kWStages x kWBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(wring + kWStages * kWBytes);
  uint64_t* wfull = bars;
  uint64_t* wempty = wfull + kWStages;
  uint64_t* bfull = wempty + kWStages;
  uint64_t* afull = bfull + kBStages;
  uint64_t* sdone = afull + kABufs;  // MMAs of the stage done: its A buffer and B slot are free
  uint64_t* dfull = sdone + kABufs;
  uint64_t* dempty = dfull + 2;
  uint64_t* drain = dempty + 2;
  uint32_t* tbase_s = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = a.ws.dev_err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(smem_u32(wfull + s), 1);
      mbar_init(smem_u32(wempty + s), kDqWarps);
    }
    for (int s = 0; s < kBStages; ++s) mbar_init(smem_u32(bfull + s), 1);
    for (int b = 0; b < kABufs; ++b) {
      mbar_init(smem_u32(afull + b), kDqWarps);
      mbar_init(smem_u32(sdone + b), 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(smem_u32(dfull + d), 1);
      mbar_init(smem_u32(dempty + d), kEpWarps);
    }
    mbar_init(smem_u32(drain), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tbase_s), kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tb = *tbase_s;

  const int total = a.n_sh_chunks * a.mt_s + *a.ws.n_rchunks * a.mt_r;

  // The producer and MMA warps run converged: every lane takes the waits and
  // one elected lane (the same lane each time) issues the copies, the MMAs
  // and their commits.  Issuing from a converged warp keeps tcgen05.mma on
  // the fast path; issuing from a lone divergent lane costs several times more.
  if (warp == kWarpWProd) {
    // ---------------- TMA producer: weight tiles ----------------
    const uint64_t pol = policy_evict_first();  // weights are read once
    uint32_t it = 0;
    bool failed = false;
    Item tn = item_or_empty(a, blockIdx.x, total);
    for (int i = blockIdx.x; i < total && !failed; i += gridDim.x) {
      const Item t = tn;
      tn = item_or_empty(a, i + gridDim.x, total);
      const int sh = t.e < 0 ? 1 : 0;
      const int KS = sh ? a.ks_s : a.ks_r;
      const int ya = MODE == 0 ? (sh ? 0 : t.e * a.I) + 64 * t.mt
                               : (sh ? 0 : t.e * a.H) + 128 * t.mt;
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int s = it % kWStages;
        if (!warp_wait(smem_u32(wempty + s), ((it / kWStages) & 1) ^ 1, err)) {
          failed = true;
          break;
        }
        if (elect_one()) {
          fence_proxy_async_smem();
          const uint32_t full = smem_u32(wfull + s);
          const uint32_t base = smem_u32(wring + s * kWBytes);
          mbar_arrive_expect_tx(full, RS ? kAQBytes : kWBytes);
          if (MODE == 0) {
            tma_load_2d_hint(base, &a.aq[sh][0], ks * 128, ya, full, pol);
            tma_load_2d_hint(base + 8192, &a.aq[sh][1], ks * 128, ya, full, pol);
            if (!RS) {
              tma_load_2d_hint(base + kAQBytes, &a.as[sh][0], ks * 8, ya, full, pol);
              tma_load_2d_hint(base + kAQBytes + 1024, &a.as[sh][1], ks * 8, ya, full, pol);
            }
          } else {
            tma_load_2d_hint(base, &a.aq[sh][0], ks * 128, ya, full, pol);
            if (!RS)
              tma_load_2d_hint(base + kAQBytes, &a.as[sh][0], ks * 8, ya, full, pol);
          }
        }
        __syncwarp();
      }
    }
    // let copies in flight land before the CTA exits
    const uint32_t n_wait = it < kWStages ? it : kWStages;
    for (uint32_t j = it - n_wait; j < it; ++j)
      warp_wait(smem_u32(wfull + j % kWStages), (j / kWStages) & 1, err);
  } else if (warp == kWarpBProd) {
    // ---------------- TMA producer: activation rows ----------------
    if (elect_one()) prefetch_tmap(&a.b);
    __syncwarp();
    const uint64_t pol = policy_evict_last();  // activation rows are re-read by other CTAs
    uint32_t it = 0;
    bool failed = false;
    Item tn = item_or_empty(a, blockIdx.x, total);
    for (int i = blockIdx.x; i < total && !failed; i += gridDim.x) {
      const Item t = tn;
      tn = item_or_empty(a, i + gridDim.x, total);
      const int KS = t.e < 0 ? a.ks_s : a.ks_r;
      const int nb = (t.n + 15) >> 4;
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int s = it % kBStages;
        if (!warp_wait(smem_u32(sdone + s), ((it / kBStages) & 1) ^ 1, err)) {
          failed = true;
          break;
        }
        if (elect_one()) {
          const uint32_t full = smem_u32(bfull + s);
          const uint32_t base = smem_u32(bring + s * kBBytes);
          mbar_arrive_expect_tx(full, nb * 4 * 2048);
          for (int j = 0; j < 4; ++j)
            for (int b = 0; b < nb; ++b)
              tma_load_2d_hint(base + j * kSlabBytes + b * 2048, &a.b, ks * kKS + 64 * j,
                               t.row0 + 16 * b, full, pol);
        }
        __syncwarp();
      }
    }
    const uint32_t n_wait = it < kBStages ? it : kBStages;
    for (uint32_t j = it - n_wait; j < it; ++j)
      warp_wait(smem_u32(bfull + j % kBStages), (j / kBStages) & 1, err);
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    uint32_t it = 0, ic = 0;
    bool failed = false;
    Item tn = item_or_empty(a, blockIdx.x, total);
    for (int i = blockIdx.x; i < total && !failed; i += gridDim.x, ++ic) {
      const Item t = tn;
      tn = item_or_empty(a, i + gridDim.x, total);
      const int KS = t.e < 0 ? a.ks_s : a.ks_r;
      const uint32_t idesc = idesc_f16(128, ((t.n + 15) >> 4) * 16);
      const int d = ic & 1;
      if (!warp_wait(smem_u32(dempty + d), ((ic >> 1) & 1) ^ 1, err)) break;
      fence_after_sync();
      const uint32_t dt = tb + NMAX * d;
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int sb = it % kBStages;  // B slot, A buffer and done barrier share the index
        if (!warp_wait(smem_u32(bfull + sb), (it / kBStages) & 1, err) ||
            !warp_wait(smem_u32(afull + sb), (it / kABufs) & 1, err)) {
          failed = true;
          break;
        }
        fence_after_sync();
        const uint32_t at = tb + 2 * NMAX + 128 * sb;
        // descriptor of slab 0; later slabs / K steps add (byte offset >> 4) to the
        // 14-bit start field, which stays below 2^14 inside shared memory
        const uint64_t bd = sdesc_sw128(smem_u32(bring + sb * kBBytes));
        if (elect_one()) {
          mma_ts_stage16<kSlabBytes>(dt, at, bd, idesc, ks == 0);
          mma_commit(smem_u32(sdone + sb));
          if (ks == KS - 1) mma_commit(smem_u32(dfull + d));
        }
        __syncwarp();
      }
    }
    // every MMA this warp issued has completed once the drain barrier flips
    if (elect_one()) mma_commit(smem_u32(drain));
    __syncwarp();
    warp_wait(smem_u32(drain), 0, err);
  } else if (warp < kDqWarps) {
    // ---------------- dequantisers ----------------
    // warp w: TMEM lane quadrant w % 4, K slab w / 4 (groups 2j, 2j+1) of every stage
    const int q = warp & 3, j = warp >> 2;
    const int R = tile_row<MODE>(32 * q + lane);  // tile row of this thread's TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    uint32_t it = 0;
    bool failed = false;
    Item tn = item_or_empty(a, blockIdx.x, total);
    for (int i = blockIdx.x; i < total && !failed; i += gridDim.x) {
      const Item t = tn;
      tn = item_or_empty(a, i + gridDim.x, total);
      const int KS = t.e < 0 ? a.ks_s : a.ks_r;
      for (int ks = 0; ks < KS; ++ks, ++it) {
        const int s = it % kWStages, ab = it % kABufs;
        if (!warp_wait(smem_u32(wfull + s), (it / kWStages) & 1, err)) {
          failed = true;
          break;
        }
        const unsigned char* st = wring + s * kWBytes;
        const uint32_t sc =
            RS ? 0u : *reinterpret_cast<const uint32_t*>(st + kAQBytes + R * 16 + 4 * j);
        const uint4 w0 = *reinterpret_cast<const uint4*>(st + R * 128 + (((2 * j) ^ (R & 7)) << 4));
        const uint4 w1 =
            *reinterpret_cast<const uint4*>(st + R * 128 + (((2 * j + 1) ^ (R & 7)) << 4));
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(wempty + s));
        if (!warp_wait(smem_u32(sdone + ab), ((it / kABufs) & 1) ^ 1, err)) {
          failed = true;
          break;
        }
        fence_after_sync();
        uint32_t v[32];
        if (RS) {
          dq_word_f16_raw(w0.x, v + 0);
          dq_word_f16_raw(w0.y, v + 4);
          dq_word_f16_raw(w0.z, v + 8);
          dq_word_f16_raw(w0.w, v + 12);
          dq_word_f16_raw(w1.x, v + 16);
          dq_word_f16_raw(w1.y, v + 20);
          dq_word_f16_raw(w1.z, v + 24);
          dq_word_f16_raw(w1.w, v + 28);
        } else {
          const __half2 s0 = u2h((sc & 0xFFFFu) | (sc << 16));
          const __half2 s1 = u2h((sc >> 16) | (sc & 0xFFFF0000u));
          dq_word_f16(w0.x, s0, v + 0);
          dq_word_f16(w0.y, s0, v + 4);
          dq_word_f16(w0.z, s0, v + 8);
          dq_word_f16(w0.w, s0, v + 12);
          dq_word_f16(w1.x, s1, v + 16);
          dq_word_f16(w1.y, s1, v + 20);
          dq_word_f16(w1.z, s1, v + 24);
          dq_word_f16(w1.w, s1, v + 28);
        }
        tmem_st32(tb + lane_base + 2 * NMAX + 128 * ab + 32 * j, v);
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(afull + ab));
      }
    }
  } else if (warp < kDqWarps + kEpWarps) {
    // ---------------- epilogue (warps 16..19, TMEM lane quadrant warp % 4) ----------------
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // one scale a row: the scale of this thread's weight row (tile row R of
    // TMEM lane 32q + lane) multiplies its accumulator, loaded one item ahead
    const int R = tile_row<MODE>(32 * q + lane);
    auto row_scale = [&](const Item& t) -> float {
      if (!RS || t.n == 0) return 1.0f;
      const int sh = t.e < 0 ? 1 : 0;
      const size_t ya = MODE == 0 ? static_cast<size_t>(sh ? 0 : t.e) * a.I + 64 * t.mt
                                  : static_cast<size_t>(sh ? 0 : t.e) * a.H + 128 * t.mt;
      const uint16_t* p =
          MODE == 0 ? a.rs[sh][R < 64 ? 0 : 1] + ya + (R & 63) : a.rs[sh][0] + ya + R;
      return __half2float(__ushort_as_half(__ldg(p)));
    };
    uint32_t ic = 0;
    Item tn = item_or_empty(a, blockIdx.x, total);
    float srow_n = row_scale(tn);
    for (int i = blockIdx.x; i < total; i += gridDim.x, ++ic) {
      const Item t = tn;
      tn = item_or_empty(a, i + gridDim.x, total);
      const float srow = srow_n;
      srow_n = row_scale(tn);
      const int d = ic & 1;
      if (!warp_wait(smem_u32(dfull + d), (ic >> 1) & 1, err)) break;
      fence_after_sync();
      const int nch = (t.n + 15) >> 4;
      for (int c0 = 0; c0 < nch; ++c0) {
        uint32_t v[16];
        tmem_ld16(tb + lane_base + NMAX * d + 16 * c0, v);
        tmem_wait_ld();
        if (MODE == 0) {
          // lanes l < 16: gate row 16q + l; lanes l + 16: the matching up row
          const int r = 64 * t.mt + 16 * q + (lane & 15);
          __half* hrow = a.ws.h16 + static_cast<size_t>(t.row0 + 16 * c0) * a.Imax + kpos8(r);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (16 * c0 + c < t.n) {
              const float g = RS ? __uint_as_float(v[c]) * srow : __uint_as_float(v[c]);
              const float u = __shfl_down_sync(0xffffffffu, g, 16);
              if (lane < 16) {
                const float silu = g / (1.0f + expf(-g));
                hrow[static_cast<size_t>(c) * a.Imax] = __float2half_rn(silu * u);
              }
            }
        } else {
          const int m = 128 * t.mt + 32 * q + lane;
          float* orow = a.ws.obuf + static_cast<size_t>(t.row0 + 16 * c0) * a.H + m;
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (16 * c0 + c < t.n)
              orow[static_cast<size_t>(c) * a.H] = RS ? __uint_as_float(v[c]) * srow : __uint_as_float(v[c]);
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(dempty + d));
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    fence_after_sync();
    tmem_dealloc(tb, kTmemCols);
  }
}

// Routed chunk list (warp 0 of block 0) and the f16 activation rows: row p <
// T*k holds token perm[p] / k, row T*k + t token t, each in the 8-element
// order of the dequantised weights.
__global__ void __launch_bounds__(256) tc_prep_kernel(Shape sh, int T, int cr, Workspace ws) {
  const int N = T * sh.k, H = sh.H;
  const int row = blockIdx.x;
  if (row == 0) {
    // block-wide exclusive scan of the per-expert chunk counts; thread i
    // handles experts i * ept .. i * ept + ept - 1 (E <= 1024, 256 threads)
    __shared__ int wsum[8];
    const int ept = (sh.E + 255) / 256;
    const int e0 = threadIdx.x * ept;
    int mine = 0;
    for (int q = 0; q < ept; ++q)
      if (e0 + q < sh.E) mine += (ws.counts[e0 + q] + cr - 1) / cr;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < 8; ++w) {
      before += w < warp ? wsum[w] : 0;
      total += wsum[w];
    }
    int pos = before + incl - mine;
    for (int q = 0; q < ept; ++q) {
      const int e = e0 + q;
      if (e >= sh.E) break;
      const int n = ws.counts[e], off = ws.offsets[e];
      for (int c = 0; c * cr < n; ++c)
        ws.chunks[pos++] = make_int4(off + cr * c, min(cr, n - cr * c), e, 0);
    }
    if (threadIdx.x == 0) *ws.n_rchunks = total;
  }
  const int tok = row < N ? ws.perm[row] / sh.k : row - N;
  const float4* src = reinterpret_cast<const float4*>(ws.xf + static_cast<size_t>(tok) * H);
  uint4* dst = reinterpret_cast<uint4*>(ws.x16 + static_cast<size_t>(row) * H);
  for (int o = threadIdx.x; o < H / 8; o += blockDim.x) {
    const float4 lo = src[2 * o], hi = src[2 * o + 1];
    uint4 r;
    r.x = h2u(__floats2half2_rn(lo.x, hi.x));
    r.y = h2u(__floats2half2_rn(lo.y, hi.y));
    r.z = h2u(__floats2half2_rn(lo.z, hi.z));
    r.w = h2u(__floats2half2_rn(lo.w, hi.w));
    dst[o] = r;
  }
}

// ---- host side --------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// 2-D map over rows x cols elements (row stride = cols * esize bytes).
bool encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
               uint64_t cols, uint64_t rows, uint32_t box_c, uint32_t box_r, bool swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {box_c, box_r};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int imax_of(const Shape& sh) { return sh.n_shared && sh.Is > sh.I ? sh.Is : sh.I; }

}  // namespace tc

bool tc_path_ok(const Shape& sh) {
  if (sh.wfmt != MOE_W_INT4) return false;  // int4, grouped or one scale a row
  if (sh.H % 256 != 0 || sh.I % 256 != 0) return false;
  if (sh.n_shared && sh.Is % 256 != 0) return false;
  return true;
}

size_t tc_max_chunks(int Tm, int k, int E) {
  return static_cast<size_t>(Tm) * k / 64 + E + 1;  // chunks of >= 64 rows
}

TcMaps* tc_create_maps(const moe_weights_t& w, const Shape& sh, const Workspace& ws, int Tm) {
  using namespace tc;
  if (!tc_path_ok(sh)) return nullptr;
  TcMaps* m = new (std::nothrow) TcMaps;
  if (!m) return nullptr;
  memset(m, 0, sizeof(TcMaps));
  const uint64_t H = sh.H, I = sh.I, E = sh.E, Is = sh.Is;
  const uint64_t R = static_cast<uint64_t>(Tm) * sh.k + Tm;
  const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, U16 = CU_TENSOR_MAP_DATA_TYPE_UINT16,
             F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  bool ok = true;
  const bool gs = sh.gsz != 0;  // grouped scales: by TMA; one a row: read by the dequantisers
  m->row_scaled = gs ? 0 : 1;
  m->rs[0][0] = w.gate_s;
  m->rs[0][1] = w.up_s;
  m->rs[0][2] = w.down_s;
  m->rs[1][0] = w.sh_gate_s;
  m->rs[1][1] = w.sh_up_s;
  m->rs[1][2] = w.sh_down_s;
  ok = ok && encode_2d(&m->gu_q[0][0], w.gate_q, U8, 1, H / 2, E * I, 128, 64, true);
  ok = ok && encode_2d(&m->gu_q[0][1], w.up_q, U8, 1, H / 2, E * I, 128, 64, true);
  ok = ok && (!gs || encode_2d(&m->gu_s[0][0], w.gate_s, U16, 2, H / 32, E * I, 8, 64, false));
  ok = ok && (!gs || encode_2d(&m->gu_s[0][1], w.up_s, U16, 2, H / 32, E * I, 8, 64, false));
  ok = ok && encode_2d(&m->dn_q[0], w.down_q, U8, 1, I / 2, E * H, 128, 128, true);
  ok = ok && (!gs || encode_2d(&m->dn_s[0], w.down_s, U16, 2, I / 32, E * H, 8, 128, false));
  if (sh.n_shared) {
    ok = ok && encode_2d(&m->gu_q[1][0], w.sh_gate_q, U8, 1, H / 2, Is, 128, 64, true);
    ok = ok && encode_2d(&m->gu_q[1][1], w.sh_up_q, U8, 1, H / 2, Is, 128, 64, true);
    ok = ok && (!gs || encode_2d(&m->gu_s[1][0], w.sh_gate_s, U16, 2, H / 32, Is, 8, 64, false));
    ok = ok && (!gs || encode_2d(&m->gu_s[1][1], w.sh_up_s, U16, 2, H / 32, Is, 8, 64, false));
    ok = ok && encode_2d(&m->dn_q[1], w.sh_down_q, U8, 1, Is / 2, H, 128, 128, true);
    ok = ok && (!gs || encode_2d(&m->dn_s[1], w.sh_down_s, U16, 2, Is / 32, H, 8, 128, false));
  }
  ok = ok && encode_2d(&m->x16, ws.x16, F16, 2, H, R, 64, 16, true);
  ok = ok && encode_2d(&m->h16, ws.h16, F16, 2, imax_of(sh), R, 64, 16, true);
  if (!ok) {
    delete m;
    return nullptr;
  }
  return m;
}

void tc_destroy_maps(TcMaps* m) { delete m; }

// Rows per chunk for a batch: 128 when the experts average at least 64 plan
// rows (the tensor core then runs full-width MMAs), else 64.
int tc_chunk_rows(const Shape& sh, int T) {
  return static_cast<long long>(T) * sh.k >= 64LL * sh.E ? 128 : 64;
}

cudaError_t launch_tc_prep(const Shape& sh, int T, const Workspace& ws, cudaStream_t s) {
  const int rows = T * sh.k + (sh.n_shared ? T : 0);
  tc::tc_prep_kernel<<<rows, 256, 0, s>>>(sh, T, tc_chunk_rows(sh, T), ws);
  return cudaGetLastError();
}

namespace tc {
namespace {
template <int MODE, int NMAX, bool RS>
cudaError_t launch_gemm_rs(const Args& a, int n_sm, cudaStream_t s) {
  static std::atomic<size_t> attr_set[kMaxDevices];
  constexpr int smem = Cfg<NMAX>::kSmemBytes;
  const cudaError_t e =
      opt_in_smem(reinterpret_cast<const void*>(tc_gemm_kernel<MODE, NMAX, RS>), attr_set, smem);
  if (e != cudaSuccess) return e;
  tc_gemm_kernel<MODE, NMAX, RS><<<n_sm, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}
template <int MODE, int NMAX>
cudaError_t launch_gemm_inst(const Args& a, int n_sm, cudaStream_t s) {
  return a.row_scaled ? launch_gemm_rs<MODE, NMAX, true>(a, n_sm, s)
                      : launch_gemm_rs<MODE, NMAX, false>(a, n_sm, s);
}
}  // namespace
}  // namespace tc

cudaError_t launch_tc_gemm(const TcMaps& m, const Shape& sh, int T, const Workspace& ws, int mode,
                           int n_sm, cudaStream_t s) {
  using namespace tc;
  Args a;
  memset(&a, 0, sizeof(a));
  a.ws = ws;
  a.T = T;
  a.N = T * sh.k;
  a.H = sh.H;
  a.I = sh.I;
  a.Is = sh.n_shared ? sh.Is : sh.I;
  a.Imax = imax_of(sh);
  // the front end (T <= 4) builds chunks of at most 32 rows, within 64
  a.chunk = tc_chunk_rows(sh, T);
  a.n_sh_chunks = sh.n_shared ? (T + a.chunk - 1) / a.chunk : 0;
  a.row_scaled = m.row_scaled;
  for (int e = 0; e < 2; ++e) {
    a.rs[e][0] = mode == 0 ? m.rs[e][0] : m.rs[e][2];
    a.rs[e][1] = mode == 0 ? m.rs[e][1] : nullptr;
  }
  if (mode == 0) {
    a.aq[0][0] = m.gu_q[0][0];
    a.aq[0][1] = m.gu_q[0][1];
    a.as[0][0] = m.gu_s[0][0];
    a.as[0][1] = m.gu_s[0][1];
    a.aq[1][0] = m.gu_q[1][0];
    a.aq[1][1] = m.gu_q[1][1];
    a.as[1][0] = m.gu_s[1][0];
    a.as[1][1] = m.gu_s[1][1];
    a.b = m.x16;
    a.mt_r = sh.I / 64;
    a.mt_s = a.Is / 64;
    a.ks_r = a.ks_s = sh.H / kKS;
  } else {
    a.aq[0][0] = m.dn_q[0];
    a.as[0][0] = m.dn_s[0];
    a.aq[1][0] = m.dn_q[1];
    a.as[1][0] = m.dn_s[1];
    a.b = m.h16;
    a.mt_r = a.mt_s = sh.H / 128;
    a.ks_r = sh.I / kKS;
    a.ks_s = a.Is / kKS;
  }
  if (a.chunk == 128)
    return mode == 0 ? launch_gemm_inst<0, 128>(a, n_sm, s) : launch_gemm_inst<1, 128>(a, n_sm, s);
  return mode == 0 ? launch_gemm_inst<0, 64>(a, n_sm, s) : launch_gemm_inst<1, 64>(a, n_sm, s);
}

}  // namespace moe

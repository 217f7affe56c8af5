// General routed-expert path (any batch size): dequantising GEMV/GEMM-lite
// kernels over the routing plan, then the weighted combine.
//
// "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy":
// N2 (per-expert gate/up/down tensors, packed symmetric int4 with grouped
// scales), "G2 - native GLM-5.2 correctness spine" (dequant -> f32
// multiply-accumulate), "G2 implementation status" (offset-binary Q4,
// unweighted shared expert), N4 (each expert runs once over the rows that
// chose it, rows composed back in route order).
//
// Rows of the activation buffer hbuf: position p of the plan's permutation
// for routed entries (p < T*k), then T*k + t for the shared expert of token t.
// obuf uses the same row numbering with H columns.
//
// A CTA owns a tile of kNT consecutive plan positions (or kNT tokens of the
// shared expert) and 64 output rows; positions of one expert inside the tile
// form one run that streams each weight row once for all of its tokens.  For
// T <= 4 the runs of a tile are spread over blockIdx.z, one CTA each.
//
// Every expert format runs here (N2: symmetric int4/int8, per-row or grouped
// scales): packed offset-binary int4 or signed int8 weights, one fp16 scale
// per 32 values or one per row.
//
// The expert tier (tier.cu) runs the same kernels with a slot table: each
// routed expert reads its weights from the HBM slot the table names, and a
// launch takes only the experts of one phase (resident ones first, loaded
// ones once their copies have landed).
#include "moe_internal.cuh"
#include "tier_internal.cuh"

namespace moe {
namespace {

constexpr int kNT = 4;        // plan positions per CTA tile
constexpr int kRows = 64;     // output rows per CTA
constexpr int kWarps = 8;
constexpr int kGS = 36;       // smem stride of one 32-element group (bank padding)

__device__ __forceinline__ float half_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// sum_{j<32} (u_j - 8) * x_j for one group (16 packed bytes) and NT tokens;
// xs: token-major smem rows of (K/32)*kGS floats, g: group index.
template <int NT>
__device__ __forceinline__ void group_dot(const uint4 q, const float* xs, int row_len, int g,
                                          float (&part)[NT]) {
  const uint32_t wds[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int t = 0; t < NT; ++t) part[t] = 0.0f;
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    float qv[8];
#pragma unroll
    for (int n = 0; n < 8; ++n)
      qv[n] = static_cast<float>(static_cast<int>((wds[wi] >> (4 * n)) & 15u) - 8);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float* xp = xs + t * row_len + g * kGS + wi * 8;
      const float4 a = *reinterpret_cast<const float4*>(xp);
      const float4 b = *reinterpret_cast<const float4*>(xp + 4);
      float s = part[t];
      s = fmaf(qv[0], a.x, s);
      s = fmaf(qv[1], a.y, s);
      s = fmaf(qv[2], a.z, s);
      s = fmaf(qv[3], a.w, s);
      s = fmaf(qv[4], b.x, s);
      s = fmaf(qv[5], b.y, s);
      s = fmaf(qv[6], b.z, s);
      s = fmaf(qv[7], b.w, s);
      part[t] = s;
    }
  }
}

// sum_{j<32} q_j * x_j for one group of 32 signed int8 weights (32 bytes,
// element j in byte j: two's complement, "G2 implementation status" Q8).
template <int NT>
__device__ __forceinline__ void group_dot_i8(const uint4 q0, const uint4 q1, const float* xs,
                                             int row_len, int g, float (&part)[NT]) {
  const uint32_t wds[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int t = 0; t < NT; ++t) part[t] = 0.0f;
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {
    float qv[4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
      qv[n] = static_cast<float>(static_cast<int8_t>((wds[wi] >> (8 * n)) & 0xFFu));
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float4 a = *reinterpret_cast<const float4*>(xs + t * row_len + g * kGS + wi * 4);
      float s = part[t];
      s = fmaf(qv[0], a.x, s);
      s = fmaf(qv[1], a.y, s);
      s = fmaf(qv[2], a.z, s);
      s = fmaf(qv[3], a.w, s);
      part[t] = s;
    }
  }
}

// One group of a weight row in either format: int4 (16 bytes) or int8 (32).
template <int FMT, int NT>
__device__ __forceinline__ void group_dot_fmt(const uint8_t* row, const float* xs, int row_len,
                                              int g, float (&part)[NT]) {
  if (FMT == MOE_W_INT8) {
    const uint4* q = reinterpret_cast<const uint4*>(row) + 2 * g;
    group_dot_i8<NT>(__ldg(q), __ldg(q + 1), xs, row_len, g, part);
  } else {
    group_dot<NT>(__ldg(reinterpret_cast<const uint4*>(row) + g), xs, row_len, g, part);
  }
}

// Tile of the CTA: which rows of hbuf/obuf it produces, from which expert.
struct Run {
  int e;       // expert (-1: shared)
  int n;       // tokens in the run (1..kNT)
  int tok[kNT];
  int row[kNT];  // output row (plan position, or T*k + t)
};

// Splits the CTA's tile into runs of one expert each; returns the count.
__device__ inline int tile_runs(const Workspace& ws, int T, int k, int y, Run* runs) {
  const int N = T * k;
  const int Yr = (N + kNT - 1) / kNT;
  int nr = 0;
  if (y < Yr) {
    const int p0 = y * kNT, p1 = min(N, p0 + kNT);
    for (int p = p0; p < p1; ++p) {
      const int i = ws.perm[p];
      const int e = ws.ids[i];
      if (nr == 0 || runs[nr - 1].e != e) {
        runs[nr].e = e;
        runs[nr].n = 0;
        ++nr;
      }
      Run& r = runs[nr - 1];
      r.tok[r.n] = i / k;
      r.row[r.n] = p;
      ++r.n;
    }
  } else {
    const int t0 = (y - Yr) * kNT, t1 = min(T, t0 + kNT);
    runs[0].e = -1;
    runs[0].n = t1 - t0;
    for (int t = t0; t < t1; ++t) {
      runs[0].tok[t - t0] = t;
      runs[0].row[t - t0] = N + t;
    }
    nr = t1 > t0 ? 1 : 0;
  }
  return nr;
}

// Row strides of a K-long row in the shape's format: weight bytes, scales,
// and the scale index step per group (0: one scale for the whole row).
struct RowFmt {
  size_t qb, ns;
  int sstep;
};
__device__ __forceinline__ RowFmt row_fmt(const Shape& sh, int K) {
  return RowFmt{row_bytes(sh, K), row_scales(sh, K), sh.gsz == 0 ? 0 : 1};
}

template <int FMT, int NT>
__device__ void gate_up_rows(const uint8_t* gq, const uint16_t* gs, const uint8_t* uq,
                             const uint16_t* us, int H, int I, const RowFmt& f, int r0,
                             const float* xs, const Run& run, const Workspace& ws) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = H / 32, row_len = G * kGS;
  for (int rr = warp; rr < kRows; rr += kWarps) {
    const int r = r0 + rr;
    if (r >= I) break;
    const uint8_t* gr = gq + static_cast<size_t>(r) * f.qb;
    const uint8_t* ur = uq + static_cast<size_t>(r) * f.qb;
    const uint16_t* gsr = gs + static_cast<size_t>(r) * f.ns;
    const uint16_t* usr = us + static_cast<size_t>(r) * f.ns;
    float ga[NT], ua[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) ga[t] = ua[t] = 0.0f;
    for (int g = lane; g < G; g += 32) {
      const float sa = half_to_f32(__ldg(gsr + g * f.sstep));
      const float sb = half_to_f32(__ldg(usr + g * f.sstep));
      float pa[NT], pb[NT];
      group_dot_fmt<FMT, NT>(gr, xs, row_len, g, pa);
      group_dot_fmt<FMT, NT>(ur, xs, row_len, g, pb);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        ga[t] = fmaf(sa, pa[t], ga[t]);
        ua[t] = fmaf(sb, pb[t], ua[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float g = warp_sum(ga[t]), u = warp_sum(ua[t]);
      if (lane == 0) {
        const float silu = g / (1.0f + expf(-g));
        ws.hbuf[static_cast<size_t>(run.row[t]) * ws.hstride + r] = silu * u;
      }
    }
  }
}

template <int FMT, int NT>
__device__ void down_rows(const uint8_t* dq, const uint16_t* ds, int H, int I, const RowFmt& f,
                          int r0, const float* hs, const Run& run, const Workspace& ws) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = I / 32, row_len = G * kGS;
  for (int rr = warp; rr < kRows; rr += kWarps) {
    const int r = r0 + rr;
    if (r >= H) break;
    const uint8_t* dr = dq + static_cast<size_t>(r) * f.qb;
    const uint16_t* dsr = ds + static_cast<size_t>(r) * f.ns;
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    for (int g = lane; g < G; g += 32) {
      const float sa = half_to_f32(__ldg(dsr + g * f.sstep));
      float pa[NT];
      group_dot_fmt<FMT, NT>(dr, hs, row_len, g, pa);
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = fmaf(sa, pa[t], acc[t]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float o = warp_sum(acc[t]);
      if (lane == 0) ws.obuf[static_cast<size_t>(run.row[t]) * H + r] = o;
    }
  }
}

// Stage NT rows of length K (floats, from src rows) into padded smem.
__device__ inline void stage_rows(float* xs, const float* src, size_t src_stride,
                                  const int* rows, int n, int K) {
  const int G = K / 32, row_len = G * kGS;
  for (int t = 0; t < n; ++t) {
    const float* s = src + static_cast<size_t>(rows[t]) * src_stride;
    for (int i = threadIdx.x * 4; i < K; i += blockDim.x * 4) {
      const float4 v = *reinterpret_cast<const float4*>(s + i);
      *reinterpret_cast<float4*>(xs + t * row_len + (i / 32) * kGS + (i % 32)) = v;
    }
  }
}

// Whether a run belongs to this launch, and the weight index of its expert.
// phase < 0: every run, expert e at index e.  Otherwise the routed run of
// expert e belongs to phase slot_tab[e] >> kSlotPhaseShift and reads slot
// slot_tab[e] & mask; the shared expert belongs to phase 0.  The same for
// every thread of the CTA.
__device__ __forceinline__ bool run_in_phase(int e, const int32_t* slot_tab, int phase,
                                             int& slot) {
  slot = e;
  if (phase < 0) return true;
  if (e < 0) return phase == 0;
  const int v = __ldg(slot_tab + e);
  slot = v & ((1 << kSlotPhaseShift) - 1);
  return (v >> kSlotPhaseShift) == phase;
}

template <int FMT>
__global__ void __launch_bounds__(kWarps * 32)
gate_up_kernel(moe_weights_t w, Shape sh, int T, int n_tiles, Workspace ws,
               const int32_t* __restrict__ slot_tab, int phase) {
  extern __shared__ float xs[];
  __shared__ Run runs[kNT];
  __shared__ int n_runs;
  for (int y = blockIdx.y; y < n_tiles; y += gridDim.y) {
  __syncthreads();
  if (threadIdx.x == 0) n_runs = tile_runs(ws, T, sh.k, y, runs);
  __syncthreads();
  for (int ri = blockIdx.z; ri < n_runs; ri += gridDim.z) {
    const Run& run = runs[ri];
    const bool shared = run.e < 0;
    int slot = run.e;
    if (!run_in_phase(run.e, slot_tab, phase, slot)) continue;
    const int I = shared ? sh.Is : sh.I;
    const int r0 = blockIdx.x * kRows;
    if (r0 >= I) continue;
    __syncthreads();
    stage_rows(xs, ws.xf, sh.H, run.tok, run.n, sh.H);
    __syncthreads();
    const RowFmt f = row_fmt(sh, sh.H);
    const size_t eq = shared ? 0 : static_cast<size_t>(slot) * I * f.qb;
    const size_t es = shared ? 0 : static_cast<size_t>(slot) * I * f.ns;
    const uint8_t* gq = (shared ? w.sh_gate_q : w.gate_q) + eq;
    const uint16_t* gs = (shared ? w.sh_gate_s : w.gate_s) + es;
    const uint8_t* uq = (shared ? w.sh_up_q : w.up_q) + eq;
    const uint16_t* us = (shared ? w.sh_up_s : w.up_s) + es;
    switch (run.n) {
      case 1: gate_up_rows<FMT, 1>(gq, gs, uq, us, sh.H, I, f, r0, xs, run, ws); break;
      case 2: gate_up_rows<FMT, 2>(gq, gs, uq, us, sh.H, I, f, r0, xs, run, ws); break;
      case 3: gate_up_rows<FMT, 3>(gq, gs, uq, us, sh.H, I, f, r0, xs, run, ws); break;
      default: gate_up_rows<FMT, 4>(gq, gs, uq, us, sh.H, I, f, r0, xs, run, ws); break;
    }
  }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kWarps * 32)
down_kernel(moe_weights_t w, Shape sh, int T, int n_tiles, Workspace ws,
            const int32_t* __restrict__ slot_tab, int phase) {
  extern __shared__ float hs[];
  __shared__ Run runs[kNT];
  __shared__ int n_runs;
  const int r0 = blockIdx.x * kRows;
  for (int y = blockIdx.y; y < n_tiles; y += gridDim.y) {
  __syncthreads();
  if (threadIdx.x == 0) n_runs = tile_runs(ws, T, sh.k, y, runs);
  __syncthreads();
  for (int ri = blockIdx.z; ri < n_runs; ri += gridDim.z) {
    const Run& run = runs[ri];
    const bool shared = run.e < 0;
    int slot = run.e;
    if (!run_in_phase(run.e, slot_tab, phase, slot)) continue;
    const int I = shared ? sh.Is : sh.I;
    __syncthreads();
    stage_rows(hs, ws.hbuf, ws.hstride, run.row, run.n, I);
    __syncthreads();
    const RowFmt f = row_fmt(sh, I);
    const size_t eq = shared ? 0 : static_cast<size_t>(slot) * sh.H * f.qb;
    const size_t es = shared ? 0 : static_cast<size_t>(slot) * sh.H * f.ns;
    const uint8_t* dq = (shared ? w.sh_down_q : w.down_q) + eq;
    const uint16_t* ds = (shared ? w.sh_down_s : w.down_s) + es;
    switch (run.n) {
      case 1: down_rows<FMT, 1>(dq, ds, sh.H, I, f, r0, hs, run, ws); break;
      case 2: down_rows<FMT, 2>(dq, ds, sh.H, I, f, r0, hs, run, ws); break;
      case 3: down_rows<FMT, 3>(dq, ds, sh.H, I, f, r0, hs, run, ws); break;
      default: down_rows<FMT, 4>(dq, ds, sh.H, I, f, r0, hs, run, ws); break;
    }
  }
  }
}

// y_t = (acc ? y_t : 0) + (sum_j w_tj * o_(t,j), slot order) + o_shared_t;
// block (t, c) covers columns [1024 c, 1024 c + 1024) of token t.
__global__ void __launch_bounds__(256)
combine_kernel(Shape sh, int T, Workspace ws, float* __restrict__ y, int accumulate) {
  const int t = blockIdx.x;
  const int H = sh.H, k = sh.k, N = T * k;
  {
    const int r = blockIdx.y * 1024 + threadIdx.x * 4;
    if (r >= H) return;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int p = ws.inv[t * k + j];
      const float wj = ws.topw[t * k + j];
      const float4 o = *reinterpret_cast<const float4*>(ws.obuf + static_cast<size_t>(p) * H + r);
      v.x = fmaf(wj, o.x, v.x);
      v.y = fmaf(wj, o.y, v.y);
      v.z = fmaf(wj, o.z, v.z);
      v.w = fmaf(wj, o.w, v.w);
    }
    if (sh.n_shared) {
      const float4 o =
          *reinterpret_cast<const float4*>(ws.obuf + static_cast<size_t>(N + t) * H + r);
      v.x += o.x;
      v.y += o.y;
      v.z += o.z;
      v.w += o.w;
    }
    float4* yp = reinterpret_cast<float4*>(y + static_cast<size_t>(t) * H + r);
    if (accumulate) {
      const float4 b = *yp;
      v.x += b.x;
      v.y += b.y;
      v.z += b.z;
      v.w += b.w;
    }
    *yp = v;
  }
}

cudaError_t set_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

// Small batches (T <= 4): the runs of a tile (distinct experts, at most kNT)
// go to kNT CTAs (blockIdx.z) instead of one CTA in turn, so that a call's
// few experts stream in parallel.  Larger batches keep one CTA per tile.
int runs_z(int T) { return T <= 4 ? kNT : 1; }

int tiles_y(const Shape& sh, int T) {
  return (T * sh.k + kNT - 1) / kNT + (sh.n_shared ? (T + kNT - 1) / kNT : 0);
}

}  // namespace

cudaError_t launch_gate_up_slots(const moe_weights_t& w, const Shape& sh, int T,
                                 const Workspace& ws, const int32_t* slot_tab, int phase,
                                 cudaStream_t s) {
  const int Imax = sh.n_shared ? max(sh.I, sh.Is) : sh.I;
  const size_t smem = static_cast<size_t>(kNT) * (sh.H / 32) * kGS * sizeof(float);
  auto kern = sh.wfmt == MOE_W_INT8 ? gate_up_kernel<MOE_W_INT8> : gate_up_kernel<MOE_W_INT4>;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int nt = tiles_y(sh, T);
  const dim3 grid((Imax + kRows - 1) / kRows, min(nt, 65535), runs_z(T));
  kern<<<grid, kWarps * 32, smem, s>>>(w, sh, T, nt, ws, slot_tab, phase);
  return cudaGetLastError();
}

cudaError_t launch_down_slots(const moe_weights_t& w, const Shape& sh, int T, const Workspace& ws,
                              const int32_t* slot_tab, int phase, cudaStream_t s) {
  const int Imax = sh.n_shared ? max(sh.I, sh.Is) : sh.I;
  const size_t smem = static_cast<size_t>(kNT) * (Imax / 32) * kGS * sizeof(float);
  auto kern = sh.wfmt == MOE_W_INT8 ? down_kernel<MOE_W_INT8> : down_kernel<MOE_W_INT4>;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int nt = tiles_y(sh, T);
  const dim3 grid((sh.H + kRows - 1) / kRows, min(nt, 65535), runs_z(T));
  kern<<<grid, kWarps * 32, smem, s>>>(w, sh, T, nt, ws, slot_tab, phase);
  return cudaGetLastError();
}

cudaError_t launch_gate_up(const moe_weights_t& w, const Shape& sh, int T, const Workspace& ws,
                           cudaStream_t s) {
  return launch_gate_up_slots(w, sh, T, ws, nullptr, -1, s);
}

cudaError_t launch_down(const moe_weights_t& w, const Shape& sh, int T, const Workspace& ws,
                        cudaStream_t s) {
  return launch_down_slots(w, sh, T, ws, nullptr, -1, s);
}

cudaError_t launch_combine(const Shape& sh, int T, const Workspace& ws, float* y,
                           int accumulate, cudaStream_t s) {
  combine_kernel<<<dim3(T, (sh.H + 1023) / 1024), 256, 0, s>>>(sh, T, ws, y, accumulate);
  return cudaGetLastError();
}

}  // namespace moe

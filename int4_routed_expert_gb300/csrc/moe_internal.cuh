// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Per-handle device workspace, carved out of one cudaMalloc at create time.
struct Workspace {
  float* xf;         // [Tm][H]      fp32 copy (or RMSNorm) of the input
  float* logits;     // [Tm][E]
  int32_t* ids;      // [Tm][k]
  float* topw;       // [Tm][k]
  int32_t* counts;   // [E]
  int32_t* offsets;  // [E+1]
  int32_t* perm;     // [Tm*k]
  int32_t* inv;      // [Tm*k]  position of entry i inside perm
  int32_t* active;   // [E]
  int32_t* n_active; // [1]
  float* hbuf;       // [Tm*k + Tm][hstride] SwiGLU activations (routed, then shared)
  float* obuf;       // [Tm*k + Tm][H]       expert outputs before the combine
  float* sval;       // [min(Tm,4)][E] un-biased router scores (in-kernel routers)
  float* skey;       // [min(Tm,4)][E] selection keys s + bias (in-kernel routers)
  int32_t* dev_err;  // device error word (bounded waits that gave up)
  int32_t* dslot;    // [3][32] single-token slot table: expert, first position, entries
  unsigned long long* gbar;  // grid barrier counter of the single-token kernel (monotonic)
  __half* x16;       // [Tm*k + Tm][H]    f16 activation rows of the tensor-core path
  __half* h16;       // [Tm*k + Tm][Imax] f16 SwiGLU rows of the tensor-core path
  int4* chunks;      // routed chunks of <= 64 plan rows: {first row, rows, expert, 0}
  int32_t* n_rchunks;  // [1] number of routed chunks
  // single-token tensor-core kernel (decode_mma.cu): two-part sums of the
  // octets and tiles cut by CTA ranges [unit][2][16], per-octet corrections
  // of the h fragments [slot][I/8], and the parts' counters (monotonic)
  float* dm_part;
  float* dm_cpart;
  unsigned* dm_cnt;
  // the selection of a single-token call, published by CTA 0 of either
  // single-token kernel: generation word, ids, weights
  unsigned long long* dm_pub_gen;
  int32_t* dm_pub_id;
  float* dm_pub_w;
  int hstride;       // row stride of hbuf in floats (>= Imax, multiple of 1024)
};

struct Shape {
  int H, I, Is, E, k, n_group, topk_group, n_shared;
  float rsf;
  int wfmt = 0;  // moe_wformat_t of the experts
  int gsz = 32;  // scale group along K: 32, or 0 for one scale a row
};

// Bytes of one K-long weight row and its scales in the shape's format.
__host__ __device__ inline size_t row_bytes(const Shape& sh, int K) {
  return sh.wfmt == MOE_W_INT8 ? static_cast<size_t>(K) : static_cast<size_t>(K) / 2;
}
__host__ __device__ inline size_t row_scales(const Shape& sh, int K) {
  return sh.gsz == 0 ? 1 : static_cast<size_t>(K) / 32;
}
// grouped int4: the format of the tensor-core paths
__host__ __device__ inline bool grouped_int4(const Shape& sh) { return sh.wfmt == MOE_W_INT4 && sh.gsz == 32; }

}  // namespace moe

// Phase ids of the trace API (a call records only the phases it runs).
#define MOE_N_PHASES 12

namespace moe {
struct TcMaps;  // TMA tensor maps of the tensor-core grouped GEMM (tc_gemm.cu)
namespace dm {
struct Maps;    // TMA tensor maps of the single-token tensor-core kernel (decode_mma.cu)
}
}

struct moe_layer {
  moe_config_t cfg;
  moe_weights_t w;
  moe::Shape sh;
  void* ws_base;
  size_t ws_bytes;
  moe::Workspace ws;
  int device;
  char err[512];
  int n_sm;
  unsigned long long decode_calls;  // single-token barrier rounds so far (grid barrier targets)
  moe::TcMaps* tc;                  // NULL when the shape does not fit the tensor-core path
  moe::dm::Maps* dm;                // NULL when the shape does not fit the single-token MMA kernel
  // phase tracing: trace_cap calls x (MOE_N_PHASES + 1) events, and per call
  // the phase id recorded after each launched phase
  cudaEvent_t* trace_ev;
  int* trace_phase;  // [trace_cap][MOE_N_PHASES]
  int* trace_nrec;   // [trace_cap]
  int trace_cap;
  int trace_used;
};

namespace moe {

// Sets the message moe_last_error(NULL) returns on this thread.
void set_thread_error(const char* fmt, ...);

// Why a configuration is rejected (NULL when it is valid), as moe_layer_create
// and moe_workspace_bytes judge it.
const char* config_error(const moe_config_t* c);

// NULL when [p, p + bytes) lies in device (or managed) memory of `device`
// inside allocations that hold all of it; else why not.  Needs a current
// context on `device`.
const char* device_extent_error(const void* p, size_t bytes, int device);

// ---- launchers (each returns the cudaError_t of its launch) --------------

// x (fp32 or bf16) -> xf fp32, optionally RMSNorm'd with gamma (fp64 sum of
// squares in the fixed order of the router).
cudaError_t launch_prep(const void* x, moe_dtype_t dtype, int T, int H,
                        const float* gamma, float eps, float* xf, cudaStream_t s);

// logits[t][e] = x_t . Wr_e in the fixed summation order.
cudaError_t launch_router_logits(const float* xf, int T, int H, const float* Wr, int E,
                                 float* logits, cudaStream_t s);

// warp-per-token noaux_tc selection -> ids, topw.
cudaError_t launch_select(const float* logits, const float* bias, int T, const Shape& sh,
                          int32_t* ids, float* topw, cudaStream_t s);

// single-CTA stable routing plan.
cudaError_t launch_plan(const int32_t* ids, int T, int k, int E, int32_t* counts,
                        int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active,
                        int32_t* n_active, cudaStream_t s);

// SwiGLU gate/up projections over the plan (+ shared expert): hbuf.
cudaError_t launch_gate_up(const moe_weights_t& w, const Shape& sh, int T,
                           const Workspace& ws, cudaStream_t s);

// down projection over the plan (+ shared expert): obuf.
cudaError_t launch_down(const moe_weights_t& w, const Shape& sh, int T,
                        const Workspace& ws, cudaStream_t s);

// y = (acc ? y : 0) + sum_j w_tj * o_(t,j) + o_shared_t.
cudaError_t launch_combine(const Shape& sh, int T, const Workspace& ws, float* y,
                           int accumulate, cudaStream_t s);

// Tensor-core grouped GEMM path (tc_gemm.cu): any T, shapes with H, I and
// the shared I multiples of 256.
bool tc_path_ok(const Shape& sh);
size_t tc_max_chunks(int Tm, int k, int E);
TcMaps* tc_create_maps(const moe_weights_t& w, const Shape& sh, const Workspace& ws, int Tm);
void tc_destroy_maps(TcMaps* m);
// routed chunk list + f16 activation rows
cudaError_t launch_tc_prep(const Shape& sh, int T, const Workspace& ws, cudaStream_t s);
// mode 0: gate/up -> h16; mode 1: down -> obuf
cudaError_t launch_tc_gemm(const TcMaps& m, const Shape& sh, int T, const Workspace& ws, int mode,
                           int n_sm, cudaStream_t s);

// Small-batch routing front end of the grouped GEMM (front.cu): prep,
// logits, selection, plan, chunk list and f16 rows in one cooperative
// kernel for T <= 4.  calls: as for launch_decode.
bool front_path_ok(const Shape& sh, int T, int n_sm);
cudaError_t launch_front(const moe_weights_t& w, const Shape& sh, int T, const void* x,
                         moe_dtype_t dt, const float* gamma, float eps, const Workspace& ws,
                         int n_sm, unsigned long long* calls, cudaStream_t s);

// Fused single-token kernel.  When `marker.fn` is set (phase tracing),
// marker.fn(ctx, phase) is called after the launch.
struct PhaseMarker {
  void (*fn)(void* ctx, int phase);
  void* ctx;
  void mark(int phase) const {
    if (fn) fn(ctx, phase);
  }
};
bool decode_path_ok(const Shape& sh, int T, int n_sm);

// Single-token kernel on the tensor cores (decode_mma.cu): H and I
// multiples of 1024, the shared expert as wide as a routed one.
bool dm_shape_ok(const Shape& sh);
dm::Maps* dm_create_maps(const moe_weights_t& w, const Shape& sh);
void dm_destroy_maps(dm::Maps* m);
bool dm_path_ok(const Shape& sh, int T, int n_sm, const dm::Maps* maps);
// workspace sizes of Workspace::dm_part (+ dm_cpart) and dm_cnt
size_t dm_part_floats(int H, int I, int Is, int k, int n_shared);
size_t dm_cnt_words(int H, int I, int Is, int k, int n_shared);
cudaError_t launch_dm(const dm::Maps& maps, const moe_weights_t& w, const Shape& sh, const void* x,
                      moe_dtype_t dt, const float* gamma, float eps, const Workspace& ws, float* y,
                      int accumulate, int n_sm, unsigned long long* calls, const PhaseMarker& pm,
                      cudaStream_t s);
// calls: the handle's count of grid-barrier rounds (read and advanced).
// write_plan: 0 leaves the workspace's plan arrays unwritten (no plan output).
cudaError_t launch_decode(const moe_weights_t& w, const Shape& sh, int T, const void* x,
                          moe_dtype_t dt, const float* gamma, float eps, const Workspace& ws,
                          float* y, int accumulate, int write_plan, int n_sm,
                          unsigned long long* calls, const PhaseMarker& pm, cudaStream_t s);

}  // namespace moe

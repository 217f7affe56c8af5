// Host side of the fused single-token kernel (decode_fused.cuh): which
// shapes it takes, and its launch.
#include "decode_fused.cuh"

namespace moe {
namespace dec {

// fused single-token kernel; returns cudaErrorInvalidValue for an
// uninstantiated (H, I) chunk combination
cudaError_t launch_dec_fused_i1(const DecArgs& a, int cpl_h, size_t smem, int n_sm,
                                cudaStream_t s);
cudaError_t launch_dec_fused_i2(const DecArgs& a, int cpl_h, size_t smem, int n_sm,
                                cudaStream_t s);

namespace {
constexpr size_t kSmemLimit = 227 * 1024 - 1024;  // per-CTA opt-in limit, minus static smem
}  // namespace

}  // namespace dec

bool decode_path_ok(const Shape& sh, int T, int n_sm) {
  using namespace dec;
  if (T != 1 || sh.k > kMaxEntries) return false;
  if (sh.wfmt != MOE_W_INT4) return false;  // int4, grouped or one scale a row
  const int epl = fast_select_epl(sh);
  if (epl < 1 || epl > 8) return false;
  if (n_sm < 1 || (sh.E + n_sm - 1) / n_sm > kMaxLocalExperts) return false;
  // a down item's 4 rows of scales (I / 4 bytes) are one bulk copy: a
  // multiple of 16 bytes
  if (sh.I % 64 != 0) return false;
  if (sh.n_shared && sh.Is != sh.I) return false;
  if (!chunks_per_lane(sh.H)) return false;
  const int ci = chunks_per_lane(sh.I);
  if (ci != 1 && ci != 2) return false;  // intermediate rows kept in registers
  return fused_smem_bytes(sh, n_sm) <= kSmemLimit;
}

cudaError_t launch_decode(const moe_weights_t& w, const Shape& sh, int T, const void* x,
                          moe_dtype_t dt, const float* gamma, float eps, const Workspace& ws,
                          float* y, int accumulate, int write_plan, int n_sm,
                          unsigned long long* calls, const PhaseMarker& pm, cudaStream_t s) {
  using namespace dec;
  DecArgs a;
  a.w = w;
  a.sh = sh;
  a.T = T;
  a.x = x;
  a.dt = static_cast<int>(dt);
  a.gamma = gamma;
  a.eps = eps;
  a.ws = ws;
  a.y = y;
  a.accumulate = accumulate;
  a.write_plan = write_plan;
  // every CTA adds one to the grid-barrier counter per barrier round;
  // *calls counts the rounds of this handle so far
  a.gtarget = (*calls + 1) * static_cast<unsigned long long>(n_sm);
  a.gtarget2 = (*calls + 2) * static_cast<unsigned long long>(n_sm);
  const int cpl_h = chunks_per_lane(sh.H), cpl_i = chunks_per_lane(sh.I);
  const size_t smem = fused_smem_bytes(sh, n_sm);
  const cudaError_t e = cpl_i == 1 ? launch_dec_fused_i1(a, cpl_h, smem, n_sm, s)
                                   : launch_dec_fused_i2(a, cpl_h, smem, n_sm, s);
  if (e != cudaSuccess) return e;
  *calls += 2;
  pm.mark(7);
  return cudaSuccess;
}

}  // namespace moe

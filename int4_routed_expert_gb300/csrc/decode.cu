// Host side of the fused small-batch path: eligibility, sizes and the
// two-kernel launch chain (see decode_common.cuh).
#include "decode_fused.cuh"

namespace moe {
namespace dec {

cudaError_t launch_dec_ab_nt1(const DecArgs& a, int cpl, size_t smem, int n_sm, cudaStream_t s);
cudaError_t launch_dec_ab_nt4(const DecArgs& a, int cpl, size_t smem, int n_sm, cudaStream_t s);
cudaError_t launch_dec_c_nt1(const DecArgs& a, int cpl, bool h_smem, size_t smem, int n_sm,
                             bool pdl, cudaStream_t s);
cudaError_t launch_dec_c_nt4(const DecArgs& a, int cpl, size_t smem, int n_sm, bool pdl,
                             cudaStream_t s);
// fused single-token kernel; returns cudaErrorInvalidValue for an
// uninstantiated (H, I) chunk combination
cudaError_t launch_dec_fused_i1(const DecArgs& a, int cpl_h, size_t smem, int n_sm,
                                cudaStream_t s);
cudaError_t launch_dec_fused_i2(const DecArgs& a, int cpl_h, size_t smem, int n_sm,
                                cudaStream_t s);

namespace {

constexpr size_t kSmemLimit = 227 * 1024 - 1024;  // per-CTA opt-in limit, minus static smem
constexpr size_t kHSmemBudget = 190 * 1024;       // activations staged in smem up to this

struct Sizes {
  int NT, warps_b, stages_b;
  size_t ab, c;
  bool h_smem;
};

Sizes sizes_for(const Shape& sh, int T, int n_sm) {
  Sizes z{};
  z.NT = T == 1 ? 1 : 4;
  z.warps_b = z.NT == 1 ? kWarpsB1 : kWarpsB4;
  z.stages_b = z.NT == 1 ? kStagesB1 : kStagesB4;
  z.ab = ab_smem_bytes(sh, z.NT, z.warps_b, z.stages_b, n_sm);
  const int hstride = swz_pad(sh.I);
  z.h_smem = z.NT == 1 &&
             c_smem_bytes(sh, T, z.NT, true, hstride) <= kHSmemBudget;
  z.c = c_smem_bytes(sh, T, z.NT, z.h_smem, hstride);
  return z;
}

// The fused kernel serves T == 1 when its shared memory fits and the
// intermediate size is one of its instantiations (h kept in registers).
bool fused_ok(const Shape& sh, int T, int n_sm) {
  if (T != 1) return false;
  const int ci = chunks_per_lane(sh.I);
  if (ci != 1 && ci != 2) return false;
  return fused_smem_bytes(sh, n_sm) <= kSmemLimit;
}

}  // namespace
}  // namespace dec

bool decode_path_ok(const Shape& sh, int T, int n_sm) {
  using namespace dec;
  if (T < 1 || T > kMaxNT || T * sh.k > kMaxEntries) return false;
  const int epl = fast_select_epl(sh);
  if (epl < 1 || epl > 8) return false;
  if (n_sm < 1 || (sh.E + n_sm - 1) / n_sm > kMaxLocalExperts) return false;
  if (sh.I % 256 != 0) return false;
  if (sh.n_shared && sh.Is != sh.I) return false;
  if (!chunks_per_lane(sh.H) || !chunks_per_lane(sh.I)) return false;
  const Sizes z = sizes_for(sh, T, n_sm);
  return z.ab <= kSmemLimit && z.c <= kSmemLimit;
}

cudaError_t launch_decode(const moe_weights_t& w, const Shape& sh, int T, const void* x,
                          moe_dtype_t dt, const float* gamma, float eps, const Workspace& ws,
                          float* y, int accumulate, int n_sm, unsigned long long* calls,
                          const PhaseMarker& pm, cudaStream_t s) {
  using namespace dec;
  const Sizes z = sizes_for(sh, T, n_sm);
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
  // every CTA adds one to the grid-barrier counter per barrier round;
  // *calls counts the rounds of this handle so far
  a.gtarget = (*calls + 1) * static_cast<unsigned long long>(n_sm);
  a.gtarget2 = (*calls + 2) * static_cast<unsigned long long>(n_sm);
  const int cpl_h = chunks_per_lane(sh.H), cpl_i = chunks_per_lane(sh.I);
  if (fused_ok(sh, T, n_sm)) {
    const size_t smem = fused_smem_bytes(sh, n_sm);
    cudaError_t e = cpl_i == 1 ? launch_dec_fused_i1(a, cpl_h, smem, n_sm, s)
                               : launch_dec_fused_i2(a, cpl_h, smem, n_sm, s);
    if (e != cudaSuccess) return e;
    *calls += 2;
    pm.mark(7);
    return cudaSuccess;
  }
  cudaError_t e = z.NT == 1 ? launch_dec_ab_nt1(a, cpl_h, z.ab, n_sm, s)
                            : launch_dec_ab_nt4(a, cpl_h, z.ab, n_sm, s);
  if (e != cudaSuccess) return e;
  *calls += 1;
  pm.mark(8);
  const bool pdl = pm.fn == nullptr;
  e = z.NT == 1 ? launch_dec_c_nt1(a, cpl_i, z.h_smem, z.c, n_sm, pdl, s)
                : launch_dec_c_nt4(a, cpl_i, z.c, n_sm, pdl, s);
  if (e != cudaSuccess) return e;
  pm.mark(9);
  return cudaSuccess;
}

}  // namespace moe

// dec_c instantiations for one token.
#include "decode_c.cuh"

namespace moe {
namespace dec {

cudaError_t launch_dec_c_nt1(const DecArgs& a, int cpl, bool h_smem, size_t smem, int n_sm,
                             bool pdl, cudaStream_t s) {
  return h_smem ? launch_c_cpl<1, true>(a, cpl, smem, n_sm, pdl, s)
                : launch_c_cpl<1, false>(a, cpl, smem, n_sm, pdl, s);
}

}  // namespace dec
}  // namespace moe

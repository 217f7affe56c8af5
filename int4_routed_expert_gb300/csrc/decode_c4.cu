// dec_c instantiations for two to four tokens (activations read through L2).
#include "decode_c.cuh"

namespace moe {
namespace dec {

cudaError_t launch_dec_c_nt4(const DecArgs& a, int cpl, size_t smem, int n_sm, bool pdl,
                             cudaStream_t s) {
  return launch_c_cpl<4, false>(a, cpl, smem, n_sm, pdl, s);
}

}  // namespace dec
}  // namespace moe

// dec_ab instantiations for one token.
#include "decode_ab.cuh"

namespace moe {
namespace dec {

cudaError_t launch_dec_ab_nt1(const DecArgs& a, int cpl, size_t smem, int n_sm, cudaStream_t s) {
  return launch_ab_cpl<1, kStagesB1, kWarpsB1>(a, cpl, smem, n_sm, s);
}

}  // namespace dec
}  // namespace moe

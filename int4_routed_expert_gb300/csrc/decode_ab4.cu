// dec_ab instantiations for two to four tokens.
#include "decode_ab.cuh"

namespace moe {
namespace dec {

cudaError_t launch_dec_ab_nt4(const DecArgs& a, int cpl, size_t smem, int n_sm, cudaStream_t s) {
  return launch_ab_cpl<4, kStagesB4, kWarpsB4>(a, cpl, smem, n_sm, s);
}

}  // namespace dec
}  // namespace moe

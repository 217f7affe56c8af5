// dec_fused instantiations for I = up to 1024 (1 chunk(s) of 32 groups per lane).
#include "decode_fused.cuh"

namespace moe {
namespace dec {

cudaError_t launch_dec_fused_i1(const DecArgs& a, int cpl_h, size_t smem, int n_sm,
                                cudaStream_t s) {
  switch (cpl_h) {
    case 1: return launch_fused<1, 1>(a, smem, n_sm, s);
    case 2: return launch_fused<2, 1>(a, smem, n_sm, s);
    case 4: return launch_fused<4, 1>(a, smem, n_sm, s);
    case 6: return launch_fused<6, 1>(a, smem, n_sm, s);
    case 8: return launch_fused<8, 1>(a, smem, n_sm, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dec
}  // namespace moe

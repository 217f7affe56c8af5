// dec_fused instantiations for I = 2048 (2 chunk(s) of 32 groups per lane).
#include "decode_fused.cuh"

namespace moe {
namespace dec {

cudaError_t launch_dec_fused_i2(const DecArgs& a, int cpl_h, size_t smem, int n_sm,
                                cudaStream_t s) {
  switch (cpl_h) {
    case 1: return launch_fused<1, 2>(a, smem, n_sm, s);
    case 2: return launch_fused<2, 2>(a, smem, n_sm, s);
    case 4: return launch_fused<4, 2>(a, smem, n_sm, s);
    case 6: return launch_fused<6, 2>(a, smem, n_sm, s);
    case 8: return launch_fused<8, 2>(a, smem, n_sm, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dec
}  // namespace moe

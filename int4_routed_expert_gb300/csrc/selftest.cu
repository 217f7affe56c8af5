// Self-test of the bounded waits (moe_selftest_bounded_wait in moe.h): the
// kernels' grid-barrier and mbarrier waits give up after about one second,
// set bit 0 of an error word and return, so that a wait that can never
// complete ends the kernel instead of hanging the GPU.  Here one warp waits
// on a counter that stays below its target, or on an mbarrier phase nobody
// arrives on, and the host reads the error word.
#include "decode_common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(
    int which, unsigned long long* counter, int* err) {
  __shared__ uint64_t bar;
  if (which == 0) {
    // the counter stays at 0; the target 1 is never reached
    dec::gbar_wait(counter, 1ull, err);
  } else {
    if (threadIdx.x == 0) {
      mbar_init(smem_u32(&bar), 1);
      fence_barrier_init();
    }
    __syncwarp();
    // phase 0 needs one arrival that never comes
    const bool ok = mbar_wait(smem_u32(&bar), 0, err);
    __all_sync(0xffffffffu, ok);
  }
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_selftest_bounded_wait(int which, int32_t* flags) {
  if ((which != 0 && which != 1) || flags == nullptr) {
    moe::set_thread_error("moe_selftest_bounded_wait: which must be 0 or 1 and flags non-NULL");
    return MOE_ERR_INVALID_ARG;
  }
  void* buf = nullptr;
  cudaError_t e = cudaMalloc(&buf, 256);
  if (e == cudaSuccess) e = cudaMemset(buf, 0, 256);
  if (e == cudaSuccess) {
    unsigned long long* counter = static_cast<unsigned long long*>(buf);
    int* err = reinterpret_cast<int*>(static_cast<char*>(buf) + 128);
    moe::bounded_wait_selftest_kernel<<<1, 32>>>(which, counter, err);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int32_t v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) *flags = v;
  }
  if (buf) cudaFree(buf);
  if (e != cudaSuccess) {
    moe::set_thread_error("moe_selftest_bounded_wait: %s", cudaGetErrorString(e));
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

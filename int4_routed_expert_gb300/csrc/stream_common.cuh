// Building blocks of the small-batch streaming kernels: mbarrier-guarded
// 1-D TMA bulk copies into per-warp shared-memory rings, bounded waits,
// programmatic dependent launch, and the exact int4 dequantisation used by
// the SIMT dot products.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kErrWaitTimeout = 1;             // device error bit: a bounded wait gave up
constexpr long long kWaitClocks = 2000000000;  // about one second at the SM clock

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or about 0.1 ms pass, so that waiting warps take no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// kWaitClocks, sets kErrWaitTimeout in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity)) {
    if (clock64() - t0 > kWaitClocks) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// global -> shared bulk copy completing on an mbarrier.  dst, src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- swizzled, pre-scaled activation layout ------------------------------
//
// A K-vector is stored as groups of 32 (g = k / 32, i = k % 32) so that lane
// (g & 31) reads its group as 8 conflict-free 16-byte loads:
//   index(g, i) = (((g >> 5) * 8 + i / 4) * 32 + (g & 31)) * 4 + i % 4
// and element i is multiplied by 2^-p(i % 8), p = 0,4,8,12,16,8,12,16: the
// power of two that the matching dequantised nibble carries (see dq_word).
__host__ __device__ constexpr int swz_pad(int K) { return ((K / 32 + 31) / 32) * 1024; }

__device__ __forceinline__ int swz_index(int g, int i) {
  return (((g >> 5) * 8 + (i >> 2)) * 32 + (g & 31)) * 4 + (i & 3);
}

__device__ __forceinline__ float swz_prescale(int i) {
  const int n = i & 7;
  const int p = n < 5 ? 4 * n : 4 * n - 12;
  return __int_as_float((127 - p) << 23);
}

// ---- exact int4 dequantisation --------------------------------------------
//
// For a 32-bit word holding nibbles u_0..u_7 (u_n at bits 4n): OR-ing the
// masked nibble into the bits of 2^23 gives the float 2^23 + u * 2^p exactly
// (p = bit position, at most 16 so the field stays inside the mantissa);
// nibbles 5..7 are taken from w >> 12 at p = 8, 12, 16.  Subtracting
// 2^23 + 8 * 2^p (exact) leaves (u - 8) * 2^p, the offset-binary value times
// a power of two that the pre-scaled activation cancels exactly.
constexpr uint32_t kMagic = 0x4B000000u;  // 2^23

template <uint32_t MASK>
__device__ __forceinline__ float lop_mask_or(uint32_t a, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "n"(MASK), "r"(magic));
  return __uint_as_float(r);
}

struct DqWord {
  float2 a, b, c, d;  // elements (0,1) (2,3) (4,5) (6,7), each (u - 8) * 2^p
};

__device__ __forceinline__ DqWord dq_word(uint32_t v, uint32_t magic) {
  const uint32_t v2 = v >> 12;
  DqWord r;
  r.a = __fadd2_rn(make_float2(lop_mask_or<0xFu>(v, magic), lop_mask_or<0xF0u>(v, magic)),
                   make_float2(-8388616.0f, -8388736.0f));
  r.b = __fadd2_rn(make_float2(lop_mask_or<0xF00u>(v, magic), lop_mask_or<0xF000u>(v, magic)),
                   make_float2(-8390656.0f, -8421376.0f));
  r.c = __fadd2_rn(make_float2(lop_mask_or<0xF0000u>(v, magic), lop_mask_or<0xF00u>(v2, magic)),
                   make_float2(-8912896.0f, -8390656.0f));
  r.d = __fadd2_rn(make_float2(lop_mask_or<0xF000u>(v2, magic), lop_mask_or<0xF0000u>(v2, magic)),
                   make_float2(-8421376.0f, -8912896.0f));
  return r;
}

// acc += dequantised word . pre-scaled x (x0: elements 0..3, x1: 4..7)
__device__ __forceinline__ float2 dq_fma(const DqWord& q, float4 x0, float4 x1, float2 acc) {
  acc = __ffma2_rn(q.a, make_float2(x0.x, x0.y), acc);
  acc = __ffma2_rn(q.b, make_float2(x0.z, x0.w), acc);
  acc = __ffma2_rn(q.c, make_float2(x1.x, x1.y), acc);
  acc = __ffma2_rn(q.d, make_float2(x1.z, x1.w), acc);
  return acc;
}

// Group dot products of two rows (qa, qb: 32 nibbles each) against one
// pre-scaled group xg[0..7]; returns the pair sums in da, db.
__device__ __forceinline__ void dq_dot2(const uint4 qa, const uint4 qb, const float4* xg,
                                        uint32_t magic, float2& da, float2& db) {
  float2 a0 = make_float2(0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
  a0 = dq_fma(dq_word(qa.x, magic), xg[0], xg[1], a0);
  b0 = dq_fma(dq_word(qb.x, magic), xg[0], xg[1], b0);
  a1 = dq_fma(dq_word(qa.y, magic), xg[2], xg[3], a1);
  b1 = dq_fma(dq_word(qb.y, magic), xg[2], xg[3], b1);
  a0 = dq_fma(dq_word(qa.z, magic), xg[4], xg[5], a0);
  b0 = dq_fma(dq_word(qb.z, magic), xg[4], xg[5], b0);
  a1 = dq_fma(dq_word(qa.w, magic), xg[6], xg[7], a1);
  b1 = dq_fma(dq_word(qb.w, magic), xg[6], xg[7], b1);
  da = __fadd2_rn(a0, a1);
  db = __fadd2_rn(b0, b1);
}

__device__ __forceinline__ float half_bits_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

}  // namespace moe

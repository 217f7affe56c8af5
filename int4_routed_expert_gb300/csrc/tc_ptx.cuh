// Inline-PTX building blocks of the tensor-core grouped GEMM: tensor memory
// (TMEM) allocation, loads and stores, tcgen05.mma with the A operand in
// TMEM and the B operand in shared memory, completion through mbarriers, and
// 2-D and 3-D TMA tensor loads.
//
// Descriptor formats (PTX ISA, tcgen05 "shared memory descriptor" and
// "instruction descriptor" for .kind::f16):
//   shared memory descriptor (64 bit): start address >> 4 in bits 0..13,
//   leading-dimension byte offset >> 4 in 16..29, stride-dimension byte
//   offset >> 4 in 32..45, the fixed version value 1 in bits 46..47, base
//   offset 49..51, layout (swizzle) type in 61..63 (2 = 128-byte swizzle).
//   instruction descriptor (32 bit): D format in bits 4..5 (1 = f32), A and B
//   formats in 7..9 and 10..12 (0 = f16), A / B major-ness in bits 15 / 16
//   (0 = K-major), N >> 3 in 17..22, M >> 4 in 24..28.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "stream_common.cuh"

namespace moe {
namespace tc {

// ---- TMEM allocation (one warp, .sync.aligned) ----------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- TMEM stores / loads, 32 lanes x 32 bit shape --------------------------
// Thread i of warp w addresses TMEM lane 32 * (w % 4) + i; register j goes to
// column (taddr & 0xffff) + j.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- MMA -------------------------------------------------------------------
// D[tmem] (+)= A[tmem] * B[smem]; issued by one thread.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The 16 MMAs of one 256-wide K stage: A columns at + 8i (i = 0..15), B
// slabs of 64 rows x 128 bytes at descriptor start + (slab_bytes * (i / 4) +
// 32 * (i % 4)) >> 4.  The first MMA overwrites D when `first` is set.
template <int SLAB_BYTES>
__device__ __forceinline__ void mma_ts_stage16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t first) {
#define MOE_MMA_ONE(I)                                                                        \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1 + " #I "*8], bd" #I ", %3, 1;\n\t"
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd<16>;\n\t"
      "setp.eq.b32 p, %4, 0;\n\t"
      "mov.b64 bd0, %2;\n\t"
      "add.s64 bd1, %2, 2;\n\t add.s64 bd2, %2, 4;\n\t add.s64 bd3, %2, 6;\n\t"
      "add.s64 bd4, %2, %5;\n\t add.s64 bd5, bd4, 2;\n\t add.s64 bd6, bd4, 4;\n\t"
      "add.s64 bd7, bd4, 6;\n\t"
      "add.s64 bd8, bd4, %5;\n\t add.s64 bd9, bd8, 2;\n\t add.s64 bd10, bd8, 4;\n\t"
      "add.s64 bd11, bd8, 6;\n\t"
      "add.s64 bd12, bd8, %5;\n\t add.s64 bd13, bd12, 2;\n\t add.s64 bd14, bd12, 4;\n\t"
      "add.s64 bd15, bd12, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd0, %3, p;\n\t"
      MOE_MMA_ONE(1) MOE_MMA_ONE(2) MOE_MMA_ONE(3) MOE_MMA_ONE(4) MOE_MMA_ONE(5)
      MOE_MMA_ONE(6) MOE_MMA_ONE(7) MOE_MMA_ONE(8) MOE_MMA_ONE(9) MOE_MMA_ONE(10)
      MOE_MMA_ONE(11) MOE_MMA_ONE(12) MOE_MMA_ONE(13) MOE_MMA_ONE(14) MOE_MMA_ONE(15)
      "}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(first), "l"(static_cast<uint64_t>(SLAB_BYTES >> 4))
      : "memory");
#undef MOE_MMA_ONE
}

// Arrives once on the mbarrier when every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// f32 accumulator, f16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// K-major operand in the 128-byte swizzled layout: rows of 128 bytes (64
// f16 along K), 8-row atoms of 1024 bytes; start must lie in a 1024-byte
// aligned atom (plus a multiple of 32 bytes to step K by 16 inside it).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused): 16 B
  d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride between 8-row atoms
  d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
  return d;
}

// ---- TMA tensor loads --------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 3-D tensor tile load: box of the map at element coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Same as tma_load_2d, with an L2 eviction-priority policy (createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policies: data read once (evicted first) and data re-read soon (kept).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 32 lanes x 32 bit, 32 columns
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// named barrier among `count` threads
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace tc
}  // namespace moe

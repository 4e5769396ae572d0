// Inline-PTX helpers for the 5th-generation tensor cores of sm_103a (tcgen05: MMA into tensor
// memory, TMEM allocation and loads) and for tiled tensor-map TMA loads.
//
// Operand layout used throughout: K-major tiles in the 128-byte-swizzled canonical layout, i.e.
// rows of 64 bf16 (128 bytes) with the 16-byte chunks of row r XOR-permuted by (r mod 8), 8-row
// groups 1024 bytes apart.  A TMA box of {64 elements, R rows} with 128-byte swizzle writes
// exactly this layout; the tile base must be 1024-byte aligned.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace s2 {

// ------------------------------------------------------------------ TMA (tensor maps)

// Box at element coordinates (x innermost, y) of a 2-D tensor map into shared memory, completion
// counted on `bar` (complete_tx).  x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ dependent launches

// Wait until the grids this one depends on (programmatic stream serialisation) have completed and
// their memory operations are visible; a no-op without such a dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid of the stream to be scheduled (it still waits for this grid in pdl_wait).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ tensor memory

// Whole warp: allocate `ncols` TMEM columns (a power of two >= 32); the base address goes to
// shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// Whole warp (the allocating one).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand starting at byte
// address `addr` (advance by 32 bytes per 16-element K step inside the 128-byte row):
// start address >> 4 in bits 0-13, leading byte offset (unused for this layout) 16 B in bits
// 16-29, stride byte offset 1024 B (between 8-row groups) >> 4 in bits 32-45, descriptor
// version 1 in bits 46-47, swizzle mode 2 (128 bytes) in bits 61-63.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16 (bits 7-9 and
// 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ MMA

// D[tmem] = A·B^T (+ D when accum != 0); issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

// D[tmem] = A·B^T (+ D when accum != 0) with A read from tensor memory at `a_tmem` (row m of the
// 128-row tile in lane m, 32-bit column c holding K elements 2c (low half) and 2c+1 (high half))
// and B from shared memory; issued by one thread.
__device__ __forceinline__ void tc_mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

// `bar` receives one arrival when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Warp-wide: thread t reads TMEM lane (lane base + t), 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-wide: thread t writes TMEM lane (lane base + t), 32 consecutive 32-bit columns, then waits
// until the writes are complete.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ fp8 e4m3 expansion

// Four e4m3 codes (bytes of w, K order from the low byte) as two bf16x2 words, exactly.
// e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is the subnormal range
// m·2^-9.  Moving the 7 magnitude bits to bits 4..10 of a bf16 pattern (sign to bit 15) gives the
// bf16 whose exponent field is the e4m3 one and whose mantissa starts with the e4m3 mantissa, i.e.
// the code's value times 2^-120 for every code (subnormal codes become bf16 subnormals); one bf16x2
// multiply by 2^120 restores the value.  Per half-word with the code b in the low byte:
// b + 15·(b & 0x80) puts the sign at bit 11 and leaves the magnitude in bits 0..6, and << 4 moves
// both into place.
__device__ __forceinline__ uint32_t e4m3x2_pattern(uint32_t x) {
  const uint32_t t = x & 0x00800080u;
  return (x + 15u * t) << 4;
}
__device__ __forceinline__ uint32_t bf16x2_mul_2p120(uint32_t p) {
  uint32_t r;
  // 0x7B80 = 2^120 in bf16; the addend -0 keeps the product's sign and value
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(p), "r"(0x7B807B80u), "r"(0x80008000u));
  return r;
}
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = bf16x2_mul_2p120(e4m3x2_pattern(__byte_perm(w, 0u, 0x4140)));
  hi = bf16x2_mul_2p120(e4m3x2_pattern(__byte_perm(w, 0u, 0x4342)));
}

}  // namespace s2

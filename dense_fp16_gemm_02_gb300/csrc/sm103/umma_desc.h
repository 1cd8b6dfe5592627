// Encoders for the two descriptors a tcgen05.mma reads: the 64-bit shared-
// memory matrix descriptor and the 32-bit instruction descriptor of
// .kind::f16. Plain constexpr functions, compiled for host and device, so
// the host tests can pin them.
//
// Shared-memory descriptor fields (PTX ISA, "Shared memory descriptor" of the
// tcgen05 matrix operands):
//   bits  0–13  start address >> 4
//   bits 16–29  leading-dimension byte offset >> 4 (unused for swizzled
//               K-major operands; set to 1)
//   bits 32–45  stride-dimension byte offset >> 4 (distance between 8-row
//               groups: 1024 B for 128-byte rows)
//   bits 46–48  fixed 0b001
//   bits 49–51  base offset (0: every stage starts on a 1024-byte boundary)
//   bit  52     leading-dimension mode (0: relative offsets)
//   bits 61–63  swizzle mode (0 none, 1 128B with 32B atoms, 2 128B, 4 64B,
//               6 32B)
// "SASS-Level Kernel Generation for Blackwell" (section "Addresses from
// layouts") works one example: a stage of A of 128 rows × 64 fp16, K-major,
// 128-byte swizzle, has the high word 0x40004040.
//
// Instruction descriptor for .kind::f16 (PTX ISA, "Instruction descriptor"):
//   bits 4–5 D format (1 = f32), bits 7–9 A format and 10–12 B format
//   (0 = f16, 1 = bf16), bit 13/14 negate A/B, bit 15/16 A/B major
//   (0 = K-major), bits 17–22 N >> 3, bits 24–28 M >> 4.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define WG_HD __host__ __device__ __forceinline__
#else
#define WG_HD inline
#endif

namespace wg {

enum : uint32_t {
  kSwizzleNone = 0,
  kSwizzle128B = 2,
};

// Descriptor of a K-major operand tile stored as 128-byte rows with the
// 128-byte swizzle, 8-row groups `sbo_bytes` apart, starting at shared-memory
// byte address `smem_addr`.
WG_HD constexpr uint64_t umma_smem_desc_sw128(uint32_t smem_addr, uint32_t sbo_bytes = 1024) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu)            // start address
         | ((uint64_t)1u << 16)                             // LBO (unused) = 1
         | ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32)   // SBO
         | ((uint64_t)1u << 46)                             // fixed 0b001
         | ((uint64_t)kSwizzle128B << 61);                  // 128-byte swizzle
}

// Instruction descriptor: f32 accumulator, A and B both f16 (or both bf16),
// both K-major, shape M × N (K = 16 per instruction for .kind::f16).
WG_HD constexpr uint32_t umma_idesc_f16(uint32_t M, uint32_t N, bool bf16_inputs = false) {
  return (1u << 4)                                  // D = f32
         | ((bf16_inputs ? 1u : 0u) << 7)           // A format
         | ((bf16_inputs ? 1u : 0u) << 10)          // B format
         | (0u << 15) | (0u << 16)                  // both K-major
         | (((N >> 3) & 0x3Fu) << 17)
         | (((M >> 4) & 0x1Fu) << 24);
}

// Byte offset, inside a 128-byte-swizzled K-major tile whose base is
// 1024-byte aligned, of element (row, k) of 2-byte type: the 16-byte chunk
// index (k / 8) is XORed with row mod 8. Used by the host tests to rebuild
// the image a descriptor describes.
WG_HD constexpr uint32_t sw128_offset_f16(uint32_t row, uint32_t k) {
  return row * 128u + ((((k >> 3) ^ (row & 7u)) & 7u) << 4) + (k & 7u) * 2u;
}

}  // namespace wg

// 16-bit-output kernels (C in fp16 or bf16, rounded from the fp32
// accumulator once, data parallel only): single-CTA and 256-column pair
// tiles, the configurations the per-shape choice takes most often.
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesOut16A[] = {
    WG_ENTRY_H("g1_128x256_s4_a2_direct", 1, 1, 256, 4, 2, kEpiDirect, 1, kSchedStatic),
    WG_ENTRY_H("g1_128x128_s6_a2_tma", 1, 1, 128, 6, 2, kEpiTma, 1, kSchedStatic),
    WG_ENTRY_H("g1_128x64_s8_a2_direct", 1, 1, 64, 8, 2, kEpiDirect, 1, kSchedStatic),
    WG_ENTRY_H("g2_256x256_s6_a2_direct", 2, 1, 256, 6, 2, kEpiDirect, 1, kSchedStatic),
    WG_ENTRY_H("g2_256x256_s6_a2_tma", 2, 1, 256, 6, 2, kEpiTma, 1, kSchedStatic),
    WG_ENTRY_H("g2_256x224_s7_a2_direct", 2, 1, 224, 7, 2, kEpiDirect, 1, kSchedStatic),
    WG_ENTRY_H("g2_256x224_s6_a2_tma", 2, 1, 224, 6, 2, kEpiTma, 1, kSchedStatic),
    WG_ENTRY_H("g2_256x192_s8_a2_direct", 2, 1, 192, 8, 2, kEpiDirect, 1, kSchedStatic),
};
const int kNumEntriesOut16A = sizeof(kEntriesOut16A) / sizeof(kEntriesOut16A[0]);

}  // namespace wg

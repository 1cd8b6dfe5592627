// 16-bit-output kernels (C in fp16 or bf16, data parallel only): 512-column
// pair tiles, A multicast across two MMA groups, and cluster launch control.
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesOut16B[] = {
    WG_ENTRY_H("g2_256x128_s8_a2_tma", 2, 1, 128, 8, 2, kEpiTma, 1, kSchedStatic),
    WG_ENTRY_H("g2_512x256_s4_a1_tma", 2, 2, 256, 4, 1, kEpiTma, 1, kSchedStatic),
    WG_ENTRY_H("g2m2_512x256_s6_a2_tma", 2, 1, 256, 6, 2, kEpiTma, 2, kSchedStatic),
    WG_ENTRY_H("g2m2_512x224_s6_a2_tma", 2, 1, 224, 6, 2, kEpiTma, 2, kSchedStatic),
    WG_ENTRY_H("g2_256x256_s6_a2_direct_clc", 2, 1, 256, 6, 2, kEpiDirect, 1, kSchedClc),
    WG_ENTRY_H("g2_512x256_s4_a1_tma_clc", 2, 2, 256, 4, 1, kEpiTma, 1, kSchedClc),
};
const int kNumEntriesOut16B = sizeof(kEntriesOut16B) / sizeof(kEntriesOut16B[0]);

}  // namespace wg

// Kernel configurations whose cluster holds two MMA groups stacked along C's
// rows: the groups need the same rows of B (the MMA's A operand, 16 KB per
// CTA and k-block), so each CTA loads half of its B slice and multicasts it
// to the CTA in the same position of the other group (TMA multicast within
// the cluster; stage releases go to all CTAs). Each CTA then reads 8 KB of B
// per k-block from L2 instead of 16.
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesRowMc[] = {
    WG_ENTRY_MR("g1r2_128x128_s8_a2_direct", 1, 1, 64, 8, 2, kEpiDirect, 2, kSchedStatic),
    WG_ENTRY_MR("g1r2_128x256_s6_a2_direct", 1, 1, 128, 6, 2, kEpiDirect, 2, kSchedStatic),
    WG_ENTRY_X2("g1r2_128x256_s3x2_a2_direct", 1, 1, 128, 3, 2, kEpiDirect, 2),
    WG_ENTRY_X2("g1r2_128x128_s4x2_a2_direct", 1, 1, 64, 4, 2, kEpiDirect, 2),
    WG_ENTRY_MR("g2r2_256x128_s10_a2_direct", 2, 1, 64, 10, 2, kEpiDirect, 2, kSchedStatic),
    WG_ENTRY_MR("g2r2_256x256_s8_a2_direct", 2, 1, 128, 8, 2, kEpiDirect, 2, kSchedStatic),
    WG_ENTRY_MR("g2r2_256x384_s7_a2_direct", 2, 1, 192, 7, 2, kEpiDirect, 2, kSchedStatic),
    WG_ENTRY_MR("g2r2_256x448_s7_a2_direct", 2, 1, 224, 7, 2, kEpiDirect, 2, kSchedStatic),
    WG_ENTRY_MR("g2r2_256x512_s6_a2_direct", 2, 1, 256, 6, 2, kEpiDirect, 2, kSchedStatic),
    WG_ENTRY_MR("g2r2_256x256_s7_a2_tma", 2, 1, 128, 7, 2, kEpiTma, 2, kSchedStatic),
    WG_ENTRY_MR("g2r2_256x448_s6_a2_tma", 2, 1, 224, 6, 2, kEpiTma, 2, kSchedStatic),
    WG_ENTRY_MR("g2r2_256x512_s5_a2_tma", 2, 1, 256, 5, 2, kEpiTma, 2, kSchedStatic),
};
const int kNumEntriesRowMc = sizeof(kEntriesRowMc) / sizeof(kEntriesRowMc[0]);

}  // namespace wg

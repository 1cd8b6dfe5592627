// Kernel configurations with a CTA pair per MMA (tcgen05.mma.cta_group::2,
// M = 256 over two SMs): 256-wide pair tiles (one atom per CTA).
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesPair[] = {
    WG_ENTRY("g2_256x256_s6_a2_tma", 2, 1, 256, 6, 2, kEpiTma),
    WG_ENTRY("g2_256x256_s6_a2_direct", 2, 1, 256, 6, 2, kEpiDirect),
    WG_ENTRY("g2_256x224_s6_a2_tma", 2, 1, 224, 6, 2, kEpiTma),
    WG_ENTRY("g2_256x224_s7_a2_direct", 2, 1, 224, 7, 2, kEpiDirect),
    WG_ENTRY("g2_256x192_s6_a2_tma", 2, 1, 192, 6, 2, kEpiTma),
    WG_ENTRY("g2_256x192_s8_a2_direct", 2, 1, 192, 8, 2, kEpiDirect),
    WG_ENTRY("g2_256x160_s8_a2_direct", 2, 1, 160, 8, 2, kEpiDirect),
    WG_ENTRY("g2_256x128_s8_a2_tma", 2, 1, 128, 8, 2, kEpiTma),
    WG_ENTRY("g2_256x64_s10_a2_direct", 2, 1, 64, 10, 2, kEpiDirect),
    WG_ENTRY_X2("g2_256x64_s5x2_a2_direct", 2, 1, 64, 5, 2, kEpiDirect, 1),
};
const int kNumEntriesPair = sizeof(kEntriesPair) / sizeof(kEntriesPair[0]);

}  // namespace wg

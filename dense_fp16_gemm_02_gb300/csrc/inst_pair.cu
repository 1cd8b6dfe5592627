// Kernel configurations with a CTA pair per MMA (tcgen05.mma.cta_group::2,
// M = 256 over two SMs).
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesPair[] = {
    WG_ENTRY("g2_256x256_s6_a2_tma", 2, 1, 256, 6, 2, kEpiTma),
    WG_ENTRY("g2_256x256_s6_a2_direct", 2, 1, 256, 6, 2, kEpiDirect),
    WG_ENTRY("g2_512x256_s4_a1_tma", 2, 2, 256, 4, 1, kEpiTma),
    WG_ENTRY("g2_512x128_s4_a2_tma", 2, 2, 128, 4, 2, kEpiTma),
    WG_ENTRY("g2_256x128_s8_a2_tma", 2, 1, 128, 8, 2, kEpiTma),
    WG_ENTRY("g2_256x64_s10_a2_direct", 2, 1, 64, 10, 2, kEpiDirect),
};
const int kNumEntriesPair = sizeof(kEntriesPair) / sizeof(kEntriesPair[0]);

}  // namespace wg

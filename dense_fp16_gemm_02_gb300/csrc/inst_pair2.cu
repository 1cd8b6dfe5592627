// Kernel configurations with a CTA pair per MMA and two stacked M = 256 atoms
// per CTA: 512-wide pair tiles.
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesPair2[] = {
    WG_ENTRY("g2_512x256_s4_a1_tma", 2, 2, 256, 4, 1, kEpiTma),
    WG_ENTRY("g2_512x224_s4_a1_tma", 2, 2, 224, 4, 1, kEpiTma),
    WG_ENTRY("g2_512x128_s4_a2_tma", 2, 2, 128, 4, 2, kEpiTma),
};
const int kNumEntriesPair2 = sizeof(kEntriesPair2) / sizeof(kEntriesPair2[0]);

}  // namespace wg

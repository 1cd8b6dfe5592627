// Kernel configurations whose cluster holds two MMA groups side by side along
// C's columns: the groups need the same rows of A, so each CTA loads half of
// its A slice and multicasts it to the CTA in the same position of the other
// group (TMA multicast within the cluster; stage releases go to all CTAs).
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesMulticast[] = {
    WG_ENTRY_MC("g2m2_512x224_s6_a2_tma", 2, 1, 224, 6, 2, kEpiTma, 2),
    WG_ENTRY_MC("g2m2_512x256_s6_a2_tma", 2, 1, 256, 6, 2, kEpiTma, 2),
    WG_ENTRY_MC("g2m2_512x256_s6_a2_direct", 2, 1, 256, 6, 2, kEpiDirect, 2),
    WG_ENTRY_MC("g2m2_1024x256_s4_a1_tma", 2, 2, 256, 4, 1, kEpiTma, 2),
    WG_ENTRY_MC("g1m2_256x256_s4_a2_tma", 1, 1, 256, 4, 2, kEpiTma, 2),
};
const int kNumEntriesMulticast = sizeof(kEntriesMulticast) / sizeof(kEntriesMulticast[0]);

}  // namespace wg

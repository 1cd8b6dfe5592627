// Kernel configurations that take their tiles through cluster launch control:
// one cluster per tile is launched, and a running cluster that finishes a tile
// cancels a cluster that has not launched yet and computes its tile instead
// (tiles in serpentine order within raster groups).
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesClc[] = {
    WG_ENTRY_FULL("g2_256x224_s6_a2_tma_clc", 2, 1, 224, 6, 2, kEpiTma, 1, kSchedClc),
    WG_ENTRY_FULL("g2_256x256_s6_a2_direct_clc", 2, 1, 256, 6, 2, kEpiDirect, 1, kSchedClc),
    WG_ENTRY_FULL("g2_512x256_s4_a1_tma_clc", 2, 2, 256, 4, 1, kEpiTma, 1, kSchedClc),
    WG_ENTRY_FULL("g1_128x256_s4_a2_direct_clc", 1, 1, 256, 4, 2, kEpiDirect, 1, kSchedClc),
};
const int kNumEntriesClc = sizeof(kEntriesClc) / sizeof(kEntriesClc[0]);

}  // namespace wg

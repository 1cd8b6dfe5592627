// Kernel configurations with one CTA per MMA (tcgen05.mma.cta_group::1, M = 128).
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesSingle[] = {
    WG_ENTRY("g1_128x256_s4_a2_tma", 1, 1, 256, 4, 2, kEpiTma),
    WG_ENTRY("g1_128x256_s4_a2_direct", 1, 1, 256, 4, 2, kEpiDirect),
    WG_ENTRY("g1_128x128_s6_a2_tma", 1, 1, 128, 6, 2, kEpiTma),
    WG_ENTRY("g1_128x64_s8_a2_direct", 1, 1, 64, 8, 2, kEpiDirect),
    // Two k-blocks per stage: at N = 64 the MMA thread's per-stage hand-off,
    // not the tensor pipe, paces the k-loop.
    WG_ENTRY_X2("g1_128x64_s4x2_a2_direct", 1, 1, 64, 4, 2, kEpiDirect, 1),
    WG_ENTRY_X2("g1_128x256_s2x2_a2_direct", 1, 1, 256, 2, 2, kEpiDirect, 1),
};
const int kNumEntriesSingle = sizeof(kEntriesSingle) / sizeof(kEntriesSingle[0]);

}  // namespace wg

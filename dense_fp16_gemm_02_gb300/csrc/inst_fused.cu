// Kernels with the alpha/beta/bias epilogue (D = alpha·A·Bᵀ + beta·Cin +
// bias[column]), static data-parallel schedule. The register-store kernels
// ("_ab2", "_ab4") prefetch their Cin blocks (32×32) through a TMA ring per
// epilogue warp of 2 or 4 slots that runs on into the worker's next tile;
// the ring takes shared memory from the stage ring, so these run one or two
// stages fewer than their plain twins. The TMA-epilogue kernels ("_tma_ab1")
// serve the in-place form D += alpha·A·Bᵀ + bias (beta = 1, Cin = D, fp32):
// they add alpha·acc + bias into D with TMA reduce-adds and read no Cin. The
// rule picks among them from measured rates.
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"

namespace wg {

const KernelEntry kEntriesFused[] = {
    // fp32 D (4 KB Cin blocks)
    WG_ENTRY_AB("g2_256x224_s6_a2_direct", 2, 1, 224, 6, 2, 2),
    WG_ENTRY_AB("g2_256x224_s5_a2_direct", 2, 1, 224, 5, 2, 4),
    WG_ENTRY_AB("g2_256x256_s6_a2_direct", 2, 1, 256, 6, 2, 2),
    WG_ENTRY_AB("g2_256x128_s7_a2_direct", 2, 1, 128, 7, 2, 2),
    WG_ENTRY_AB("g1_128x256_s4_a2_direct", 1, 1, 256, 4, 2, 2),
    WG_ENTRY_AB("g1_128x128_s6_a2_direct", 1, 1, 128, 6, 2, 2),
    // fp32 D in place with beta = 1: reduce-adds into D, no Cin ring
    WG_ENTRY_AB_RED("g2_256x224_s6_a2_tma", 2, 1, 224, 6, 2),
    WG_ENTRY_AB_RED("g2_256x256_s6_a2_tma", 2, 1, 256, 6, 2),
    WG_ENTRY_AB_RED("g2_256x128_s8_a2_tma", 2, 1, 128, 8, 2),
    WG_ENTRY_AB_RED("g1_128x256_s4_a2_tma", 1, 1, 256, 4, 2),
    WG_ENTRY_AB_RED("g1_128x128_s6_a2_tma", 1, 1, 128, 6, 2),
    // 16-bit D (2 KB Cin blocks)
    WG_ENTRY_AB_H("g2_256x224_s6_a2_direct", 2, 1, 224, 6, 2, 4),
    WG_ENTRY_AB_H("g2_256x256_s6_a2_direct", 2, 1, 256, 6, 2, 4),
    WG_ENTRY_AB_H("g2_256x128_s7_a2_direct", 2, 1, 128, 7, 2, 4),
    WG_ENTRY_AB_H("g1_128x128_s6_a2_direct", 1, 1, 128, 6, 2, 4),
};
const int kNumEntriesFused = sizeof(kEntriesFused) / sizeof(kEntriesFused[0]);

}  // namespace wg

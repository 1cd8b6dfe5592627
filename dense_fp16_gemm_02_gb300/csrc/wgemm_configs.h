// The table of compiled kernel configurations. Each instantiation unit
// (inst_*.cu) contributes entries; the host library (wgemm_host.cu) picks one
// per call.
#pragma once
#include <stdint.h>

namespace wg {

struct KernelEntry {
  const char* name;
  int cg, reps, bn, stages, acc, epi;
  int tile_rows, tile_cols;  // C rows / columns of one worker tile
  uint32_t smem_bytes;
  const void* func;          // the __global__ function (host stub)
};

// Instantiation units fill these (defined in inst_*.cu).
extern const KernelEntry kEntriesPair[];
extern const int kNumEntriesPair;
extern const KernelEntry kEntriesSingle[];
extern const int kNumEntriesSingle;
extern const KernelEntry kEntriesPair2[];
extern const int kNumEntriesPair2;

}  // namespace wg

// Builds the entry of one configuration (only in .cu files that include the
// kernel template).
#define WG_ENTRY(NAME, CG, REPS, BN, STAGES, ACC, EPI)                                          \
  wg::KernelEntry {                                                                             \
    NAME, CG, REPS, BN, STAGES, ACC, EPI, wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI>::kTileRows,   \
        wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI>::kTileCols,                                     \
        wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI>::kSmemBytes,                                    \
        reinterpret_cast<const void*>(&wg::wgemm_kernel<wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI>>) \
  }

// The table of compiled kernel configurations. Each instantiation unit
// (inst_*.cu) contributes entries; the host library (wgemm_host.cu) picks one
// per call.
#pragma once
#include <stdint.h>

namespace wg {

struct KernelEntry {
  const char* name;
  int cg, reps, bn, stages, acc, epi;
  int mc;                    // MMA groups per cluster side by side along C's columns (sharing A)
  int mr;                    // MMA groups per cluster stacked along C's rows (sharing B)
  int sched;                 // 0: static persistent grid, 1: cluster launch control
  int tile_rows, tile_cols;  // C rows / columns of one worker tile
  int out;                   // 0: fp32 C; 1: 16-bit C (fp16 or bf16), data parallel only
  int fuse;                  // > 0: alpha/beta/bias epilogue (its Cin ring depth), data parallel only
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
extern const KernelEntry kEntriesMulticast[];
extern const int kNumEntriesMulticast;
extern const KernelEntry kEntriesClc[];
extern const int kNumEntriesClc;
extern const KernelEntry kEntriesOut16A[];
extern const int kNumEntriesOut16A;
extern const KernelEntry kEntriesOut16B[];
extern const int kNumEntriesOut16B;
extern const KernelEntry kEntriesFused[];
extern const int kNumEntriesFused;
extern const KernelEntry kEntriesRowMc[];
extern const int kNumEntriesRowMc;

}  // namespace wg

// Builds the entry of one configuration (only in .cu files that include the
// kernel template). MC = MMA groups per cluster side by side along C's
// columns (sharing the A tile), MR = groups stacked along C's rows (sharing
// the B tile); SCHED = kSchedStatic or kSchedClc; OUT = kOut32 or kOut16;
// FUSE = 0 or the Cin ring depth; KPS = k-blocks per stage (1 or 2).
#define WG_ENTRY_GEN(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE, MR, KPS)           \
  wg::KernelEntry {                                                                                 \
    NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, MR, SCHED,                                            \
        wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE, MR, KPS>::kTileRows,          \
        wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE, MR, KPS>::kTileCols, OUT,     \
        FUSE, wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE, MR, KPS>::kSmemBytes,   \
        reinterpret_cast<const void*>(&wg::wgemm_kernel<                                            \
                                      wg::Cfg<CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE, \
                                              MR, KPS>>)                                            \
  }
#define WG_ENTRY_ANY(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE) \
  WG_ENTRY_GEN(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE, 1, 1)
// MR groups stacked along C's rows sharing the B tile (fp32 C).
#define WG_ENTRY_MR(NAME, CG, REPS, BN, STAGES, ACC, EPI, MR, SCHED) \
  WG_ENTRY_GEN(NAME, CG, REPS, BN, STAGES, ACC, EPI, 1, SCHED, wg::kOut32, 0, MR, 1)
// Stages of two k-blocks ("_s<STAGES>x2_"), fp32 C, static schedule.
#define WG_ENTRY_X2(NAME, CG, REPS, BN, STAGES, ACC, EPI, MR) \
  WG_ENTRY_GEN(NAME, CG, REPS, BN, STAGES, ACC, EPI, 1, wg::kSchedStatic, wg::kOut32, 0, MR, 2)
#define WG_ENTRY_OUT(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT) \
  WG_ENTRY_ANY(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, 0)
#define WG_ENTRY_FULL(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED) \
  WG_ENTRY_OUT(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, wg::kOut32)
#define WG_ENTRY_MC(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC) \
  WG_ENTRY_FULL(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, wg::kSchedStatic)
#define WG_ENTRY(NAME, CG, REPS, BN, STAGES, ACC, EPI) \
  WG_ENTRY_FULL(NAME, CG, REPS, BN, STAGES, ACC, EPI, 1, wg::kSchedStatic)
// 16-bit C: the same configuration with "_h" appended to its name.
#define WG_ENTRY_H(NAME, CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED) \
  WG_ENTRY_OUT(NAME "_h", CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, wg::kOut16)
// alpha/beta/bias epilogue (register stores, static schedule) with a Cin
// ring of SLOTS blocks per epilogue warp: "_ab<SLOTS>", and "_ab<SLOTS>_h"
// with a 16-bit C.
#define WG_ENTRY_AB(NAME, CG, REPS, BN, STAGES, ACC, SLOTS) \
  WG_ENTRY_ANY(NAME "_ab" #SLOTS, CG, REPS, BN, STAGES, ACC, wg::kEpiDirect, 1, wg::kSchedStatic, \
               wg::kOut32, SLOTS)
// The in-place form D += alpha·A·Bᵀ + bias (beta = 1, Cin = D, fp32 D) with
// the TMA epilogue: its stores are reduce-adds into D and it reads no Cin.
// "_ab1" after a "_tma" name.
#define WG_ENTRY_AB_RED(NAME, CG, REPS, BN, STAGES, ACC) \
  WG_ENTRY_ANY(NAME "_ab1", CG, REPS, BN, STAGES, ACC, wg::kEpiTma, 1, wg::kSchedStatic, \
               wg::kOut32, 1)
#define WG_ENTRY_AB_H(NAME, CG, REPS, BN, STAGES, ACC, SLOTS) \
  WG_ENTRY_ANY(NAME "_ab" #SLOTS "_h", CG, REPS, BN, STAGES, ACC, wg::kEpiDirect, 1, \
               wg::kSchedStatic, wg::kOut16, SLOTS)

// The GEMM kernel family: one warp-specialised persistent kernel, templated on
// its tile, pair mode, ring depth, accumulator count, epilogue and C element
// width (fp32, or a 16-bit type: fp16 or bf16, chosen at run time). The
// operand type (fp16 or bf16, both the same) is the instruction descriptor's
// and the tensor maps' business alone, so one kernel serves both.
//
// Roles ("SASS-Level Kernel Generation for Blackwell", sections "What a
// Blackwell GEMM is" and "Writing a kernel"), 256 threads per CTA:
//   warp 0     TMA producer: fills the stage ring with tiles of B and A.
//   warp 1     MMA issuer (the pair leader's, for pair MMAs): one thread
//              issues tcgen05.mma into a TMEM accumulator and frees stages
//              with tcgen05.commit. Warp 1 also owns the TMEM allocation.
//   warps 2-3  idle.
//   warps 4-7  epilogue: TMEM → registers → C (direct stores, or a shared-
//              memory staging tile written out by TMA store / reduce-add).
// Hand-offs are mbarrier pipes: stage full / stage empty between producer and
// MMA, accumulator full / accumulator empty between MMA and epilogue.
//
// Operand orientation is "SwapAB" (same page, section "Inside the kernels"):
// the tile of B (rows = columns of C) is the MMA's A operand and the tile of A
// (rows = rows of C) is its B operand. The accumulator is the C block
// transposed: TMEM lane = column of C, TMEM column = row of C, so one warp's
// tcgen05.ld row of 32 lanes is 32 consecutive floats of one row of C.
//
// With CG == 2 one MMA of M = 256 spans the two CTAs of a cluster pair: each
// CTA holds 128 rows of the MMA's A operand (128·REPS columns of C) and half
// of its B operand (BN/2 rows of C); each CTA's TMEM holds its 128 lanes of
// the accumulator for all BN rows of C. The leader (cluster rank 0) issues.
//
// Every wait is bounded: after kWaitTimeoutNs the waiting role records the
// site in the device status word, raises the CTA's abort flag, and returns;
// the CTA then tears down normally (TMEM freed) and exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103/ptx.cuh"
#include "sm103/umma_desc.h"
#include "wgemm_plan.h"

namespace wg {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr int kThreads = 256;
constexpr int kBK = 64;  // K per stage: one 128-byte swizzle row of 16-bit operands

enum EpilogueMode : int { kEpiDirect = 0, kEpiTma = 1 };

// Device status word (one per device, written by the first failing wait).
struct DeviceStatus {
  int32_t code;    // 0 = fine, else a negative WGEMM_ERR_* value
  int32_t block;
  int32_t warp;
  int32_t site;    // role · 16 + barrier kind
  int32_t parity;
  int32_t pad[3];
};

enum WaitSite : int32_t {
  kSiteProducerEmpty = 0x01,
  kSiteProducerTail = 0x02,
  kSiteMmaFull = 0x11,
  kSiteMmaAccEmpty = 0x12,
  kSiteMmaDrain = 0x13,
  kSiteEpiAccFull = 0x21,
  kSiteEpiFlagOwner = 0x22,
  kSiteEpiFlagZero = 0x23,
  kSiteEpiSync = 0x24,
  kSiteEpiCinFull = 0x25,
  // index checks of debug builds
  kCheckPlan = 0x31,
  kCheckTmemMma = 0x32,
  kCheckTmemLd = 0x33,
  kCheckStore = 0x34,
  kCheckStaging = 0x35,
  kCheckFlag = 0x36,
  kCheckZero = 0x37,
  kSiteClcEmpty = 0x41,
  kSiteClcFull = 0x42,
  kSiteAbortLoads = 0x51,
  kSiteAbortClc = 0x52,
  kSiteAbortCin = 0x53,
};

struct KParams {
  CUtensorMap tmA;  // A (M×K fp16 or bf16): the MMA's B operand, box {64, BN/CG}
  CUtensorMap tmB;  // B (N×K, A's type): the MMA's A operand, box {64, 128·REPS}
  CUtensorMap tmC;  // C (M×N, fp32 or 16-bit): box {32, 32}, for the TMA epilogue
  Plan plan;
  void* C;          // fp32 C, or 16-bit C in 16-bit-output kernels
  int64_t ldc;      // in elements
  uint32_t idesc;   // tcgen05.mma instruction descriptor (operand types, M, N)
  int32_t c_bf16;   // 16-bit-output kernels: 1 = bf16, 0 = fp16
  // Fused epilogue (FUSE kernels): D = alpha·acc + beta·Cin + bias[column].
  CUtensorMap tmCin;    // Cin (M×N, C's type): box {32, 32}; read when load_cin
  const float* bias;    // N fp32 values, or null
  float alpha, beta;
  int32_t load_cin;     // 1: read Cin (beta != 0)
  uint32_t* flags;  // split-K / stream-K flags (monotone epochs)
  uint32_t epoch;
  int32_t flag_words;  // words the flag array holds
  DeviceStatus* status;
  uint32_t wait_skew;  // added to the epoch the flag waits expect (0; tests use 1)
  int32_t trace_ctas;  // CTAs the trace buffer holds (trace builds only)
  uint64_t* trace;     // per-CTA event timestamps (trace builds only), else null
};

// Timeline trace (builds with -DWGEMM_TRACE=1): %globaltimer at fixed points
// of each CTA's life, kTraceEvents per CTA, written by one thread per event.
#ifndef WGEMM_TRACE
#define WGEMM_TRACE 0
#endif
enum TraceEvent : int {
  kTrEntry = 0,        // kernel entry (thread 0)
  kTrSetUp = 1,        // after the set-up barrier (thread 0)
  kTrFirstData = 2,    // MMA thread: first stage landed
  kTrLastCommit = 3,   // MMA thread: last accumulator committed
  kTrEpiFirst = 4,     // epilogue warp 4: first accumulator full
  kTrEpiDone = 5,      // epilogue warp 4: last unit written
  kTrExit = 6,         // after the teardown barrier (thread 0)
  kTrUnits = 7,        // number of units this CTA ran (a count, not a time)
  kTraceEvents = 8,
};
__device__ __forceinline__ void trace_event(const KParams& p, int ev, uint64_t value = 0) {
  if (WGEMM_TRACE && p.trace != nullptr && (int32_t)blockIdx.x < p.trace_ctas) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[(size_t)blockIdx.x * kTraceEvents + ev] = ev == kTrUnits ? value : t;
  }
}

constexpr uint32_t pow2_at_least_32(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

enum SchedMode : int { kSchedStatic = 0, kSchedClc = 1 };

enum OutWidth : int { kOut32 = 0, kOut16 = 1 };

template <int CG_, int REPS_, int BN_, int STAGES_, int ACC_, int EPI_, int MC_ = 1,
          int SCHED_ = kSchedStatic, int OUT_ = kOut32, int FUSE_ = 0, int MR_ = 1, int KPS_ = 1>
struct Cfg {
  static constexpr int OUT = OUT_;        // OutWidth: fp32 C, or 16-bit C (data parallel only)
  // FUSE > 0: alpha/beta/bias epilogue (data parallel only). With register
  // stores its Cin ring has FUSE slots per epilogue warp; with the TMA
  // epilogue (fp32 D) it is the in-place form D += alpha·acc + bias, added
  // into D by TMA reduce-adds, with no Cin ring.
  static constexpr int FUSE = FUSE_;
  static constexpr int SCHED = SCHED_;    // SchedMode
  static constexpr int CG = CG_;          // CTAs per MMA: 1, or 2 (pair)
  static constexpr int MC = MC_;          // MMA groups per cluster side by side along C's columns
  static constexpr int MR = MR_;          // MMA groups per cluster stacked along C's rows
  static constexpr int REPS = REPS_;      // stacked MMA atoms per CTA (C columns 128·REPS)
  static constexpr int BN = BN_;          // MMA N = C rows of a tile
  static constexpr int STAGES = STAGES_;  // ring depth
  // k-blocks per stage (1 or 2). With two, a stage's barrier hand-off and
  // MMA commit serve eight MMAs instead of four: where the MMA thread, not
  // the tensor pipe, sets the k-loop's pace (small N), that pace rises.
  static constexpr int KPS = KPS_;
  static constexpr int ACC = ACC_;        // TMEM accumulators
  static constexpr int EPI = EPI_;        // EpilogueMode

  static constexpr int kCtaCols = 128 * REPS;       // C columns per CTA
  static constexpr int kGroupCols = kCtaCols * CG;  // C columns per MMA group (CTA or pair)
  static constexpr int kTileCols = kGroupCols * MC; // C columns per worker (cluster) tile
  static constexpr int kTileRows = BN * MR;         // C rows per worker tile
  static constexpr int kGroups = MC * MR;           // MMA groups per cluster
  static constexpr int kClusterSize = CG * kGroups;
  static constexpr int kArows = 128 * REPS;         // MMA-A rows (of B) per CTA stage
  static constexpr int kBrows = BN / CG;            // MMA-B rows (of A) per CTA stage
  // With MC groups side by side along C's columns, the groups of a cluster
  // need the same rows of A: each CTA loads 1/MC of its A slice and multicasts
  // it to the CTA in the same position of every group.
  static constexpr int kBrowsPart = kBrows / MC;
  // With MR groups stacked along C's rows, the groups need the same rows of
  // B: each CTA loads 1/MR of its B slice and multicasts it the same way.
  static constexpr int kArowsPart = kArows / MR;
  static constexpr uint32_t kAbytes = kArows * 128;
  static constexpr uint32_t kBbytes = kBrows * 128;
  static constexpr uint32_t kKbBytes = kAbytes + kBbytes;  // one k-block of both operands
  static constexpr uint32_t kStageBytes = KPS * kKbBytes;   // k-block q at q · kKbBytes
  static constexpr uint32_t kAccCols = REPS * BN;   // TMEM columns per accumulator
  static constexpr uint32_t kTmemCols = pow2_at_least_32(kAccCols * ACC);
  static constexpr uint32_t kCBytes = OUT == kOut16 ? 2 : 4;  // bytes per C element
  static constexpr uint32_t kEpiSlotBytes = 32 * 32 * kCBytes;  // one 32×32 staging tile
  // TMEM chunks (32 columns each) drained per wait: 4 when storing from
  // registers, 2 when staging through shared memory (one slot per chunk).
  static constexpr int kEpiBatch = EPI == kEpiTma ? (BN / 32 >= 2 ? 2 : 1)
                                                  : (BN / 32 >= 4 ? 4 : BN / 32);
  static constexpr uint32_t kEpiBytes = EPI == kEpiTma ? 4 * kEpiBatch * kEpiSlotBytes : 0;
  // A worker's last unit (static schedule) is drained after every MMA has
  // read its stages, so the stage ring is idle: its TMA epilogue stages
  // through kTailGroups groups of kEpiBatch slots per warp carved from the
  // ring, with that many bulk stores / reduce-adds in flight instead of one.
  static constexpr uint32_t kTailGroupsFit =
      EPI == kEpiTma ? (STAGES * kStageBytes / 4) / (kEpiBatch * kEpiSlotBytes) : 1;
  static constexpr int kTailGroups =
      (EPI == kEpiTma && SCHED == kSchedStatic) ? (kTailGroupsFit < 8 ? (int)kTailGroupsFit : 8)
                                                : 1;
  static constexpr uint32_t kTailWarpBytes = kTailGroups * kEpiBatch * kEpiSlotBytes;
  // Fused epilogue: each epilogue warp prefetches its 32×32 blocks of Cin
  // with TMA into a private ring of kCinSlots slots.
  static constexpr bool kFuseReduce = FUSE > 0 && EPI == kEpiTma;
  static constexpr int kCinSlots = kFuseReduce ? 0 : FUSE;
  static constexpr uint32_t kCinBytes = 4 * kCinSlots * kEpiSlotBytes;

  // Shared-memory layout (offsets from a 1024-byte-aligned base).
  static constexpr uint32_t kOffStages = 0;
  static constexpr uint32_t kOffEpi = STAGES * kStageBytes;
  static constexpr uint32_t kOffCin = kOffEpi + kEpiBytes;
  static constexpr uint32_t kOffBars = kOffCin + kCinBytes;
  // Cluster launch control: a ring of kClcDepth 16-byte responses, each with a
  // full barrier (bytes of the response) and an empty barrier (releases of
  // every consumer in the cluster, gathered in the cluster leader).
  static constexpr int kClcDepth = SCHED == kSchedClc ? 4 : 0;
  static constexpr uint32_t kClcConsumers = kClusterSize * 6 + kGroups;
  static constexpr uint32_t kNumBars = 2 * STAGES + 2 * ACC + 2 + 2 * kClcDepth + 4 * kCinSlots;
  static constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
  static constexpr uint32_t kOffResp = (kOffMisc + 16 + 15) / 16 * 16;
  static constexpr uint32_t kSmemBytes = kOffResp + 16 * kClcDepth + 1024;  // + alignment slack

  // The configurations the host may give a split-K or stream-K plan; every
  // other one runs data-parallel plans only and compiles just that path.
  // With row multicast (MR = 2) a worker is the cluster: both MMA groups walk
  // the same units, so they always need the same k-blocks of B.
  static constexpr bool kKSplit =
      EPI == kEpiTma && SCHED == kSchedStatic && MC == 1 && OUT == kOut32 && FUSE == 0;

  static_assert(CG == 1 || CG == 2, "CG");
  static_assert(OUT == kOut32 || OUT == kOut16, "OUT");
  static_assert(!FUSE || EPI == kEpiDirect || OUT == kOut32,
                "the reduce-add fused epilogue writes fp32 D");
  static_assert(kTailGroups >= 1 && 4 * kTailWarpBytes <= STAGES * kStageBytes,
                "tail staging inside the stage ring");
  static_assert(!FUSE || SCHED == kSchedStatic, "the Cin ring prefetches the next unit");
  static_assert(FUSE >= 0 && FUSE <= 8, "Cin ring depth");
  static_assert(MC == 1 || MC == 2, "MC");
  static_assert(MR == 1 || MR == 2, "MR");
  static_assert(MC == 1 || MR == 1, "one multicast direction per configuration");
  static_assert(kBrowsPart % 8 == 0 && kArowsPart % 8 == 0, "multicast part in 8-row groups");
  static_assert(REPS == 1 || REPS == 2, "REPS");
  static_assert(BN % 32 == 0 && BN % (16 * CG) == 0 && BN >= 32 && BN <= 256, "MMA N");
  static_assert(kBrows % 8 == 0, "operand rows in 8-row groups");
  static_assert(kAccCols * ACC <= 512, "TMEM capacity");
  static_assert(kSmemBytes <= 232448, "shared memory");
  // The MMA thread offsets one descriptor per stage (16-byte units in a
  // 14-bit field): shared-window addresses of the buffer, reserved space and
  // alignment slack included, must stay below 256 KB.
  static_assert(kSmemBytes + 4096 <= (1u << 18), "descriptor address field");
  static_assert(kKbBytes % 1024 == 0, "stage and k-block alignment");
  static_assert(KPS == 1 || KPS == 2, "KPS");
};

// An fp32 accumulator value (its bits) rounded to the 16-bit C type, to
// nearest with ties to even: bf16 or fp16.
__device__ __forceinline__ uint16_t to_c16(uint32_t bits, bool bf16) {
  const float f = __uint_as_float(bits);
  return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f))
              : __half_as_ushort(__float2half_rn(f));
}

// Out of line: it runs only when a wait has given up, and every bounded wait
// site would otherwise carry its own copy (less code ahead of the first loads
// measured faster on small shapes).
static __device__ __noinline__ void record_error(DeviceStatus* st, int32_t code, int32_t site,
                                                 uint32_t parity) {
  if (atomicCAS(&st->code, 0, code) == 0) {
    st->block = (int32_t)blockIdx.x;
    st->warp = (int32_t)(threadIdx.x / 32);
    st->site = site;
    st->parity = (int32_t)parity;
    __threadfence();
  }
}

// Debug builds (-DWGEMM_CHECKED=1) verify every index the kernel derives
// (plan coordinates, TMEM columns, shared-memory offsets, global addresses,
// flag indices) before use; a violation is recorded in the device status word
// (code -9, the site, and the offending value) and the access is skipped.
#ifndef WGEMM_CHECKED
#define WGEMM_CHECKED 0
#endif
#define WG_CHECK(st, cond, site, value)                            \
  (!WGEMM_CHECKED || (cond) ||                                     \
   (record_error((st), -9, (site), (uint32_t)(value)), false))

// Bounded wait for the phase of parity `parity` of `bar`. False on timeout or
// when another role of the CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity,
                                         volatile uint32_t* abort_flag, DeviceStatus* st,
                                         int32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        record_error(st, -5, site, parity);
        return false;
      }
    }
  }
}

// Bounded wait used after an abort: waits for this CTA's own operations in
// flight (copies, responses) to land before the CTA exits, ignoring the
// abort flag; gives up after the same time limit. Out of line: only abort
// paths call it.
static __device__ __noinline__ bool wait_bar_final(uint32_t bar, uint32_t parity,
                                                   DeviceStatus* st, int32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0 && global_timer_ns() - t0 > kWaitTimeoutNs) {
      record_error(st, -5, site, parity);
      return false;
    }
  }
}

// Bounded wait until the flag word has reached `epoch` (monotone, wrap-safe).
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t epoch,
                                          volatile uint32_t* abort_flag, DeviceStatus* st,
                                          int32_t site) {
  if ((int32_t)(ld_acquire_gpu(flag) - epoch) >= 0) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(64);
    if ((int32_t)(ld_acquire_gpu(flag) - epoch) >= 0) return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        record_error(st, -5, site, epoch);
        return false;
      }
    }
  }
}

// Fused epilogue state of one epilogue warp (warp-uniform, except `bias`):
// the current unit's geometry, its Cin blocks, and the ring counters.
struct CinUnit {
  int32_t col_cta, row0;  // the unit's first C column of this CTA, first C row
  int32_t lc;             // chunks (32 rows) of the unit holding rows of C, per atom
  int32_t nblk;           // Cin blocks of this warp in the unit: atoms with columns × lc
};
struct FuseState {
  CinUnit cur, next;      // this unit, and the worker's next unit (nblk 0: none)
  int32_t t;              // next block of the unit to consume
  int32_t cur_issued;     // blocks of this unit issued so far (in order)
  int32_t pre;            // blocks of the next unit issued so far (in order)
  uint32_t issued, consumed;  // Cin loads issued / consumed since kernel start
  float bias[2];          // bias of this lane's column, per atom (0 without bias)
};

template <class K>
struct Kernel {
  // Barrier addresses.
  __device__ static uint32_t bar_full(uint32_t base, int s) { return base + K::kOffBars + 8 * s; }
  __device__ static uint32_t bar_empty(uint32_t base, int s) {
    return base + K::kOffBars + 8 * (K::STAGES + s);
  }
  __device__ static uint32_t bar_accf(uint32_t base, int a) {
    return base + K::kOffBars + 8 * (2 * K::STAGES + a);
  }
  __device__ static uint32_t bar_acce(uint32_t base, int a) {
    return base + K::kOffBars + 8 * (2 * K::STAGES + K::ACC + a);
  }
  __device__ static uint32_t bar_drain(uint32_t base) {
    return base + K::kOffBars + 8 * (2 * K::STAGES + 2 * K::ACC);
  }
  // Rendezvous of the four epilogue warps (arrival count 4).
  __device__ static uint32_t bar_epi(uint32_t base) {
    return base + K::kOffBars + 8 * (2 * K::STAGES + 2 * K::ACC + 1);
  }
  __device__ static uint32_t bar_clc_full(uint32_t base, int j) {
    return base + K::kOffBars + 8 * (2 * K::STAGES + 2 * K::ACC + 2 + j);
  }
  __device__ static uint32_t bar_clc_empty(uint32_t base, int j) {
    return base + K::kOffBars + 8 * (2 * K::STAGES + 2 * K::ACC + 2 + K::kClcDepth + j);
  }
  __device__ static uint32_t clc_resp(uint32_t base, int j) { return base + K::kOffResp + 16 * j; }
  // Fused epilogue: Cin slot s of epilogue warp q, and its full barrier.
  __device__ static uint32_t bar_cin(uint32_t base, uint32_t q, uint32_t s) {
    return base + K::kOffBars +
           8 * (2 * K::STAGES + 2 * K::ACC + 2 + 2 * K::kClcDepth + q * K::kCinSlots + s);
  }
  __device__ static uint32_t cin_slot(uint32_t base, uint32_t q, uint32_t s) {
    return base + K::kOffCin + (q * K::kCinSlots + s) * K::kEpiSlotBytes;
  }

  // Unit i of the worker in the plan (see plan_unit).
  __device__ static bool unit_at(const Plan& plan, int32_t worker, int32_t i, Unit& u) {
    if constexpr (K::kKSplit) return plan_unit(plan, worker, i, u);
    else return plan_unit_dp(plan, worker, i, u);
  }

  // Unit i of this CTA's worker (cluster). Static scheduling: the plan's
  // order. Cluster launch control: unit 0 is the worker's own tile, unit
  // i > 0 is the tile of the cluster that CLC response i−1 cancelled; the
  // response is read once it has landed and then released to the cluster
  // leader (`release`: one thread per consuming role; `warp_wide`: the whole
  // warp reads, then its releasing lane arrives). False when there are no
  // more units (or, with ok = false, when a wait gave up).
  __device__ static bool next_unit(const KParams& p, uint32_t base, int32_t worker, int32_t i,
                                   bool release, bool warp_wide, Unit& u, bool& ok,
                                   volatile uint32_t* abort_flag, int32_t site) {
    if constexpr (K::SCHED == kSchedStatic) {
      return unit_at(p.plan, worker, i, u);
    } else {
      if (i == 0) {
        if (worker >= p.plan.num_tiles) return false;
        plan_tile_unit(p.plan, worker, u);
        return true;
      }
      const int32_t e = i - 1;
      const int j = e % K::kClcDepth;
      const uint32_t ph = (uint32_t)(e / K::kClcDepth) & 1u;
      if (!wait_bar(bar_clc_full(base, j), ph, abort_flag, p.status, site)) {
        ok = false;
        return false;
      }
      uint32_t x = 0;
      const bool got = clc_query(clc_resp(base, j), x);
      if (warp_wide) __syncwarp();
      if (release) mbar_arrive_cluster(mapa_shared(bar_clc_empty(base, j), 0));
      if (!got) return false;
      const int32_t t = (int32_t)(x / K::kClusterSize);
      if (!WG_CHECK(p.status, t >= 0 && t < p.plan.num_tiles, kCheckPlan, t)) {
        ok = false;
        return false;
      }
      plan_tile_unit(p.plan, t, u);
      return true;
    }
  }

  // Cluster launch control scheduler (one thread of warp 2 in every CTA): the
  // cluster leader asks for the next tile by cancelling a cluster that has not
  // launched yet, the response is multicast to every CTA of the cluster, and
  // each CTA's thread accounts the response bytes on its own full barrier.
  // One request is in flight at a time, and none is issued after a failure.
  __device__ static void scheduler(const KParams& p, uint32_t base, uint32_t crank,
                                   volatile uint32_t* abort_flag) {
    for (int32_t e = 0;; ++e) {
      const int j = e % K::kClcDepth;
      const uint32_t ph = (uint32_t)(e / K::kClcDepth) & 1u;
      if (crank == 0) {
        // Every consumer in the cluster has read the slot's previous response.
        if (!wait_bar(bar_clc_empty(base, j), ph ^ 1, abort_flag, p.status, kSiteClcEmpty)) return;
        fence_proxy_async_shared();
        if constexpr (K::kClusterSize > 1) clc_try_cancel_multicast(clc_resp(base, j), bar_clc_full(base, j));
        else clc_try_cancel(clc_resp(base, j), bar_clc_full(base, j));
      }
      mbar_arrive_expect_tx(bar_clc_full(base, j), 16);
      if (!wait_bar(bar_clc_full(base, j), ph, abort_flag, p.status, kSiteClcFull)) {
        // Aborted with a response possibly in flight: let it land here first.
        wait_bar_final(bar_clc_full(base, j), ph, p.status, kSiteAbortClc);
        return;
      }
      uint32_t x;
      const bool got = clc_query(clc_resp(base, j), x);
      mbar_arrive_cluster(mapa_shared(bar_clc_empty(base, j), 0));
      if (!got) return;
    }
  }

  __device__ static uint32_t stage_a(uint32_t base, int s) {
    return base + K::kOffStages + s * K::kStageBytes;
  }
  __device__ static uint32_t stage_b(uint32_t base, int s) {
    return stage_a(base, s) + K::kAbytes;
  }

  __device__ static bool unit_ok(const KParams& p, const Unit& u) {
    return WG_CHECK(p.status, u.tm >= 0 && u.tm < p.plan.tiles_m, kCheckPlan, u.tm) &&
           WG_CHECK(p.status, u.tn >= 0 && u.tn < p.plan.tiles_n, kCheckPlan, u.tn) &&
           WG_CHECK(p.status, u.kb_begin >= 0 && u.kb_begin < u.kb_end && u.kb_end <= p.plan.kblocks,
                    kCheckPlan, u.kb_end) &&
           WG_CHECK(p.status, u.tile >= 0 && u.tile < p.plan.num_tiles, kCheckPlan, u.tile);
  }

  // ------------------------------------------------------------ producer
  // CTA position in its cluster: `rank` within the MMA group (0 = the group's
  // leader, which issues the MMAs), `grp` = the group's index in the cluster.
  __device__ static uint32_t group_leader(uint32_t grp) { return grp * K::CG; }
  __device__ static uint16_t same_rank_mask(uint32_t rank) {
    uint16_t m = 0;
#pragma unroll
    for (int q = 0; q < K::kGroups; ++q) m |= (uint16_t)(1u << (q * K::CG + rank));
    return m;
  }
  // The group's position along C's columns and along C's rows.
  __device__ static int32_t col_group(uint32_t grp) { return K::MR == 1 ? (int32_t)grp : 0; }
  __device__ static int32_t row_group(uint32_t grp) { return K::MR == 1 ? 0 : (int32_t)grp; }
  __device__ static uint16_t group_mask(uint32_t grp) {
    return (uint16_t)(((1u << K::CG) - 1u) << (grp * K::CG));
  }

  // Loads k-block `kb` of a unit into k-block slot q of stage s (the stage's
  // bytes are accounted once, by load_stage).
  __device__ static void load_kb(const KParams& p, uint32_t base, uint32_t s, uint32_t q,
                                 int32_t kb, int32_t b_row0, int32_t a_row0, uint32_t rank,
                                 uint32_t grp) {
    const uint32_t full = bar_full(base, s);
    const uint32_t sa = stage_a(base, s) + q * K::kKbBytes, sb = sa + K::kAbytes;
    const uint32_t a_dst = sb + grp * K::kBrowsPart * 128;
    if constexpr (K::MR > 1) {
      // Part grp of the B slice goes to this rank of every group; the A rows
      // are this CTA's own. b_row0 is the slice's first row.
      const uint32_t b_dst = sa + grp * K::kArowsPart * 128;
      const int32_t b_part = b_row0 + (int32_t)grp * K::kArowsPart;
      if constexpr (K::CG == 1) {
        tma_load_2d_multicast(b_dst, &p.tmB, full, kb * kBK, b_part, same_rank_mask(rank));
        tma_load_2d(sb, &p.tmA, full, kb * kBK, a_row0);
      } else {
        const uint32_t full_leader = mapa_shared(full, group_leader(grp));
        tma_load_2d_pair_multicast(b_dst, &p.tmB, full_leader, kb * kBK, b_part,
                                   same_rank_mask(rank));
        tma_load_2d_pair(sb, &p.tmA, full_leader, kb * kBK, a_row0);
      }
      return;
    }
    if constexpr (K::kKSplit) {
      // K-split plans: each k-block of an operand has few readers, and C's
      // lines, zeroed or stored early and reduce-added at the end, must stay
      // in L2 meanwhile: the operand loads are marked evict-first.
      if (p.plan.mode != kDataParallel) {
        const uint64_t pol = l2_policy_evict_first();
        if constexpr (K::CG == 1) {
          tma_load_2d_hint(sa, &p.tmB, full, kb * kBK, b_row0, pol);
          tma_load_2d_hint(a_dst, &p.tmA, full, kb * kBK, a_row0, pol);
        } else {
          const uint32_t full_leader = mapa_shared(full, group_leader(grp));
          tma_load_2d_pair_hint(sa, &p.tmB, full_leader, kb * kBK, b_row0, pol);
          tma_load_2d_pair_hint(a_dst, &p.tmA, full_leader, kb * kBK, a_row0, pol);
        }
        return;
      }
    }
    if constexpr (K::CG == 1) {
      tma_load_2d(sa, &p.tmB, full, kb * kBK, b_row0);
      if constexpr (K::MC == 1)
        tma_load_2d(a_dst, &p.tmA, full, kb * kBK, a_row0);
      else
        tma_load_2d_multicast(a_dst, &p.tmA, full, kb * kBK, a_row0, same_rank_mask(rank));
    } else {
      // Every byte that lands in either CTA of a pair is counted on the
      // pair leader's full barrier.
      const uint32_t full_leader = mapa_shared(full, group_leader(grp));
      tma_load_2d_pair(sa, &p.tmB, full_leader, kb * kBK, b_row0);
      if constexpr (K::MC == 1)
        tma_load_2d_pair(a_dst, &p.tmA, full_leader, kb * kBK, a_row0);
      else
        tma_load_2d_pair_multicast(a_dst, &p.tmA, full_leader, kb * kBK, a_row0,
                                   same_rank_mask(rank));
    }
  }

  // Loads k-blocks kb0 .. kb0 + nk − 1 (nk <= KPS) of a unit into stage s: one
  // arrival on the stage's full barrier counts the bytes of all of them (in
  // a pair, both CTAs' bytes, on the leader's barrier), then each k-block's
  // loads.
  __device__ static void load_stage(const KParams& p, uint32_t base, uint32_t s, int32_t kb0,
                                    int32_t nk, int32_t b_row0, int32_t a_row0, uint32_t rank,
                                    uint32_t grp) {
    if (K::CG == 1 || rank == 0)
      mbar_arrive_expect_tx(bar_full(base, s), (uint32_t)nk * K::kKbBytes * (uint32_t)K::CG);
    for (int32_t q = 0; q < nk; ++q)
      load_kb(p, base, s, (uint32_t)q, kb0 + q, b_row0, a_row0, rank, grp);
  }

  // Kernels without a cluster start filling the ring as soon as the barriers
  // exist, before the CTA-wide set-up barrier and the TMEM allocation: the
  // thread that initialised the barriers loads the first unit's first
  // min(STAGES, k-blocks) stages (all empty at that point) and returns how
  // many. (Doing the same for a pair's leader measured no gain.)
  __device__ static uint32_t prefill(const KParams& p, uint32_t base, int32_t worker,
                                     uint32_t rank, uint32_t grp) {
    if constexpr (K::kClusterSize != 1) {
      return 0;
    } else {
      Unit u;
      bool have;
      if constexpr (K::SCHED == kSchedClc) {
        have = worker < p.plan.num_tiles;
        if (have) plan_tile_unit(p.plan, worker, u);
      } else {
        have = unit_at(p.plan, worker, 0, u);
      }
      if (!have || !unit_ok(p, u)) return 0;
      const int32_t b_row0 = u.tn * K::kTileCols + (int32_t)rank * K::kCtaCols;
      const int32_t a_row0 = u.tm * K::kTileRows + (int32_t)rank * K::kBrows;
      uint32_t n = 0;
      for (int32_t kb = u.kb_begin; kb < u.kb_end && n < (uint32_t)K::STAGES; kb += K::KPS, ++n)
        load_stage(p, base, n, kb, min(K::KPS, u.kb_end - kb), b_row0, a_row0, rank, grp);
      return n;
    }
  }

  __device__ static void producer(const KParams& p, uint32_t base, uint32_t rank, uint32_t grp,
                                  int32_t worker, uint32_t prefilled,
                                  volatile uint32_t* abort_flag) {
    // The first `prefilled` stages of unit 0 were loaded before set-up.
    uint32_t s = prefilled % (uint32_t)K::STAGES, ph = prefilled / (uint32_t)K::STAGES;
    uint32_t fills = prefilled;  // stages filled so far
    bool ok = true;
    for (int32_t i = 0; ok; ++i) {
      Unit u;
      if (!next_unit(p, base, worker, i, true, false, u, ok, abort_flag, kSiteClcFull)) break;
      if (!unit_ok(p, u)) { ok = false; break; }
      const int32_t b_row0 = u.tn * K::kTileCols + col_group(grp) * K::kGroupCols +
                             (int32_t)rank * K::kCtaCols;                     // rows of B
      const int32_t a_row0 = u.tm * K::kTileRows + row_group(grp) * K::BN +
                             (int32_t)rank * K::kBrows +
                             (K::MC > 1 ? (int32_t)grp * K::kBrowsPart : 0);  // rows of A
      // Stages of KPS k-blocks from the unit's start (the last one may be
      // short); unit 0's first `prefilled` stages are already loaded.
      const int32_t kb_first =
          i == 0 ? min(u.kb_end, u.kb_begin + (int32_t)prefilled * K::KPS) : u.kb_begin;
      for (int32_t kb = kb_first; kb < u.kb_end; kb += K::KPS) {
        if (!wait_bar(bar_empty(base, s), ph ^ 1, abort_flag, p.status, kSiteProducerEmpty)) {
          ok = false;
          break;
        }
        load_stage(p, base, s, kb, min(K::KPS, u.kb_end - kb), b_row0, a_row0, rank, grp);
        ++fills;
        if (++s == (uint32_t)K::STAGES) { s = 0; ph ^= 1; }
      }
    }
    if (ok) {
      // Tail: wait until the MMA has released every stage this CTA filled, so
      // that no commit aimed at this CTA's barriers is still in flight at exit.
      for (int j = 0; j < K::STAGES; ++j) {
        if (!wait_bar(bar_empty(base, s), ph ^ 1, abort_flag, p.status, kSiteProducerTail)) break;
        if (++s == (uint32_t)K::STAGES) { s = 0; ph ^= 1; }
      }
    } else if (rank == 0) {
      // Aborted: let the loads already issued land before the CTA (and, in a
      // pair, its peer, which waits at the final cluster barrier) can exit.
      // The leader's full barrier counts the bytes of both CTAs of the pair.
      for (uint32_t x = 0; x < (uint32_t)K::STAGES && x < fills; ++x) {
        const uint32_t last = x + (uint32_t)K::STAGES * ((fills - 1 - x) / (uint32_t)K::STAGES);
        wait_bar_final(bar_full(base, x), (last / (uint32_t)K::STAGES) & 1u, p.status,
                       kSiteAbortLoads);
      }
    }
  }

  // ------------------------------------------------------------ MMA issuer
  __device__ static void mma(const KParams& p, uint32_t base, uint32_t tmem, uint32_t grp,
                             int32_t worker, volatile uint32_t* abort_flag) {
    // A stage is free once every group of the cluster has read it (other
    // groups' multicasts write into it), so its release goes to all CTAs.
    constexpr uint16_t kAllCtas = (uint16_t)((1u << K::kClusterSize) - 1u);
    const uint16_t own = group_mask(grp);
    const uint32_t idesc = p.idesc;
    uint32_t s = 0, ph = 0, ab = 0, aph = 0;
    bool ok = true;
    for (int32_t i = 0; ok; ++i) {
      Unit u;
      if (!next_unit(p, base, worker, i, true, false, u, ok, abort_flag, kSiteClcFull)) break;
      if (!wait_bar(bar_acce(base, ab), aph ^ 1, abort_flag, p.status, kSiteMmaAccEmpty)) {
        ok = false;
        break;
      }
      tcgen05_fence_after();
      const uint32_t d = tmem + ab * K::kAccCols;
      if (!unit_ok(p, u) ||
          !WG_CHECK(p.status, (ab + 1) * K::kAccCols <= K::kTmemCols, kCheckTmemMma, ab)) {
        ok = false;
        break;
      }
      for (int32_t kb = u.kb_begin; kb < u.kb_end; kb += K::KPS) {
        if (!wait_bar(bar_full(base, s), ph, abort_flag, p.status, kSiteMmaFull)) {
          ok = false;
          break;
        }
        if (WGEMM_TRACE && i == 0 && kb == u.kb_begin) trace_event(p, kTrFirstData);
        tcgen05_fence_after();
        // The stage's k-blocks (the same split as the producer's).
        const int32_t nk = min(K::KPS, u.kb_end - kb);
        // One descriptor for the stage; every operand slice of it lies a
        // constant number of 16-byte units further. The stage starts
        // 1024-byte aligned and all of shared memory lies below 256 KB, so
        // the descriptor's 14-bit address field never carries into the
        // fields above it (host test: `wgemm_debug_smem_desc` offsets).
        const uint64_t desc0 = umma_smem_desc_sw128(stage_a(base, s));
#pragma unroll
        for (int32_t q = 0; q < K::KPS; ++q) {
          if (q >= nk) break;
#pragma unroll
          for (int r = 0; r < K::REPS; ++r) {
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j) {
              const uint32_t a_off = (uint32_t)q * K::kKbBytes + r * 128 * 128 + j * 32;
              const uint32_t b_off = (uint32_t)q * K::kKbBytes + K::kAbytes + j * 32;
              umma_f16<K::CG>(d + r * K::BN, desc0 + (a_off >> 4), desc0 + (b_off >> 4), idesc,
                              (kb + q > u.kb_begin || j > 0) ? 1u : 0u);
            }
          }
        }
        if constexpr (K::kClusterSize == 1) umma_commit(bar_empty(base, s));
        else if constexpr (K::CG == 1) umma_commit_multicast(bar_empty(base, s), kAllCtas);
        else umma_commit_pair_multicast(bar_empty(base, s), kAllCtas);
        if (++s == (uint32_t)K::STAGES) { s = 0; ph ^= 1; }
      }
      if (!ok) break;
      if constexpr (K::CG == 1) umma_commit(bar_accf(base, ab));
      else umma_commit_pair_multicast(bar_accf(base, ab), own);
      if (WGEMM_TRACE) trace_event(p, kTrLastCommit);
      if (++ab == (uint32_t)K::ACC) { ab = 0; aph ^= 1; }
    }
    if (!ok) {
      // Let the MMAs already issued finish before TMEM is freed.
      if constexpr (K::CG == 1) umma_commit(bar_drain(base));
      else umma_commit_pair_multicast(bar_drain(base), own);
      wait_bar(bar_drain(base), 0, abort_flag, p.status, kSiteMmaDrain);
    }
  }

  // Bounded rendezvous of the four epilogue warps: every lane's earlier
  // memory operations happen before every lane's later ones.
  __device__ static bool epi_sync(uint32_t base, uint32_t& phase, volatile uint32_t* abort_flag,
                                  DeviceStatus* st) {
    __syncwarp();
    if (lane_id() == 0) mbar_arrive(bar_epi(base));
    const bool ok = wait_bar(bar_epi(base), phase, abort_flag, st, kSiteEpiSync);
    phase ^= 1;
    __syncwarp();
    return ok;
  }

  // One batch of the epilogue: chunks [c0, c0 + NBB) of one atom of the
  // accumulator (TMEM columns from `tatom`) go to C rows row0 + 32·c0 ...,
  // columns col_warp + lane. Chunks wholly outside C are skipped. When
  // `release` is set the accumulator is handed back to the MMA warp once the
  // batch's TMEM reads are complete.
  // Fused epilogue, lane 0: load Cin block t of unit `g` (atom t / lc, chunk
  // t % lc) of epilogue warp q into the next ring slot.
  __device__ static void cin_issue(const KParams& p, uint32_t base, uint32_t q, const CinUnit& g,
                                   uint32_t issued, int32_t t) {
    const int32_t r = t / g.lc, c = t - r * g.lc;
    const uint32_t slot = issued % (uint32_t)K::kCinSlots;
    const uint32_t bar = bar_cin(base, q, slot);
    mbar_arrive_expect_tx(bar, K::kEpiSlotBytes);
    tma_load_2d(cin_slot(base, q, slot), &p.tmCin, bar, g.col_cta + r * 128 + (int32_t)q * 32,
                g.row0 + 32 * c);
  }

  // The Cin geometry of unit i of `worker` for epilogue warp q (nblk = 0 when
  // the worker has no unit i).
  __device__ static CinUnit cin_unit(const KParams& p, uint32_t q, uint32_t rank, uint32_t grp,
                                     int32_t worker, int32_t i) {
    CinUnit g{0, 0, 0, 0};
    Unit u;
    if (!unit_at(p.plan, worker, i, u)) return g;
    const int32_t M = p.plan.M, N = p.plan.N;
    constexpr int kChunks = K::BN / 32;
    g.col_cta = u.tn * K::kTileCols + col_group(grp) * K::kGroupCols + (int32_t)rank * K::kCtaCols;
    g.row0 = u.tm * K::kTileRows + row_group(grp) * K::BN;
    const int32_t rows = M - g.row0;
    g.lc = rows <= 0 ? 0 : ((rows + 31) / 32 < kChunks ? (rows + 31) / 32 : kChunks);
    int32_t atoms = 0;
#pragma unroll
    for (int r = 0; r < K::REPS; ++r)
      if (g.col_cta + r * 128 + (int32_t)q * 32 < N) atoms = r + 1;
    g.nblk = atoms * g.lc;
    return g;
  }

  // Fused epilogue, at the start of unit i (before its accumulator is full):
  // this lane's bias, the next unit's geometry, and the unit's first Cin
  // loads (those the previous unit did not already issue).
  __device__ static void fuse_begin(const KParams& p, uint32_t base, uint32_t q, uint32_t rank,
                                    uint32_t grp, int32_t worker, int32_t i, FuseState& f) {
    const uint32_t lane = threadIdx.x % 32;
    const int32_t N = p.plan.N;
    f.cur = i == 0 ? cin_unit(p, q, rank, grp, worker, 0) : f.next;
    f.next = cin_unit(p, q, rank, grp, worker, i + 1);
#pragma unroll
    for (int r = 0; r < K::REPS; ++r) {
      const int32_t col = f.cur.col_cta + r * 128 + (int32_t)q * 32 + (int32_t)lane;
      f.bias[r] = (p.bias != nullptr && col < N) ? p.bias[col] : 0.f;
    }
    f.t = 0;
    f.cur_issued = i == 0 ? 0 : f.pre;  // issued while the previous unit drained
    f.pre = 0;
    // The reduce-add form reads no Cin: D's old values are added in L2.
    if constexpr (K::kCinSlots > 0) {
      if (!p.load_cin) return;
      // The slots were last read by this warp's generic loads: order those
      // reads before the TMA writes that refill them.
      fence_proxy_async_shared();
      __syncwarp();
      // Fill the ring: at most kCinSlots loads in flight.
      while (f.cur_issued < f.cur.nblk && f.issued - f.consumed < (uint32_t)K::kCinSlots) {
        if (lane == 0) cin_issue(p, base, q, f.cur, f.issued, f.cur_issued);
        ++f.issued;
        ++f.cur_issued;
      }
    }
  }

  // Fused epilogue: turn the accumulator values of chunks [c0, c0 + nb) of
  // atom r into alpha·acc + beta·Cin + bias, consuming the Cin blocks in
  // ring order and refilling each slot with the block kCinSlots ahead (of
  // this unit, else of the next one). False if a wait gave up.
  template <int NBB>
  __device__ static bool fuse_apply(const KParams& p, uint32_t base, uint8_t* smem, uint32_t q,
                                    int r, int c0, int nb, uint32_t (&v)[NBB][32], FuseState& f,
                                    volatile uint32_t* abort_flag) {
    const uint32_t lane = threadIdx.x % 32;
    const float alpha = p.alpha, beta = p.beta, bias = f.bias[r];
#pragma unroll
    for (int b = 0; b < NBB; ++b) {
      if (b >= nb) break;
      const int32_t c = c0 + b;
      if (c >= f.cur.lc) break;  // rows past M: nothing of this chunk is stored
      bool with_cin = false;
      if constexpr (K::kCinSlots > 0) with_cin = p.load_cin != 0;
      if (with_cin) {
        if constexpr (K::kCinSlots > 0) {
          const uint32_t slot = f.consumed % (uint32_t)K::kCinSlots;
          if (!wait_bar(bar_cin(base, q, slot), (f.consumed / (uint32_t)K::kCinSlots) & 1u,
                        abort_flag, p.status, kSiteEpiCinFull))
            return false;
          const uint8_t* sp = smem + (cin_slot(base, q, slot) - base);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float cin;
            if constexpr (K::OUT == kOut16) {
              const uint16_t h = reinterpret_cast<const uint16_t*>(sp)[e * 32 + lane];
              cin = p.c_bf16 ? __bfloat162float(__ushort_as_bfloat16(h))
                             : __half2float(__ushort_as_half(h));
            } else {
              cin = reinterpret_cast<const float*>(sp)[e * 32 + lane];
            }
            v[b][e] = __float_as_uint(fmaf(alpha, __uint_as_float(v[b][e]), fmaf(beta, cin, bias)));
          }
          ++f.consumed;
          fence_proxy_async_shared();
          __syncwarp();
          // The freed slot takes the next block in consumption order: this
          // unit's, else the next unit's.
          if (f.cur_issued < f.cur.nblk) {
            if (lane == 0) cin_issue(p, base, q, f.cur, f.issued, f.cur_issued);
            ++f.issued;
            ++f.cur_issued;
          } else if (f.pre < f.next.nblk) {
            if (lane == 0) cin_issue(p, base, q, f.next, f.issued, f.pre);
            ++f.issued;
            ++f.pre;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          v[b][e] = __float_as_uint(fmaf(alpha, __uint_as_float(v[b][e]), bias));
      }
      ++f.t;
    }
    return true;
  }

  // WAITN: bulk groups (batches) that may still be reading staging slots
  // when this batch's slots are written: 0 with the two per-warp slots,
  // kTailGroups - 1 when staging rotates through the idle stage ring.
  template <int NBB, int WAITN>
  __device__ static bool drain(const KParams& p, uint32_t base, uint8_t* smem, uint32_t tmem,
                               uint32_t tatom, int c0, int nb, int32_t col_warp, int32_t row0,
                               bool add, uint32_t stage_base, bool release, uint32_t ab,
                               uint32_t grp, int r, FuseState& fs,
                               volatile uint32_t* abort_flag) {
    const uint32_t lane = threadIdx.x % 32;
    const int32_t M = p.plan.M, N = p.plan.N;
    const int64_t ldc = p.ldc;
    bool live = col_warp < N && row0 + c0 * 32 < M;  // warp-uniform
    live = live && WG_CHECK(p.status,
                            (tatom & 0xFFFFu) - (tmem & 0xFFFFu) + (c0 + nb) * 32u <= K::kTmemCols,
                            kCheckTmemLd, tatom);
    uint32_t v[NBB][32];
    // tcgen05.ld / wait::ld are .sync.aligned: the whole warp must execute
    // them together, so reconverge after any lane-divergent stores before.
    __syncwarp();
    if (live) {
#pragma unroll
      for (int b = 0; b < NBB; ++b)
        if (b < nb) tmem_ld_32x32b_x32(tatom + (c0 + b) * 32, v[b]);
      tmem_ld_wait();
    }
    if (release) {
      tcgen05_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (K::CG == 1) mbar_arrive(bar_acce(base, ab));
        else mbar_arrive_cluster(mapa_shared(bar_acce(base, ab), group_leader(grp)));
      }
    }
    if (!live) return true;
    if constexpr (K::FUSE) {
      if (!fuse_apply<NBB>(p, base, smem, (threadIdx.x / 32) & 3u, r, c0, nb, v, fs, abort_flag))
        return false;
    }
    if constexpr (K::EPI == kEpiDirect && K::OUT == kOut16) {
      const int32_t col = col_warp + (int32_t)lane;
      if (col < N) {
        const bool bf = p.c_bf16 != 0;
#pragma unroll
        for (int b = 0; b < NBB; ++b) {
          if (b >= nb) break;
          const int32_t row_c = row0 + (c0 + b) * 32;
          uint16_t* dst = static_cast<uint16_t*>(p.C) + (int64_t)row_c * ldc + col;
          if (WGEMM_CHECKED) {
            for (int e = 0; e < 32; ++e) {
              const int64_t off = (int64_t)(row_c + e) * ldc + col;
              if (row_c + e < M &&
                  WG_CHECK(p.status, col >= 0 && off >= 0 && off < (int64_t)(M - 1) * ldc + N,
                           kCheckStore, off))
                dst[e * ldc] = to_c16(v[b][e], bf);
            }
          } else if (row_c + 32 <= M) {
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[e * ldc] = to_c16(v[b][e], bf);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (row_c + e < M) dst[e * ldc] = to_c16(v[b][e], bf);
          }
        }
      }
      __syncwarp();
    } else if constexpr (K::EPI == kEpiDirect) {
      const int32_t col = col_warp + (int32_t)lane;
      if (col < N) {
#pragma unroll
        for (int b = 0; b < NBB; ++b) {
          if (b >= nb) break;
          const int32_t row_c = row0 + (c0 + b) * 32;
          float* dst = static_cast<float*>(p.C) + (int64_t)row_c * ldc + col;
          if (WGEMM_CHECKED) {
            for (int e = 0; e < 32; ++e) {
              const int64_t off = (int64_t)(row_c + e) * ldc + col;
              if (row_c + e < M &&
                  WG_CHECK(p.status, col >= 0 && off >= 0 && off < (int64_t)(M - 1) * ldc + N,
                           kCheckStore, off))
                dst[e * ldc] = __uint_as_float(v[b][e]);
            }
          } else if (row_c + 32 <= M) {
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[e * ldc] = __uint_as_float(v[b][e]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (row_c + e < M) dst[e * ldc] = __uint_as_float(v[b][e]);
          }
        }
      }
      __syncwarp();
    } else {
      // Stage each 32 rows × 32 columns block row-major (one slot per chunk,
      // reused once the previous batch's stores have read it), then one lane
      // writes them out with TMA stores or reduce-adds; TMA clips what lies
      // outside M × N.
      const uint32_t soff = stage_base - base;
      if (!WG_CHECK(p.status,
                    (soff >= K::kOffEpi && soff + nb * K::kEpiSlotBytes <= K::kOffBars) ||
                        (WAITN > 0 && soff + nb * K::kEpiSlotBytes <=
                                          (uint32_t)K::STAGES * K::kStageBytes),
                    kCheckStaging, soff))
        return true;
      if (lane == 0) bulk_wait_group_read<WAITN>();
      __syncwarp();
#pragma unroll
      for (int b = 0; b < NBB; ++b) {
        if (b >= nb) break;
        if constexpr (K::OUT == kOut16) {
          const bool bf = p.c_bf16 != 0;
          uint16_t* sp =
              reinterpret_cast<uint16_t*>(smem + (stage_base - base) + b * K::kEpiSlotBytes);
#pragma unroll
          for (int e = 0; e < 32; ++e) sp[e * 32 + lane] = to_c16(v[b][e], bf);
        } else {
          float* sp = reinterpret_cast<float*>(smem + (stage_base - base) + b * K::kEpiSlotBytes);
#pragma unroll
          for (int e = 0; e < 32; ++e) sp[e * 32 + lane] = __uint_as_float(v[b][e]);
        }
      }
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int b = 0; b < NBB; ++b) {
          if (b >= nb) break;
          const uint32_t sbuf = stage_base + b * K::kEpiSlotBytes;
          const int32_t row_c = row0 + (c0 + b) * 32;
          // 16-bit C is written by data-parallel units only: partial sums
          // are never rounded to 16 bits before they are added.
          // K-split partial sums, and the in-place fused form, add into C.
          if ((K::kKSplit && add) || K::kFuseReduce) tma_reduce_add_2d(&p.tmC, sbuf, col_warp, row_c);
          else tma_store_2d(&p.tmC, sbuf, col_warp, row_c);
        }
        bulk_commit_group();
      }
    }
    return true;
  }

  // ------------------------------------------------------------ epilogue
  // 128 threads (warps 4..7); warp q = warp % 4 reads TMEM lanes 32q..32q+31.
  __device__ static void epilogue(const KParams& p, uint32_t base, uint8_t* smem, uint32_t tmem,
                                  uint32_t rank, uint32_t grp, int32_t worker,
                                  volatile uint32_t* abort_flag) {
    const uint32_t crank = grp * K::CG + rank;  // rank in the cluster
    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t q = warp & 3;
    bool ok = true;
    uint32_t sync_phase = 0;

    if constexpr (K::kKSplit) {
      if (p.plan.mode == kSplitK || p.plan.zero_first)
        ok = zero_slices(p, base, rank, grp, worker, sync_phase, abort_flag);
    }

    uint32_t ab = 0, aph = 0;
    const uint32_t stage_base = base + K::kOffEpi + q * K::kEpiBatch * K::kEpiSlotBytes;
    const uint32_t tail_base = base + K::kOffStages + q * K::kTailWarpBytes;
    FuseState fs{};
    for (int32_t i = 0; ok; ++i) {
      Unit u;
      bool got = next_unit(p, base, worker, i, lane == 0, true, u, ok, abort_flag, kSiteClcFull);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!got || !ok) break;
      if constexpr (K::FUSE) {
        // Start this unit's Cin loads before its accumulator is full.
        fuse_begin(p, base, q, rank, grp, worker, i, fs);
      }
      if (!wait_bar(bar_accf(base, ab), aph, abort_flag, p.status, kSiteEpiAccFull)) {
        ok = false;
        break;
      }
      __syncwarp();
      if (WGEMM_TRACE && i == 0 && threadIdx.x == 128) trace_event(p, kTrEpiFirst);
      tcgen05_fence_after();
      if (!unit_ok(p, u)) { ok = false; break; }
      const int32_t col_cta =
          u.tn * K::kTileCols + col_group(grp) * K::kGroupCols + (int32_t)rank * K::kCtaCols;
      const int32_t row0 = u.tm * K::kTileRows + row_group(grp) * K::BN;
      // Only K-split units add into C (data-parallel units store).
      const bool add = K::kKSplit && (u.kind == kUnitAddAfterOwner || u.kind == kUnitAddAfterZero ||
                                      u.kind == kUnitAddAfterZeroed);
      if constexpr (K::kKSplit) {
        if (add) {
          if (u.kind == kUnitAddAfterOwner) {
            if (lane == 0)
              ok = WG_CHECK(p.status, (int32_t)(u.tile * K::kClusterSize + crank) < p.flag_words,
                            kCheckFlag, u.tile) &&
                   wait_flag(p.flags + (u.tile * K::kClusterSize + crank), p.epoch + p.wait_skew,
                             abort_flag, p.status, kSiteEpiFlagOwner);
          } else {
            // Every slice's zeroing flag of the tile, one lane per flag, so the
            // acquire loads' round trips overlap instead of adding up.
            const int32_t f0 = (u.tile * K::kClusterSize + crank) * p.plan.splits;
            for (int32_t s0 = 0; s0 < p.plan.splits && ok; s0 += 32) {
              const int32_t s = s0 + (int32_t)lane;
              bool mine = true;
              if (s < p.plan.splits)
                mine = WG_CHECK(p.status, f0 + s < p.flag_words, kCheckFlag, u.tile) &&
                       wait_flag(p.flags + (f0 + s), p.epoch + p.wait_skew, abort_flag, p.status,
                                 kSiteEpiFlagZero);
              ok = __all_sync(0xffffffffu, mine);
            }
          }
          // The lanes' acquires cover the generic zero stores (the warp
          // barrier carries them to lane 0); order them before the
          // async-proxy reduce-adds that lane 0 issues.
          if (lane == 0) {
            fence_acq_rel_gpu();
            fence_proxy_async_global();
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      // TMEM is drained in batches of NB chunks of 32 columns (32 rows of C):
      // all loads of a batch are issued before one wait, so their latency is
      // paid once per batch; a shorter batch takes the remainder of an atom.
      constexpr int kChunks = K::BN / 32;
      constexpr int NB = K::kEpiBatch;
      const uint32_t tacc = tmem + ((q * 32u) << 16) + ab * K::kAccCols;
      // The worker's last unit stages through the idle stage ring.
      bool tail = false;
      if constexpr (K::kTailGroups > 1) {
        Unit u_next;
        tail = !unit_at(p.plan, worker, i + 1, u_next);
      }
      int32_t batch = 0;
#pragma unroll 1
      for (int r = 0; r < K::REPS; ++r) {
        const int32_t col_warp = col_cta + r * 128 + (int32_t)q * 32;
        const bool last_atom = r == K::REPS - 1;
#pragma unroll 1
        for (int c0 = 0; c0 < kChunks; c0 += NB) {
          // The last batch of an atom may be short (kChunks not a multiple of
          // NB); one register array of NB chunks serves every batch.
          const int nb = kChunks - c0 < NB ? kChunks - c0 : NB;
          const bool rel = last_atom && c0 + nb == kChunks;
          bool dok;
          if (tail) {
            const uint32_t sb = tail_base + (uint32_t)(batch % K::kTailGroups) * NB *
                                                K::kEpiSlotBytes;
            dok = drain<NB, K::kTailGroups - 1>(p, base, smem, tmem, tacc + r * K::BN, c0, nb,
                                                  col_warp, row0, add, sb, rel, ab, grp, r, fs,
                                                  abort_flag);
          } else {
            dok = drain<NB, 0>(p, base, smem, tmem, tacc + r * K::BN, c0, nb, col_warp, row0,
                               add, stage_base, rel, ab, grp, r, fs, abort_flag);
          }
          ++batch;
          if (!dok) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
      }
      if (!ok) break;
      if constexpr (K::kKSplit) {
        if (u.kind == kUnitStoreRaise) {
          // Owner of the tile's first k-block: make the stores complete and
          // visible, then raise the flag for the CTAs that add to this tile.
          if (lane == 0) {
            bulk_wait_group<0>();
            fence_proxy_async_global();
          }
          if (!epi_sync(base, sync_phase, abort_flag, p.status)) { ok = false; break; }
          if (threadIdx.x == 128 &&
              WG_CHECK(p.status, (int32_t)(u.tile * K::kClusterSize + crank) < p.flag_words, kCheckFlag,
                       u.tile)) {
            fence_acq_rel_gpu();
            st_release_gpu(p.flags + (u.tile * K::kClusterSize + crank), p.epoch);
          }
        }
      }
      if (++ab == (uint32_t)K::ACC) { ab = 0; aph ^= 1; }
    }
    if constexpr (K::EPI == kEpiTma) {
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
    if constexpr (K::kCinSlots > 0) {
      // Aborted: let this warp's Cin loads in flight land before exit.
      if (!ok && p.load_cin && lane == 0)
        for (uint32_t j = fs.consumed; j != fs.issued; ++j)
          wait_bar_final(bar_cin(base, q, j % (uint32_t)K::kCinSlots),
                         (j / (uint32_t)K::kCinSlots) & 1u, p.status, kSiteAbortCin);
      __syncwarp();
    }
    if (WGEMM_TRACE && threadIdx.x == 128) trace_event(p, kTrEpiDone);
  }


  // Split-K and zero-first stream-K: before any unit of this worker runs,
  // zero this CTA's share of every tile slice its zeroing units (kind
  // kUnitAddAfterZero) own and raise each slice's flag.
  __device__ static bool zero_slices(const KParams& p, uint32_t base, uint32_t rank, uint32_t grp,
                                     int32_t worker, uint32_t& sync_phase,
                                     volatile uint32_t* abort_flag) {
    const uint32_t crank = grp * K::CG + rank;  // rank in the cluster
    const int32_t M = p.plan.M, N = p.plan.N;
    const int64_t ldc = p.ldc;
    const int32_t t = (int32_t)threadIdx.x - 128;  // 0..127
    for (int32_t i = 0;; ++i) {
      Unit u;
      if (!unit_at(p.plan, worker, i, u)) break;
      if (u.kind != kUnitAddAfterZero) continue;
      int32_t r0, r1;
      plan_zero_rows(K::BN, p.plan.splits, u.split, r0, r1);
      const int32_t group_row0 = u.tm * K::kTileRows + row_group(grp) * K::BN;
      const int32_t row_begin = group_row0 + r0;
      int32_t row_end = group_row0 + r1;
      if (row_end > M) row_end = M;
      const int32_t col_begin =
          u.tn * K::kTileCols + col_group(grp) * K::kGroupCols + (int32_t)rank * K::kCtaCols;
      int32_t col_end = col_begin + K::kCtaCols;
      if (col_end > N) col_end = N;
      if (row_begin >= row_end || col_begin >= col_end) continue;
      const int32_t ncols = col_end - col_begin;
      const int32_t nvec = ncols / 4;  // ldc % 4 == 0 and C is 16-byte aligned
      if (!WG_CHECK(p.status, row_begin >= 0 && row_end <= M && col_begin >= 0 && col_end <= N,
                    kCheckZero, row_end))
        continue;
      for (int32_t r = row_begin; r < row_end; ++r) {
        float* row = static_cast<float*>(p.C) + (int64_t)r * ldc + col_begin;
        for (int32_t v = t; v < nvec; v += 128)
          reinterpret_cast<float4*>(row)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t c = nvec * 4 + t; c < ncols; c += 128) row[c] = 0.f;
      }
    }
    fence_proxy_async_global();
    if (!epi_sync(base, sync_phase, abort_flag, p.status)) return false;
    if (t == 0) {
      fence_acq_rel_gpu();
      for (int32_t i = 0;; ++i) {
        Unit u;
        if (!unit_at(p.plan, worker, i, u)) break;
        if (u.kind != kUnitAddAfterZero) continue;
        const int32_t fi = (u.tile * K::kClusterSize + crank) * p.plan.splits + u.split;
        if (WG_CHECK(p.status, fi < p.flag_words, kCheckFlag, fi))
          st_release_gpu(p.flags + fi, p.epoch);
      }
    }
    return true;
  }
};

template <class K>
__global__ void __launch_bounds__(kThreads, 1) wgemm_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t warp = threadIdx.x / 32;
  const uint32_t crank = K::kClusterSize > 1 ? cluster_ctarank() : 0u;
  const uint32_t rank = crank % K::CG;  // position in the MMA group (0 = leader)
  const uint32_t grp = crank / K::CG;   // MMA group in the cluster
  const int32_t worker = (int32_t)(blockIdx.x / K::kClusterSize);

  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + K::kOffMisc);
  volatile uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;

  uint32_t prefilled = 0;  // meaningful in thread 0, the producer
  if (threadIdx.x == 0) {
    if (WGEMM_TRACE) trace_event(p, kTrEntry);
    prefetch_tensormap(&p.tmA);
    prefetch_tensormap(&p.tmB);
    if (K::EPI == kEpiTma) prefetch_tensormap(&p.tmC);
    for (int s = 0; s < K::STAGES; ++s) {
      mbar_init(Kernel<K>::bar_full(base, s), 1);
      mbar_init(Kernel<K>::bar_empty(base, s), K::kGroups);  // one release per MMA group
    }
    for (int a = 0; a < K::ACC; ++a) {
      mbar_init(Kernel<K>::bar_accf(base, a), 1);
      mbar_init(Kernel<K>::bar_acce(base, a), 4 * K::CG);
    }
    mbar_init(Kernel<K>::bar_drain(base), 1);
    mbar_init(Kernel<K>::bar_epi(base), 4);
    for (int j = 0; j < K::kClcDepth; ++j) {
      mbar_init(Kernel<K>::bar_clc_full(base, j), 1);
      mbar_init(Kernel<K>::bar_clc_empty(base, j), K::kClcConsumers);
    }
    if constexpr (K::kCinSlots > 0) {
      for (int j = 0; j < 4 * K::kCinSlots; ++j)
        mbar_init(Kernel<K>::bar_cin(base, j / K::kCinSlots, j % K::kCinSlots), 1);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    // Programmatic dependent launch: everything above touches no global
    // memory that an earlier grid writes, so it overlaps that grid's tail;
    // the first operand load waits for it. A grid that depends on this one
    // may be scheduled from now on: it cannot start on an SM before this
    // grid's CTA there exits (shared memory), and it waits for this grid's
    // completion before it touches memory.
    griddep_wait();
    griddep_launch_dependents();
    if constexpr (K::kClusterSize == 1) prefilled = Kernel<K>::prefill(p, base, worker, rank, grp);
  }
  if (warp == 1) {
    tmem_alloc<K::CG>(smem_addr(misc), K::kTmemCols);
    tmem_relinquish<K::CG>();
  }
  tcgen05_fence_before();
  if constexpr (K::kClusterSize > 1) cluster_sync();
  else __syncthreads();
  tcgen05_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (WGEMM_TRACE && threadIdx.x == 0) trace_event(p, kTrSetUp);
  griddep_wait();  // every role reads or writes global memory only after this

  if (warp == 0) {
    // Thread 0 initialised the barriers and prefilled the ring, so it produces.
    if (threadIdx.x == 0) Kernel<K>::producer(p, base, rank, grp, worker, prefilled, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0) {
      if (elect_one()) Kernel<K>::mma(p, base, tmem, grp, worker, abort_flag);
      __syncwarp();
    }
  } else if (warp == 2) {
    if constexpr (K::SCHED == kSchedClc) {
      if (elect_one()) Kernel<K>::scheduler(p, base, crank, abort_flag);
      __syncwarp();
    }
  } else if (warp >= 4) {
    Kernel<K>::epilogue(p, base, smem, tmem, rank, grp, worker, abort_flag);
  }

  tcgen05_fence_before();
  if constexpr (K::kClusterSize > 1) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tcgen05_fence_after();
    tmem_dealloc<K::CG>(tmem, K::kTmemCols);
  }
  if (WGEMM_TRACE && threadIdx.x == 0) trace_event(p, kTrExit);
}

// K == 0: C := 0 (the empty sum), for C elements of `elem_bytes` (4 or 2).
__global__ void wgemm_zero_kernel(void* C, int32_t M, int32_t N, int64_t ldc, int32_t elem_bytes);

}  // namespace wg

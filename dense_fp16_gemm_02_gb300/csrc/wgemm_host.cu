// Host side of the C-ABI library: argument checks, per-shape configuration
// choice, tensor-map encoding, the split-K / stream-K flag workspace, and the
// launch. Declarations and their contracts are in include/wgemm.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "wgemm.h"
#include "wgemm_configs.h"
#include "wgemm_kernel.cuh"
#include "wgemm_plan.h"

namespace wg {

// The per-device status word the kernels write on a failed wait.
__device__ DeviceStatus g_device_status;

__global__ void wgemm_zero_kernel(void* C, int32_t M, int32_t N, int64_t ldc,
                                  int32_t elem_bytes) {
  const int64_t total = (int64_t)M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / N, c = i - r * N;
    if (elem_bytes == 4) static_cast<float*>(C)[r * ldc + c] = 0.f;
    else static_cast<uint16_t*>(C)[r * ldc + c] = 0;  // +0 in fp16 and in bf16
  }
}

// K == 0 with the fused epilogue: D := beta·Cin + bias[column] (the product
// of an empty sum is 0), D and Cin of `elem_bytes` (4: fp32; 2: fp16 or bf16
// by `bf16`). Cin is read only when beta != 0; bias may be null.
__global__ void wgemm_axpby_kernel(void* D, int64_t ldd, const void* Cin, int64_t ldcin,
                                   const float* bias, float beta, int32_t M, int32_t N,
                                   int32_t elem_bytes, int32_t bf16) {
  const int64_t total = (int64_t)M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / N, c = i - r * N;
    float v = bias ? bias[c] : 0.f;
    if (beta != 0.f) {
      float x;
      if (elem_bytes == 4) {
        x = static_cast<const float*>(Cin)[r * ldcin + c];
      } else {
        const uint16_t h = static_cast<const uint16_t*>(Cin)[r * ldcin + c];
        x = bf16 ? __bfloat162float(__ushort_as_bfloat16(h)) : __half2float(__ushort_as_half(h));
      }
      v = fmaf(beta, x, v);
    }
    if (elem_bytes == 4) {
      static_cast<float*>(D)[r * ldd + c] = v;
    } else {
      static_cast<uint16_t*>(D)[r * ldd + c] =
          bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
    }
  }
}

namespace {

constexpr int kMaxDevices = 64;

// The fused epilogue's operands (plain calls: fused = false).
struct EpiArgs {
  bool fused = false;
  const void* cin = nullptr;
  int ldcin = 0;
  const float* bias = nullptr;
  float alpha = 1.f, beta = 0.f;
};

struct Registry {
  std::vector<const KernelEntry*> entries;
  Registry() {
    for (int i = 0; i < kNumEntriesSingle; ++i) entries.push_back(&kEntriesSingle[i]);
    for (int i = 0; i < kNumEntriesPair; ++i) entries.push_back(&kEntriesPair[i]);
    for (int i = 0; i < kNumEntriesPair2; ++i) entries.push_back(&kEntriesPair2[i]);
    for (int i = 0; i < kNumEntriesMulticast; ++i) entries.push_back(&kEntriesMulticast[i]);
    for (int i = 0; i < kNumEntriesClc; ++i) entries.push_back(&kEntriesClc[i]);
    for (int i = 0; i < kNumEntriesOut16A; ++i) entries.push_back(&kEntriesOut16A[i]);
    for (int i = 0; i < kNumEntriesOut16B; ++i) entries.push_back(&kEntriesOut16B[i]);
    for (int i = 0; i < kNumEntriesFused; ++i) entries.push_back(&kEntriesFused[i]);
    for (int i = 0; i < kNumEntriesRowMc; ++i) entries.push_back(&kEntriesRowMc[i]);
  }
};

const Registry& registry() {
  static Registry r;
  return r;
}

struct DeviceState {
  bool init = false;
  bool supported = false;
  int sm_count = 0;
  DeviceStatus* status = nullptr;      // device address of g_device_status
  std::vector<int> max_workers;        // per config: co-resident clusters (0 = not queried)
  DeviceStatus last_error{};
};

struct Workspace {
  uint32_t* flags = nullptr;
  size_t bytes = 0;
  uint32_t epoch = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
uint32_t g_debug_wait_skew = 0;  // see wgemm_debug_set_flag_wait_skew
bool g_cooperative = true;          // see wgemm_debug_set_cooperative
uint64_t* g_debug_trace = nullptr;  // see wgemm_debug_set_trace
bool g_pdl = false;                 // see wgemm_set_pdl
int g_debug_trace_ctas = 0;

bool env_log() {
  static const bool on = [] {
    const char* v = std::getenv("WGEMM_LOG");
    return v && v[0] == '1';
  }();
  return on;
}

// Requires g_mu.
int device_state(int* dev_out, DeviceState** st_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return WGEMM_ERR_NO_DEVICE;
  }
  DeviceState& st = g_dev[dev];
  if (!st.init) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return WGEMM_ERR_NO_DEVICE;
    }
    st.supported = prop.major == 10 && prop.minor == 3;
    st.sm_count = prop.multiProcessorCount;
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
        cudaGetLastError();
        return WGEMM_ERR_LAUNCH;
      }
      st.status = static_cast<DeviceStatus*>(p);
      if (cudaMemset(st.status, 0, sizeof(DeviceStatus)) != cudaSuccess) return WGEMM_ERR_LAUNCH;
    }
    st.max_workers.assign(registry().entries.size(), 0);
    st.init = true;
  }
  if (!st.supported) return WGEMM_ERR_NO_DEVICE;
  *dev_out = dev;
  *st_out = &st;
  return WGEMM_OK;
}

int encoder() {
  if (g_encode) return WGEMM_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return WGEMM_ERR_LAUNCH;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return WGEMM_OK;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t elem_strides[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaLaunchConfig_t launch_config(const KernelEntry& e, int workers, cudaStream_t stream,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(workers * e.cg * e.mc * e.mr), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = e.smem_bytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)(e.cg * e.mc * e.mr);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// K-split grids (split-K, stream-K and their mixes) wait on flags that other
// CTAs of the same grid raise, so every CTA must be resident at once. A
// cooperative launch guarantees that: the grid starts only when all of its
// CTAs fit on the GPU beside whatever else runs there (a grid that cannot fit
// at all fails to launch). The grid never exceeds the co-resident count.
// `attr` is the array cfg.attrs points to, with room for one more entry.
void cooperative(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr) {
  attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
  attr[cfg.numAttrs].val.cooperative = 1;
  ++cfg.numAttrs;
}

// Requires g_mu. Co-resident workers (clusters) of a configuration on this
// device; sets the kernel's shared-memory attribute on first use.
int max_workers(DeviceState& st, int id) {
  if (st.max_workers[id] > 0) return st.max_workers[id];
  const KernelEntry& e = *registry().entries[id];
  if (cudaFuncSetAttribute(e.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)e.smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return WGEMM_ERR_LAUNCH;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config(e, st.sm_count / (e.cg * e.mc * e.mr), nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, e.func, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return WGEMM_ERR_LAUNCH;
  }
  st.max_workers[id] = n;
  return n;
}

int find_config(const char* name) {
  const auto& es = registry().entries;
  for (size_t i = 0; i < es.size(); ++i)
    if (std::strcmp(es[i]->name, name) == 0) return (int)i;
  return -1;
}

// The per-shape choice. A measured table of winners first, then a rule.
struct Choice {
  int config, mode, splits;
};

struct TunedRow {
  int M, N, K;
  const char* config;
  int mode, splits;
  double us;
};

const TunedRow kTuned[] = {
#include "wgemm_tuned.inc"
};

// Measured cost of each data-parallel configuration (tune.py --rates):
// a call of `waves` full waves over `kblocks` k-blocks takes about
// t0 + waves · (a + b · kblocks) microseconds. Two fits per configuration:
// operand rows that start on 32-byte sectors, and rows 16 bytes off them
// (every 128-byte TMA row then touches five L2 sectors instead of four,
// which costs tiles with more operand bytes per flop up to 40%).
struct RateRow {
  const char* config;
  double t0_us, a_us, b_us;     // rows on 32-byte sectors
  double t0u_us, au_us, bu_us;  // rows 16 bytes off
};

const RateRow kRates[] = {
#include "wgemm_rates.inc"
    {nullptr, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0},
};

// A 16-bit-output configuration ("..._h") without rates of its own takes
// those of its fp32 twin (same main loop; its epilogue writes half the bytes).
const RateRow* rate_of(const char* name) {
  for (const RateRow& r : kRates)
    if (r.config && std::strcmp(r.config, name) == 0) return &r;
  const size_t n = std::strlen(name);
  if (n > 2 && std::strcmp(name + n - 2, "_h") == 0) {
    const std::string twin(name, n - 2);
    for (const RateRow& r : kRates)
      if (r.config && twin == r.config) return &r;
  }
  return nullptr;
}

// Operand rows of both A and B start on 32-byte sectors.
bool rows_on_sectors(int lda, int ldb) { return lda % 16 == 0 && ldb % 16 == 0; }

// The fused epilogue of a configuration: 0 none, 1 the Cin ring (register
// stores; any alpha, beta, Cin), 2 the reduce-add form (TMA epilogue; only
// D += alpha·A·Bᵀ + bias in place, fp32).
int fuse_kind(const KernelEntry& e) { return e.fuse == 0 ? 0 : (e.epi == kEpiTma ? 2 : 1); }

// Whether a configuration serves a call whose epilogue is `fuse` (0 plain, 1
// general fused, 2 fused in place with beta = 1 and fp32 D, which either
// fused form can compute).
bool fuse_fits(const KernelEntry& e, int fuse) {
  const int k = fuse_kind(e);
  return fuse == 2 ? k != 0 : k == fuse;
}

// Configurations that may run split-K or stream-K plans: TMA epilogue (the
// reduce-adds), static schedule (every worker resident and owning its own
// units), no column multicast, fp32 C and no fused epilogue. Row-multicast
// clusters qualify: the cluster is the worker and its groups share every
// unit. The kernel compiles its split-K and stream-K paths for exactly these
// (Cfg::kKSplit).
bool can_split_k(const KernelEntry& e) {
  return e.epi == kEpiTma && e.mc == 1 && e.sched == 0 && e.out == 0 && !e.fuse;
}

// Predicted microseconds of a configuration and K-decomposition from the
// measured rates, with `workers` co-resident workers; < 0 if not modelled.
double predict_us(const KernelEntry& e, int M, int N, int K, bool aligned, int mode, int splits,
                  int workers) {
  const RateRow* r = rate_of(e.name);
  if (!r || workers <= 0) return -1.0;
  const double t0 = aligned ? r->t0_us : r->t0u_us;
  const double a = aligned ? r->a_us : r->au_us;
  const double b = aligned ? r->b_us : r->bu_us;
  const int64_t tiles = (int64_t)((M + e.tile_rows - 1) / e.tile_rows) *
                        ((N + e.tile_cols - 1) / e.tile_cols);
  const int64_t kblocks = (K + kBK - 1) / kBK;
  if (mode == kSplitK) {
    const int64_t units = tiles * splits;
    const int64_t waves = (units + workers - 1) / workers;
    // Zeroing C and one reduce-add of every partial tile in L2 (measured
    // ≈3 µs plus ≈0.5 µs per split on GB300).
    return t0 + 3.0 + 0.5 * splits + waves * a +
           waves * b * (double)((kblocks + splits - 1) / splits);
  }
  if (mode == kStreamK) {
    const int64_t per_worker = (tiles * kblocks + workers - 1) / workers;
    // The owner's store and flag, then the other units' reduce-adds, one
    // after the other (measured ≈6 µs on GB300).
    return t0 + 6.0 + a + b * (double)per_worker;
  }
  if (mode != kDataParallel) return -1.0;  // the waves + stream-K tail mix is not modelled
  const int64_t waves = (tiles + workers - 1) / workers;
  return t0 + waves * (a + b * (double)kblocks);
}

Choice choose(DeviceState& st, int M, int N, int K, int lda, int ldb, bool c_tma_ok, int out,
              int fuse = 0, bool dp_only = false) {
  // The table was measured with fp32 C, the plain epilogue and rows on
  // 32-byte sectors.
  const bool aligned = rows_on_sectors(lda, ldb);
  for (const TunedRow& r : kTuned) {
    if (out == 0 && fuse == 0 && aligned && r.M == M && r.N == N && r.K == K &&
        (!dp_only || r.mode == kDataParallel)) {
      const int id = find_config(r.config);
      const bool tma = std::strstr(r.config, "_tma") != nullptr;
      if (id >= 0 && (c_tma_ok || !tma)) return {id, r.mode, r.splits};
    }
  }
  // Not in the table: the configuration and K-decomposition with the least
  // predicted time from the measured per-configuration rates. Split-K is
  // taken only when it predicts at least 10% less time than the best
  // data-parallel choice: its fix-up cost (zeroing, reduce-adds in L2, flag
  // waits) varies more from shape to shape than one fitted constant.
  // Stream-K is not chosen here. Its model assumes the data-parallel k-loop
  // rate, but stream-K's ranges start at scattered k offsets, and measured
  // k-loops run 12-35% slower than that; split-K's units stay in step.
  // Calls predicted at kLongCallUs or more run under the power cap when they
  // come back to back, and there the lone-call rates mislead. The 512-column
  // tiles with cluster launch control read the fewest operand bytes per flop
  // and hand out tiles in serpentine order, which keeps the tiles in flight
  // adjacent and cuts DRAM reads (16384³: 7.9 against 17.9 GB per call for
  // the 256×256 static tile), so they spend less energy per call and run at
  // a higher clock. Back to back (blocks of consecutive calls) the 512×256
  // CLC tile beat the rule's lone-call choice by 2–5 % at 12288³ and
  // 8192×8192×16384, and the 256×256 static tile by 9 % at 16384³; the
  // 256-column CLC tiles did not (12288³: 2299 against 2260 µs). The rates,
  // fitted on calls of up to 4 waves and K = 4096, put the 512×256 CLC tile
  // 14–22 % behind there; at 12288³ they predict 1750 µs for the static
  // choice, which took 2260–2323 µs back to back. So for such calls the best
  // 512-column CLC configuration is taken when its prediction is within 30 %
  // of the best and the shape gives it at least two waves of tiles.
  constexpr double kLongCallUs = 500.0, kClcMargin = 1.30;
  const auto& es = registry().entries;
  Choice best{-1, kDataParallel, 1}, best_split{-1, kDataParallel, 1},
      best_clc{-1, kDataParallel, 1};
  double best_us = 0.0, best_split_us = 0.0, best_clc_us = 0.0;
  for (int id = 0; id < (int)es.size(); ++id) {
    const KernelEntry& e = *es[id];
    if (e.out != out || !fuse_fits(e, fuse) || (e.epi == kEpiTma && !c_tma_ok)) continue;
    const int w = max_workers(st, id);
    if (w <= 0) continue;
    auto consider = [&](int mode, int splits) {
      const double us = predict_us(e, M, N, K, aligned, mode, splits, w);
      Choice& c = mode == kDataParallel ? best : best_split;
      double& c_us = mode == kDataParallel ? best_us : best_split_us;
      if (us >= 0.0 && (c.config < 0 || us < c_us)) {
        c = {id, mode, splits};
        c_us = us;
      }
      const int64_t clc_tiles = (int64_t)((M + e.tile_rows - 1) / e.tile_rows) *
                                ((N + e.tile_cols - 1) / e.tile_cols);
      if (mode == kDataParallel && e.sched == 1 && e.tile_cols >= 512 && us >= 0.0 &&
          clc_tiles >= 2 * (int64_t)w && (best_clc.config < 0 || us < best_clc_us)) {
        best_clc = {id, mode, splits};
        best_clc_us = us;
      }
    };
    consider(kDataParallel, 1);
    const bool ksplit = can_split_k(e);
    const int64_t tiles = (int64_t)((M + e.tile_rows - 1) / e.tile_rows) *
                          ((N + e.tile_cols - 1) / e.tile_cols);
    const int kblocks = (K + kBK - 1) / kBK;
    if (ksplit && !dp_only && kblocks >= 32 && tiles < w) {
      for (int sp = 2; sp <= 16 && sp <= kblocks / 8 && tiles * sp <= w; ++sp)
        consider(kSplitK, sp);
    }
  }
  if (best_split.config >= 0 && (best.config < 0 || best_split_us < 0.9 * best_us))
    return best_split;
  if (best.config >= 0 && best_us >= kLongCallUs && best_clc.config >= 0 &&
      best_clc_us <= kClcMargin * best_us)
    return best_clc;
  if (best.config >= 0) return best;
  // No rates compiled in: a plain fallback.
  if (fuse) {
    return {find_config(out == 0 ? "g2_256x256_s6_a2_direct_ab2" : "g2_256x256_s6_a2_direct_ab4_h"),
            kDataParallel, 1};
  }
  const char* fb = c_tma_ok ? "g2_256x256_s6_a2_tma" : "g2_256x256_s6_a2_direct";
  if (out == 0) return {find_config(fb), kDataParallel, 1};
  return {find_config((std::string(fb) + "_h").c_str()), kDataParallel, 1};
}

// Tile rows per raster group (WGEMM_RASTER_GROUP overrides the default 8).
int raster_group() {
  static const int g = [] {
    const char* v = std::getenv("WGEMM_RASTER_GROUP");
    const int x = v ? std::atoi(v) : 0;
    return x > 0 ? x : 8;
  }();
  return g;
}

// Element types of the typed entry points (WGEMM_F32 / WGEMM_F16 / WGEMM_BF16).
bool ab_type_ok(int t) { return t == WGEMM_F16 || t == WGEMM_BF16; }
bool c_type_ok(int t) { return t == WGEMM_F32 || t == WGEMM_F16 || t == WGEMM_BF16; }
int c_bytes(int t) { return t == WGEMM_F32 ? 4 : 2; }
CUtensorMapDataType tma_type(int t) {
  return t == WGEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
         : t == WGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

int check_args(const void* A, const void* B, const void* C, int M, int N, int K, int lda, int ldb,
               int ldc, int c_elem_bytes = 4) {
  if (M < 0 || N < 0 || K < 0) return WGEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WGEMM_OK;
  if (!C) return WGEMM_ERR_INVALID_ARG;
  if (ldc < N) return WGEMM_ERR_INVALID_ARG;
  if (K > 0) {
    if (!A || !B || lda < K || ldb < K) return WGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (lda % 8) || (ldb % 8))
      return WGEMM_ERR_ALIGNMENT;
  }
  if (reinterpret_cast<uintptr_t>(C) & (uintptr_t)(c_elem_bytes - 1)) return WGEMM_ERR_ALIGNMENT;
  return WGEMM_OK;
}

// C can be written by TMA (16-byte aligned base and row stride).
bool c_tma_ok(const void* C, int ldc, int c_elem_bytes = 4) {
  return !(reinterpret_cast<uintptr_t>(C) & 15) && !(((int64_t)ldc * c_elem_bytes) % 16);
}

// Fills the plan for a configuration; WGEMM_ERR_CONFIG if the mode cannot run.
int make_plan(const KernelEntry& e, int M, int N, int K, int mode, int splits, int max_w,
              Plan* p) {
  std::memset(p, 0, sizeof(*p));
  p->M = M;
  p->N = N;
  p->K = K;
  p->tile_rows = e.tile_rows;
  p->tile_cols = e.tile_cols;
  p->tiles_m = (M + e.tile_rows - 1) / e.tile_rows;
  p->tiles_n = (N + e.tile_cols - 1) / e.tile_cols;
  p->num_tiles = p->tiles_m * p->tiles_n;
  p->kblocks = (K + kBK - 1) / kBK;
  p->mode = mode;
  p->splits = 1;
  p->group = raster_group();
  if (mode != kDataParallel && !can_split_k(e)) return WGEMM_ERR_CONFIG;
  p->sched = e.sched;
  if (mode == kDataParallel && e.sched == 1) {
    p->workers = p->num_tiles;  // one cluster per tile; running clusters take the rest
  } else if (mode == kDataParallel) {
    p->workers = std::min(p->num_tiles, max_w);
  } else if (mode == kSplitK) {
    if (splits < 1) return WGEMM_ERR_CONFIG;
    p->splits = std::min(splits, p->kblocks);
    p->workers = (int32_t)std::min<int64_t>((int64_t)p->num_tiles * p->splits, max_w);
  } else if (mode == kStreamK) {
    p->total_iters = (int64_t)p->num_tiles * p->kblocks;
    p->workers = (int32_t)std::min<int64_t>(p->total_iters, max_w);
  } else if (mode == kHybridK) {
    // Whole waves of tiles data parallel; the partial last wave and the
    // `splits` − 1 full waves before it by stream-K over all workers. Fewer
    // tiles than workers leaves no whole wave: plain stream-K.
    if (splits < 1) return WGEMM_ERR_CONFIG;
    p->mode = kStreamK;
    if (p->num_tiles < max_w) {
      p->total_iters = (int64_t)p->num_tiles * p->kblocks;
      p->workers = (int32_t)std::min<int64_t>(p->total_iters, max_w);
    } else {
      p->workers = max_w;
      const int32_t waves = p->num_tiles / max_w;
      const int32_t dp_waves = std::max(0, waves - (splits - 1));
      p->dp_tiles = dp_waves * max_w;
      p->total_iters = (int64_t)(p->num_tiles - p->dp_tiles) * p->kblocks;
    }
  } else if (mode == kStreamKZero) {
    // Stream-K ranges with split-K's fix-up: owners zero their tile first.
    p->mode = kStreamK;
    p->zero_first = 1;
    p->total_iters = (int64_t)p->num_tiles * p->kblocks;
    p->workers = (int32_t)std::min<int64_t>(p->total_iters, max_w);
  } else {
    return WGEMM_ERR_CONFIG;
  }
  return p->workers > 0 ? WGEMM_OK : WGEMM_ERR_CONFIG;
}

// Requires g_mu. Flags for a call on (dev, stream): at least `words` words.
int workspace(int dev, cudaStream_t stream, size_t words, Workspace** out) {
  Workspace& ws = g_ws[{dev, stream}];
  const size_t bytes = std::max<size_t>(words * sizeof(uint32_t), 4096);
  if (ws.bytes < bytes) {
    if (ws.flags) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return WGEMM_ERR_LAUNCH;
      cudaFree(ws.flags);
      ws.flags = nullptr;
      ws.bytes = 0;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
      cudaGetLastError();
      return WGEMM_ERR_WORKSPACE;
    }
    if (cudaMemset(p, 0, bytes) != cudaSuccess) {
      cudaFree(p);
      return WGEMM_ERR_WORKSPACE;
    }
    ws.flags = static_cast<uint32_t*>(p);
    ws.bytes = bytes;
    ws.epoch = 0;
  }
  *out = &ws;
  return WGEMM_OK;
}

// True while `stream` is being captured into a CUDA graph. K-split plans
// are not captured: their flags carry a per-call epoch that the kernel
// parameters fix at capture, and a replayed graph would find the flags of
// its previous replay already up.
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return cs != cudaStreamCaptureStatusNone;
}

int run(const void* A, const void* B, void* C, int ab_type, int c_type, int M, int N, int K,
        int lda, int ldb, int ldc, int config_id, int mode, int splits, cudaStream_t stream,
        const EpiArgs& ep = EpiArgs()) {
  if (!ab_type_ok(ab_type) || !c_type_ok(c_type)) return WGEMM_ERR_INVALID_ARG;
  const int cb = c_bytes(c_type), out = c_type == WGEMM_F32 ? 0 : 1;
  // D += alpha·A·Bᵀ + bias in place (Cin = D, beta = 1, fp32 D) may also
  // run the reduce-add kernels.
  const bool in_place = ep.fused && ep.beta == 1.f && ep.cin == C && ep.ldcin == ldc &&
                        c_type == WGEMM_F32;
  const int fuse = ep.fused ? (in_place ? 2 : 1) : 0;
  int rc = check_args(A, B, C, M, N, K, lda, ldb, ldc, cb);
  if (rc != WGEMM_OK) return rc;
  const bool load_cin = ep.fused && ep.beta != 0.f;
  if (load_cin) {
    if (M > 0 && N > 0 && (!ep.cin || ep.ldcin < N)) return WGEMM_ERR_INVALID_ARG;
    // Cin is read by TMA: 16-byte aligned base and row pitch.
    if (M > 0 && N > 0 && !c_tma_ok(ep.cin, ep.ldcin, cb)) return WGEMM_ERR_ALIGNMENT;
  }
  if (M == 0 || N == 0) return WGEMM_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* st;
  if ((rc = device_state(&dev, &st)) != WGEMM_OK) return rc;
  if (K == 0) {
    const int64_t total = (int64_t)M * N;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)st->sm_count * 8);
    if (ep.fused)
      wgemm_axpby_kernel<<<blocks, 256, 0, stream>>>(C, ldc, ep.cin, ep.ldcin, ep.bias,
                                                     load_cin ? ep.beta : 0.f, M, N, cb,
                                                     c_type == WGEMM_BF16 ? 1 : 0);
    else
      wgemm_zero_kernel<<<blocks, 256, 0, stream>>>(C, M, N, ldc, cb);
    return cudaGetLastError() == cudaSuccess ? WGEMM_OK : WGEMM_ERR_LAUNCH;
  }
  const auto& es = registry().entries;
  const bool c_ok = c_tma_ok(C, ldc, cb);
  const bool in_graph = capturing(stream);
  if (config_id < 0) {
    Choice c = choose(*st, M, N, K, lda, ldb, c_ok, out, fuse, in_graph);
    config_id = c.config;
    mode = c.mode;
    splits = c.splits;
  }
  if (config_id < 0 || config_id >= (int)es.size()) return WGEMM_ERR_CONFIG;
  const KernelEntry& e = *es[config_id];
  if (e.out != out || !fuse_fits(e, fuse)) return WGEMM_ERR_CONFIG;
  if (e.epi == kEpiTma && !c_ok) return WGEMM_ERR_ALIGNMENT;
  if (mode < 0) {
    Choice c = choose(*st, M, N, K, lda, ldb, c_ok, out, fuse, in_graph);
    mode = c.mode;
    splits = c.splits;
    if (mode != kDataParallel && e.epi != kEpiTma) mode = kDataParallel;
  }
  if (in_graph && mode != kDataParallel) return WGEMM_ERR_CONFIG;
  // 16-bit C is rounded once from the full fp32 sum, and the fused epilogue
  // applies alpha, beta and bias to the full sum: no K split.
  if ((out != 0 || fuse) && mode != kDataParallel) return WGEMM_ERR_CONFIG;
  const int mw = max_workers(*st, config_id);
  if (mw < 0) return mw;
  if ((rc = encoder()) != WGEMM_OK) return rc;

  KParams params;
  std::memset(&params, 0, sizeof(params));
  if ((rc = make_plan(e, M, N, K, mode, splits, mw, &params.plan)) != WGEMM_OK) return rc;
  const int brows_a = e.bn / e.cg / e.mc, rows_b = 128 * e.reps / e.mr;
  if (!encode_2d(&params.tmA, tma_type(ab_type), A, (uint64_t)K, (uint64_t)M, (uint64_t)lda * 2,
                 kBK, (uint32_t)brows_a, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&params.tmB, tma_type(ab_type), B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb * 2,
                 kBK, (uint32_t)rows_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
      (e.epi == kEpiTma &&
       !encode_2d(&params.tmC, tma_type(c_type), C, (uint64_t)N, (uint64_t)M,
                  (uint64_t)ldc * cb, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE)))
    return WGEMM_ERR_LAUNCH;
  params.C = C;
  params.ldc = ldc;
  params.idesc = umma_idesc_f16(128u * e.cg, (uint32_t)e.bn, ab_type == WGEMM_BF16);
  params.c_bf16 = c_type == WGEMM_BF16 ? 1 : 0;
  if (ep.fused) {
    params.alpha = ep.alpha;
    params.beta = ep.beta;
    params.bias = ep.bias;
    // The reduce-add form adds into D's old values in L2: no Cin read.
    params.load_cin = load_cin && fuse_kind(e) == 1 ? 1 : 0;
    if (params.load_cin && !encode_2d(&params.tmCin, tma_type(c_type), ep.cin, (uint64_t)N, (uint64_t)M,
                               (uint64_t)ep.ldcin * cb, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
      return WGEMM_ERR_LAUNCH;
  }
  params.status = st->status;
  params.trace = g_debug_trace;
  params.trace_ctas = g_debug_trace_ctas;
  if (params.plan.mode != kDataParallel) {
    Workspace* ws;
    const size_t words = (size_t)params.plan.num_tiles * e.cg * e.mc * e.mr * params.plan.splits;
    if ((rc = workspace(dev, stream, words, &ws)) != WGEMM_OK) return rc;
    params.flags = ws->flags;
    params.flag_words = (int32_t)(ws->bytes / sizeof(uint32_t));
    params.epoch = ++ws->epoch;
    params.wait_skew = g_debug_wait_skew;
  }
  if (env_log())
    std::fprintf(stderr, "wgemm: %dx%dx%d config %s mode %d splits %d workers %d tiles %d\n", M, N,
                 K, e.name, params.plan.mode, params.plan.splits, params.plan.workers,
                 params.plan.num_tiles);
  cudaLaunchAttribute attr[3];
  cudaLaunchConfig_t cfg = launch_config(e, params.plan.workers, stream, attr);
  if (e.cg * e.mc * e.mr == 1) cfg.numAttrs = 0;  // no cluster: a plain launch
  if (params.plan.mode != kDataParallel && g_cooperative) cooperative(cfg, attr);
  if (g_pdl) {
    // May start (set-up only; loads wait) while the previous kernel on the
    // stream finishes, once that kernel allows its dependents to launch.
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  void* args[] = {&params};
  if (cudaLaunchKernelExC(&cfg, e.func, args) != cudaSuccess) {
    cudaGetLastError();
    return WGEMM_ERR_LAUNCH;
  }
  return WGEMM_OK;
}

}  // namespace
}  // namespace wg

using namespace wg;

extern "C" {

int wgemm_f16f32(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C, int M, int N, int K,
                 int lda, int ldb, int ldc, wgemm_stream_t stream) {
  return run(A, B, C, WGEMM_F16, WGEMM_F32, M, N, K, lda, ldb, ldc, -1, -1, 1,
             reinterpret_cast<cudaStream_t>(stream));
}

int wgemm_f16f32_config(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C, int M, int N, int K,
                        int lda, int ldb, int ldc, int config_id, int mode, int splits,
                        wgemm_stream_t stream) {
  return wgemm_gemm_config(A, B, C, WGEMM_F16, WGEMM_F32, M, N, K, lda, ldb, ldc, config_id, mode,
                           splits, stream);
}

int wgemm_gemm(const void* A, const void* B, void* C, int ab_type, int c_type, int M, int N, int K,
               int lda, int ldb, int ldc, wgemm_stream_t stream) {
  return run(A, B, C, ab_type, c_type, M, N, K, lda, ldb, ldc, -1, -1, 1,
             reinterpret_cast<cudaStream_t>(stream));
}

int wgemm_gemm_config(const void* A, const void* B, void* C, int ab_type, int c_type, int M, int N,
                      int K, int lda, int ldb, int ldc, int config_id, int mode, int splits,
                      wgemm_stream_t stream) {
  if (config_id < 0 || config_id >= (int)registry().entries.size()) return WGEMM_ERR_CONFIG;
  if (mode < -1 || mode > kStreamKZero) return WGEMM_ERR_CONFIG;
  return run(A, B, C, ab_type, c_type, M, N, K, lda, ldb, ldc, config_id, mode, splits,
             reinterpret_cast<cudaStream_t>(stream));
}

int wgemm_gemm_ex(const void* A, const void* B, void* D, const void* Cin, const float* bias,
                  float alpha, float beta, int ab_type, int c_type, int M, int N, int K, int lda,
                  int ldb, int ldd, int ldcin, wgemm_stream_t stream) {
  return wgemm_gemm_ex_config(A, B, D, Cin, bias, alpha, beta, ab_type, c_type, M, N, K, lda,
                              ldb, ldd, ldcin, -1, stream);
}

int wgemm_gemm_ex_config(const void* A, const void* B, void* D, const void* Cin,
                         const float* bias, float alpha, float beta, int ab_type, int c_type,
                         int M, int N, int K, int lda, int ldb, int ldd, int ldcin,
                         int config_id, wgemm_stream_t stream) {
  if (config_id < -1 || config_id >= (int)registry().entries.size()) return WGEMM_ERR_CONFIG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return WGEMM_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // alpha = 1, beta = 0 and no bias is the plain product: every kernel.
  if (config_id < 0 && alpha == 1.f && beta == 0.f && bias == nullptr)
    return run(A, B, D, ab_type, c_type, M, N, K, lda, ldb, ldd, -1, -1, 1, s);
  EpiArgs ep;
  ep.fused = true;
  ep.cin = Cin;
  ep.ldcin = ldcin;
  ep.bias = bias;
  ep.alpha = alpha;
  ep.beta = beta;
  return run(A, B, D, ab_type, c_type, M, N, K, lda, ldb, ldd, config_id,
             config_id < 0 ? -1 : kDataParallel, 1, s, ep);
}

int wgemm_bf16f32(const wgemm_bf16_t* A, const wgemm_bf16_t* B, float* C, int M, int N, int K,
                  int lda, int ldb, int ldc, wgemm_stream_t stream) {
  return wgemm_gemm(A, B, C, WGEMM_BF16, WGEMM_F32, M, N, K, lda, ldb, ldc, stream);
}

int wgemm_f16f16(const wgemm_f16_t* A, const wgemm_f16_t* B, wgemm_f16_t* C, int M, int N, int K,
                 int lda, int ldb, int ldc, wgemm_stream_t stream) {
  return wgemm_gemm(A, B, C, WGEMM_F16, WGEMM_F16, M, N, K, lda, ldb, ldc, stream);
}

int wgemm_bf16bf16(const wgemm_bf16_t* A, const wgemm_bf16_t* B, wgemm_bf16_t* C, int M, int N,
                   int K, int lda, int ldb, int ldc, wgemm_stream_t stream) {
  return wgemm_gemm(A, B, C, WGEMM_BF16, WGEMM_BF16, M, N, K, lda, ldb, ldc, stream);
}

int wgemm_set_pdl(int enable) {
  if (enable != 0 && enable != 1) return WGEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  const int prev = g_pdl ? 1 : 0;
  g_pdl = enable == 1;
  return prev;
}

int wgemm_num_configs(void) { return (int)registry().entries.size(); }

const char* wgemm_config_name(int id) {
  const auto& es = registry().entries;
  return (id >= 0 && id < (int)es.size()) ? es[id]->name : "";
}

int wgemm_select(int M, int N, int K, int lda, int ldb, int c_type, int fused, int* config_id,
                 int* mode, int* splits) {
  if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || !c_type_ok(c_type) || fused < 0 ||
      fused > 2 || (fused == 2 && c_type != WGEMM_F32))
    return WGEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* st;
  const int rc = device_state(&dev, &st);
  if (rc != WGEMM_OK) return rc;
  Choice c = choose(*st, M, N, K, lda, ldb, true, c_type == WGEMM_F32 ? 0 : 1, fused);
  if (config_id) *config_id = c.config;
  if (mode) *mode = c.mode;
  if (splits) *splits = c.splits;
  return WGEMM_OK;
}

int wgemm_check(wgemm_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return WGEMM_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* st;
  int rc = device_state(&dev, &st);
  if (rc != WGEMM_OK) return rc;
  DeviceStatus s;
  if (cudaMemcpy(&s, st->status, sizeof(s), cudaMemcpyDeviceToHost) != cudaSuccess)
    return WGEMM_ERR_LAUNCH;
  if (s.code != 0) {
    st->last_error = s;
    if (cudaMemset(st->status, 0, sizeof(DeviceStatus)) != cudaSuccess) return WGEMM_ERR_LAUNCH;
    return s.code;
  }
  return WGEMM_OK;
}

int wgemm_last_device_error(int* block, int* warp, int* site, int* parity) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return WGEMM_ERR_NO_DEVICE;
  }
  const DeviceStatus& s = g_dev[dev].last_error;
  if (block) *block = s.block;
  if (warp) *warp = s.warp;
  if (site) *site = s.site;
  if (parity) *parity = s.parity;
  return s.code;
}

const char* wgemm_status_string(int status) {
  switch (status) {
    case WGEMM_OK: return "ok";
    case WGEMM_ERR_INVALID_ARG: return "invalid argument";
    case WGEMM_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case WGEMM_ERR_LAUNCH: return "CUDA error while preparing or launching";
    case WGEMM_ERR_NO_DEVICE: return "no current device of compute capability 10.3";
    case WGEMM_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel expired";
    case WGEMM_ERR_CONFIG: return "configuration cannot run this shape or mode";
    case WGEMM_ERR_WORKSPACE: return "flag workspace allocation failed";
    default: return "unknown status";
  }
}

size_t wgemm_workspace_bytes(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  size_t total = 0;
  for (const auto& kv : g_ws)
    if (kv.first.first == dev) total += kv.second.bytes;
  return total;
}

int wgemm_release_workspace(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return WGEMM_ERR_NO_DEVICE;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return WGEMM_ERR_LAUNCH;
  for (auto it = g_ws.begin(); it != g_ws.end();) {
    if (it->first.first == dev) {
      if (it->second.flags) cudaFree(it->second.flags);
      it = g_ws.erase(it);
    } else {
      ++it;
    }
  }
  return WGEMM_OK;
}

int wgemm_debug_set_trace(uint64_t* device_buffer, int ctas) {
  if (ctas < 0 || (ctas > 0 && !device_buffer)) return WGEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_debug_trace = ctas > 0 ? device_buffer : nullptr;
  g_debug_trace_ctas = ctas;
  return WGEMM_OK;
}

int wgemm_debug_trace_build(void) { return WGEMM_TRACE; }

int wgemm_debug_max_workers(int config_id) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (config_id < 0 || config_id >= (int)registry().entries.size()) return WGEMM_ERR_CONFIG;
  int dev;
  DeviceState* st;
  const int rc = device_state(&dev, &st);
  if (rc != WGEMM_OK) return rc;
  return max_workers(*st, config_id);
}

double wgemm_debug_predict_us(int M, int N, int K, int lda, int ldb, int config_id, int mode,
                              int splits, int workers) {
  const auto& es = registry().entries;
  if (config_id < 0 || config_id >= (int)es.size() || M <= 0 || N <= 0 || K <= 0 || lda < K ||
      ldb < K)
    return -1.0;
  return predict_us(*es[config_id], M, N, K, rows_on_sectors(lda, ldb), mode, splits, workers);
}

int wgemm_debug_set_cooperative(int enable) {
  if (enable != 0 && enable != 1) return WGEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  const int prev = g_cooperative ? 1 : 0;
  g_cooperative = enable == 1;
  return prev;
}

int wgemm_debug_set_flag_wait_skew(int skew) {
  if (skew < 0) return WGEMM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  g_debug_wait_skew = (uint32_t)skew;
  return WGEMM_OK;
}

uint64_t wgemm_debug_smem_desc(uint32_t smem_addr) { return umma_smem_desc_sw128(smem_addr); }

uint32_t wgemm_debug_idesc(int M, int N, int bf16) {
  return umma_idesc_f16((uint32_t)M, (uint32_t)N, bf16 != 0);
}

int wgemm_debug_config_out(int config_id) {
  const auto& es = registry().entries;
  return (config_id >= 0 && config_id < (int)es.size()) ? es[config_id]->out : WGEMM_ERR_CONFIG;
}

int wgemm_debug_config_fused(int config_id) {
  const auto& es = registry().entries;
  return (config_id >= 0 && config_id < (int)es.size()) ? (es[config_id]->fuse != 0 ? 1 : 0)
                                                          : WGEMM_ERR_CONFIG;
}

uint32_t wgemm_debug_sw128_offset(uint32_t row, uint32_t k) { return sw128_offset_f16(row, k); }

int wgemm_debug_plan(int M, int N, int K, int config_id, int mode, int splits, int workers,
                     int32_t* out, int max_units, int* tile_rows, int* tile_cols) {
  const auto& es = registry().entries;
  if (config_id < 0 || config_id >= (int)es.size() || M <= 0 || N <= 0 || K <= 0 || workers <= 0)
    return WGEMM_ERR_INVALID_ARG;
  const KernelEntry& e = *es[config_id];
  Plan p;
  const int rc = make_plan(e, M, N, K, mode, splits, workers, &p);
  if (rc != WGEMM_OK) return rc;
  if (tile_rows) *tile_rows = e.tile_rows;
  if (tile_cols) *tile_cols = e.tile_cols;
  int n = 0;
  for (int w = 0; w < p.workers; ++w) {
    for (int i = 0;; ++i) {
      Unit u;
      // The unit walk the configuration's kernel compiles (Cfg::kKSplit).
      if (!(can_split_k(e) ? plan_unit(p, w, i, u) : plan_unit_dp(p, w, i, u))) break;
      if (out && n < max_units) {
        int32_t* o = out + 7 * n;
        o[0] = u.tile; o[1] = u.tm; o[2] = u.tn; o[3] = u.kb_begin; o[4] = u.kb_end;
        o[5] = u.kind; o[6] = u.split;
      }
      ++n;
    }
  }
  return n;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free split-K entry point (wgemm_f16f32_splitk_noalloc).
//
// Its split-K flags live in a fixed array in device memory that belongs to the
// library image itself: every device that loads the library holds these
// 64 KiB until the process exits. Host code must not use the array's name as
// a device address (on the host it names a stand-in); the device address is
// taken once per device with cudaGetSymbolAddress, with that device current.
namespace wg {

constexpr uint32_t kNoAllocFlagWords = 16384;  // 64 KiB of split-K flags
static __device__ __align__(256) uint32_t g_noalloc_flags[kNoAllocFlagWords];

namespace {

struct NoAllocState {
  uint32_t* flags = nullptr;  // device address of g_noalloc_flags on this device
  uint32_t epoch = 0;         // flags only grow, so nothing is ever cleared
};
NoAllocState g_noalloc[kMaxDevices];

// Requires g_mu. First call on a device: look up the array's device address.
int noalloc_flags(int dev, NoAllocState** out) {
  NoAllocState& s = g_noalloc[dev];
  if (!s.flags) {
    uint32_t* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_noalloc_flags) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return WGEMM_ERR_LAUNCH;
    }
    s.flags = ptr;
  }
  *out = &s;
  return WGEMM_OK;
}

int run_noalloc(const uint16_t* A, const uint16_t* B, float* C, int M, int N, int K, int lda,
                int ldb, int ldc, int splits, cudaStream_t stream) {
  int rc = check_args(A, B, C, M, N, K, lda, ldb, ldc);
  if (rc != WGEMM_OK) return rc;
  if (splits < 1) return WGEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WGEMM_OK;
  if (!c_tma_ok(C, ldc)) return WGEMM_ERR_ALIGNMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  DeviceState* st;
  if ((rc = device_state(&dev, &st)) != WGEMM_OK) return rc;
  NoAllocState* na;
  if ((rc = noalloc_flags(dev, &na)) != WGEMM_OK) return rc;
  if (K == 0) {
    const int64_t total = (int64_t)M * N;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)st->sm_count * 8);
    wgemm_zero_kernel<<<blocks, 256, 0, stream>>>(C, M, N, ldc, 4);
    return cudaGetLastError() == cudaSuccess ? WGEMM_OK : WGEMM_ERR_LAUNCH;
  }
  const int config_id = find_config("g2_512x256_s4_a1_tma");
  if (config_id < 0) return WGEMM_ERR_CONFIG;
  // Its flags carry a per-call epoch: not a call to capture in a graph.
  if (capturing(stream)) return WGEMM_ERR_CONFIG;
  const KernelEntry& e = *registry().entries[config_id];
  const int mw = max_workers(*st, config_id);
  if (mw < 0) return mw;
  if ((rc = encoder()) != WGEMM_OK) return rc;
  KParams params;
  std::memset(&params, 0, sizeof(params));
  if ((rc = make_plan(e, M, N, K, kSplitK, splits, mw, &params.plan)) != WGEMM_OK) return rc;
  const size_t words = (size_t)params.plan.num_tiles * e.cg * params.plan.splits;
  if (words > kNoAllocFlagWords) return WGEMM_ERR_NOALLOC_TOO_LARGE;
  const int brows_a = e.bn / e.cg / e.mc, rows_b = 128 * e.reps / e.mr;
  if (!encode_2d(&params.tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, (uint64_t)K, (uint64_t)M,
                 (uint64_t)lda * 2, kBK, (uint32_t)brows_a, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&params.tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, (uint64_t)K, (uint64_t)N,
                 (uint64_t)ldb * 2, kBK, (uint32_t)rows_b, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&params.tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, (uint64_t)N, (uint64_t)M,
                 (uint64_t)ldc * 4, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
    return WGEMM_ERR_LAUNCH;
  params.C = C;
  params.ldc = ldc;
  params.idesc = umma_idesc_f16(128u * e.cg, (uint32_t)e.bn, false);
  params.status = st->status;
  params.flags = na->flags;
  params.flag_words = (int32_t)kNoAllocFlagWords;
  params.epoch = ++na->epoch;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(e, params.plan.workers, stream, attr);
  if (g_cooperative) cooperative(cfg, attr);
  void* args[] = {&params};
  if (cudaLaunchKernelExC(&cfg, e.func, args) != cudaSuccess) {
    cudaGetLastError();
    return WGEMM_ERR_LAUNCH;
  }
  return WGEMM_OK;
}

}  // namespace
}  // namespace wg

extern "C" int wgemm_f16f32_splitk_noalloc(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C,
                                           int M, int N, int K, int lda, int ldb, int ldc,
                                           int splits, wgemm_stream_t stream) {
  return wg::run_noalloc(A, B, C, M, N, K, lda, ldb, ldc, splits,
                         reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- host buffers
// wgemm_f16f32_host: A and B in host memory, C returned to host memory, through
// the caller's device buffers. A goes up in row panels and B in blocks of its
// rows (C's column blocks; one block unless B is large): first the first half
// of B's blocks, then every panel of A, then B's other blocks. Each (panel,
// block) GEMM starts as soon as its operands have landed, and each block of C
// goes down as soon as it is computed, so the copies in both directions
// overlap the GEMMs of the other blocks. Uploads and downloads run on two streams of the
// library's own (one per direction and device: the two copy directions use
// separate copy engines); the GEMMs run on the caller's stream, which waits
// for the last download before the call's end.
namespace wg {
namespace {

constexpr int kMaxHostPanels = 8;
constexpr int64_t kHostPanelBytes = 8ll << 20;  // A and C bytes per panel, at least
constexpr int kMaxHostBlocks = 4;
constexpr int64_t kHostBlockBytes = 128ll << 20;  // B bytes per block, at least
int g_debug_host_panels = 0;                     // see wgemm_debug_set_host_panels
int g_debug_host_blocks = 0;                     // see wgemm_debug_set_host_blocks

struct HostCopyStreams {
  bool init = false;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t landed[kMaxHostPanels] = {}, landed_b[kMaxHostBlocks] = {};
  cudaEvent_t computed[kMaxHostPanels * kMaxHostBlocks] = {};
};
std::mutex g_host_mu;  // one host-buffer call issues at a time
HostCopyStreams g_host[kMaxDevices];

int host_streams(int dev, HostCopyStreams** out) {
  HostCopyStreams& h = g_host[dev];
  if (!h.init) {
    bool ok = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.done, cudaEventDisableTiming) == cudaSuccess;
    for (int p = 0; ok && p < kMaxHostPanels; ++p)
      ok = cudaEventCreateWithFlags(&h.landed[p], cudaEventDisableTiming) == cudaSuccess;
    for (int b = 0; ok && b < kMaxHostBlocks; ++b)
      ok = cudaEventCreateWithFlags(&h.landed_b[b], cudaEventDisableTiming) == cudaSuccess;
    for (int q = 0; ok && q < kMaxHostPanels * kMaxHostBlocks; ++q)
      ok = cudaEventCreateWithFlags(&h.computed[q], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return WGEMM_ERR_LAUNCH;
    }
    h.init = true;
  }
  *out = &h;
  return WGEMM_OK;
}

// Panels of A's rows: as many as min(A bytes, C bytes) holds 8 MiB, 1 to 8,
// each a multiple of 256 rows (every configuration's tile height divides it).
// More panels overlap more of the copies with the GEMMs; the partly idle last
// wave of each panel's tiles costs less than that gains (one call at 16384³
// took 15.3, 11.7, 10.0 and 9.4 ms with 1, 2, 4 and 8 panels; 4096³ 0.77
// and 0.63 ms with 1 and 8). Returns the rows per panel.
int host_panel_rows(int M, int N, int K, int mode) {
  int64_t p = std::min<int64_t>(2ll * M * K, 4ll * M * N) / kHostPanelBytes;
  if (g_debug_host_panels > 0) p = g_debug_host_panels;
  if (mode != kDataParallel) p = 1;  // a K split keeps one launch
  p = std::max<int64_t>(1, std::min<int64_t>(p, kMaxHostPanels));
  int rows = (int)((M + p - 1) / p);
  rows = (rows + 255) / 256 * 256;
  return std::min(std::max(rows, 1), M);
}

// Blocks of B's rows (C's columns): as many as B's bytes hold 128 MiB, 1 to
// 4, each a multiple of 256 rows. The first half of the blocks goes up before
// A and the rest after it. No GEMM starts before its B block has landed, and
// after the last upload only the GEMMs of the last block remain, with their
// share of C to download: smaller blocks shorten both ends of the pipeline.
// One call at 16384³ (eight panels) took 9.3 ms with one block, 8.9 with two
// (the second after A). Returns B's rows (C's columns) per block.
int host_block_cols(int N, int K, int mode) {
  int64_t b = 2ll * N * K / kHostBlockBytes;
  if (g_debug_host_blocks > 0) b = g_debug_host_blocks;
  if (mode != kDataParallel) b = 1;  // a K split keeps one launch
  b = std::max<int64_t>(1, std::min<int64_t>(b, kMaxHostBlocks));
  int cols = (int)((N + b - 1) / b);
  cols = (cols + 255) / 256 * 256;
  return std::min(std::max(cols, 1), N);
}

int run_host(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C, int M, int N, int K, int lda,
             int ldb, int ldc, wgemm_f16_t* dA, wgemm_f16_t* dB, float* dC, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0) return WGEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return WGEMM_OK;
  if (!C || !dC || ldc < N) return WGEMM_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B || !dA || !dB || lda < K || ldb < K)) return WGEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dA) & 15) || (reinterpret_cast<uintptr_t>(dB) & 15) ||
      (reinterpret_cast<uintptr_t>(dC) & 15))
    return WGEMM_ERR_ALIGNMENT;
  const int64_t kd = ((int64_t)K + 7) / 8 * 8, nd = ((int64_t)N + 3) / 4 * 4;
  int config = -1, mode = -1, splits = 1;  // K == 0: the zero kernel, no configuration
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DeviceState* st;
    const int rc = device_state(&dev, &st);
    if (rc != WGEMM_OK) return rc;
    if (K > 0) {
      const Choice c = choose(*st, M, N, K, (int)kd, (int)kd, true, 0, 0, capturing(stream));
      config = c.config;
      mode = c.mode;
      splits = c.splits;
    }
  }
  std::lock_guard<std::mutex> lock(g_host_mu);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return WGEMM_ERR_NO_DEVICE;
  }
  HostCopyStreams* h;
  int rc = host_streams(dev, &h);
  if (rc != WGEMM_OK) return rc;
  const int rows = K > 0 ? host_panel_rows(M, N, K, mode) : M;
  const int panels = (M + rows - 1) / rows;
  const int cols = K > 0 ? host_block_cols(N, K, mode) : N;
  const int blocks = (N + cols - 1) / cols;
  // Everything before the call on the caller's stream comes first (the
  // caller's earlier use of dA, dB and dC included).
  if (cudaEventRecord(h->start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(h->up, h->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(h->down, h->start, 0) != cudaSuccess) {
    cudaGetLastError();
    return WGEMM_ERR_LAUNCH;
  }
  rc = WGEMM_OK;
  // Uploads in the order the GEMMs need them: the first half of B's blocks,
  // every panel of A, then B's other blocks. Each landing is marked by an
  // event.
  auto up_b = [&](int b) {
    const int c0 = b * cols, nb = std::min(cols, N - c0);
    if ((K > 0 && cudaMemcpy2DAsync(dB + (int64_t)c0 * kd, kd * 2, B + (int64_t)c0 * ldb,
                                    (size_t)ldb * 2, (size_t)K * 2, nb, cudaMemcpyHostToDevice,
                                    h->up) != cudaSuccess) ||
        cudaEventRecord(h->landed_b[b], h->up) != cudaSuccess)
      rc = WGEMM_ERR_LAUNCH;
  };
  const int head = (blocks + 1) / 2;  // B's blocks that go up before A
  for (int b = 0; b < head && rc == WGEMM_OK; ++b) up_b(b);
  for (int p = 0; p < panels && rc == WGEMM_OK; ++p) {
    const int r0 = p * rows, mp = std::min(rows, M - r0);
    if ((K > 0 && cudaMemcpy2DAsync(dA + (int64_t)r0 * kd, kd * 2, A + (int64_t)r0 * lda,
                                    (size_t)lda * 2, (size_t)K * 2, mp, cudaMemcpyHostToDevice,
                                    h->up) != cudaSuccess) ||
        cudaEventRecord(h->landed[p], h->up) != cudaSuccess)
      rc = WGEMM_ERR_LAUNCH;
  }
  for (int b = head; b < blocks && rc == WGEMM_OK; ++b) up_b(b);
  // The GEMM of rows [r0, r0 + mp) and columns [c0, c0 + nb) of the same
  // product (so the configuration chosen for the whole shape serves it), once
  // both operands have landed; then that piece of C goes down. Pieces run in
  // the order their operands land: panel by panel over the first blocks,
  // then block by block over the panels.
  auto piece = [&](int p, int b) {
    const int r0 = p * rows, mp = std::min(rows, M - r0);
    const int c0 = b * cols, nb = std::min(cols, N - c0);
    const int q = b * panels + p;
    rc = run(dA + (int64_t)r0 * kd, dB + (int64_t)c0 * kd, dC + (int64_t)r0 * nd + c0, WGEMM_F16,
             WGEMM_F32, mp, nb, K, (int)kd, (int)kd, (int)nd, config, mode, splits, stream);
    if (rc == WGEMM_OK &&
        (cudaEventRecord(h->computed[q], stream) != cudaSuccess ||
         cudaStreamWaitEvent(h->down, h->computed[q], 0) != cudaSuccess ||
         cudaMemcpy2DAsync(C + (int64_t)r0 * ldc + c0, (size_t)ldc * 4,
                           dC + (int64_t)r0 * nd + c0, nd * 4, (size_t)nb * 4, mp,
                           cudaMemcpyDeviceToHost, h->down) != cudaSuccess))
      rc = WGEMM_ERR_LAUNCH;
  };
  auto wait = [&](cudaEvent_t e) {
    if (rc == WGEMM_OK && cudaStreamWaitEvent(stream, e, 0) != cudaSuccess) rc = WGEMM_ERR_LAUNCH;
  };
  for (int b = 0; b < head; ++b) wait(h->landed_b[b]);
  for (int p = 0; p < panels && rc == WGEMM_OK; ++p) {
    wait(h->landed[p]);
    for (int b = 0; b < head && rc == WGEMM_OK; ++b) piece(p, b);
  }
  for (int b = head; b < blocks && rc == WGEMM_OK; ++b) {
    wait(h->landed_b[b]);
    for (int p = 0; p < panels && rc == WGEMM_OK; ++p) piece(p, b);
  }
  if (rc != WGEMM_OK) cudaGetLastError();
  // The caller's stream waits for both copy streams, also after an error,
  // so that synchronising it covers every copy this call enqueued.
  if (cudaEventRecord(h->done, h->down) != cudaSuccess ||
      cudaStreamWaitEvent(stream, h->done, 0) != cudaSuccess ||
      cudaEventRecord(h->done, h->up) != cudaSuccess ||
      cudaStreamWaitEvent(stream, h->done, 0) != cudaSuccess) {
    cudaGetLastError();
    if (rc == WGEMM_OK) rc = WGEMM_ERR_LAUNCH;
  }
  return rc;
}

}  // namespace
}  // namespace wg

extern "C" int wgemm_f16f32_host(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C, int M,
                                 int N, int K, int lda, int ldb, int ldc, wgemm_f16_t* dA,
                                 wgemm_f16_t* dB, float* dC, wgemm_stream_t stream) {
  return wg::run_host(A, B, C, M, N, K, lda, ldb, ldc, dA, dB, dC,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int wgemm_host_device_elems(int M, int N, int K, size_t* a_elems, size_t* b_elems,
                                       size_t* c_elems) {
  if (M < 0 || N < 0 || K < 0) return WGEMM_ERR_INVALID_ARG;
  const size_t kd = ((size_t)K + 7) / 8 * 8, nd = ((size_t)N + 3) / 4 * 4;
  if (a_elems) *a_elems = (size_t)M * kd;
  if (b_elems) *b_elems = (size_t)N * kd;
  if (c_elems) *c_elems = (size_t)M * nd;
  return WGEMM_OK;
}

extern "C" int wgemm_debug_set_host_panels(int panels) {
  if (panels < 0 || panels > wg::kMaxHostPanels) return WGEMM_ERR_INVALID_ARG;
  const int prev = wg::g_debug_host_panels;
  wg::g_debug_host_panels = panels;
  return prev;
}

extern "C" int wgemm_debug_host_panel_rows(int M, int N, int K) {
  if (M <= 0 || N < 0 || K <= 0) return WGEMM_ERR_INVALID_ARG;
  return wg::host_panel_rows(M, N, K, wg::kDataParallel);
}

extern "C" int wgemm_debug_set_host_blocks(int blocks) {
  if (blocks < 0 || blocks > wg::kMaxHostBlocks) return WGEMM_ERR_INVALID_ARG;
  const int prev = wg::g_debug_host_blocks;
  wg::g_debug_host_blocks = blocks;
  return prev;
}

extern "C" int wgemm_debug_host_block_cols(int N, int K) {
  if (N <= 0 || K <= 0) return WGEMM_ERR_INVALID_ARG;
  return wg::host_block_cols(N, K, wg::kDataParallel);
}

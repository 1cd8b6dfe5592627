// Which on-SM traffic slows tcgen05.mma? Every CTA pair of a full-chip grid
// runs the dominant kernel's MMA shape (pair M256 N224, K = 64 per
// iteration) back to back on operands resident in shared memory, as the
// tensor-pipe ceiling benchmark does, while four more warps of each CTA make
// one kind of traffic for exactly as long as the MMAs run:
//
//   none      nothing
//   gst       scalar fp32 global stores, 128 B per warp instruction, to a
//             per-warp 64 KB region (the chip's regions stay in L2)
//   gst_v4    the same with 16-byte vector stores (512 B per instruction)
//   epi       the register-store epilogue's pattern: tcgen05.ld of 32 × 32
//             accumulator values, then 32 stores of 128 B to 32 rows 16 KB apart
//   sts       shared-memory stores, 128 B per warp instruction
//   lds       shared-memory loads, 128 B per warp instruction
//   tmem_ld   tcgen05.ld 32x32b.x32 from TMEM columns the MMAs do not use
//   tmem_x16  the same bytes in 32x32b.x16 loads (half the columns per load)
//   tmem_x64  the same bytes in 32x32b.x64 loads (twice the columns per load)
//   bulk      cp.async.bulk global → shared, 16 KB copies, four in flight
//             per CTA (what the TMA producer does in the k-loop)
//
// For each mode: MMA TFLOP/s and the traffic's bytes per µs per SM over the
// MMA window. Prints one JSON line per mode.
//
// Every wait is bounded (2 s) and sets a failure flag; the traffic loops
// stop when the CTA's MMAs complete, or after 2 s. All accesses stay inside
// their buffers: global offsets are taken modulo the region sizes, shared
// offsets stay inside the 64 KB traffic region, TMEM columns inside the
// 512 allocated.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "../csrc/sm103/ptx.cuh"
#include "../csrc/sm103/umma_desc.h"

using namespace wg;

namespace {

constexpr int kSrcElems = 1 << 20;
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr int kN = 224;                        // MMA N (pair: 112 B rows per CTA)
constexpr int kAbytes = 128 * 128;             // 128 rows × 64 fp16
constexpr int kBbytes = (kN / 2) * 128;        // this CTA's half of B
constexpr int kOpBytes = 32 * 1024;            // operand region (A + B, rounded up)
constexpr int kTrafficBytes = 64 * 1024;       // shared-memory traffic region
constexpr int kSmem = kOpBytes + kTrafficBytes + 1024 + 1024;
constexpr int kWarpRegion = 64 * 1024;         // global bytes per traffic warp
constexpr int kEpiPitch = 4096;                // floats per row in the epi pattern
constexpr int kEpiColBlocks = 8;               // 32-column blocks cycled through
constexpr int kBulkBytes = 16 * 1024;
constexpr int kBulkSrcBytes = 1 << 20;

enum Mode { kNone, kGst, kGstV4, kEpi, kSts, kLds, kTmemLd, kBulk, kTmemX16, kTmemX64, kModes };
const char* const kModeNames[kModes] = {"none", "gst",  "gst_v4",   "epi",     "sts",
                                        "lds",  "tmem_ld", "bulk", "tmem_x16", "tmem_x64"};

// 32 lanes × 16 / 64 consecutive 32-bit columns per thread (cf. the x32 load).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}

__device__ bool wait_parity(uint32_t bar, uint32_t parity) {
  const unsigned long long w0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - w0 > kWaitNs) return false;
  return true;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}

// 256 threads: warps 0-3 set up and warp 0 issues the MMAs; warps 4-7 make
// the traffic of `mode`.
__global__ void __launch_bounds__(256, 1)
    mma_with_traffic(const uint16_t* src, const uint8_t* bulk_src, float* gdst, int mode,
                     int iters, unsigned long long* t, unsigned long long* bytes, int* failed) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw), base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t traffic = base + kOpBytes;
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ __align__(8) uint64_t bar_bulk[4];
  __shared__ volatile int done;
  const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank() & 1u;
  for (int i = threadIdx.x; i < (kAbytes + kBbytes) / 2; i += blockDim.x)
    reinterpret_cast<uint16_t*>(smem)[i] = src[(blockIdx.x * 977 + i) % kSrcElems];
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar_mma), 1);
    for (int s = 0; s < 4; ++s) mbar_init(smem_addr(&bar_bulk[s]), 1);
    done = 0;
    fence_mbarrier_init();
  }
  fence_proxy_async_shared();
  if (warp == 0) {
    tmem_alloc<2>(smem_addr(&tmem_slot), 512);
    tmem_relinquish<2>();
  }
  tcgen05_fence_before();
  cluster_sync();
  tcgen05_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    const unsigned long long t0 = global_timer_ns();
    if (rank == 0) {
      constexpr uint32_t idesc = umma_idesc_f16(256, kN);
      for (int it = 0; it < iters; ++it)
        for (int j = 0; j < 4; ++j)
          umma_f16<2>(tmem, umma_smem_desc_sw128(base + j * 32),
                      umma_smem_desc_sw128(base + kAbytes + j * 32), idesc, 1u);
      umma_commit_pair_multicast(smem_addr(&bar_mma), 3);
    }
    // Both CTAs of the pair receive the commit.
    const bool ok = wait_parity(smem_addr(&bar_mma), 0);
    done = 1;
    if (rank == 0) {
      t[2 * blockIdx.x] = t0;
      t[2 * blockIdx.x + 1] = ok ? global_timer_ns() : 0ull;
    }
    if (!ok) atomicExch(failed, 1);
  } else if (warp >= 4 && mode != kNone) {
    const uint32_t q = warp - 4;
    const unsigned long long t0 = global_timer_ns();
    unsigned long long n = 0;  // bytes moved by this warp
    float acc = 0.f;
    uint32_t r[32];
    float* region = gdst + ((size_t)blockIdx.x * 4 + q) * (kWarpRegion / 4);
    const uint32_t taddr = tmem + ((32u * q) << 16) + 256u;  // columns 256-511: not the MMA's
    bool quit = false;  // lane 0 of the bulk mode gave up on a wait
    for (uint32_t it = 0;; ++it) {
      // The warp leaves together: tcgen05.ld is .sync.aligned.
      if ((it & 15u) == 0u) {
        bool stop = done != 0 || quit;
        if (global_timer_ns() - t0 > kWaitNs) {
          stop = true;
          if (lane == 0) atomicExch(failed, 2);
        }
        if (__any_sync(0xFFFFFFFFu, stop)) break;
      }
      switch (mode) {
        case kGst: {
          region[(it * 32u + lane) % (kWarpRegion / 4)] = (float)it;
          n += 128;
          break;
        }
        case kGstV4: {
          float4* p = reinterpret_cast<float4*>(region);
          p[(it * 32u + lane) % (kWarpRegion / 16)] = make_float4(1.f, 2.f, 3.f, (float)it);
          n += 512;
          break;
        }
        case kEpi: {
          tmem_ld_32x32b_x32(taddr + (it % 8u) * 32u, r);
          tmem_ld_wait();
          // 32 rows of a kEpiPitch-float matrix; this warp's 32 rows start at
          // row 32·q of the CTA's slab, the column block cycles.
          float* slab = gdst + (size_t)blockIdx.x * 128 * kEpiPitch;
          const uint32_t col = (it % kEpiColBlocks) * 32u + lane;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            slab[(size_t)(32u * q + e) * kEpiPitch + col] = __uint_as_float(r[e]);
          n += 32 * 128;
          break;
        }
        case kSts: {
          sts_f32(traffic + q * 16384u + ((it * 128u) & 16383u) + lane * 4u, (float)it);
          n += 128;
          break;
        }
        case kLds: {
          acc += lds_f32(traffic + q * 16384u + ((it * 128u) & 16383u) + lane * 4u);
          n += 128;
          break;
        }
        case kTmemLd: {
          tmem_ld_32x32b_x32(taddr + (it % 8u) * 32u, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) acc += __uint_as_float(r[e]);
          n += 32 * 128;
          break;
        }
        case kTmemX16: {  // two x16 loads per iteration: the bytes of one x32
          uint32_t r16a[16], r16b[16];
          tmem_ld_x16(taddr + (it % 8u) * 32u, r16a);
          tmem_ld_x16(taddr + (it % 8u) * 32u + 16u, r16b);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) acc += __uint_as_float(r16a[e]) + __uint_as_float(r16b[e]);
          n += 32 * 128;
          break;
        }
        case kTmemX64: {  // one x64 load per iteration: the bytes of two x32
          uint32_t r64[64];
          tmem_ld_x64(taddr + (it % 4u) * 64u, r64);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 64; ++e) acc += __uint_as_float(r64[e]);
          n += 64 * 128;
          break;
        }
        case kBulk: {
          // Warp 4, lane 0 only: 16 KB copies into four 16 KB slots of the
          // traffic region, at most four in flight.
          if (q == 0 && lane == 0 && !quit) {
            const uint32_t k = (uint32_t)(n / kBulkBytes);  // copies issued so far
            const uint32_t slot = k % 4u, use = k / 4u;
            if (use > 0 && !wait_parity(smem_addr(&bar_bulk[slot]), (use - 1) & 1u)) {
              atomicExch(failed, 3);
              quit = true;  // stop issuing; the drain below still waits
            } else {
              mbar_arrive_expect_tx(smem_addr(&bar_bulk[slot]), kBulkBytes);
              bulk_g2s(traffic + slot * kBulkBytes,
                       bulk_src + (size_t)(k % (kBulkSrcBytes / kBulkBytes)) * kBulkBytes,
                       kBulkBytes, smem_addr(&bar_bulk[slot]));
              n += kBulkBytes;
            }
          }
          break;
        }
        default:
          break;
      }
    }
    if (mode == kBulk && q == 0 && lane == 0) {
      // Wait for every copy still in flight: slot s was used uses(s) times.
      const unsigned long long issued = n / kBulkBytes;
      for (uint32_t s = 0; s < 4 && s < issued; ++s) {
        const unsigned long long uses = (issued - s + 3) / 4;
        if (!wait_parity(smem_addr(&bar_bulk[s]), (uint32_t)((uses - 1) & 1u)))
          atomicExch(failed, 4);
      }
    }
    if (acc == 12345.678f) gdst[0] = acc;  // keeps the loads
    if (mode == kBulk) {
      if (lane == 0 && q == 0) atomicAdd(bytes, n);
    } else if (lane == 0) {
      atomicAdd(bytes, n);
    }
  }
  __syncwarp();
  tcgen05_fence_before();
  cluster_sync();
  if (warp == 0) {
    tcgen05_fence_after();
    tmem_dealloc<2>(tmem, 512);
  }
}

#define CHECK(x)                                                              \
  do {                                                                        \
    cudaError_t e_ = (x);                                                     \
    if (e_ != cudaSuccess) {                                                  \
      std::fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));           \
      std::exit(1);                                                           \
    }                                                                         \
  } while (0)

}  // namespace

int main(int argc, char** argv) {
  const int iters = argc > 1 ? std::atoi(argv[1]) : 10000;
  int sms = 0;
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  const int grid = (sms / 2) * 2;
  std::vector<uint16_t> h(kSrcElems);
  std::srand(1);
  for (auto& x : h)  // fp16 magnitudes in [0.125, 0.5), both signs
    x = (uint16_t)((0x3000 + (std::rand() & 0x7FF)) ^ ((std::rand() & 1) << 15));
  uint16_t* src = nullptr;
  uint8_t* bulk_src = nullptr;
  float* gdst = nullptr;
  unsigned long long *t = nullptr, *bytes = nullptr;
  int* failed = nullptr;
  // Global traffic buffer: the larger of the store regions (4 × 64 KB per
  // CTA) and the epi slabs (128 rows × kEpiPitch floats per CTA).
  const size_t gdst_bytes =
      std::max((size_t)grid * 4 * kWarpRegion, (size_t)grid * 128 * kEpiPitch * sizeof(float));
  CHECK(cudaMalloc(&src, h.size() * sizeof(uint16_t)));
  CHECK(cudaMemcpy(src, h.data(), h.size() * sizeof(uint16_t), cudaMemcpyHostToDevice));
  CHECK(cudaMalloc(&bulk_src, kBulkSrcBytes));
  CHECK(cudaMemset(bulk_src, 0x3c, kBulkSrcBytes));
  CHECK(cudaMalloc(&gdst, gdst_bytes));
  CHECK(cudaMalloc(&t, grid * 2 * sizeof(unsigned long long)));
  CHECK(cudaMalloc(&bytes, sizeof(unsigned long long)));
  CHECK(cudaMalloc(&failed, sizeof(int)));
  CHECK(cudaFuncSetAttribute(mma_with_traffic, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             std::max(kSmem, 120 * 1024)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = std::max(kSmem, 120 * 1024);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int reps = 4;  // the first launch of each mode warms up
  for (int mode = 0; mode < kModes; ++mode) {
    std::vector<double> tfs, gbs;
    for (int rep = 0; rep < reps; ++rep) {
      CHECK(cudaMemset(t, 0, grid * 2 * sizeof(unsigned long long)));
      CHECK(cudaMemset(bytes, 0, sizeof(unsigned long long)));
      CHECK(cudaMemset(failed, 0, sizeof(int)));
      CHECK(cudaLaunchKernelEx(&cfg, mma_with_traffic, (const uint16_t*)src,
                               (const uint8_t*)bulk_src, gdst, mode, iters, t, bytes, failed));
      CHECK(cudaDeviceSynchronize());
      int hf = 0;
      unsigned long long hb = 0;
      CHECK(cudaMemcpy(&hf, failed, sizeof(int), cudaMemcpyDeviceToHost));
      CHECK(cudaMemcpy(&hb, bytes, sizeof(hb), cudaMemcpyDeviceToHost));
      if (hf) {
        std::fprintf(stderr, "%s: a bounded wait expired (%d)\n", kModeNames[mode], hf);
        return 1;
      }
      std::vector<unsigned long long> ht(grid * 2);
      CHECK(cudaMemcpy(ht.data(), t, ht.size() * sizeof(unsigned long long),
                       cudaMemcpyDeviceToHost));
      unsigned long long lo = ~0ull, hi = 0;
      int n = 0;
      for (int b = 0; b < grid; ++b)
        if (ht[2 * b + 1]) {
          lo = std::min(lo, ht[2 * b]);
          hi = std::max(hi, ht[2 * b + 1]);
          ++n;
        }
      const double us = (hi - lo) * 1e-3;
      const double flops = 2.0 * 256 * kN * 64 * (double)iters * n;
      if (rep > 0) {
        tfs.push_back(flops / (us * 1e-6) / 1e12);
        gbs.push_back((double)hb / grid / us * 1e-3);  // GB/s per SM
      }
    }
    std::sort(tfs.begin(), tfs.end());
    std::sort(gbs.begin(), gbs.end());
    std::printf("{\"mode\": \"%s\", \"tflops\": %.1f, \"traffic_gbs_per_sm\": %.1f}\n",
                kModeNames[mode], tfs[tfs.size() / 2], gbs[gbs.size() / 2]);
    std::fflush(stdout);
  }
  CHECK(cudaFree(src));
  CHECK(cudaFree(bulk_src));
  CHECK(cudaFree(gdst));
  CHECK(cudaFree(t));
  CHECK(cudaFree(bytes));
  CHECK(cudaFree(failed));
  return 0;
}

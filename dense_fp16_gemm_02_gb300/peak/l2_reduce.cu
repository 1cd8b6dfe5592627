// How fast do bulk reduce-adds into C run in L2? The split-K and stream-K
// epilogues add fp32 partial tiles into C with TMA reduce-adds, several
// units into one tile at about the same time. Here lane 0 of `issuers` warps
// per CTA of a full-chip grid (one CTA per SM) writes blocks of fp32 (4 KB by
// default, the epilogue's 32 × 32 block) from shared memory to global memory
// with the bulk copy engine, up to 16 groups in flight per issuing thread, the
// way the epilogue's tail staging does:
//
//   store        plain bulk stores, every CTA to its own 256 KB region
//   add          bulk reduce-adds (.add.f32), every CTA to its own region
//   add_shared9  bulk reduce-adds, nine CTAs into the same region in the same
//                block order (a tile's nine split-K units)
//   add_rot9     as add_shared9, each of the nine starting at a different
//                block (rotated by its index in the group)
//   red_v4       no bulk copies: warps 1–3 add their blocks from registers
//                with red.global.add.v4.f32 (16 bytes per lane), every CTA
//                into its own region
//   add_mixed    both paths at once: lane 0 of warp 0 bulk-adds the blocks
//                b ≡ 0 (mod 4), warps 1–3 red-add the others from registers
//
// In red_v4 and add_mixed the block size is 4 KB and `issuers` is ignored.
// Each CTA covers its region `passes` times; its issuing warps take its
// blocks in turn. Usage: l2_reduce [passes] [block bytes] [issuing warps]
// [CTAs] (default: every SM, in whole groups of nine).
// Prints one JSON line per mode: bytes moved, kernel time (CUDA events,
// median of five after one warm-up) and GB/s, and whether C holds the
// expected values afterwards.
//
// All addresses stay inside their buffers (block indices are taken modulo
// the region's blocks; regions are allocated for the grid); there are no
// spin-waits, only the bulk-group waits of the copies each thread issued.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

namespace {

constexpr int kRegionBytes = 256 * 1024;  // a CTA's half of a 512 × 256 pair tile
constexpr int kSrcBytes = 64 * 1024;      // shared-memory source
constexpr int kGroup = 9;                 // CTAs adding into one region
constexpr float kValue = 1.0f;

enum Mode { kStore, kAdd, kAddShared9, kAddRot9, kRedV4, kAddMixed, kModes };
const char* const kModeNames[kModes] = {"store",    "add",    "add_shared9",
                                        "add_rot9", "red_v4", "add_mixed"};

// Warps 1–3 add 4 KB blocks of the value from registers: every lane adds 16
// bytes per instruction, a warp covers a block in 8 instructions. With `all`
// set, block b goes to warp 1 + b mod 3; otherwise blocks b ≡ w (mod 4) go
// to warp w and the blocks b ≡ 0 are left to the bulk path.
__device__ void red_blocks(unsigned char* base, int passes, int warp, bool all) {
  const int lane = (int)threadIdx.x % 32;
  constexpr int kBlk = 4096, kBlocksR = kRegionBytes / kBlk;
  for (int p = 0; p < passes; ++p) {
    for (int b = 0; b < kBlocksR; ++b) {
      const int owner = all ? 1 + b % 3 : b % 4;
      if (owner != warp) continue;
      float* blk = reinterpret_cast<float*>(base + (size_t)b * kBlk);
#pragma unroll
      for (int i = 0; i < kBlk / 512; ++i) {
        float* d = blk + (i * 32 + lane) * 4;
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
                     :: "l"(__cvta_generic_to_global(d)), "f"(kValue), "f"(kValue),
                        "f"(kValue), "f"(kValue) : "memory");
      }
    }
  }
}

#define CHECK(x)                                                                   \
  do {                                                                             \
    cudaError_t e_ = (x);                                                          \
    if (e_ != cudaSuccess) {                                                       \
      std::fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                \
      std::exit(1);                                                                \
    }                                                                              \
  } while (0)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__global__ void __launch_bounds__(128) bulk_kernel(float* dst, int mode, int passes,
                                                   int block_bytes, int issuers) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* src = reinterpret_cast<float*>(smem);
  for (int i = threadIdx.x; i < kSrcBytes / 4; i += blockDim.x) src[i] = kValue;
  // Make the generic-proxy writes visible to the bulk copies.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  const int warp = (int)threadIdx.x / 32;
  if (mode == kRedV4 || mode == kAddMixed) {
    unsigned char* own = reinterpret_cast<unsigned char*>(dst) + (size_t)blockIdx.x * kRegionBytes;
    if (warp >= 1) {
      red_blocks(own, passes, warp, mode == kRedV4);
      return;
    }
    if (mode == kRedV4 || threadIdx.x != 0) return;
    // Lane 0 of warp 0: bulk reduce-adds of the blocks b ≡ 0 (mod 4).
    for (int p = 0; p < passes; ++p) {
      for (int b = 0; b < kRegionBytes / 4096; b += 4) {
        const uint32_t s = smem_addr(smem + (b % (kSrcBytes / 4096)) * 4096);
        const size_t d = __cvta_generic_to_global(own + (size_t)b * 4096);
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
                     :: "l"(d), "r"(s), "r"(4096) : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 15;" ::: "memory");
      }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    return;
  }
  if (threadIdx.x % 32 != 0 || warp >= issuers) return;
  const int blocks = kRegionBytes / block_bytes;
  const int src_blocks = kSrcBytes / block_bytes;
  const bool shared9 = mode == kAddShared9 || mode == kAddRot9;
  const int region = shared9 ? (int)blockIdx.x / kGroup : (int)blockIdx.x;
  const int rot = mode == kAddRot9 ? ((int)blockIdx.x % kGroup) * (blocks / kGroup) : 0;
  unsigned char* base = reinterpret_cast<unsigned char*>(dst) + (size_t)region * kRegionBytes;
  for (int p = 0; p < passes; ++p) {
    for (int b = warp; b < blocks; b += issuers) {
      const int blk = (b + rot) % blocks;
      const uint32_t s = smem_addr(smem + (b % src_blocks) * block_bytes);
      const size_t d = __cvta_generic_to_global(base + (size_t)blk * block_bytes);
      if (mode == kStore)
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                     :: "l"(d), "r"(s), "r"(block_bytes) : "memory");
      else
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
                     :: "l"(d), "r"(s), "r"(block_bytes) : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      // At most 16 groups in flight (the source blocks are never rewritten).
      asm volatile("cp.async.bulk.wait_group.read 15;" ::: "memory");
    }
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace

int main(int argc, char** argv) {
  const int passes = argc > 1 ? std::max(1, std::atoi(argv[1])) : 8;
  // Block size: a power of two from 1 KB to 64 KB; issuing warps: 1 to 4.
  const int block_bytes = argc > 2 ? std::atoi(argv[2]) : 4096;
  if (block_bytes < 1024 || block_bytes > kSrcBytes || (block_bytes & (block_bytes - 1))) {
    std::fprintf(stderr, "block bytes: a power of two in [1024, %d]\n", kSrcBytes);
    return 2;
  }
  const int issuers = argc > 3 ? std::min(4, std::max(1, std::atoi(argv[3]))) : 1;
  int dev = 0, sms = 0;
  CHECK(cudaSetDevice(dev));
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  int grid = sms / kGroup * kGroup;  // whole groups of nine
  if (argc > 4) grid = std::min(grid, std::max(1, std::atoi(argv[4]) / kGroup) * kGroup);
  const int smem = kSrcBytes;
  CHECK(cudaFuncSetAttribute(bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  const size_t elems = (size_t)grid * kRegionBytes / 4;
  float* dst = nullptr;
  CHECK(cudaMalloc(&dst, elems * 4));
  std::vector<float> host(elems);
  cudaEvent_t e0, e1;
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));
  for (int mode = 0; mode < kModes; ++mode) {
    const bool shared9 = mode == kAddShared9 || mode == kAddRot9;
    std::vector<float> ms;
    bool ok = true;
    for (int rep = 0; rep < 6; ++rep) {
      CHECK(cudaMemset(dst, 0, elems * 4));
      CHECK(cudaEventRecord(e0));
      bulk_kernel<<<grid, 128, smem>>>(dst, mode, passes, block_bytes, issuers);
      CHECK(cudaEventRecord(e1));
      CHECK(cudaEventSynchronize(e1));
      CHECK(cudaGetLastError());
      float t = 0.f;
      CHECK(cudaEventElapsedTime(&t, e0, e1));
      if (rep > 0) ms.push_back(t);
      if (rep == 0) {
        // Every element of a written region holds the expected value.
        CHECK(cudaMemcpy(host.data(), dst, elems * 4, cudaMemcpyDeviceToHost));
        const int regions = shared9 ? grid / kGroup : grid;
        const float want = mode == kStore ? kValue
                           : shared9     ? kValue * (float)(kGroup * passes)
                                         : kValue * (float)passes;  // every block once per pass
        for (size_t i = 0; i < (size_t)regions * kRegionBytes / 4; ++i)
          if (host[i] != want) {
            ok = false;
            break;
          }
      }
    }
    std::sort(ms.begin(), ms.end());
    const double us = ms[ms.size() / 2] * 1e3;
    const double bytes = (double)grid * passes * kRegionBytes;
    std::printf("{\"mode\": \"%s\", \"ctas\": %d, \"passes\": %d, \"block_bytes\": %d, "
                "\"issuers\": %d, \"bytes\": %.0f, \"us\": %.2f, \"gbs\": %.1f, "
                "\"gbs_per_sm\": %.2f, \"result_ok\": %s}\n",
                kModeNames[mode], grid, passes, block_bytes, issuers, bytes, us,
                bytes / us / 1e3, bytes / us / 1e3 / grid, ok ? "true" : "false");
  }
  CHECK(cudaFree(dst));
  return 0;
}

// Tensor-pipe ceiling of this GPU for tcgen05.mma.kind::f16: every CTA (or
// CTA pair) issues back-to-back MMAs on operands resident in its shared
// memory, with no global-memory traffic inside the timed loop. One thread per
// MMA group issues; the loop's start and end (after a commit that waits for
// every issued MMA) are read from %globaltimer. The figure bounds what any
// kernel of the GEMM family can reach on the same MMA shape, and is the
// denominator of no reported fraction (the roofline uses the driver-measured
// peak); it shows how far that peak sits below the pipe itself.
//
// Prints one JSON line per MMA shape: {"shape", "issuers", "us", "tflops"}.
// Every wait is bounded (2 s), and all memory accesses stay inside the
// buffers: operands come from a 1 Mi-element source array indexed modulo its
// size, and the timing array holds two values per CTA.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "../csrc/sm103/ptx.cuh"
#include "../csrc/sm103/umma_desc.h"

using namespace wg;

namespace {

constexpr int kSrcElems = 1 << 20;
constexpr unsigned long long kWaitNs = 2000000000ull;

// Bounded wait for phase 0 of an mbarrier; false if it did not complete.
__device__ bool wait_phase0(uint32_t bar) {
  const unsigned long long w0 = global_timer_ns();
  while (!mbar_try_wait(bar, 0))
    if (global_timer_ns() - w0 > kWaitNs) return false;
  return true;
}

// CG CTAs per MMA (1, or a pair), MMA N, and REPS stacked M atoms per CTA.
template <int CG, int N, int REPS>
__global__ void __launch_bounds__(128, 1)
    mma_loop(const uint16_t* src, int iters, unsigned long long* t, int* failed) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw), base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  constexpr int kAbytes = 128 * 128 * REPS;  // MMA-A: 128 rows × 64 fp16 per atom
  constexpr int kBbytes = (N / CG) * 128;    // this CTA's share of MMA-B
  // Real fp16 values (not zeros) so that the tensor pipe does real work.
  for (int i = threadIdx.x; i < (kAbytes + kBbytes) / 2; i += blockDim.x)
    reinterpret_cast<uint16_t*>(smem)[i] = src[(blockIdx.x * 977 + i) % kSrcElems];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bar;
  const uint32_t rank = CG == 2 ? (cluster_ctarank() & 1u) : 0u;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbarrier_init();
  }
  fence_proxy_async_shared();  // operands written by the generic proxy, read by the MMA
  if (threadIdx.x / 32 == 0) {
    tmem_alloc<CG>(smem_addr(&tmem_slot), 512);
    tmem_relinquish<CG>();
  }
  tcgen05_fence_before();
  if (CG == 2) cluster_sync(); else __syncthreads();
  tcgen05_fence_after();
  const uint32_t tmem = tmem_slot;
  constexpr uint32_t idesc = umma_idesc_f16(128 * CG, N);
  if (threadIdx.x == 0 && rank == 0) {
    const unsigned long long t0 = global_timer_ns();
    for (int it = 0; it < iters; ++it)
      for (int r = 0; r < REPS; ++r)
        for (int j = 0; j < 4; ++j)  // K = 64 per iteration: four MMAs of K = 16
          umma_f16<CG>(tmem + r * N, umma_smem_desc_sw128(base + r * 16384 + j * 32),
                       umma_smem_desc_sw128(base + kAbytes + j * 32), idesc, 1u);
    if (CG == 1) umma_commit(smem_addr(&bar));
    else umma_commit_pair_multicast(smem_addr(&bar), 3);
    const bool ok = wait_phase0(smem_addr(&bar));
    t[2 * blockIdx.x] = t0;
    t[2 * blockIdx.x + 1] = ok ? global_timer_ns() : 0ull;
    if (!ok) atomicExch(failed, 1);
  }
  if (CG == 2 && rank == 1 && threadIdx.x == 0) {
    // The pair's commit also arrives here; wait so TMEM is not freed early.
    if (!wait_phase0(smem_addr(&bar))) atomicExch(failed, 1);
  }
  tcgen05_fence_before();
  if (CG == 2) cluster_sync(); else __syncthreads();
  if (threadIdx.x / 32 == 0) {
    tcgen05_fence_after();
    tmem_dealloc<CG>(tmem, 512);
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

template <int CG, int N, int REPS>
void measure(const char* name, const uint16_t* src, int sms, int iters, int reps) {
  const int grid = (sms / CG) * CG;
  // At least 120 KB of shared memory: one CTA, and one 512-column TMEM
  // allocation, per SM.
  const int smem = std::max(128 * 128 * REPS + (N / CG) * 128 + 2048, 120 * 1024);
  CHECK(cudaFuncSetAttribute(mma_loop<CG, N, REPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem));
  unsigned long long* t = nullptr;
  int* failed = nullptr;
  CHECK(cudaMalloc(&t, grid * 2 * sizeof(unsigned long long)));
  CHECK(cudaMalloc(&failed, sizeof(int)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  std::vector<double> tfs, uss;
  int issuers = 0;
  for (int rep = 0; rep < reps; ++rep) {
    CHECK(cudaMemset(t, 0, grid * 2 * sizeof(unsigned long long)));
    CHECK(cudaMemset(failed, 0, sizeof(int)));
    CHECK(cudaLaunchKernelEx(&cfg, mma_loop<CG, N, REPS>, src, iters, t, failed));
    CHECK(cudaDeviceSynchronize());
    int hf = 0;
    CHECK(cudaMemcpy(&hf, failed, sizeof(int), cudaMemcpyDeviceToHost));
    if (hf) {
      std::fprintf(stderr, "%s: a bounded wait expired\n", name);
      std::exit(1);
    }
    std::vector<unsigned long long> h(grid * 2);
    CHECK(cudaMemcpy(h.data(), t, h.size() * sizeof(unsigned long long),
                     cudaMemcpyDeviceToHost));
    unsigned long long lo = ~0ull, hi = 0;
    int n = 0;
    for (int b = 0; b < grid; ++b)
      if (h[2 * b + 1]) {
        lo = std::min(lo, h[2 * b]);
        hi = std::max(hi, h[2 * b + 1]);
        ++n;
      }
    const double flops = 2.0 * 128 * CG * N * 64 * REPS * (double)iters * n;
    const double tf = flops / ((hi - lo) * 1e-9) / 1e12;
    if (rep > 0) {  // the first launch warms up
      tfs.push_back(tf);
      uss.push_back((hi - lo) / 1e3);
      issuers = n;
    }
  }
  // Median of the timed launches.
  std::sort(tfs.begin(), tfs.end());
  std::sort(uss.begin(), uss.end());
  std::printf("{\"shape\": \"%s\", \"issuers\": %d, \"us\": %.1f, \"tflops\": %.1f}\n", name,
              issuers, uss[uss.size() / 2], tfs[tfs.size() / 2]);
  std::fflush(stdout);
  CHECK(cudaFree(t));
  CHECK(cudaFree(failed));
}

}  // namespace

int main(int argc, char** argv) {
  const int iters = argc > 1 ? std::atoi(argv[1]) : 20000;
  int sms = 0;
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  std::vector<uint16_t> h(kSrcElems);
  std::srand(1);
  for (auto& x : h)  // fp16 magnitudes in [0.125, 0.5), both signs
    x = (uint16_t)((0x3000 + (std::rand() & 0x7FF)) ^ ((std::rand() & 1) << 15));
  uint16_t* src = nullptr;
  CHECK(cudaMalloc(&src, h.size() * sizeof(uint16_t)));
  CHECK(cudaMemcpy(src, h.data(), h.size() * sizeof(uint16_t), cudaMemcpyHostToDevice));
  measure<2, 256, 1>("pair M256 N256", src, sms, iters, 4);
  measure<2, 224, 1>("pair M256 N224", src, sms, iters, 4);
  measure<2, 192, 1>("pair M256 N192", src, sms, iters, 4);
  measure<2, 256, 2>("pair M256 N256, 2 atoms", src, sms, iters / 2, 4);
  measure<1, 256, 1>("single M128 N256", src, sms, iters, 4);
  measure<1, 128, 1>("single M128 N128", src, sms, iters, 4);
  // The small shapes' tiles: N = 64 per MMA.
  measure<1, 64, 1>("single M128 N64", src, sms, iters, 4);
  measure<2, 64, 1>("pair M256 N64", src, sms, iters, 4);
  CHECK(cudaFree(src));
  return 0;
}

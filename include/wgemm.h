/*
 * wgemm — dense GEMM C = A·Bᵀ for NVIDIA GB300 (sm_103a): fp16 A and B,
 * fp32 accumulation, fp32 C; and the same with bf16 A and B and/or a 16-bit
 * (fp16 or bf16) C.
 *
 * The operation is the one "SASS-Level Kernel Generation for Blackwell"
 * measures (section "The numbers", Setup paragraph: fp16 inputs, fp32
 * accumulation and output, C = A·Bᵀ), with its M × N × K shape convention
 * (table of section "The numbers"):
 *
 *     C[i·ldc + j] = Σ_{k<K} A[i·lda + k] · B[j·ldb + k]
 *     for 0 ≤ i < M, 0 ≤ j < N.
 *
 * A is M×K and B is N×K, both row-major (K contiguous); C is M×N row-major.
 * C is overwritten (no alpha/beta). The sum is accumulated in fp32 on the
 * tensor cores; its rounding order is unspecified.
 *
 * Memory. Every matrix pointer is a DEVICE pointer into the current CUDA
 * device's memory, owned by the caller. The library never frees or keeps a
 * caller pointer past the call's completion on `stream`.
 *
 * Asynchrony. Calls enqueue work on `stream` (a cudaStream_t; NULL = the
 * legacy default stream) and return without synchronising. Argument errors are
 * reported before anything is enqueued. A kernel that fails at run time (a
 * bounded wait that expired) records it in a per-device status word that
 * wgemm_check() reads.
 *
 * No CPU fallback, no vendor BLAS: an unsupported argument is an error.
 *
 * Library state. The library keeps, per device: the kernel attributes and
 * occupancy it queried, and, per (device, stream), a small flag workspace for
 * the split-K and stream-K paths (allocated on first need with cudaMalloc,
 * grown when needed, freed by wgemm_release_workspace()). Calls on different
 * streams may run concurrently. The split-K and stream-K kernels (and their
 * mixes) wait on flags that other CTAs of the same grid raise, so they are
 * launched cooperatively: such a grid starts only once all of its CTAs fit on
 * the GPU beside whatever else runs there, and then all are resident at once.
 * A K-split call beside a long-running kernel from another stream therefore
 * waits for room instead of running part of its grid.
 *
 * Host threads. The GEMM entry points may be called from several host threads
 * at once; the library's state is guarded by its own locks (a call holds them
 * while it chooses and enqueues, not while the GPU runs). The wgemm_debug_*
 * hooks set process-wide values without a lock: set them while no call is in
 * progress.
 *
 * CUDA graphs. The calls may be captured into a CUDA graph (stream
 * capture) after one call of the same shape outside the capture has set up
 * the library's per-device state. While `stream` is capturing, the choice
 * takes data-parallel plans only: a K-split plan's flags carry a per-call
 * epoch fixed in the kernel parameters, which a replayed graph would repeat.
 * A K-split mode forced during capture, and wgemm_f16f32_splitk_noalloc,
 * return WGEMM_ERR_CONFIG there, with nothing enqueued.
 */
#ifndef WGEMM_H
#define WGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same struct tag as CUDA's runtime and driver headers). */
typedef struct CUstream_st* wgemm_stream_t;

/* An fp16 (IEEE binary16) value, passed as its bit pattern. */
typedef uint16_t wgemm_f16_t;

/* A bf16 (bfloat16: the upper 16 bits of an IEEE binary32) value, as its bit pattern. */
typedef uint16_t wgemm_bf16_t;

/* Element types of wgemm_gemm. */
#define WGEMM_F32 0
#define WGEMM_F16 1
#define WGEMM_BF16 2

/* Status codes. */
#define WGEMM_OK 0
#define WGEMM_ERR_INVALID_ARG -1      /* M/N/K < 0, NULL with a non-empty operand, lda < K, ldb < K, ldc < N, an unknown element type */
#define WGEMM_ERR_ALIGNMENT -2        /* A or B not 16-byte aligned, lda or ldb not a multiple of 8, C not aligned to its element size, or a TMA-epilogue configuration forced on a C whose base or row pitch (ldc · element size) is not a multiple of 16 bytes */
#define WGEMM_ERR_LAUNCH -3           /* a CUDA call failed while preparing or launching */
#define WGEMM_ERR_NO_DEVICE -4        /* no current device, or it is not compute capability 10.3 */
#define WGEMM_ERR_DEVICE_TIMEOUT -5   /* a bounded wait inside a kernel expired (see wgemm_last_device_error) */
#define WGEMM_ERR_CONFIG -6           /* the forced configuration id does not exist, is for the other C width, or cannot run this shape or mode */
#define WGEMM_ERR_WORKSPACE -7        /* the flag workspace could not be allocated */
#define WGEMM_ERR_NOALLOC_TOO_LARGE -8 /* the problem needs more split-K flags than wgemm_f16f32_splitk_noalloc's fixed array holds */

/*
 * C = A·Bᵀ on `stream`.
 *   A: M×K fp16, row stride lda elements (lda ≥ K, lda % 8 == 0, 16-byte aligned)
 *   B: N×K fp16, row stride ldb elements (ldb ≥ K, ldb % 8 == 0, 16-byte aligned)
 *   C: M×N fp32, row stride ldc elements (ldc ≥ N, 4-byte aligned). When C is
 *      16-byte aligned and ldc % 4 == 0 the epilogue may write C with TMA
 *      stores or reduce-adds (needed by split-K and stream-K); otherwise a
 *      configuration that stores from registers is chosen.
 * M == 0 or N == 0: nothing to do, returns WGEMM_OK. K == 0: C := 0 (the empty
 * sum). C must not overlap A or B. The kernel configuration (tile shape, pair
 * MMA, depth, scheduler, split-K) is chosen per shape from a measured table,
 * else by a rule; stream-K runs when forced (wgemm_f16f32_config). Returns
 * WGEMM_OK once the work is enqueued, else a negative WGEMM_ERR_* code
 * (nothing enqueued).
 */
int wgemm_f16f32(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C,
                 int M, int N, int K, int lda, int ldb, int ldc,
                 wgemm_stream_t stream);

/*
 * As wgemm_f16f32, but with the kernel configuration `config_id`
 * (0 ≤ config_id < wgemm_num_configs()) and the K-decomposition forced:
 * mode 0 = data parallel, 1 = split-K into `splits` ways (splits ≥ 1),
 * 2 = stream-K, 3 = whole waves of tiles data parallel and the rest (the
 * partial last wave and `splits` − 1 full waves before it, splits ≥ 1) by
 * stream-K, 4 = stream-K with zeroing first (the stream-K ranges; the unit
 * holding a tile's first k-block zeroes the tile when its kernel starts,
 * and every unit, that one included, adds its partial into C; `splits` is
 * ignored), -1 = what the configuration table picks. Used by the tests and the
 * per-shape sweep. WGEMM_ERR_CONFIG if the combination cannot run.
 */
int wgemm_f16f32_config(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C,
                        int M, int N, int K, int lda, int ldb, int ldc,
                        int config_id, int mode, int splits,
                        wgemm_stream_t stream);

/*
 * The same product for other element types. Page 1's measured operation has
 * fp16 operands and fp32 C; bf16 operands and a 16-bit C are the adjacent
 * variants of the same tensor-core instruction (tcgen05.mma .kind::f16 takes
 * fp16 or bf16 operands, both of the same type, and accumulates in fp32).
 *   ab_type: WGEMM_F16 or WGEMM_BF16 — the type of both A and B.
 *   c_type:  WGEMM_F32, WGEMM_F16 or WGEMM_BF16. A 16-bit C holds the fp32
 *            sum rounded once to nearest, ties to even; it is computed data
 *            parallel only (K is never split, so no partial sum is rounded).
 * Layout, strides and alignment as wgemm_f16f32, with C's alignment and TMA
 * conditions taken in C's element size: C aligned to its element size; the
 * TMA epilogue wants a 16-byte aligned C and ldc · element size a multiple
 * of 16. Returns as wgemm_f16f32; WGEMM_ERR_INVALID_ARG for an unknown type.
 * wgemm_gemm(A, B, C, WGEMM_F16, WGEMM_F32, ...) is wgemm_f16f32.
 */
int wgemm_gemm(const void* A, const void* B, void* C, int ab_type, int c_type,
               int M, int N, int K, int lda, int ldb, int ldc,
               wgemm_stream_t stream);

/*
 * As wgemm_gemm with the configuration and K-decomposition forced (see
 * wgemm_f16f32_config). A configuration serves one C width: those whose
 * name ends in "_h" write a 16-bit C and run data parallel only (mode 0 or
 * -1); the others write fp32. WGEMM_ERR_CONFIG otherwise.
 */
int wgemm_gemm_config(const void* A, const void* B, void* C, int ab_type, int c_type,
                      int M, int N, int K, int lda, int ldb, int ldc,
                      int config_id, int mode, int splits,
                      wgemm_stream_t stream);

/*
 * The product with a fused epilogue (page 1 has no counterpart; it is the
 * usual GEMM epilogue of a linear layer):
 *
 *     D[i·ldd + j] = alpha · Σ_k A[i·lda + k]·B[j·ldb + k] + beta · Cin[i·ldcin + j] + bias[j]
 *
 * computed in fp32 from the fp32 sum (fmaf(alpha, sum, fmaf(beta, Cin, bias))),
 * then, for a 16-bit D, rounded once to nearest-even.
 *   D:    M×N of c_type (WGEMM_F32, WGEMM_F16 or WGEMM_BF16), row pitch ldd.
 *   Cin:  M×N of c_type, row pitch ldcin; read only when beta != 0 (it may
 *         then be NULL). It is read with TMA: a 16-byte aligned base and
 *         ldcin · element size a multiple of 16, else WGEMM_ERR_ALIGNMENT.
 *         Cin may be D itself (ldcin == ldd): every element is read before it
 *         is written. Any other overlap of Cin and D is undefined.
 *   bias: N fp32 values (device memory), or NULL for none.
 *   alpha, beta: finite fp32 scalars (WGEMM_ERR_INVALID_ARG otherwise).
 * A, B, types and alignment as wgemm_gemm. K == 0 gives D = beta·Cin + bias.
 * alpha = 1, beta = 0 and bias = NULL is exactly wgemm_gemm (any kernel);
 * otherwise the call runs one of the fused configurations (names containing
 * "_ab"), data parallel. In the register-store ones ("_direct_ab<F>") each
 * epilogue warp prefetches its blocks of Cin with TMA while the unit's main
 * loop runs. The in-place form D += alpha·A·Bᵀ + bias (Cin == D, ldcin == ldd,
 * beta == 1, fp32 D) may also run the reduce-add ones ("_tma_ab1"): they
 * add alpha·sum + bias (one fmaf) into D's old values with TMA reduce-adds
 * in L2 and read no Cin, so D's element is rounded twice (the fmaf and the
 * add), as in the general form.
 * wgemm_gemm_ex_config forces a fused configuration (config_id ≥ 0), or
 * chooses (-1); WGEMM_ERR_CONFIG for a configuration that is not fused, is
 * of the other D width, or is a reduce-add one for a call that is not of
 * the in-place form.
 */
int wgemm_gemm_ex(const void* A, const void* B, void* D, const void* Cin, const float* bias,
                  float alpha, float beta, int ab_type, int c_type,
                  int M, int N, int K, int lda, int ldb, int ldd, int ldcin,
                  wgemm_stream_t stream);
int wgemm_gemm_ex_config(const void* A, const void* B, void* D, const void* Cin,
                         const float* bias, float alpha, float beta, int ab_type, int c_type,
                         int M, int N, int K, int lda, int ldb, int ldd, int ldcin,
                         int config_id, wgemm_stream_t stream);

/* Typed shorthands of wgemm_gemm: bf16 → fp32, fp16 → fp16, bf16 → bf16. */
int wgemm_bf16f32(const wgemm_bf16_t* A, const wgemm_bf16_t* B, float* C,
                  int M, int N, int K, int lda, int ldb, int ldc,
                  wgemm_stream_t stream);
int wgemm_f16f16(const wgemm_f16_t* A, const wgemm_f16_t* B, wgemm_f16_t* C,
                 int M, int N, int K, int lda, int ldb, int ldc,
                 wgemm_stream_t stream);
int wgemm_bf16bf16(const wgemm_bf16_t* A, const wgemm_bf16_t* B, wgemm_bf16_t* C,
                   int M, int N, int K, int lda, int ldb, int ldc,
                   wgemm_stream_t stream);

/*
 * Programmatic dependent launch, process-wide, off by default. When on,
 * wgemm_f16f32 and wgemm_gemm launch their kernel with CUDA's programmatic
 * stream serialization: the kernel may be scheduled before the previous
 * kernel on the stream has finished (once that kernel allows it: every wgemm
 * kernel does so right after its set-up), runs its set-up (barriers, tensor
 * memory, tensor-map prefetch) and then waits, in griddepcontrol.wait, for
 * the previous kernel to complete and its writes to be visible before its
 * first load or store. Results are those of ordinary stream order; only
 * launch latency and set-up overlap the previous call's tail. (PTX ISA,
 * griddepcontrol; "SASS-Level Kernel Generation for Blackwell" measures with
 * it off.) The split-K no-allocation entry point and the K = 0 path ignore
 * the setting. Returns the previous setting (0 or 1), or
 * WGEMM_ERR_INVALID_ARG unless enable is 0 or 1.
 */
int wgemm_set_pdl(int enable);

/*
 * Number of compiled kernel configurations, and the name of one ("" if out
 * of range). A name reads g<G>[m2|r2]_<C>x<R>_s<S>_a<A>_<E>[_clc][_ab<F>][_h]:
 * G CTAs per MMA (1, or 2 for a CTA pair); m2 = two MMA groups per cluster
 * side by side along C's columns sharing the A tile, r2 = two groups stacked
 * along C's rows sharing the B tile; C × R the C columns × rows of one
 * worker (cluster) tile; S ring stages; A TMEM accumulators; E the epilogue
 * (direct: stores from registers, tma: staged TMA stores); _clc tiles taken
 * by cluster launch control (else a static persistent schedule); _ab<F> the
 * fused alpha/beta/bias epilogue (direct: with an F-block Cin ring; tma_ab1:
 * the in-place reduce-add form); _h a 16-bit C.
 * Split-K and stream-K run on the static, fp32, unfused "tma" configurations
 * without m2 (an r2 cluster runs them as one worker).
 */
int wgemm_num_configs(void);
const char* wgemm_config_name(int config_id);

/*
 * The choice wgemm_f16f32 (c_type WGEMM_F32, fused 0), wgemm_gemm (any
 * c_type; the operand type does not enter) or wgemm_gemm_ex (fused 1: among
 * the fused configurations; fused 2: the in-place form with beta = 1 and
 * fp32 D, which may also take the reduce-add ones) makes for a shape and
 * operand row pitches
 * (lda, ldb, in elements) on the current device: for fp32 C, the measured
 * per-shape table if the shape is in it and both pitches are multiples of 16
 * elements (rows on 32-byte sectors, as the table was measured); else the
 * configuration of C's width and
 * K-decomposition with the least time predicted from measured
 * per-configuration rates (waves of tiles × per-k-block cost + fixed costs),
 * fitted separately for rows on and off 32-byte sectors. A K split is chosen
 * only when it predicts at least 20% less time than the best data-parallel
 * configuration. Writes the configuration id, mode and splits (any pointer
 * may be NULL). Returns WGEMM_OK, WGEMM_ERR_INVALID_ARG (negative size, a
 * pitch below K, an unknown c_type, fused not 0, 1 or 2, fused 2 with a
 * 16-bit c_type) or a device error.
 */
int wgemm_select(int M, int N, int K, int lda, int ldb, int c_type, int fused, int* config_id,
                 int* mode, int* splits);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. Returns WGEMM_OK, WGEMM_ERR_DEVICE_TIMEOUT, or WGEMM_ERR_LAUNCH if a
 * CUDA error is pending.
 */
int wgemm_check(wgemm_stream_t stream);

/*
 * Details of the last device error wgemm_check saw on the current device:
 * the block, the warp, the wait site (role·16 + barrier kind) and the phase
 * parity it waited for. Any pointer may be NULL. Returns the error code.
 */
int wgemm_last_device_error(int* block, int* warp, int* site, int* parity);

/* A short English description of a status code. Never NULL. */
const char* wgemm_status_string(int status);

/* Bytes of flag workspace currently held for the current device (all streams). */
size_t wgemm_workspace_bytes(void);

/* Frees the current device's flag workspaces after synchronising the device. */
int wgemm_release_workspace(void);

/*
 * Split-K C = A·Bᵀ that allocates nothing. The paper has no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc or cudaFree
 * while they run, for example a process whose framework allocator has
 * reserved the device memory for itself (a new allocation can fail), a
 * latency-bound serving loop that cannot afford the device-wide
 * synchronisation cudaFree implies when a workspace grows, or a host
 * application that forbids plug-in libraries from owning device allocations.
 *
 * Same arguments and result as wgemm_f16f32 (A, B, C device pointers owned by
 * the caller), computed by the pair-MMA configuration g2_512x256_s4_a1_tma
 * with K split `splits` ways (splits >= 1, clamped to ceil(K / 64)). C must
 * be 16-byte aligned with ldc % 4 == 0 (the partial sums are added into C
 * with TMA reduce-adds), else WGEMM_ERR_ALIGNMENT.
 *
 * Scratch: the split-K flags live in a fixed array of 16384 32-bit words
 * (64 KiB) of device memory inside the library image, which every device that
 * loads the library holds until the process exits. A call needs
 * ceil(M / 256) · ceil(N / 512) · 2 · splits words; a larger problem is
 * rejected with WGEMM_ERR_NOALLOC_TOO_LARGE before anything is enqueued.
 * The array keeps the previous call's contents; the flags hold a per-device
 * call counter that only grows, so nothing needs clearing between calls.
 * Every call on a device shares the one array: calls that overlap on the GPU
 * (for example on two streams at once) race on it and give wrong results;
 * order them on one stream or with events.
 *
 * Set-up: the first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and the kernel's attributes
 * and occupancy; make that first call before any stream capture. The call
 * never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * wgemm_set_pdl does not apply to this call: it is always launched without
 * programmatic dependent launch, so it starts only after the previous kernel
 * on the stream has finished.
 */
int wgemm_f16f32_splitk_noalloc(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C,
                                int M, int N, int K, int lda, int ldb, int ldc,
                                int splits, wgemm_stream_t stream);

/*
 * wgemm_f16f32_host: the same product, C = A·Bᵀ with fp16 A and B and fp32
 * accumulation and C ("SASS-Level Kernel Generation for Blackwell", section
 * "The numbers", the setup paragraph), with A, B and C in HOST memory: the
 * call uploads A and B, computes, and downloads C, all asynchronously on
 * `stream`.
 *
 * A (M×K, row pitch lda >= K), B (N×K, pitch ldb >= K) and C (M×N, pitch
 * ldc >= N) are host pointers, any alignment; they should be page-locked
 * (cudaHostAlloc or cudaHostRegister) for the copies to overlap anything,
 * and must stay valid and untouched until `stream` reaches the call's end.
 * dA, dB and dC are device buffers the caller owns, 16-byte aligned, of at
 * least the element counts wgemm_host_device_elems gives: M·kd, N·kd and
 * M·nd with kd = K rounded up to a multiple of 8 and nd = N rounded up to a
 * multiple of 4 (the pitches the call uses on the device). Their contents
 * on return are the device copies of A, B and C.
 *
 * How it runs: A goes up in row panels (a multiple of 256 rows each; as
 * many as min(A bytes, C bytes) holds 8 MiB, 1 to 8) and B in blocks of its
 * rows, that is C's columns (a multiple of 256 rows each; as many as B's
 * bytes hold 128 MiB, 1 to 4); a product that splits K has one panel and one
 * block. The uploads run in the order the GEMMs need them: the first half of
 * B's blocks, every panel of A, then B's other blocks. The GEMM of each
 * (panel, block) runs on `stream` as soon as both have landed, with the
 * configuration chosen for the whole shape, and each such block of C goes
 * down as soon as it is computed. So the uploads and downloads overlap the
 * other blocks' GEMMs. The copies run on two streams
 * the library creates per device (one per direction); they wait for
 * everything enqueued on `stream` before the call, and `stream` waits for
 * the last download, so work enqueued on `stream` after the call sees C in
 * host memory. Consecutive calls on one stream therefore do not overlap;
 * calls on different streams overlap their copies with each other's GEMMs.
 * Calls from several host threads are serialised inside the library.
 *
 * Returns WGEMM_OK (also for M == 0 or N == 0, which enqueue nothing; K == 0
 * downloads zeros), WGEMM_ERR_INVALID_ARG (negative sizes, a NULL pointer
 * with a non-empty operand, a pitch below its row length),
 * WGEMM_ERR_ALIGNMENT (a device buffer not 16-byte aligned), or an error of
 * the GEMM call or WGEMM_ERR_LAUNCH from a failed copy or event. After an
 * error part of the work may be enqueued and C is undefined, but `stream`
 * still waits for every copy the call enqueued, so synchronising it is
 * enough before the buffers are freed.
 */
int wgemm_f16f32_host(const wgemm_f16_t* A, const wgemm_f16_t* B, float* C, int M, int N,
                      int K, int lda, int ldb, int ldc, wgemm_f16_t* dA, wgemm_f16_t* dB,
                      float* dC, wgemm_stream_t stream);

/*
 * Device buffer sizes for wgemm_f16f32_host, in elements: a_elems = M·kd
 * (fp16), b_elems = N·kd (fp16), c_elems = M·nd (fp32), kd and nd as above.
 * Any output pointer may be NULL. Host only. Returns WGEMM_OK or
 * WGEMM_ERR_INVALID_ARG (a negative size).
 */
int wgemm_host_device_elems(int M, int N, int K, size_t* a_elems, size_t* b_elems,
                            size_t* c_elems);

/*
 * Host-side introspection, no GPU needed (used by the host tests).
 *
 * wgemm_debug_smem_desc: the 64-bit tcgen05 shared-memory descriptor the
 * kernels build for a K-major fp16 operand tile with the 128-byte swizzle,
 * starting at shared byte address `smem_addr`.
 * wgemm_debug_idesc: the 32-bit instruction descriptor of a kind::f16 MMA of
 * shape M×N×16 with an f32 accumulator, fp16 operands (bf16 = 0) or bf16
 * operands (bf16 = 1).
 * wgemm_debug_config_out: 0 if a configuration writes fp32 C, 1 if 16-bit C,
 * WGEMM_ERR_CONFIG for an unknown id. wgemm_debug_config_fused: 1 if it has
 * the alpha/beta/bias epilogue, else 0 (WGEMM_ERR_CONFIG for an unknown id).
 * wgemm_debug_sw128_offset: byte offset of fp16 element (row, k) inside a
 * 1024-byte-aligned 128-byte-swizzled K-major tile.
 * wgemm_debug_plan: fills `out` (7 int32 per unit: tile, tm, tn, kb_begin,
 * kb_end, kind, split) with every unit of the plan the library would run
 * for this shape, configuration, mode and worker count, in worker-major
 * order; returns the number of units (or a negative error), writing at most
 * `max_units`. Also writes the tile shape (rows, cols) of the configuration.
 */
/*
 * Fault-path test hook: from the next call on, the split-K and stream-K
 * kernels wait for flags to reach their call's epoch + `skew` instead of the
 * epoch. A skew of 1 is a value no CTA ever writes, so the flag waits run out
 * their time limit (2 s), record WGEMM_ERR_DEVICE_TIMEOUT in the device status
 * word and return; the kernel tears down normally. 0 (the default) restores
 * normal operation. Returns WGEMM_OK, or WGEMM_ERR_INVALID_ARG for skew < 0.
 */
int wgemm_debug_set_flag_wait_skew(int skew);

/*
 * Profiling hook: enable = 0 launches the split-K and stream-K grids from
 * the next call on without the cooperative attribute, 1 (the default)
 * restores it. Nsight Compute cannot profile a cooperative cluster launch
 * (the launch fails with an error), but it runs every profiled kernel alone
 * on the GPU, so all of a grid's CTAs are resident there anyway. Outside a
 * profiler keep the default: a plain K-split launch beside another
 * long-running kernel may start only part of its grid, whose flag waits then
 * expire (WGEMM_ERR_DEVICE_TIMEOUT). Returns the previous setting, or
 * WGEMM_ERR_INVALID_ARG.
 */
int wgemm_debug_set_cooperative(int enable);

/*
 * Test hook: panels > 0 makes wgemm_f16f32_host split A into that many row
 * panels (before the rounding to 256 rows), whatever the shape's bytes; 0
 * (the default) restores the rule. Returns the previous setting, or
 * WGEMM_ERR_INVALID_ARG for panels outside 0..8.
 * wgemm_debug_host_panel_rows: the rows per panel wgemm_f16f32_host uses for
 * a data-parallel product of this shape (host only), or
 * WGEMM_ERR_INVALID_ARG.
 */
int wgemm_debug_set_host_panels(int panels);
int wgemm_debug_host_panel_rows(int M, int N, int K);

/*
 * Test hook: blocks > 0 makes wgemm_f16f32_host split B's rows (C's columns)
 * into that many blocks (before the rounding to 256 rows), whatever B's
 * bytes; 0 (the default) restores the rule. Returns the previous setting, or
 * WGEMM_ERR_INVALID_ARG for blocks outside 0..4.
 * wgemm_debug_host_block_cols: B's rows (C's columns) per block that
 * wgemm_f16f32_host uses for a data-parallel product with this N and K
 * (host only), or WGEMM_ERR_INVALID_ARG.
 */
int wgemm_debug_set_host_blocks(int blocks);
int wgemm_debug_host_block_cols(int N, int K);

/*
 * Timeline tracing (a library built with WGEMM_TRACE=1 only; other builds
 * ignore the buffer). wgemm_debug_set_trace: from the next call on, CTA b of
 * each GEMM kernel writes %globaltimer values (ns) into
 * device_buffer[b·8 + e] for b < ctas, at e = 0 kernel entry, 1 after the
 * set-up barrier, 2 first stage landed (MMA thread), 3 last accumulator
 * committed, 4 epilogue's first accumulator full, 5 epilogue done, 6 after the
 * teardown barrier. The caller owns the device buffer; ctas = 0 turns tracing
 * off. wgemm_debug_trace_build: 1 in a tracing build, else 0.
 */
int wgemm_debug_set_trace(uint64_t* device_buffer, int ctas);
int wgemm_debug_trace_build(void);

/*
 * The per-shape rule. wgemm_debug_max_workers: co-resident workers (CTAs or
 * clusters) of a configuration on the current device (a negative status on
 * error). wgemm_debug_predict_us: the time the rule predicts for a shape,
 * configuration and K-decomposition with `workers` workers and operand row
 * pitches lda, ldb, from the measured per-configuration rates compiled into
 * the library (-1 if the configuration has none, the mode is not modelled
 * (3, the data-parallel + stream-K tail mix) or an argument is invalid).
 * Host arithmetic only.
 */
int wgemm_debug_max_workers(int config_id);
double wgemm_debug_predict_us(int M, int N, int K, int lda, int ldb, int config_id, int mode,
                              int splits, int workers);

uint64_t wgemm_debug_smem_desc(uint32_t smem_addr);
uint32_t wgemm_debug_idesc(int M, int N, int bf16);
int wgemm_debug_config_out(int config_id);
int wgemm_debug_config_fused(int config_id);
uint32_t wgemm_debug_sw128_offset(uint32_t row, uint32_t k);
int wgemm_debug_plan(int M, int N, int K, int config_id, int mode, int splits, int workers,
                     int32_t* out, int max_units, int* tile_rows, int* tile_cols);

#ifdef __cplusplus
}
#endif

#endif /* WGEMM_H */

/*
 * gemm.h -- C ABI of the GB300 (sm_103a) TN GEMM library  libgemm_gb300.so
 *
 * The operation (HGEMM and its int8 variant):
 *
 *     C[i][j] = sum_{k<K} A[i][k] * B[j][k]          0 <= i < M, 0 <= j < N
 *
 * with A an M x K row-major matrix, B an N x K row-major matrix (both contiguous
 * along K: the "row-major A, column-major B" layout of the HGEMM kernels in
 * "RL驱动CUDA L2 GEMM内核自动调优：A100/H100 tile size与融合优化", paragraph on tile
 * size and data layout) and C an M x N row-major matrix that is overwritten
 * (no alpha/beta, C is never read).  Other operand storages (B stored K x N, A
 * stored K x M) are selected with gemm_layout_t: the kernels then load
 * M/N-contiguous tiles and use M/N-major shared-memory matrix descriptors.
 *
 *   GEMM_F16    : fp16 A, B;  fp32 accumulation;  fp16 C (round to nearest even)
 *   GEMM_BF16   : bf16 A, B;  fp32 accumulation;  bf16 C (round to nearest even)
 *   GEMM_I8_I32 : int8 A, B;  exact integer sum;  int32 C (two's-complement wrap
 *                 modulo 2^32 if a sum leaves the int32 range)
 *   (fp16 / int8 precision switch of the same post, paragraph on multi-precision
 *    adaptation; the fp32 accumulator is this library's reading where the post
 *    is silent.)
 *
 * Ownership and threading
 *   - A plan is created for one (M, N, K, dtype, layout) on the device that is
 *     current at creation time and must be used with that device current.
 *   - The plan owns its device memory (error word, split-K partials and
 *     counters, int8 conversion buffers).  A, B and C are owned by the caller,
 *     are device pointers, and must stay valid until the stream work finishes.
 *   - gemm_run is asynchronous on the caller's stream.  A plan holds one set of
 *     scratch buffers: do not run the same plan on two streams at once.
 *   - No host locks are taken; distinct plans may be used from distinct threads.
 *
 * Errors
 *   Every call returns a gemm_status_t.  Argument and alignment problems are
 *   reported before any device work is queued.  No call falls back to another
 *   backend or to the CPU.  Kernels bound every wait; a wait that runs out sets
 *   the plan's device error word, which gemm_plan_check reports as
 *   GEMM_ERR_DEVICE_TIMEOUT.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_ABI_VERSION 1

typedef enum {
    GEMM_F16 = 0,
    GEMM_BF16 = 1,
    GEMM_I8_I32 = 2
} gemm_dtype_t;

/*
 * Operand storage.  C is always M x N row-major; the math is always
 * C[i][j] = sum_k a(i,k) * b(k,j) with a, b the logical M x K and K x N operands.
 */
typedef enum {
    GEMM_LAYOUT_TN = 0,  /* A stored M x K, B stored N x K (both K contiguous): C = A * B^T */
    GEMM_LAYOUT_NN = 1,  /* A stored M x K, B stored K x N (N contiguous):      C = A * B   */
    GEMM_LAYOUT_TT = 2,  /* A stored K x M (M contiguous), B stored N x K:      C = A^T * B^T */
    GEMM_LAYOUT_NT = 3   /* A stored K x M, B stored K x N:                     C = A^T * B */
} gemm_layout_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,     /* negative size, NULL pointer, bad config, wrong device */
    GEMM_ERR_UNSUPPORTED = 2,     /* unknown dtype or layout */
    GEMM_ERR_ALIGNMENT = 3,       /* pointer not 16-byte aligned or row stride not a multiple of 16 B */
    GEMM_ERR_NO_DEVICE = 4,       /* no CUDA device / driver */
    GEMM_ERR_ARCH = 5,            /* current device is not compute capability 10.3 */
    GEMM_ERR_OOM = 6,             /* device allocation for the plan failed */
    GEMM_ERR_TENSORMAP = 7,       /* cuTensorMapEncodeTiled rejected a descriptor */
    GEMM_ERR_LAUNCH = 8,          /* kernel launch failed */
    GEMM_ERR_DEVICE_TIMEOUT = 9,  /* a kernel wait ran out (reported by gemm_plan_check) */
    GEMM_ERR_CUDA = 10,           /* any other CUDA runtime error */
    GEMM_ERR_SCRATCH_LIMIT = 11   /* gemm_run_splitk_noalloc: problem exceeds its fixed scratch */
} gemm_status_t;

/*
 * Kernel configuration (what the per-shape table chooses; see gemm_select_config).
 *   block_n      : output tile width, 64, 128, 224 or 256 (tile height is 128
 *                  rows; 224 only with cta_pair, split_k 1, no multicast and B
 *                  stored N x K; int8 wider than 128 only with cta_pair, split_k 1
 *                  and no multicast)
 *   stages       : depth of the shared-memory ring; 0 = the default for block_n
 *   split_k      : number of K slices per output tile (>= 1); slices are summed
 *                  in a fixed order, so results are run-to-run identical
 *   raster_group : m-blocks per band of the L2-friendly tile order (>= 1)
 *   max_ctas     : persistent grid cap; 0 = one CTA per SM
 *   split_mode   : how K slices are combined when split_k > 1:
 *                  0 = partials in plan memory, summed by the last slice to finish;
 *                  1 = the slices of a tile run as one thread-block cluster and are
 *                      summed through distributed shared memory (split_k must
 *                      come out as 2, 4 or 8; one tile slice per CTA, no scratch)
 *   cta_pair     : 1 = 256-row tiles computed by an SM pair (tcgen05 cta_group::2
 *                  thread-block cluster of two CTAs): block_n 128, 224 or 256;
 *                  0 = 128-row tiles on one SM
 *   direct_store : epilogue store path: 0 = TMA tensor stores from a swizzled
 *                  shared-memory buffer; 1 = 16-byte global stores from each
 *                  thread's row (one-SM kernel only)
 *   multicast    : 0/1 = off; 2 or 4 = clusters of that many CTAs compute
 *                  adjacent N-tiles of the same rows, each loading 1/multicast
 *                  of the shared A tile and multicasting it to the others
 *                  (one-SM kernel, split_k 1; 4 needs A stored M x K).  With
 *                  cta_pair, 2 = clusters of two SM pairs computing adjacent
 *                  N-tiles of the same 256 rows, each CTA loading 64 of its 128
 *                  A rows for both pairs (split_k 1, kblocks_per_stage 1).
 *                  Multicast copies stay within this GPU's own memory.
 *   kblocks_per_stage : 0 = the table's choice; 1, 2 or 4 = 64-wide k-blocks
 *                  per ring slot.  2: one-SM kernel with block_n 64 or 128 or
 *                  the SM-pair kernel; 4: one-SM kernel with block_n 64 or the
 *                  SM-pair kernel with block_n 128 (two slots).  Both need no
 *                  multicast and K % 64 == 0 when an operand is K-contiguous;
 *                  each operand's k-blocks of a slot arrive in one copy per
 *                  64-element block
 *   l2_prefetch  : 0 = off; d in 1..64 = while loading k-block kb, also ask L2
 *                  to fetch k-block kb + d of the same tile (hides DRAM latency
 *                  on long K)
 */
typedef struct {
    int32_t block_n;
    int32_t stages;
    int32_t split_k;
    int32_t raster_group;
    int32_t max_ctas;
    int32_t split_mode;
    int32_t cta_pair;
    int32_t direct_store;
    int32_t multicast;
    int32_t l2_prefetch;
    int32_t kblocks_per_stage;
} gemm_config_t;

typedef struct gemm_plan *gemm_plan_t;

/* Activation of the fused epilogue (gemm_run_bias_act). */
typedef enum {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1,   /* max(x, 0) */
    GEMM_ACT_GELU = 2,   /* x * Phi(x), Phi = standard normal CDF (erf form) */
    GEMM_ACT_SILU = 3    /* x / (1 + exp(-x)) */
} gemm_activation_t;

/*
 * Create a plan.  Validates the arguments (sizes >= 0; every stored row of A,
 * B and C a multiple of 16 bytes: for fp16/bf16 the contiguous dimension of A
 * and of B (K for TN, M or N for the other layouts) a multiple of 8 and N a
 * multiple of 8; for int8 multiples of 16 and N of 4), checks the current
 * device is an sm_103 part, picks the kernel
 * configuration from the built-in table and allocates the plan's scratch
 * memory.  On success *plan receives a handle that gemm_plan_destroy frees.
 * Row-stride rule: "TMA/2D tensor" alignment of "B-08. Hopper TMA：从单线程 Bulk
 * Copy 到吞吐墙" (www.lqnn.cn), section 6.1 (global base 16 B, strides multiples
 * of 16 B).
 */
gemm_status_t gemm_plan_create(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                               gemm_layout_t layout, gemm_plan_t *plan);

/* As gemm_plan_create, with an explicit configuration instead of the table's. */
gemm_status_t gemm_plan_create_with_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                           gemm_layout_t layout, const gemm_config_t *config,
                                           gemm_plan_t *plan);

/*
 * Queue C = A * B^T on `stream` (a cudaStream_t; NULL = the legacy default
 * stream).  A, B, C: device pointers, 16-byte aligned, in the plan's layout and
 * element types.  M == 0 or N == 0 queues nothing; K == 0 writes zeros to C.
 * Returns after queueing; errors of the queued work surface through
 * gemm_plan_check or the CUDA stream.
 */
gemm_status_t gemm_run(gemm_plan_t plan, const void *A, const void *B, void *C, void *stream);

/*
 * Linear-layer epilogue fused into the GEMM (fp16/bf16 plans):
 *     C[i][j] = act(sum_k A[i][k] * B[j][k] + bias[j])
 * evaluated in fp32 before the conversion to the output type.  bias: device
 * pointer to N fp32 values, 16-byte aligned, or NULL (no bias); act: a
 * gemm_activation_t.  Otherwise as gemm_run.  The pages list the order of
 * fused operations among the tuning dimensions of the HGEMM kernels ("RL驱动
 * CUDA L2 GEMM内核自动调优", paragraph on tile size and fusion order) without
 * naming them; bias + activation is what follows FFN-shaped GEMMs.
 * int8 plans return GEMM_ERR_UNSUPPORTED unless bias is NULL and act is NONE.
 */
gemm_status_t gemm_run_bias_act(gemm_plan_t plan, const void *A, const void *B, void *C,
                                const float *bias, gemm_activation_t act, void *stream);

/*
 * Synchronise `stream`, then read and clear the plan's device error word.
 * GEMM_ERR_DEVICE_TIMEOUT if a kernel of this plan gave up on a wait,
 * GEMM_ERR_CUDA if the stream reported an error, else GEMM_OK.
 */
gemm_status_t gemm_plan_check(gemm_plan_t plan, void *stream);

/* Free a plan and its device memory.  NULL is a no-op. */
gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* The configuration a plan runs with. */
gemm_status_t gemm_plan_get_config(gemm_plan_t plan, gemm_config_t *config);

/*
 * How the plan launches its GEMM kernel: `grid` CTAs in thread-block clusters
 * of `cluster` CTAs, of which at most `max_active_clusters` fit on the device
 * at once (as the CUDA occupancy calculator reports for the kernel, its block
 * size and shared memory; 0 if that query failed).  A grid above
 * cluster * max_active_clusters runs in more than one wave.  Any output pointer
 * may be NULL.  GEMM_ERR_INVALID_ARG for a NULL plan.
 */
gemm_status_t gemm_plan_get_launch(gemm_plan_t plan, int32_t *grid, int32_t *cluster,
                                   int32_t *max_active_clusters);

/*
 * Set the limit, in nanoseconds, after which a kernel wait of this plan gives
 * up (default 2e9).  ns == 0 restores the default.
 */
gemm_status_t gemm_plan_set_timeout(gemm_plan_t plan, uint64_t ns);

/*
 * Test hook for failure reporting: make every shared-memory ring slot of this
 * plan's GEMM kernel wait for `extra_bytes` more than its copies deliver, so
 * the slot never completes, the kernel's bounded wait runs out (see
 * gemm_plan_set_timeout), the kernel unwinds and frees its resources, and
 * gemm_plan_check reports GEMM_ERR_DEVICE_TIMEOUT.  The GPU context stays
 * usable.  0 restores normal operation.  Output C is undefined while it is set.
 */
gemm_status_t gemm_plan_set_wait_test(gemm_plan_t plan, uint32_t extra_bytes);

/*
 * Host-only query (no device work): the configuration the table picks for a
 * shape on a GPU with `num_sms` SMs, after validating the shape as
 * gemm_plan_create does.
 */
gemm_status_t gemm_select_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                 int32_t num_sms, gemm_config_t *config);

/*
 * Host-only: the output tile (m_blk, n_blk) that the persistent scheduler
 * assigns to linear tile index `tile` for an m_blocks x n_blocks tile grid in
 * bands of `raster_group` m-blocks (the same function the kernels evaluate).
 */
gemm_status_t gemm_tile_coords(int64_t m_blocks, int64_t n_blocks, int32_t raster_group,
                               int64_t tile, int64_t *m_blk, int64_t *n_blk);

/* Bytes of device memory a plan for this shape/config allocates (host-only). */
gemm_status_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                   const gemm_config_t *config, size_t *bytes);

/* Static description of a status code. */
const char *gemm_status_string(gemm_status_t status);

/* GEMM_ABI_VERSION of the built library. */
int32_t gemm_abi_version(void);

/*
 * Measurement aid: queue one empty kernel of `grid` CTAs x 192 threads on
 * `stream`, launched like the GEMM kernels (same block size, programmatic
 * dependent launch, grid-dependency wait).  Back-to-back launches of it give
 * the launch-latency floor that bounds the smallest GEMMs.
 */
gemm_status_t gemm_launch_empty(int32_t grid, void *stream);

/*
 * Split-K GEMM that allocates no device memory (no counterpart on the pages:
 * this exists for callers that may not allocate -- plugins whose host framework
 * owns all device memory and offers no allocator, services that reserve their
 * memory budget up front, loops where cudaMalloc's possible device
 * synchronisation or failure is not acceptable).
 *
 * Computes C = A * B^T exactly as gemm_run does for GEMM_F16 / GEMM_BF16 (same
 * kernel, 128 x 64 output tiles, K cut into `split_k` slices summed in a fixed
 * order), with the split-K partials, counters and error word in one fixed
 * 16 MiB array compiled into the library instead of plan memory.  A, B, C are
 * caller-owned device pointers with the gemm_run layout and alignment rules;
 * no plan is needed.  split_k >= 1 (clamped to the number of 64-wide K blocks).
 *
 * Limit: with split_k > 1 the partials need ceil(M/128) * ceil(N/64) * split_k
 * * 32 KiB <= 16 MiB - 32 KiB (at most 511 tile-slices) and at most 4096
 * tiles; larger problems return GEMM_ERR_SCRATCH_LIMIT.  split_k == 1 needs no
 * partials.  GEMM_I8_I32 returns GEMM_ERR_UNSUPPORTED.
 *
 * The array occupies 16 MiB on every GPU where the library's device code is
 * loaded, until the process exits.  The first call on a device (that device
 * current) looks up the array's device address (cudaGetSymbolAddress) and
 * prepares the kernel; make it before any stream capture.  Every call clears
 * the array's split-K counters on `stream`; all calls share the one array, so
 * calls whose work overlaps on the GPU (different streams, or different host
 * threads) race and must be serialised by the caller.  A wait that runs out
 * sets the array's error word, which no call clears: gemm_noalloc_check
 * reports and clears it.  Calls no cudaMalloc, cudaFree or allocating library
 * routine.
 */
gemm_status_t gemm_run_splitk_noalloc(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                      int32_t split_k, const void *A, const void *B, void *C,
                                      void *stream);

/*
 * The failure report of gemm_run_splitk_noalloc on the current device (no
 * counterpart on the pages; the no-alloc path has no plan whose error word
 * gemm_plan_check could read).  Synchronises `stream`, then reads and clears
 * the fixed array's error word: GEMM_ERR_DEVICE_TIMEOUT if a kernel of any
 * no-alloc call since the last check gave up on a wait (its C is then
 * undefined), GEMM_ERR_CUDA if the stream or the read failed, else GEMM_OK
 * (also when no no-alloc call has run on this device).  Allocates nothing.
 */
gemm_status_t gemm_noalloc_check(void *stream);

/*
 * Failure-test hook of gemm_run_splitk_noalloc, process-wide (no counterpart on
 * the pages): later no-alloc calls make every ring slot wait for `extra_bytes`
 * (a multiple of 16, at most 4096) more than its copies deliver, so the slot
 * never completes and the kernel's bounded wait runs out after `timeout_ns`
 * (0 = the default 2 s); the kernel unwinds, frees its TMEM and records the
 * failure for gemm_noalloc_check.  extra_bytes = 0 restores normal operation.
 */
gemm_status_t gemm_noalloc_set_wait_test(uint32_t extra_bytes, uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */

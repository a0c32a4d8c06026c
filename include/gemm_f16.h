/*
 * gemm_f16 — dense tiled fp16 matrix multiply for NVIDIA GB300 (sm_103a).
 *
 *   C[m, n] = fp16( sum_{k < K} A[m, k] * B[k, n] ),  0 <= m < M, 0 <= n < N
 *
 * with fp16 operands, fp32 accumulation and one rounding to fp16 (round to
 * nearest even; values past the fp16 range become +-inf).
 *
 * The operation and its contract follow the pages this library is built from:
 *  - the definition and the fp16-in / fp32-accumulate / fp16-out precision
 *    points: "Triton GEMM: from one output tile to addresses, boundaries and
 *    data reuse" (charlestar.github.io), the opening problem statement and the
 *    paragraph on the three precision positions; TileLang tutorial ch. 14
 *    "GEMM operators", section 1.1;
 *  - strides in elements for both operands and an explicit output pitch: the
 *    same Triton page, section "Shape states the meaning, stride decides the
 *    address" (transposed views such as B = X.T are ordinary strided views);
 *  - dimensions the tile does not divide, with the K tail zero-filled (never
 *    wrapped modulo K) and only the M x N outputs written: section "Three
 *    non-divisible dimensions need different boundary handling";
 *  - 64-bit address arithmetic: section "Putting addresses and boundaries into
 *    a short kernel";
 *  - the argument checks (positive sizes and strides, outputs not sharing
 *    storage with inputs): the wrapper on the same page;
 *  - split-K with an fp32 partial-sum reduction for shapes whose output tiles
 *    cannot fill the device: TileLang tutorial ch. 14, section 4.1.
 *
 * All functions are thread-safe unless stated.  No function allocates or frees
 * the caller's memory.
 */
#ifndef GEMM_F16_H
#define GEMM_F16_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GEMM_F16_ABI_VERSION 3

/* Largest M, N or K (and total rows of a grouped call): 2^31 - 2^16.  The
   copies' tile coordinates are 32-bit; element offsets are 64-bit and may
   exceed 2^32 freely. */
#define GEMM_F16_MAX_DIM ((int64_t)2147418112)

typedef enum {
    GEMM_F16_OK = 0,
    /* A null pointer, M/N/K <= 0 or > GEMM_F16_MAX_DIM, a stride <= 0, ldc < N, an fp16 pointer that
       is not 2-byte aligned, a size whose extent overflows int64, a pointer
       that is not device (or managed) memory of the current device (host
       memory, pinned or not, and another GPU's memory are refused), or a view
       that runs past the end of the allocation it points into. */
    GEMM_F16_ERR_INVALID_VALUE = 1,
    /* The bytes C's M x N view spans overlap the bytes spanned by A or B. */
    GEMM_F16_ERR_ALIAS = 2,
    /* The current device is not compute capability 10.3 (GB300). */
    GEMM_F16_ERR_UNSUPPORTED_DEVICE = 3,
    /* The split-K workspace could not be allocated, or the caller-supplied
       workspace is smaller than gemm_f16_workspace_size() reports or not
       256-byte aligned. */
    GEMM_F16_ERR_OUT_OF_MEMORY = 4,
    /* A CUDA runtime/driver call failed while setting up or launching. */
    GEMM_F16_ERR_LAUNCH = 5,
    /* Reported through gemm_f16_device_status(): a kernel gave up on a bounded
       wait (a lost pipeline arrival) and returned early; C is undefined. */
    GEMM_F16_ERR_TIMEOUT = 6,
    /* Reported through gemm_f16_device_status() with GEMM_F16_OPT_DEBUG_BOUNDS on: a
       gathered load or a per-thread store of C would have left the byte range its
       view spans and was skipped; C is undefined. */
    GEMM_F16_ERR_BOUNDS = 7
} gemm_f16_status;

/*
 * C = A * B on `stream` (0 = the legacy default stream).  Asynchronous: the
 * call returns once the kernel is queued.
 *
 *   A        device pointer to element (0,0) of A; element (m,k) is at
 *            A + m*stride_am + k*stride_ak (strides in ELEMENTS, fp16).
 *   B        device pointer; element (k,n) is at B + k*stride_bk + n*stride_bn.
 *   C        device pointer; element (m,n) is written at C + m*ldc + n.
 *            Elements of C outside the M x N view (the pitch padding between
 *            N and ldc) are never written.
 *   M, N, K  sizes, 0 < size <= GEMM_F16_MAX_DIM; nothing needs to be a tile
 *            multiple.
 *
 * Any positive strides are accepted (row-major, column-major / transposed
 * views, pitched slices, non-unit inner strides).  Alignment is not required:
 * operands whose base is 16-byte aligned with a unit inner stride and a
 * 16-byte-multiple pitch go through TMA.  The others are either gathered by the
 * kernel with bounds-checked loads (products under 1e9 FLOPs) or first copied
 * once, by a separate HBM-bound kernel on `stream`, into an aligned buffer of
 * the library workspace (rows along the operand's smaller stride, pitch a
 * multiple of 8 elements, of 64 when the rows run along M or N) that the GEMM
 * then reads through TMA: the padding
 * form of boundary handling.  Likewise a C that TMA cannot store in place (an
 * unaligned base, a pitch or N that is not a multiple of 8 elements) is, for
 * such products, stored by TMA into an aligned buffer of the workspace and
 * then copied into the M x N view by a second HBM-bound kernel, which writes
 * no element outside the view.  Results are identical either way.
 *
 * Ownership: the caller owns A, B and C; they must stay valid until the work
 * on `stream` completes.  For shapes that use split-K, and for the aligned
 * operand copies, the library uses a per-device workspace that it allocates on
 * first need (cudaMalloc, which synchronises the device), grows on demand and
 * frees at process exit; such calls that run concurrently on different streams
 * must use gemm_f16_ws() with separate workspaces (which never copies operands:
 * it gathers them).
 *
 * Stream capture: a captured call records the workspace buffers current at
 * capture time.  Growing a buffer synchronises the device and cannot happen
 * inside a capture, so make one uncaptured call of the same shape first; and
 * since growth frees the old buffer, a later uncaptured call that needs more
 * workspace invalidates graphs that hold the old one.  Captured calls that
 * must stay replayable regardless should use gemm_f16_ws() (caller-owned
 * workspace) or gemm_f16_noalloc().
 *
 * Errors: argument errors are returned before any device work is queued;
 * launch errors after.  A device-side bounded-wait expiry does not show here:
 * see gemm_f16_device_status().
 */
gemm_f16_status gemm_f16(const void* A, int64_t stride_am, int64_t stride_ak,
                         const void* B, int64_t stride_bk, int64_t stride_bn,
                         void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                         cudaStream_t stream);

/*
 * Same as gemm_f16() with a caller-owned workspace: device memory of at least
 * gemm_f16_workspace_size() bytes, 256-byte aligned (else
 * GEMM_F16_ERR_OUT_OF_MEMORY), any contents.  When the
 * call uses split-K it first clears the workspace's counter block with
 * cudaMemsetAsync on `stream`, then the kernel writes fp32 partial sums into
 * the rest.  `workspace` may be NULL when the size query returns 0.  Calls
 * sharing one workspace must not overlap in time on the device.
 */
gemm_f16_status gemm_f16_ws(const void* A, int64_t stride_am, int64_t stride_ak,
                            const void* B, int64_t stride_bk, int64_t stride_bn,
                            void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes a call with these sizes needs on the current device (0 when
 * no tile is cut along K).  An upper bound over operand layouts; depends on
 * M, N, K, the options and the device's SM count. */
gemm_f16_status gemm_f16_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * Batched GEMM: `batch` problems of the same shape in one launch,
 *
 *   C_b[m, n] = fp16( sum_k A_b[m, k] * B_b[k, n] ),  0 <= b < batch,
 *
 * with A_b at A + b*stride_ab, B_b at B + b*stride_bb, C_b at C + b*stride_cb
 * (element offsets; inside a problem the addressing of gemm_f16()).  Follows
 * the TileLang tutorial ch. 14 "GEMM operators", section 4.4 (batched GEMM:
 * identical shapes, the (batch, m-tile, n-tile) space flattened into one tile
 * space).  A stride of 0 for A or B shares that operand across the batch
 * (e.g. one weight matrix); stride_cb must be at least the span of one C view,
 * so the problems' outputs do not overlap.  batch >= 1.
 * Operands whose batch stride is a multiple of 16 bytes keep the TMA path;
 * others are gathered.  Precision, tails, workspace, errors and asynchrony are
 * those of gemm_f16().
 */
gemm_f16_status gemm_f16_batched(const void* A, int64_t stride_ab, int64_t stride_am, int64_t stride_ak,
                                 const void* B, int64_t stride_bb, int64_t stride_bk, int64_t stride_bn,
                                 void* C, int64_t stride_cb, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 int64_t batch, cudaStream_t stream);

/* Most groups of one gemm_f16_grouped() call. */
#define GEMM_F16_MAX_GROUPS 64

/*
 * Grouped GEMM (the MoE expert layer): `groups` problems that share K and N
 * and differ in M.  Group g owns group_rows[g] consecutive rows of A and C
 * (the groups' rows concatenated in group order, starting at row 0) and
 * multiplies them by its own B_g at B + g*stride_bg:
 *
 *   C[r, n] = fp16( sum_k A[r, k] * B_g[k, n] )   for row r of group g.
 *
 * Follows the TileLang tutorial ch. 14 "GEMM operators", section 4.3 (grouped
 * GEMM: concatenated A and C with a per-group offset table, the scheduler
 * walking every group's tiles in one launch); the offset table is built here
 * from group_rows.
 *
 *   group_rows  HOST array of `groups` row counts (>= 0; empty groups allowed).
 *   groups      1 .. GEMM_F16_MAX_GROUPS.
 *   stride_bg   element distance between consecutive groups' B (0 shares one B).
 *   A, C        addressed as in gemm_f16() with M = sum of group_rows.
 * A tile never mixes groups: rows past a group's end are computed from the
 * next group's A rows but never stored.  With every group empty the call does
 * nothing and returns GEMM_F16_OK.  Other behaviour is that of gemm_f16().
 */
gemm_f16_status gemm_f16_grouped(const void* A, int64_t stride_am, int64_t stride_ak,
                                 const void* B, int64_t stride_bg, int64_t stride_bk, int64_t stride_bn,
                                 void* C, int64_t ldc, const int64_t* group_rows, int64_t groups,
                                 int64_t N, int64_t K, cudaStream_t stream);

/*
 * Fused output stage.  The pages name bias and activation fused into the
 * GEMM's output stage (TileLang tutorial ch. 14 "GEMM operators", section 6.3,
 * item 4, the epilogue of the comparison checklist; AI-infra knowledge base
 * "Matrix multiplication and memory-access optimisation", section 05) and, for
 * MoE layers, a gate/up GEMM fusing the two projections, with the activation
 * and the multiply ("C500 TileLang GEMM review", section 17.3).  They fix no
 * arithmetic; the library's reading:
 *
 *   B_up == NULL:  C[m,n] = fp16( act( sum_k A[m,k] B[k,n] + bias[n] ) )
 *   B_up != NULL:  C[m,n] = fp16( act( sum_k A[m,k] B[k,n] + bias[n] )
 *                                 * ( sum_k A[m,k] B_up[k,n] + bias_up[n] ) )
 *
 * B is the gate projection.  B_up is read with B's strides (and B's batch or
 * group stride): the two projections share a layout.  bias and bias_up are
 * fp16 vectors of N elements (unit stride) or NULL for zero; bias_up needs
 * B_up.  The sums accumulate in fp32; bias, activation and product are
 * evaluated in fp32 on them and rounded once to fp16.
 *
 * act: GEMM_F16_ACT_NONE (identity), _RELU (x < 0 ? 0 : x), _SILU
 * (x / (1 + e^-x)), _GELU (exact: x * Phi(x), Phi(x) = erfc(-x / sqrt 2) / 2).
 *
 * Execution: the gate/up form computes both products in one MMA stream per
 * tile (each stage holds the A rows once and both projections' columns; the
 * accumulator holds the gate columns, then the up columns of the same output
 * columns), so A is read once for both and neither product is written to
 * memory.  Its tiles are never cut along K and never swapped (small M runs
 * unswapped).  The bias/activation form runs every plan gemm_f16() runs,
 * including the swapped form (the bias then runs along the kernel view's
 * rows) and split-K / stream-K, where the stage is applied after the last
 * partial is added.
 *
 * Errors: those of gemm_f16(), plus GEMM_F16_ERR_INVALID_VALUE for an unknown
 * act, bias_up without B_up, an odd B_up / bias address or a negative
 * stride_bias, and GEMM_F16_ERR_ALIAS when C overlaps B_up, bias or bias_up.
 * Ownership and asynchrony are those of gemm_f16().
 */
enum {
    GEMM_F16_ACT_NONE = 0,
    GEMM_F16_ACT_RELU = 1,
    GEMM_F16_ACT_SILU = 2,
    GEMM_F16_ACT_GELU = 3
};

gemm_f16_status gemm_f16_fused(const void* A, int64_t stride_am, int64_t stride_ak,
                               const void* B, int64_t stride_bk, int64_t stride_bn,
                               const void* B_up, const void* bias, const void* bias_up, int act,
                               void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                               cudaStream_t stream);

/* gemm_f16_batched() with the fused output stage; problem b uses the bias
 * vectors at bias + b*stride_bias and bias_up + b*stride_bias (0 shares one). */
gemm_f16_status gemm_f16_batched_fused(const void* A, int64_t stride_ab, int64_t stride_am, int64_t stride_ak,
                                       const void* B, int64_t stride_bb, int64_t stride_bk, int64_t stride_bn,
                                       const void* B_up, const void* bias, const void* bias_up,
                                       int64_t stride_bias, int act, void* C, int64_t stride_cb, int64_t ldc,
                                       int64_t M, int64_t N, int64_t K, int64_t batch, cudaStream_t stream);

/* gemm_f16_grouped() with the fused output stage (the MoE expert layer: group g
 * multiplies its rows by B + g*stride_bg and B_up + g*stride_bg, with the bias
 * vectors at bias + g*stride_bias and bias_up + g*stride_bias). */
gemm_f16_status gemm_f16_grouped_fused(const void* A, int64_t stride_am, int64_t stride_ak,
                                       const void* B, int64_t stride_bg, int64_t stride_bk, int64_t stride_bn,
                                       const void* B_up, const void* bias, const void* bias_up,
                                       int64_t stride_bias, int act, void* C, int64_t ldc,
                                       const int64_t* group_rows, int64_t groups, int64_t N, int64_t K,
                                       cudaStream_t stream);

/* Size of the fixed scratch array behind gemm_f16_noalloc(). */
#define GEMM_F16_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * Same as gemm_f16(), but the library allocates nothing, ever.  (The pages
 * this library follows have no counterpart: this entry point exists for
 * callers, not for the method.)
 *
 * For callers that must not call cudaMalloc: a process that has handed all
 * device memory to its own pool, code that runs where a device allocation is
 * forbidden or where the device synchronisation cudaMalloc implies cannot be
 * afforded.  gemm_f16() grows a workspace with cudaMalloc the first time a
 * call cuts tiles along K (split-K or stream-K); this variant instead keeps
 * those counters and partial sums in one file-scope device array of
 * GEMM_F16_NOALLOC_SCRATCH_BYTES (8 MiB) that every device loading the library
 * holds until the process exits.  The caller still passes A, B and C.
 *
 * - Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it with the
 *   device's current context; make that first call before any stream capture
 *   on the device.  A call made in a different context (after
 *   cudaDeviceReset(), for instance) looks the address up again.
 * - Operands TMA cannot address are always gathered by the kernel, never
 *   copied to an aligned buffer (gemm_f16() copies them for large products).
 *   The plan this entry point runs is therefore the one gemm_f16_get_plan()
 *   reports while GEMM_F16_OPT_REPACK is 1; for aligned operands it is the
 *   plan of gemm_f16() whatever that option says.
 * - A call whose plan needs more than GEMM_F16_NOALLOC_SCRATCH_BYTES of
 *   workspace is rejected with GEMM_F16_ERR_OUT_OF_MEMORY before anything is
 *   queued (that plan's workspace_bytes, as above).
 * - Every call on a device shares the one array and finds the previous call's
 *   contents there: the call first clears the counter block with
 *   cudaMemsetAsync on `stream`.  Calls that overlap on the GPU (different
 *   streams, no ordering between them) race on the array and give undefined
 *   results; order them.
 * - Calls that cut no tile along K do not touch the array.
 * Other arguments, errors and asynchrony are those of gemm_f16().
 */
gemm_f16_status gemm_f16_noalloc(const void* A, int64_t stride_am, int64_t stride_ak,
                                 const void* B, int64_t stride_bk, int64_t stride_bn,
                                 void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 cudaStream_t stream);

/* Human-readable name of a status code; never NULL. */
const char* gemm_f16_status_string(int status);

/*
 * Read the current device's status word that kernels set on a bounded-wait
 * expiry (GEMM_F16_OK if none since the last reset).  Synchronises the device.
 * With reset != 0 the word is cleared and the library's split-K counters are
 * re-zeroed (an aborted kernel may leave them non-zero).
 */
gemm_f16_status gemm_f16_device_status(int* status, int reset);

/* How a call would be executed, for tests and profiling. */
typedef struct {
    int swap_ab;        /* computed as C^T = B^T A^T (small M) */
    int pair;           /* 2-CTA clusters sharing one 256-row tile (cta_group::2) */
    int a_tma, a_mn_major, b_tma, b_mn_major, c_tma;   /* kernel-view operands */
    int tile_m, tile_n, tiles_m, tiles_n;
    int splits, kblocks, units, grid, stages;
    int streamk_tiles;  /* trailing tiles whose K blocks are spread over all workers */
    int tail_split;     /* trailing partial wave of tiles cut along N into this many pieces */
    int smem_bytes;
    size_t workspace_bytes;
    int a_box3d, b_box3d;   /* MN-major TMA operand read as one 3-D box per stage */
    int cluster_ctas;       /* CTAs per cluster: 1, or 2 (pair form) */
    int fused;              /* the fused output stage runs (gemm_f16_fused_get_plan) */
    int gated;              /* gate/up form: tile_n output columns, 2 * tile_n accumulator columns */
    int repack;             /* bit 0: A, bit 1: B (and B_up) copied to an aligned buffer before the GEMM;
                               bit 2: C written to an aligned buffer, then copied into place */
    int two_k_loads;        /* both 64-wide K blocks of a pipeline phase come in one TMA copy per
                               operand (whole K blocks of full-width tiles; see GEMM_F16_OPT_TWO_K_LOADS) */
} gemm_f16_plan;

/* Fill *plan for the given arguments without launching anything.  Returns the
 * same validation status gemm_f16() would. */
gemm_f16_status gemm_f16_get_plan(const void* A, int64_t stride_am, int64_t stride_ak,
                                  const void* B, int64_t stride_bk, int64_t stride_bn,
                                  void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                  gemm_f16_plan* plan);

/* The plan gemm_f16_fused() would run for these arguments (same validation). */
gemm_f16_status gemm_f16_fused_get_plan(const void* A, int64_t stride_am, int64_t stride_ak,
                                        const void* B, int64_t stride_bk, int64_t stride_bn,
                                        const void* B_up, const void* bias, const void* bias_up, int act,
                                        void* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                        gemm_f16_plan* plan);

/*
 * Process-wide tuning and test knobs (not thread-safe with concurrent calls):
 *   GEMM_F16_OPT_FORCE_GATHER  bit 0: A, bit 1: B, bit 2: C never use TMA
 *   GEMM_F16_OPT_SPLITS        > 0: classic split-K, every tile cut into this many K
 *                              segments (clamped to the K blocks); replaces stream-K.
 *                              Units are numbered segment-major (all tiles' first
 *                              segments, then the second ones, ...).  0 default: none,
 *                              except for a swapped small-M pair plan whose tiles are
 *                              fewer than half the SMs but at least a quarter of them:
 *                              2, 3 or 4 segments, whichever fills the waves of units
 *                              best, when that fill is at least 80 % and each segment
 *                              keeps 8 or more K blocks
 *   GEMM_F16_OPT_TILE_N        > 0: force the tile width (multiple of 64, <= 256)
 *   GEMM_F16_OPT_PANEL         > 0: tile-rows per rasterisation panel (default 8, or 2 when the
 *                              launch has at most four waves of tiles or at most 16 tile columns)
 *   GEMM_F16_OPT_SWAP          0 auto, 1 never swap, 2 always swap
 *   GEMM_F16_OPT_TIMEOUT_MS    bounded-wait limit in ms (default 1000)
 *   GEMM_F16_OPT_MAX_CTAS      > 0: cap the persistent grid
 *   GEMM_F16_OPT_PAIR          0 default (2-CTA pair tiles for 256-wide tiles of TMA
 *                              operands without split-K, and for swapped small-M plans whose
 *                              B, the caller's A, is K-major), 1 never, 2 also for 128-wide
 *                              tiles
 *   GEMM_F16_OPT_STREAMK       0 default: stream-K tail when an operand is gathered (not
 *                              TMA-addressable) or when a swapped (small-M) plan has fewer
 *                              tiles than the device has SMs and does not take the K
 *                              segments above, whole tiles otherwise; 1: whole
 *                              tiles only; 2: stream-K tail whenever the tiles do not divide
 *                              evenly
 *   GEMM_F16_OPT_TAIL_SPLIT    0 default: cut the last partial wave of tiles along N
 *                              into narrower tiles; 1 never
 *   GEMM_F16_OPT_MAX_STAGES    >= 2: cap the pipeline depth in 64-wide K slots, rounded
 *                              down to an even count (default: as many as shared memory
 *                              holds, at most 16)
 *   GEMM_F16_OPT_REPACK        0 default: operands TMA cannot address are copied to an
 *                              aligned buffer, and a C TMA cannot store in place goes out
 *                              through one, for products of at least 1e9 FLOPs (gathered
 *                              operands and row-wise C stores below); 1 never; 2 always
 *   GEMM_F16_OPT_PDL           0 default: every kernel is launched as a programmatic dependent
 *                              of the kernel before it on the stream (its set-up overlaps that
 *                              kernel's tail; it reads and writes memory only after that kernel
 *                              has completed); 1 plain stream order
 *   GEMM_F16_OPT_DEBUG_BOUNDS  1: every gathered operand load and every per-thread store of C
 *                              is checked against the byte range its view spans (TMA
 *                              accesses are bounded by their tensor maps); one that would
 *                              leave it is skipped and gemm_f16_device_status() reports
 *                              GEMM_F16_ERR_BOUNDS.  2: the checker's own test, with each
 *                              range ending 16 bytes early.  0 default (off)
 *   GEMM_F16_OPT_L2_A, _L2_B   L2 eviction policy of the TMA loads of the kernel's A and B
 *   GEMM_F16_OPT_L2_C          operands and of the TMA stores of C (the kernel computes
 *                              C^T = B^T A^T when the plan swaps, so its A is then the
 *                              caller's B): 1 none, 2 evict first, 3 evict last; 0 default:
 *                              A evict first, B evict last and C evict first for one-problem,
 *                              non-gated launches of several waves whose A is at least 256 MB,
 *                              whose B is at most 48 MB and whose raster keeps each A row
 *                              panel within one wave (at most 16 tile columns, raster panels
 *                              of at most 2 rows); none otherwise
 *   GEMM_F16_OPT_TWO_K_LOADS   0 default: when both operands are TMA-addressable (K-major, or
 *                              MN-major read as 3-D boxes), the plan is not the single-CTA gate/up
 *                              form, and K holds at least two whole 64-wide blocks, each pipeline
 *                              phase of a full-width tile
 *                              loads its two K blocks with one copy per operand (a map with the
 *                              K block as an outer dimension), half the copies of one per K
 *                              block; a ragged last K block and narrow tail pieces keep one copy
 *                              per block.  1 one copy per K block always
 *   GEMM_F16_OPT_TEST_STALL    failure-detection test: 1 makes every CTA's MMA issuer wait
 *                              first on a barrier that nothing arrives on, so the bounded
 *                              wait runs out (after GEMM_F16_OPT_TIMEOUT_MS), the kernel
 *                              aborts cleanly and gemm_f16_device_status() reports
 *                              GEMM_F16_ERR_TIMEOUT; C is left undefined.  0 default
 * A value of 0 restores the default.  Returns GEMM_F16_ERR_INVALID_VALUE for an
 * unknown option or a value out of range.
 */
enum {
    GEMM_F16_OPT_FORCE_GATHER = 1,
    GEMM_F16_OPT_SPLITS = 2,
    GEMM_F16_OPT_TILE_N = 3,
    GEMM_F16_OPT_PANEL = 4,
    GEMM_F16_OPT_SWAP = 5,
    GEMM_F16_OPT_TIMEOUT_MS = 6,
    GEMM_F16_OPT_MAX_CTAS = 7,
    GEMM_F16_OPT_PAIR = 8,
    GEMM_F16_OPT_STREAMK = 9,
    GEMM_F16_OPT_TAIL_SPLIT = 10,
    GEMM_F16_OPT_MAX_STAGES = 11,
    /* 12 is not an option (gemm_f16_set_option() refuses it) */
    GEMM_F16_OPT_REPACK = 13,
    GEMM_F16_OPT_TEST_STALL = 14,
    GEMM_F16_OPT_PDL = 15,
    GEMM_F16_OPT_DEBUG_BOUNDS = 16,
    GEMM_F16_OPT_L2_A = 17,
    GEMM_F16_OPT_L2_B = 18,
    GEMM_F16_OPT_L2_C = 19,
    GEMM_F16_OPT_TWO_K_LOADS = 20
};
gemm_f16_status gemm_f16_set_option(int option, int64_t value);

/* GEMM_F16_ABI_VERSION of the loaded library. */
int gemm_f16_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H */

/*
 * gemm_relu -- C = ReLU(A . B) on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the GEMM+ReLU worked example of "Writing
 * High-Performance Kernels in TileLang" (atlascloud.ai guide, GEMM section,
 * listing `matmul_relu_kernel`; the same listing appears in the CSDN
 * TileLang note and the Korean edition of the guide):
 *   A is (M, K), B is (K, N), C is (M, N), all row-major IEEE binary16;
 *   products are accumulated in binary32 over the whole K range; ReLU,
 *   max(x, 0), is applied to the binary32 accumulator; the result is rounded
 *   to binary16 (round-to-nearest-even) and stored.  A ReLU result of zero
 *   is stored as +0.
 * The listing's correctness check is assert_close(c, relu(a @ b)) with
 * rtol = atol = 1e-2, which is the tolerance this library is tested to.
 *
 * All functions return a gemm_status_t value and never abort the process.
 * Device functions use the CUDA device that is current on the calling
 * thread.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream); it is declared void* so this header needs no CUDA
 * headers.
 */
#ifndef GEMM_RELU_H
#define GEMM_RELU_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* null pointer, negative or too large dimension */
    GEMM_ERR_ALIGNMENT = 2,          /* pointer not 16-byte aligned, or K % 8 or N % 8 != 0 */
    GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* no CUDA device, or not compute capability 10.3 */
    GEMM_ERR_OUT_OF_MEMORY = 4,      /* library-owned workspace could not be allocated */
    GEMM_ERR_LAUNCH = 5,             /* the kernel launch failed */
    GEMM_ERR_TIMEOUT = 6,            /* a device-side wait exceeded its limit (reported later) */
    GEMM_ERR_CUDA = 7,               /* another CUDA runtime error */
    GEMM_ERR_TOO_LARGE = 8           /* gemm_relu_noalloc: problem outside its fixed scratch */
} gemm_status_t;

/* Largest accepted M, N or K (TMA coordinates are signed 32-bit). */
#define GEMM_RELU_MAX_DIM 2147483647LL

/*
 * C = ReLU(A . B) if apply_relu != 0, else C = A . B (same rounding).
 *
 * A, B, C: device pointers to dense row-major binary16 matrices with leading
 *          dimensions K, N and N.  Each must be 16-byte aligned.  C must not
 *          overlap A or B (not checked).  The caller owns all three.
 * M, N, K: 0 <= M, N, K <= GEMM_RELU_MAX_DIM; K and N must be multiples of
 *          8 (the row pitch of A and B must be a multiple of 16 bytes for the
 *          tensor-memory-accelerator copies).  M has no constraint.
 *          M == 0 or N == 0: nothing is done.  K == 0: C is set to +0.
 *
 * Arithmetic: fp32 accumulation of the exact binary16 products, ReLU as
 * x > 0 ? x : +0 on the accumulator (so -0 and NaN become +0), then one
 * round-to-nearest-even cast (results beyond 65504 become infinities).
 * NaN and infinite inputs follow IEEE 754: a NaN operand or inf x 0 makes
 * a NaN term, infinities of both signs in one sum give NaN.
 *
 * Execution is asynchronous on `stream`; GEMM_OK means enqueued.  A device
 * fault of this call (e.g. a timed-out wait) is reported by the next
 * gemm_relu_check_device_error().  Shapes whose work is split along K use a
 * library-owned fp32 workspace and arrival counters kept per (device,
 * stream); they are grown on first need (which synchronizes that stream),
 * so issue one call of the largest shape before capturing a CUDA graph.
 * Calls on the same stream are ordered; calls on different streams use
 * different workspaces and may overlap.
 */
int gemm_relu(const void* A, const void* B, void* C,
              int64_t M, int64_t N, int64_t K, int apply_relu, void* stream);

/* Layouts of B for gemm_relu_ex. */
typedef enum {
    GEMM_B_KN = 0, /* B is K x N row-major (leading dimension N): C = ReLU(A . B) */
    GEMM_B_NK = 1  /* B is N x K row-major (leading dimension K): C = ReLU(A . B^T) */
} gemm_b_layout_t;

/* Element types of A, B and C for gemm_relu_ex (accumulation is fp32). */
typedef enum {
    GEMM_DTYPE_F16 = 0,  /* IEEE binary16 */
    GEMM_DTYPE_BF16 = 1  /* bfloat16 */
} gemm_dtype_t;

/*
 * gemm_relu with a choice of B layout and element type.  The (N, K) form of
 * B is the GEMM of "TileLang Guide: Composable Tiled AI Kernel Programming"
 * (sections "Tiles as First-Class Language Primitives" and "Production
 * Implementation", Step 1: B buffer (N, K), tile product with transpose_B);
 * bfloat16 is the element type of that page's FlashMLA listing.
 *
 * A (M x K) and C (M x N) are row-major; B is laid out as `b_layout` says;
 * all three hold `dtype` elements, and C is rounded to nearest-even in that
 * type.  Every other rule is gemm_relu's: 16-byte aligned pointers, K % 8 ==
 * 0 and N % 8 == 0, asynchronous on `stream`, the same workspace.
 * gemm_relu(...) is gemm_relu_ex(..., GEMM_B_KN, GEMM_DTYPE_F16, stream).
 * An unknown b_layout or dtype returns GEMM_ERR_INVALID_ARG.
 */
int gemm_relu_ex(const void* A, const void* B, void* C,
                 int64_t M, int64_t N, int64_t K, int apply_relu,
                 int b_layout, int dtype, void* stream);

/*
 * Same operation on HOST buffers: copies A and B to library-owned device
 * buffers, runs the GEMM, copies C back, and synchronizes `stream` before
 * returning.  Small problems run as one block on `stream`.  Problems of at
 * least 16 MiB (A, B and C together) with M >= 1024 run in up to 8 row
 * blocks (multiples of 256 rows, at least 512) pipelined over two internal
 * streams of the library: B and each block of A are copied in on one,
 * block i's GEMM runs on `stream` once its rows are in, and its rows of C
 * are copied out on the other, so the copy in of block i + 1, the GEMM of
 * block i and the copy out of block i - 1 overlap.  All of it starts after
 * the work already queued on `stream`.  (The environment variable
 * GEMM_RELU_HOST_BLOCK_ROWS=r, for tuning, sets the block height; 0 keeps
 * one block.)  Pinned host memory gives the fastest copies; pageable
 * memory also works.  Alignment rules on the host
 * pointers are waived (the device copies are aligned); K % 8 and N % 8
 * still apply.  Returns the device error status of the call as well.
 */
int gemm_relu_host(const void* A_host, const void* B_host, void* C_host,
                   int64_t M, int64_t N, int64_t K, int apply_relu, void* stream);

/*
 * Synchronizes `stream`, then reads and clears the current device's error
 * word.  Returns GEMM_ERR_TIMEOUT if a kernel of this library gave up a
 * bounded wait since the last check (the split-K counters are then reset),
 * GEMM_ERR_CUDA if the stream reports a CUDA error, else GEMM_OK.
 *
 * Every device wait of the kernels is bounded (2 s plus 2 us per k-block);
 * a CTA whose wait runs out records the error, stops its other roles, lets
 * its copies and MMAs in flight land, frees its tensor memory and returns.
 * Test hook of that path (tests only): with the environment variable
 * GEMM_RELU_TEST_DROP_KB=k set, gemm_relu, gemm_relu_ex and
 * gemm_relu_noalloc launch with every CTA leaving the copies of k-block k
 * of its first work item undone and with every wait limited to 1 ms, so
 * that the wait for that k-block runs out and the launch ends with the
 * error recorded (its C is incomplete).  A k outside [0, number of
 * k-blocks of the plan) or a plan that runs in clusters is refused with
 * GEMM_ERR_INVALID_ARG.
 */
int gemm_relu_check_device_error(void* stream);

/* Human-readable name of a gemm_status_t value (static storage). */
const char* gemm_relu_status_string(int status);

/* Frees every library-owned device buffer on every device.  Must not be
 * called while work of this library is in flight. */
void gemm_relu_shutdown(void);

/* ---- Entry point that allocates nothing -------------------------------- */

/* Bytes of the fixed device scratch array behind gemm_relu_noalloc (one per
 * device that loads the library, held until the process exits). */
#define GEMM_RELU_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * Same operation and arguments as gemm_relu, for callers that must not
 * allocate device memory.  gemm_relu grows a split-K workspace with
 * cudaMalloc the first time a shape needs one, and cudaMalloc / cudaFree
 * can synchronize the device; a caller in a loop that must never stall on
 * an allocation, or a process whose device memory is entirely reserved by
 * another allocator, cannot allow that.  This entry point never calls
 * cudaMalloc, cudaFree or any allocating routine: it runs the small-M
 * (swapped-operand) kernel with its split-K partial tiles, arrival
 * counters and error word in a fixed array of
 * GEMM_RELU_NOALLOC_SCRATCH_BYTES in device memory.  The caller still owns
 * and passes A, B and C (device pointers, same layout and alignment rules
 * as gemm_relu).  There is no counterpart on the pages: it is a deployment
 * convenience.
 *
 * Limits: 1 <= M <= 128 and K >= 1, and the split-K partials of the chosen
 * plan must fit in the array (about 8 MiB: ceil(N / 128) x round_up(M, 16)
 * x 512 bytes x the number of CTAs sharing a tile); otherwise it returns
 * GEMM_ERR_TOO_LARGE without launching anything.  M == 0 or N == 0 is a
 * no-op.
 *
 * The first call on a device does a one-time set-up there (device check,
 * the scratch array's device address via cudaGetSymbolAddress, kernel
 * attributes); make that first call before any stream capture.  With CUDA's
 * default lazy module loading, that first call is also when the driver
 * loads this code's module on the device, which reserves the array and the
 * kernel image (about GEMM_RELU_NOALLOC_SCRATCH_BYTES plus a few hundred
 * KiB of device memory): a caller that later reserves all remaining device
 * memory should make the first call at initialisation, before doing so.
 * Every call on a device shares the one array and finds it as the previous
 * call left it: each call first clears, on `stream`, the split-K counters
 * it needs to start at zero.  Calls whose execution overlaps on the GPU
 * (e.g. on two streams) race on the array and give undefined results;
 * issue them in one stream or otherwise ordered.  A timed-out device wait
 * in this variant is recorded in the array's own error word, which stays
 * set until gemm_relu_noalloc_check_device_error reads and clears it.
 */
int gemm_relu_noalloc(const void* A, const void* B, void* C,
                      int64_t M, int64_t N, int64_t K, int apply_relu, void* stream);

/*
 * The error check of gemm_relu_noalloc, which allocates nothing either:
 * synchronizes `stream`, reads the fixed array's error word on the current
 * device with one 4-byte copy, and clears the word (and the split-K
 * counters) if it was set.  Returns GEMM_ERR_TIMEOUT if a gemm_relu_noalloc
 * kernel on this device gave up a bounded wait since the last check (the C
 * of that call is incomplete), GEMM_ERR_CUDA if the stream reports a CUDA
 * error, GEMM_ERR_UNSUPPORTED_DEVICE if the device is not a GB300, else
 * GEMM_OK.  Like gemm_relu_noalloc, it has no counterpart on the pages.
 */
int gemm_relu_noalloc_check_device_error(void* stream);

/* ---- Host-only planning interface (no CUDA calls; usable without a GPU) -- */

typedef struct {
    int32_t path;        /* 0 nothing to do, 1 zero fill (K == 0), 2 tiled (one CTA per tile),
                            3 swapped operands (small M), 4 tiled by CTA pairs (256 x mma_n) */
    int32_t mma_m;       /* tcgen05 MMA M: 128, or 256 for a CTA pair (C rows; C columns for path 3) */
    int32_t mma_n;       /* tcgen05 MMA N: 128 or 256 (C columns) / padded M (path 3) */
    int32_t tile_m;      /* C tile rows */
    int32_t tile_n;      /* C tile columns */
    int32_t tiles_m, tiles_n, num_tiles;
    int32_t num_kb;      /* ceil(K / block_k) */
    int32_t block_k;     /* k-rows per shared-memory ring stage: 64, or 128 for path 3 */
    int32_t group_m;     /* tile rasterisation: tiles_m are walked in groups of group_m */
    int32_t grid;        /* persistent workers (a worker is `cluster` CTAs) */
    int32_t cluster;     /* CTAs per worker: 1, or 2 for path 4 */
    int32_t dp_tiles;    /* tiles [0, dp_tiles) are done whole, round-robin over CTAs */
    int32_t sk_tiles;    /* tiles [dp_tiles, num_tiles) are split along K (stream-K); when the
                            slots of each split tile share its reduction (every worker has at
                            most one split item, and the columns divide into whole epilogue
                            chunks per slot) the split tiles are instead [0, sk_tiles), the
                            whole ones after them, and each worker runs its split item first */
    int32_t sk_q, sk_r;  /* stream-K k-blocks per CTA: q, plus 1 for CTAs < r */
    int32_t splits;      /* > 1: tiles [dp_tiles, num_tiles) are instead cut into `splits`
                            equal K ranges; item i is (tile i % T, K range i / T), T the
                            number of such tiles, and worker c takes items c, c+grid, ... */
    int32_t max_slots;   /* most CTAs sharing one stream-K tile */
    int32_t num_stages;  /* shared-memory ring depth */
    int32_t stage_bytes; /* bytes of A and B tile per ring stage */
    int32_t smem_bytes;  /* dynamic shared memory per CTA */
    int32_t tmem_cols;   /* tensor-memory columns allocated per CTA */
    int32_t pack_a;      /* 1: A is first copied to a row pitch that is a multiple of 128 bytes (library
                            workspace), because neither A's nor B's pitch is (decided here for B stored
                            (K, N); B stored (N, K) shares A's pitch) */
    int64_t workspace_bytes; /* fp32 partial tiles for the stream-K tiles */
    int64_t counter_count;   /* arrival counters (one per split tile and CTA of a worker); the
                                counter array also holds max_slots ready flags per counter */
} gemm_relu_plan_t;

/*
 * Fills *plan with the decomposition gemm_relu uses for an M x N x K
 * problem on a device with `num_sms` multiprocessors (CTA pairs: at most
 * num_sms / 2; the runtime also caps them by the device's co-resident
 * cluster count).  Pure host code.  The environment variable
 * GEMM_RELU_FORCE_PATH (tuning and tests only) restricts the choice:
 * "tiled256", "tiled128", "tiled64" (128 x 256 / 128 x 128 / 128 x 64
 * tiles, one CTA each), "pair" (CTA pairs, 256 x 256 tiles), "swap"
 * (swapped operands, M <= 128 only), optionally followed by ":dp" to forbid
 * splitting tiles along K, by ":sN" to cut every tile into N equal K ranges
 * (the split schedule), by ":c2" to split every tile's K range between the
 * two CTAs of a cluster, which combine their halves through distributed
 * shared memory ("pair" has no ":c2": its cluster already holds one
 * 256-row tile), by ":sk" to run every tile stream-K over all workers, or
 * by ":tS" for full data-parallel waves with the leftover tiles cut into S
 * K ranges; ":no3d" keeps every TMA copy two-dimensional (one copy per
 * 64-k block or 64-column chunk); ":pk" / ":npk" force the copy of A to a
 * 128-byte pitch on (when K % 64 != 0) or off.
 * Returns GEMM_OK, or GEMM_ERR_INVALID_ARG for bad sizes / null plan.
 */
int gemm_relu_plan(int64_t M, int64_t N, int64_t K, int num_sms, gemm_relu_plan_t* plan);

/*
 * The TMA boxes of the copies the kernel issues for one ring stage under
 * *plan (host-only; used by the CPU tests, and by the library itself to
 * encode its tensor maps).  Elements are 16-bit.  An operand whose stage is
 * one 3-D copy views its row-major matrix as 64-element column blocks (a
 * third dimension 128 bytes apart); a box of several blocks lands them block
 * after block in shared memory.  b_layout is GEMM_B_KN or GEMM_B_NK; the
 * ":no3d" suffix of GEMM_RELU_FORCE_PATH keeps every copy 2-D.
 * Returns GEMM_OK, or GEMM_ERR_INVALID_ARG for a null pointer or a plan
 * without a kernel (path < 2).
 */
typedef struct {
    int32_t a_3d;           /* 1: A's stage is one 3-D copy of a_box[2] 64-k blocks */
    uint32_t a_box[3];      /* 64 (k), rows of A (128, or the padded M when swapped), 64-k blocks */
    int32_t b_3d;           /* 1: B's stage is one 3-D copy */
    uint32_t b_box[3];      /* B (K, N): 64 columns, k-rows, 64-column chunks; B (N, K): 64 (k),
                               rows of N, 64-k blocks */
    uint32_t b2_box[2];     /* B's second (2-D) map: 64 columns (or 64 k), k-rows (or rows of N) */
    int64_t b_view_inner;   /* 3-D B (K, N): the columns its view covers (whole 64-column chunks) */
} gemm_relu_boxes_t;

int gemm_relu_plan_boxes(const gemm_relu_plan_t* plan, int64_t M, int64_t N, int64_t K, int b_layout,
                         gemm_relu_boxes_t* boxes);

/*
 * The idx-th work item of worker `cta` under *plan, exactly as the kernel walks
 * it: C tile `tile` (tile_m_idx, tile_n_idx after rasterisation), k-blocks
 * [kb_begin, kb_end), and for a tile split along K its share `slot` of
 * `nslots`.  Returns 1 if the item exists, 0 past the CTA's last item,
 * negative on bad arguments.  Pure host code (used to test the schedule).
 */
int gemm_relu_plan_work_item(const gemm_relu_plan_t* plan, int cta, int idx,
                             int32_t* tile, int32_t* tile_m_idx, int32_t* tile_n_idx,
                             int32_t* kb_begin, int32_t* kb_end,
                             int32_t* slot, int32_t* nslots);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_RELU_H */

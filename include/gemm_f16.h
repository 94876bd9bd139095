/*
 * gemm_f16.h -- C ABI of the GB300 (sm_103a) dense fp16 GEMM
 *
 *     C[M,N] = A[M,K] . B[N,K]^T      fp16 operands, fp32 accumulation, fp16 result
 *
 * The operation is the one computed by "1. WGMMA: Hopper's Asynchronous Tensor
 * Core" (tilus tutorial), section "The Full Kernel": A is an [m, k] row-major
 * fp16 matrix, B an [n, k] row-major fp16 matrix used transposed, the
 * accumulator is fp32 and is cast to fp16 on the store to the [m, n]
 * row-major C.  The output cast rounds to nearest even.
 *
 * Layout: every matrix is row-major and densely packed (leading dimension =
 * number of columns): A has K contiguous elements per row, B has K contiguous
 * elements per row (it is "K-major", i.e. B^T is column-major), C has N
 * contiguous elements per row.
 *
 * Ownership: the caller owns every buffer (a, b, c, workspace) and the
 * stream.  The library never allocates or frees device memory and keeps no
 * per-call state; its only device-resident state is one 32-bit error word
 * per device (see gemm_f16_take_device_error) and the module-static scratch
 * array of gemm_f16_nt_noalloc.  Launches are asynchronous
 * on `stream`; a, b are only read; c is fully overwritten (no beta, no
 * accumulate).  Overlap of c with a or b is undefined.
 *
 * Host-side state per device (SM and cluster counts, the error word's
 * device address, the copy streams of gemm_f16_nt_host) is kept for the
 * context it was made in and made again when the current context changes,
 * so a cudaDeviceReset between calls is safe; a reset that races with a
 * call on another thread is not.  gemm_f16_nt and gemm_f16_nt_ws also keep,
 * per host thread, their last four launches (plan and encoded kernel
 * parameters), keyed on the context, the shape, the pointers a, b, c and
 * the workspace and its size: a call that repeats one of them launches it
 * again without planning and encoding (it reads nothing else; a buffer
 * freed and allocated again at the same address with the same shape is the
 * same launch).
 *
 * One GPU per call: a, b and c are memory of the current device.  The
 * variants that share one operand tile between the CTAs of a cluster by
 * multicast (see gemm_f16_variant_info) check this and return
 * GEMM_ERR_INVALID_ARG for any other pointer (a peer GPU's memory, host
 * memory); the library has no multi-GPU path.
 *
 * Errors: every entry point validates its arguments on the host before any
 * launch and returns a status code; it never exits or aborts the process.
 *   - m, n, k >= 0.  m == 0 or n == 0 is a no-op.  k == 0 writes C := 0
 *     (the empty sum) with an asynchronous memset on `stream`.
 *   - a, b, c must be non-null and 16-byte aligned when their size is > 0
 *     (GEMM_ERR_INVALID_ARG / GEMM_ERR_ALIGNMENT).
 *   - k % 8 == 0 and n % 8 == 0 (row pitches must be multiples of 16 bytes
 *     for the tensor-memory-access engine), m, n, k < 2^31
 *     (GEMM_ERR_UNSUPPORTED_SHAPE).  There is no fallback kernel.
 *   - the current device must be compute capability 10.3 (GEMM_ERR_ARCH).
 *   - a launch failure reported by the CUDA runtime -> GEMM_ERR_LAUNCH.
 *   - a pipeline wait inside the kernel that ran past its time limit is
 *     recorded on the device and reported later by gemm_f16_take_device_error
 *     as GEMM_ERR_TIMEOUT; the kernel returns instead of hanging.
 */
#ifndef GEMM_F16_H_
#define GEMM_F16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *gemm_stream_t;

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,
    GEMM_ERR_ALIGNMENT = 2,
    GEMM_ERR_UNSUPPORTED_SHAPE = 3,
    GEMM_ERR_ARCH = 4,
    GEMM_ERR_WORKSPACE = 5,
    GEMM_ERR_LAUNCH = 6,
    GEMM_ERR_TIMEOUT = 7,
    GEMM_ERR_CUDA = 8
} gemm_status_t;

/*
 * A launch plan: sizes only, no pointers, no device handles.  Produced by
 * the plan queries below, consumed by gemm_f16_nt_run.  All fields are plain
 * integers so a caller can inspect (and, for measurement, adjust) them.
 *
 * Tile rasterization follows "4. Pipeline Abstraction and Two Consumer Warp
 * Groups", section "Tile Rasterization": tile ids are walked in groups of
 * `raster_width` N-columns, row-major inside a group, the last group being
 * narrower when tiles_n is not a multiple of the width.
 */
typedef struct gemm_f16_plan {
    int32_t variant;         /* compiled kernel instance, see gemm_f16_variant_info */
    int32_t cta_group;       /* 1: one CTA per MMA tile; 2: a CTA pair (cluster of 2) shares one */
    int32_t block_m;         /* output rows per cluster tile (128 * cta_group, times the CTA pairs a
                                multicast cluster stacks along M) */
    int32_t block_n;         /* output columns per cluster tile (wide tiles: 512, 448 or 320, two MMAs of N =
                                256, 224 or 160; single CTAs sharing A by multicast: N times the CTAs along N) */
    int32_t block_k;         /* K depth of one pipeline stage (64) */
    int32_t stages;          /* shared-memory ring depth */
    int32_t raster_width;    /* N-columns per raster group (>= 1) */
    int32_t stream_k;        /* 0: every tile data-parallel; 1: data-parallel waves + stream-K tail */
    int32_t layout;          /* 0: B [N,K] and fp16 C (gemm_f16_nt*); 1: B [K,N] and fp32 D (gemm_f16_nn_f32*) */
    int32_t k_rotate;        /* 1: whole tiles walk K from a per-tile offset (set when no operand strip is
                                shared by two tiles; spreads DRAM requests; changes only summation order) */
    int64_t m, n, k;
    int64_t tiles_m, tiles_n, num_tiles;
    int64_t k_blocks;        /* ceil(k / block_k) */
    int64_t dp_tiles;        /* tiles walked data-parallel (all of them when stream_k == 0) */
    int64_t sk_iters;        /* K-block iterations of the remaining tiles, split evenly over the clusters */
    int32_t grid;            /* CTAs launched (persistent: <= resident slots) */
    int32_t cluster;         /* CTAs per cluster (cta_group times the multicast width times the K split) */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t num_sms;         /* SM count the plan was made for */
    uint64_t workspace_bytes;/* device workspace the plan needs (0 = none) */
    int32_t split_k;         /* 0: off; S > 1: split-K, each tile's K range cut into S parts (below) */
} gemm_f16_plan_t;

/*
 * Stream-K ("stream_k == 1"): the last one to two waves of tiles are not
 * given one tile per cluster; their K-block iterations are cut into equal
 * contiguous ranges, one per cluster, so no cluster idles in a partial last
 * wave.  A tile split between clusters is finished by the cluster holding
 * its first K block, which adds the fp32 partial tiles the others publish in
 * the workspace.  Workspace layout: grid partial tiles of 128 x (the
 * variant's block_n, see gemm_f16_variant_info) fp32 each, then grid 64-bit
 * flags.  A flag is set to a
 * stamp unique to the launch (a per-process random high word and a launch
 * counter), so flags left by earlier launches or found in fresh memory never
 * count and nothing needs clearing between launches; a workspace must not be
 * shared by launches that overlap on the GPU.  Every cluster of the grid
 * must be resident at once; the plan's
 * grid never exceeds that.  The fp32 partial sums change the rounding order
 * of split tiles only within the fp32 accumulation error.  For the wide tiles
 * (256 x 512, 256 x 448 and 256 x 320, block_n > 256) a requested tail
 * (stream_k = 1) covers only the partial last wave (every whole wave stays
 * data-parallel; 512 KB partials per pair); automatic plans never give them
 * one, because on GB300 it measured slower than the data-parallel waves.
 *
 * Split-K ("split_k == S > 1", stream_k 0): for products with fewer tiles
 * than resident clusters and a long K.  Each tile's K blocks are cut into S
 * equal contiguous parts; the clusters compute the tiles x S parts
 * independently and write each fp32 part to its own workspace slot (no
 * flags, no waiting between clusters); a second kernel, launched on the same
 * stream right after, adds a tile's S parts in a fixed order and writes the
 * fp16 result.  Workspace: tiles x S x (CTAs per cluster) parts of
 * 128 x block_n fp32.  Unlike the stream-K tail, no one cluster adds many
 * parts, so a tile's K can be spread over the whole GPU.  Variants with
 * fp16 C, B [N,K], tiles of whole 64-column chunks up to 256 columns and no
 * operand swap only (0-4, 11, 12, 18).
 */

/* Human-readable name of a status code (static string, never NULL).  No
 * counterpart on the pages (their only error convention is the day78 page's
 * check-and-exit macro); gemm_status_string is the same function. */
const char *gemm_f16_status_string(gemm_status_t status);
const char *gemm_status_string(gemm_status_t status);

/* Number of compiled kernel variants, and the shape of one of them: CTAs
 * per MMA (cta_group), tile N of one CTA or pair (a wide tile's two MMAs
 * together), ring depth, dynamic shared memory, CTAs
 * per cluster, layout (as in gemm_f16_plan_t), whether it computes the
 * transposed product C^T = B . A^T with the operands swapped (for products
 * with few rows of A; a plan of such a variant has tiles_m over n and
 * tiles_n over m), and its K split: 1, or the number of single CTAs of a
 * cluster that share each 128 x block_n tile, each accumulating one run of
 * its K blocks before they add the partials through distributed shared
 * memory (data-parallel plans only: no stream-K tail, no split-K).  Any
 * pointer may be NULL.  Returns GEMM_ERR_INVALID_ARG for an index out of
 * range. */
int32_t gemm_f16_variant_count(void);
gemm_status_t gemm_f16_variant_info(int32_t variant, int32_t *cta_group, int32_t *block_n,
                                    int32_t *stages, int32_t *smem_bytes, int32_t *cluster,
                                    int32_t *layout, int32_t *swapped, int32_t *k_split);

/*
 * Plan for the current CUDA device: validates the shape, checks the device
 * is compute capability 10.3, picks a variant, the grid and whether a
 * stream-K tail pays (then workspace_bytes > 0).  Host only, allocates
 * nothing, launches nothing.  The grid of tiles is the cdiv(m, BM) x
 * cdiv(n, BN) grid of "1. WGMMA", section "The Full Kernel"; the walk over
 * it is the rasterization of "4. Pipeline Abstraction and Two Consumer Warp
 * Groups", section "Tile Rasterization".
 */
gemm_status_t gemm_f16_nt_plan(int64_t m, int64_t n, int64_t k, gemm_f16_plan_t *out);

/*
 * Plan for a device with `num_sms` SMs (and `max_clusters` co-resident
 * 2-CTA clusters, or 0 for num_sms / 2) without touching any device.
 * `variant` < 0 picks automatically; `raster_width` <= 0 picks
 * automatically; `stream_k` < 0 picks automatically (stream-K tail or
 * split-K where they pay), 0 forbids both, 1 requests the stream-K tail and
 * 2 requests split-K (GEMM_ERR_INVALID_ARG for a variant without it).  Pure host code: it is the planning logic the
 * device entry points use, exposed for inspection and tests.
 */
gemm_status_t gemm_f16_nt_plan_for(int64_t m, int64_t n, int64_t k, int32_t num_sms,
                                   int32_t max_clusters, int32_t variant, int32_t raster_width,
                                   int32_t stream_k, gemm_f16_plan_t *out);

/*
 * As gemm_f16_nt_plan_for, with the co-resident cluster count of every
 * variant given, as the device entry points measure them
 * (cudaOccupancyMaxActiveClusters; a 152-SM GB300 fits 76 clusters of two
 * CTAs and 36 of four): clusters_by_variant[v] for every v below
 * gemm_f16_variant_count(), which `count` must equal; every entry >= 1
 * (for single-CTA variants, the SM count).  The automatic variant choice
 * weighs each candidate with its own count, so this reproduces a device's
 * plans on the host.  GEMM_ERR_INVALID_ARG for a NULL table, a wrong count
 * or an entry < 1.  Pure host code.
 */
gemm_status_t gemm_f16_nt_plan_for_clusters(int64_t m, int64_t n, int64_t k, int32_t num_sms,
                                            const int32_t *clusters_by_variant, int32_t count,
                                            int32_t variant, int32_t raster_width, int32_t stream_k,
                                            gemm_f16_plan_t *out);

/*
 * As gemm_f16_nt_plan, with the choices of gemm_f16_nt_plan_for overridable
 * (variant / raster_width / stream_k; negative or zero = automatic as
 * there), using the current device's SM count and co-resident cluster count.
 */
gemm_status_t gemm_f16_nt_plan_ex(int64_t m, int64_t n, int64_t k, int32_t variant,
                                  int32_t raster_width, int32_t stream_k, gemm_f16_plan_t *out);

/* Device workspace (bytes) gemm_f16_nt_ws needs for this shape on the
 * current device (the stream-K partial tiles and flags, or the split-K
 * parts); 0 when the chosen plan needs none.  No counterpart on the pages:
 * their kernels keep each tile's whole K loop in one thread block. */
gemm_status_t gemm_f16_nt_workspace_size(int64_t m, int64_t n, int64_t k, size_t *bytes);

/*
 * C = A . B^T on `stream`: the product of "1. WGMMA: Hopper's Asynchronous
 * Tensor Core", section "The Full Kernel" (its matmul(m_size, n_size,
 * k_size, a_ptr, b_ptr, c_ptr) with a stream added).  a: device pointer to
 * M*K fp16, b: device pointer to N*K fp16, c: device pointer to M*N fp16.
 * Plans automatically among the plans that need no workspace (no stream-K
 * tail, no split K).
 */
gemm_status_t gemm_f16_nt(int64_t m, int64_t n, int64_t k, const void *a, const void *b,
                          void *c, gemm_stream_t stream);

/* The product of gemm_f16_nt ("1. WGMMA", "The Full Kernel"), with a
 * caller-owned device workspace of ws_bytes bytes, 256-byte aligned: uses the automatic plan, with a stream-K tail or split K
 * when it pays.  workspace may be NULL/0 when gemm_f16_nt_workspace_size reports 0;
 * too small -> GEMM_ERR_WORKSPACE, misaligned -> GEMM_ERR_ALIGNMENT.  Calls
 * that share one workspace must not overlap on the GPU. */
gemm_status_t gemm_f16_nt_ws(int64_t m, int64_t n, int64_t k, const void *a, const void *b,
                             void *c, void *workspace, size_t ws_bytes, gemm_stream_t stream);

/* Launch a given plan (from any plan query, made for the current device's
 * SM count; either layout, c then being the plan's C or D).  The plan is
 * re-validated (GEMM_ERR_INVALID_ARG for a plan this library would not
 * make for its shape, e.g. a stream-K tail or split K on a K-split
 * variant).  Computes the product of "1. WGMMA", "The Full Kernel" (or,
 * for layout 1, of "wgmma_gemm.cu"); the plan's fields only choose how. */
gemm_status_t gemm_f16_nt_run(const gemm_f16_plan_t *plan, const void *a, const void *b, void *c,
                              void *workspace, size_t ws_bytes, gemm_stream_t stream);

/*
 * End-to-end form for host-resident data (the host-to-device copies,
 * product and copy back that "wgmma_gemm.cu" does in its main, here
 * overlapped): copies a_host (M*K fp16) and
 * b_host (N*K fp16) into the caller's device buffers a_dev / b_dev, runs
 * the GEMM into c_dev (automatic plan; the workspace, which may be NULL/0,
 * serves a stream-K tail or split K when it is large enough), and copies c_dev back to
 * c_host (M*N fp16).  Asynchronous on `stream`: the work starts after what
 * is already enqueued there and the stream continues after the last copy
 * back; pinned host memory makes the copies truly asynchronous.
 *
 * From M >= 2048 the rows of A and C go through in 2 to 8 chunks of whole
 * 256-row tiles, so that the copies overlap the GEMMs: B and the first rows
 * of A are copied in first, then chunk i's GEMM runs on `stream` while the
 * rows of chunk i+1 come in on an internal copy stream and those of chunk
 * i-1 go out on another.  The two copy streams and their events are created
 * on the first such call for each device and kept; buffers are never
 * allocated.  Calls from several host threads are enqueued one at a time.
 */
gemm_status_t gemm_f16_nt_host(int64_t m, int64_t n, int64_t k, const void *a_host,
                               const void *b_host, void *c_host, void *a_dev, void *b_dev,
                               void *c_dev, void *workspace, size_t ws_bytes, gemm_stream_t stream);

/*
 * The layout of "wgmma_gemm.cu" (its kernel and its CPU reference gemmCpu):
 *
 *     D[M,N] = A[M,K] . B[K,N]      fp16 operands, fp32 accumulation, fp32 result
 *
 * a: device pointer to M*K fp16, row-major (K contiguous); b: device pointer
 * to K*N fp16, row-major (N contiguous, i.e. B is not transposed); d: device
 * pointer to M*N fp32, row-major, fully overwritten with the fp32
 * accumulator (no rounding to fp16).  Same validation, errors, ownership and
 * asynchrony as gemm_f16_nt (k % 8 == 0, n % 8 == 0, 16-byte aligned
 * pointers); gemm_f16_nn_f32 uses a plan that needs no workspace,
 * gemm_f16_nn_f32_ws may add a stream-K tail (size from the workspace_bytes
 * of gemm_f16_nn_f32_plan_ex(m, n, k, -1, 0, -1, ...)).  Plans of this layout
 * also run through gemm_f16_nt_run.
 */
gemm_status_t gemm_f16_nn_f32(int64_t m, int64_t n, int64_t k, const void *a, const void *b,
                              void *d, gemm_stream_t stream);
gemm_status_t gemm_f16_nn_f32_ws(int64_t m, int64_t n, int64_t k, const void *a, const void *b,
                                 void *d, void *workspace, size_t ws_bytes, gemm_stream_t stream);
gemm_status_t gemm_f16_nn_f32_plan_ex(int64_t m, int64_t n, int64_t k, int32_t variant,
                                      int32_t raster_width, int32_t stream_k, gemm_f16_plan_t *out);

/*
 * Reads and clears the current device's error word after synchronizing
 * `stream`.  Returns GEMM_ERR_TIMEOUT if a kernel since the last call gave
 * up on a pipeline wait (*code, if non-NULL, receives which wait: see the
 * source), GEMM_OK otherwise, GEMM_ERR_CUDA if the runtime fails.
 */
gemm_status_t gemm_f16_take_device_error(gemm_stream_t stream, uint32_t *code);

/*
 * Host evaluation of the scheduler's arithmetic, the same inline functions
 * the kernel runs, for inspection and tests:
 *   gemm_f16_raster_coord: tile id -> (m_block, n_block) for a tiles_m x
 *     tiles_n grid walked in groups of `raster_width` N-columns.
 *   gemm_f16_fast_divmod: quotient and remainder of n by d (d >= 1) by the
 *     precomputed multiply-and-shift the kernel uses.
 */
gemm_status_t gemm_f16_raster_coord(int64_t tiles_m, int64_t tiles_n, int32_t raster_width,
                                    int64_t tile, int64_t *m_block, int64_t *n_block);
gemm_status_t gemm_f16_fast_divmod(uint32_t d, uint32_t n, uint32_t *q, uint32_t *r);

/*
 * Allocation-free form (no counterpart on the reference pages).
 *
 * Some callers cannot allocate device memory at all: code embedded in a
 * host process that owns every device allocation through its own pool (an
 * inference server, a framework plugin), where a side allocation is
 * forbidden or would break the host's memory accounting, and code on paths
 * that must not call cudaMalloc/cudaFree because those calls can
 * synchronize the device.  For them, gemm_f16_nt_noalloc computes the same
 * product as gemm_f16_nt_ws with the automatic plan (stream-K tail when it
 * pays) but takes its scratch -- the stream-K partial tiles and flags --
 * from one array that lives inside this library's device image, of
 * GEMM_F16_STATIC_SCRATCH_BYTES bytes; every GPU that loads the library
 * holds that array until the process exits.  The caller still passes the
 * operands and the output (device pointers, as for gemm_f16_nt).
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it; make that first call before any stream
 * capture.  The call allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.  All calls share the one array and it keeps
 * the last call's contents (the stream-K flags in it carry per-launch stamps,
 * so nothing there has to start at zero), so calls whose kernels overlap on
 * the GPU --
 * two streams, or two host threads -- race on it and give wrong results;
 * serialize them.  A plan that needs more scratch than the array holds is
 * rejected with GEMM_ERR_WORKSPACE before any launch (on a 152-SM GB300 the
 * largest plan needs 19.0 MiB).  Other errors as for gemm_f16_nt.
 */
#define GEMM_F16_STATIC_SCRATCH_BYTES (20u * 1024u * 1024u)
gemm_status_t gemm_f16_nt_noalloc(int64_t m, int64_t n, int64_t k, const void *a, const void *b,
                                  void *c, gemm_stream_t stream);

/*
 * Failure-detection hook for tests (no counterpart on the reference pages):
 * launches `plan` like gemm_f16_nt_run, except that the TMA producer of CTA 0
 * leaves its `skip_fill`-th ring-stage fill undone and every pipeline wait is
 * limited to `wait_limit_cycles` SM clock cycles.  The starved waits then
 * expire, the kernel records the failure in the device error word, frees its
 * tensor memory and returns; gemm_f16_take_device_error reports
 * GEMM_ERR_TIMEOUT.  C is left partly unwritten.  No fault, trap or hang.
 */
gemm_status_t gemm_f16_nt_run_stall_test(const gemm_f16_plan_t *plan, const void *a, const void *b,
                                         void *c, uint32_t skip_fill, long long wait_limit_cycles,
                                         gemm_stream_t stream);

#ifdef GEMM_F16_PHASE_TRACE
/*
 * Phase trace (only in the library built with GEMM_F16_PHASE_TRACE defined,
 * a measurement build; the product build has neither this function nor the
 * stamps).  Sets the device buffer that the single-CTA / CTA-pair kernel
 * launched by the following calls in this process writes its
 * phase stamps into, or NULL to stop.  Layout: 16 unsigned 64-bit slots per
 * CTA of the launch (slot = CTA index * 16 + phase), each overwritten with
 * %globaltimer (ns) every time its phase is passed, so a CTA that runs
 * several tiles keeps its last tile's stamps and a slot still 0 (the caller
 * zeroes the buffer) was not reached; give one buffer per traced launch.
 * Phases 0..9: kernel entry; set-up done; previous launch complete; a tile's
 * first ring stage full; its MMAs committed; its accumulator ready; its
 * stores issued; all bulk stores complete; teardown barrier; exit; for the
 * K-split variants also 10: a tile's partner slices sent, 11: the
 * partners' slices of it received.  The
 * buffer is owned by the caller and
 * must hold grid * 16 slots and stay allocated until the traced launches
 * have completed.  The wide-tile kernel is not traced.  The pointer is
 * captured at launch time (a CUDA graph keeps the value of its capture).
 */
void gemm_f16_trace_set(unsigned long long *buffer);
#endif

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_H_ */

/*
 * gemm.h -- C ABI of the GB300 (sm_103a) tiled GEMM library.
 *
 * One operation:  D = A * B + C
 *   A is M x K, B is K x N, C and D are M x N; any operand may be stored
 *   row-major or column-major with its own leading dimension.
 *
 * The operation is the matrix multiply-accumulate of the plain HIP kernel
 * "MatMulAdd_kernel2" (forum.sourcefind.cn, "DCU K100 ..." article, section
 * 5.2: each output is the K-sum of products plus C, with a column-major A and
 * a row-major B), computed the way the Triton "matmul_kernel" of the "Hopper
 * Support in Triton" slides does it (slide 5: BLOCK_M x BLOCK_N output tiles,
 * a loop over BLOCK_K slices into an fp32 accumulator, one conversion on
 * store), with the masked K tail of slides 14-15 (loads beyond K read zero)
 * and the GROUP_M tile order of the FlagGems "Hygon optimization" page
 * ("Grouped scheduling: improve L2 data reuse").
 *
 * Supported type combinations (ab_type, c_type, d_type):
 *   (F16|BF16, F16|BF16|F32 or C absent, F16|BF16|F32): fp32 accumulation,
 *       C widened to fp32 and added to the fp32 sum, one round-to-nearest-
 *       even conversion to d_type.
 *   (I8, I32 or C absent, I32): exact integer result (int32).
 *   (E4M3|E5M2, F16|BF16|F32 or C absent, F16|BF16|F32): 8-bit float
 *       operands in the OCP OFP8 encodings (E4M3: 4 exponent bits, bias 7,
 *       no infinities; E5M2: 5 exponent bits, bias 15, IEEE specials), read
 *       by the tensor core natively (tcgen05 kind::f8f6f4); fp32
 *       accumulation and the output path of the 16-bit types.  The pages
 *       name a scaled low-precision matrix product (mfma_scaled) as the next
 *       data type; this is its unscaled form.  A must be row-major and B
 *       column-major (both contiguous along K), else GEMM_ERR_UNSUPPORTED.
 *   (MXE4M3|MXE5M2, F16|BF16|F32 or C absent, F16|BF16|F32): the scaled
 *       form ("microscaled" data, the mfma_scaled entry point the "Tuning
 *       Triton" page names in its section 6, read by the OCP Microscaling
 *       definition): each element of A and B is an E4M3 / E5M2 value times
 *       the power-of-two scale of its 32-element K block, one scale per block
 *       of each row of A and of each column of B (tcgen05 kind::mxf8f6f4).
 *       Same layouts as the unscaled form; the handle runs with gemm_run_mx.
 *
 * Device pointers, caller-owned.  Every call is asynchronous on the given
 * stream.  All sizes are element counts.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
typedef enum {
  GEMM_F16 = 1,
  GEMM_BF16 = 2,
  GEMM_F32 = 3,
  GEMM_I8 = 4,
  GEMM_I32 = 5,
  GEMM_E4M3 = 6, /* OCP OFP8 E4M3 (operands only) */
  GEMM_E5M2 = 7, /* OCP OFP8 E5M2 (operands only) */
  GEMM_MXE4M3 = 8, /* E4M3 operands with E8M0 block scales (operands only; gemm_run_mx) */
  GEMM_MXE5M2 = 9  /* E5M2 operands with E8M0 block scales (operands only; gemm_run_mx) */
} gemm_dtype_t;

/* Storage order: row-major X[r,c] = X[r*ld + c]; column-major X[r + c*ld]. */
typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;

/* Status codes (0 = success, negative = failure). */
enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = -1,    /* a size, leading dimension or pointer is invalid */
  GEMM_ERR_UNSUPPORTED = -2,    /* type combination not supported */
  GEMM_ERR_MISALIGNED = -3,     /* an operand pointer is not aligned as gemm_run requires */
  GEMM_ERR_CUDA = -4,           /* a CUDA runtime/driver call or a launch failed */
  GEMM_ERR_DEVICE_TIMEOUT = -5, /* a bounded device-side wait expired (see gemm_get_status) */
  GEMM_ERR_ALLOC_FAILED = -6,   /* device or host allocation failed */
  GEMM_ERR_NO_DEVICE = -7       /* no sm_103 device is current */
};

/* Problem description.  ld* = 0 means packed (K or M for A, N or K for B,
 * N or M for C/D, by layout).  A leading dimension smaller than the packed
 * one is rejected.  c_type = 0 declares that C is always absent. */
typedef struct {
  int64_t M, N, K;
  gemm_dtype_t ab_type, c_type, d_type;
  gemm_layout_t layout_a, layout_b, layout_c, layout_d;
  int64_t lda, ldb, ldc, ldd;
} gemm_desc_t;

typedef struct gemm_plan* gemm_handle_t;

/* cudaStream_t without the CUDA headers: pass the stream handle (NULL = the
 * legacy default stream). */
typedef void* gemm_stream_t;

/*
 * gemm_create: validate desc, choose a plan (tile, stage count, raster
 * group, split-K, operand swap, repack, or the decode kernel for M <= 4
 * rows against a K-contiguous B) from the measured selection table
 * keyed on (M, N, K, types, layouts), and allocate on the current device the
 * workspace and the device status word that the plan needs.  The workspace
 * holds copies of operands whose rows the TMA unit cannot read in place
 * (rows not 16-byte aligned, or int8 widened to bf16; copy rows start on
 * 128-byte lines), aligned copies of 16-bit C and D with unaligned rows (C
 * is copied in and D copied out by extra kernels of gemm_run), split-K
 * partial sums and last-wave partials.
 *   out:  receives the handle (untouched on failure).
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED,
 * GEMM_ERR_NO_DEVICE, GEMM_ERR_ALLOC_FAILED or GEMM_ERR_CUDA.
 * Environment: GEMM_LOG=1 prints the chosen plan to stderr;
 * GEMM_FORCE_PLAN="bn=128,splits=2,group=8,swap=1" overrides fields of the
 * plan (for tuning sweeps; keys bn, splits, group, swap, grid, pair, ksub,
 * tail (the pair kernel's stream-K hybrid), skpat (0: its runs equal
 * instead of chained), sk (1: the single-CTA kernel's stream-K schedule,
 * shared tiles finished in the kernel), csk (1: a K split's CTAs reduce
 * their sums in a cluster instead of a reduce launch), kgroup (K slices
 * issued together), lsu (1: unaligned 16-bit rows loaded by producer warps
 * instead of a workspace copy), i8chunk (K of an exact int8 pass), decode,
 * dbulk: 1 takes the decode kernel's bulk-copy form whenever A's and B's
 * rows allow it, 0 never; dmma (1: the decode shapes' mma.sync form);
 * native_i8: 1 runs an int8 problem on the integer mma.sync kernel, which
 * reads A and B contiguous along K and copies them so first when they are
 * stored otherwise, instead of the exact emulation on the bf16 tensor
 * cores).
 */
GEMM_API int gemm_create(gemm_handle_t* out, const gemm_desc_t* desc);

/*
 * gemm_run: enqueue D = A*B + C on stream.  Never allocates and never
 * synchronises.  A, B, C, D must be device pointers aligned to their
 * element size; C may be NULL, which means C = 0 and C is not read.  The
 * tensor-core paths read A and B with TMA: when the description's leading
 * dimension gives rows that are not 16-byte aligned, gemm_create plans an
 * aligned workspace copy, but a base pointer that is not 16-byte aligned
 * while its rows are is rejected with GEMM_ERR_MISALIGNED (the handle has
 * no copy for it).  The decode path (M <= 4, K-contiguous B) and C / D
 * accept any element-aligned pointer.  An empty D (M or N zero) returns
 * GEMM_OK at once without looking at the pointers; K zero gives D = C
 * (A and B may then be NULL).  D may alias C only when both have the same
 * type, layout and leading dimension; D must not overlap A or B.
 * One handle must not be used by two streams at the same time (its
 * workspace and status word are shared by its calls).
 * Returns GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_MISALIGNED or
 * GEMM_ERR_CUDA (launch failure).  Device-side failures are reported by
 * gemm_get_status.
 */
GEMM_API int gemm_run(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
             gemm_stream_t stream);

/*
 * gemm_run_mx: enqueue D = (A * SA) * (B * SB) + C on stream for a handle
 * created with ab_type GEMM_MXE4M3 or GEMM_MXE5M2 (gemm_run rejects such a
 * handle, and this entry rejects any other, with GEMM_ERR_INVALID_ARG).
 * A, B, C, D as for gemm_run (A row-major, B column-major).  SA and SB are
 * device arrays of E8M0 exponents, one byte per 32-element block of K
 * (scale 2^(e - 127); e = 255 is NaN): SA holds M rows of ceil(K / 32)
 * bytes, row m for row m of A; SB holds N rows of ceil(K / 32) bytes, row n
 * for column n of B; both packed, any alignment.  A last block shorter than
 * 32 keeps its own scale.  The scales are first packed into the handle's
 * workspace by a small kernel, so SA and SB may be reused once the call's
 * work on the stream has started.  Products are exact and summed in fp32,
 * C is added and the result rounded once, as for the unscaled types.
 * Returns what gemm_run returns.
 */
GEMM_API int gemm_run_mx(gemm_handle_t h, const void* A, const uint8_t* SA, const void* B,
                         const uint8_t* SB, const void* C, void* D, gemm_stream_t stream);

/*
 * gemm_get_status: synchronise stream, then return and clear the device
 * status word of h: GEMM_OK, or GEMM_ERR_DEVICE_TIMEOUT when a kernel of an
 * earlier gemm_run gave up a bounded wait (its D is then undefined).
 * Returns GEMM_ERR_CUDA if the synchronisation itself fails.
 */
GEMM_API int gemm_get_status(gemm_handle_t h, gemm_stream_t stream);

/* gemm_destroy: free the handle's workspace and status word, and the device
 * copies, streams and events of gemm_host_io_enable (after synchronising the
 * device work that may still use them).  NULL is a no-op. */
GEMM_API int gemm_destroy(gemm_handle_t h);

/* gemm_strerror: static description of a status code. */
GEMM_API const char* gemm_strerror(int status);

/* gemm_plan_string: write a one-line description of the plan of h into buf
 * (at most n bytes including the terminator).  Returns the full length. */
GEMM_API int gemm_plan_string(gemm_handle_t h, char* buf, size_t n);

/* gemm_workspace_bytes: device workspace held by h (bytes), or -1. */
GEMM_API int64_t gemm_workspace_bytes(gemm_handle_t h);

/*
 * gemm_raster_tile: the grouped tile order, exported for host-side tests.
 * Maps the 1-D tile index t to (pid_m, pid_n) so that GROUP_M consecutive
 * tile rows share a column of B while they are in L2 (FlagGems "Hygon
 * optimization", "Grouped scheduling"); the final group is clamped to the
 * tile rows that remain.  Returns 0, or GEMM_ERR_INVALID_ARG when t is
 * outside [0, num_pid_m * num_pid_n) or a count is not positive.
 */
GEMM_API int gemm_raster_tile(int64_t t, int64_t num_pid_m, int64_t num_pid_n, int64_t group_m,
                     int64_t* pid_m, int64_t* pid_n);

/*
 * gemm_run_splitk_noalloc: D = A*B + C (fp16/bf16 A and B) with K split
 * `splits` ways (1..16), for callers that cannot allocate device memory when
 * they need the product: code running under a framework whose caching
 * allocator owns all device memory (a side cudaMalloc escapes its accounting
 * and can fail once the pool holds the device), and latency-critical paths
 * that cannot afford cudaMalloc or the device-wide synchronisation of
 * cudaFree.  The pages have no counterpart to this entry point; it exists
 * only for such callers.
 *
 * It allocates nothing: the fp32 partial sums and the device status word
 * live in one static device array of GEMM_NOALLOC_SCRATCH_BYTES that every
 * GPU loading this library holds until the process exits.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.
 * Every call shares the array (its status word is cleared by each call and
 * every partial sum is rewritten before it is read): calls whose kernels
 * overlap on the GPU race, so serialise them (one stream, or events).
 *
 * desc: as for gemm_create (layouts and leading dimensions); A and B must be
 * 16-byte aligned with 16-byte-multiple row strides (read in place by TMA).
 * Returns GEMM_OK; GEMM_ERR_INVALID_ARG for bad sizes, splits outside
 * [1, 16], or when splits * M * N * 4 bytes of partial sums exceed
 * GEMM_NOALLOC_SCRATCH_BYTES - 256; GEMM_ERR_UNSUPPORTED for other types;
 * GEMM_ERR_MISALIGNED; GEMM_ERR_NO_DEVICE; GEMM_ERR_CUDA.  A bounded
 * device-side wait that expires leaves D undefined and sets the array's
 * status word, which gemm_noalloc_status reads.
 *
 * The cached address belongs to the device's primary context: after
 * cudaDeviceReset (or any reset of that context) it no longer points at the
 * array, and this entry point must not be called again in that process.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
GEMM_API int gemm_run_splitk_noalloc(const gemm_desc_t* desc, int splits, const void* A,
                                     const void* B, const void* C, void* D,
                                     gemm_stream_t stream);

/*
 * gemm_noalloc_status: synchronise stream, then return the status word that
 * the latest gemm_run_splitk_noalloc call on the current device left in the
 * static array: GEMM_OK, or GEMM_ERR_DEVICE_TIMEOUT when one of its kernels
 * gave up a bounded wait (its D is then undefined).  Allocates nothing and
 * does not clear the word (the next call clears it).  Returns
 * GEMM_ERR_NO_DEVICE or GEMM_ERR_CUDA when the device, the synchronisation
 * or the 4-byte read fails.  The pages have no counterpart to this entry
 * point.
 */
GEMM_API int gemm_noalloc_status(gemm_stream_t stream);

/*
 * Kernel timing (a measurement hook; the operation is unchanged).
 * gemm_timing_enable(h, n): each of the next n gemm_run calls on h records a
 * pair of CUDA events on its stream, immediately before and immediately after
 * the launch of the tensor-core GEMM kernel (the repack, int8 widening and
 * split-K reduce kernels fall outside the pair).  The events are created
 * here, so gemm_run still allocates nothing; n = 0 switches timing off and
 * destroys them.  Calling it again restarts the count.  Returns GEMM_OK,
 * GEMM_ERR_INVALID_ARG (n < 0) or GEMM_ERR_CUDA.
 * gemm_timing_read(h, ms, n): waits for the recorded runs and writes the
 * kernel duration of the first min(n, runs recorded) of them, in
 * milliseconds, to the caller's host array ms; returns how many it wrote, or
 * GEMM_ERR_INVALID_ARG / GEMM_ERR_CUDA.
 */
GEMM_API int gemm_timing_enable(gemm_handle_t h, int n);
GEMM_API int gemm_timing_read(gemm_handle_t h, float* ms, int n);

/*
 * Host buffers.  The same operation, for operands that live in host memory;
 * the pages have no counterpart (their timings start from operands already
 * on the device).
 * gemm_host_io_enable(h): allocates on h's device two sets of device copies
 * of A, B, C and D (each the span of the operand in the description's
 * layout and leading dimension) and three streams owned by h.  Call once;
 * freed by gemm_destroy.  Returns GEMM_OK, GEMM_ERR_INVALID_ARG (h null or
 * another device current) or GEMM_ERR_ALLOC_FAILED.
 * gemm_run_host_batch(h, n, A, B, C, D, stream): n products D[i] = A[i] *
 * B[i] + C[i], every operand in host memory (arrays of n host pointers laid
 * out as the description says; C may be NULL, or C[i] NULL, for C = 0,
 * and is ignored when the description has no C type).
 * Host memory should be page-locked (cudaHostAlloc / cudaHostRegister);
 * pageable memory works but its copies do not overlap.  For each i: the
 * host-to-device copies of A[i], B[i], C[i] into one device set, gemm_run
 * on it, and the device-to-host copy of D into D[i].  The sets alternate,
 * so the input copies of product i+1 overlap the GEMM of product i and the
 * output copy of product i-1 (copies in and out use separate streams).
 * The call only enqueues: it starts after the work already on `stream` and
 * `stream` waits for the last output copy, so synchronising `stream` (or
 * gemm_get_status on it) completes every D[i].  Products of one call
 * overlap; a second call on the same stream starts after the first one's
 * last output copy, so pass a stream of products in one call.  The caller keeps the host
 * buffers untouched until then.  Returns GEMM_OK, GEMM_ERR_INVALID_ARG (no
 * gemm_host_io_enable, a null pointer for an operand with elements), or
 * what gemm_run returns.
 */
GEMM_API int gemm_host_io_enable(gemm_handle_t h);
GEMM_API int gemm_run_host_batch(gemm_handle_t h, int n, const void* const* A,
                                 const void* const* B, const void* const* C, void* const* D,
                                 gemm_stream_t stream);

/*
 * gemm_pair_schedule: host-side view of how the CTA-pair kernel deals its
 * work to clusters (for tests; no device needed).  For a tiles_m x tiles_n
 * grid of tiles in the grouped order (group_m), num_kb 64-wide K slices,
 * ring stages of ksub slices and `clusters` clusters, with the stream-K
 * hybrid when stream_k != 0 and it applies (a partial last wave, at least
 * one full wave) -- its runs equal (stream_k = 1), or laid out in chains of
 * at most two pieces a run where the shape allows (stream_k = 2, what the
 * kernel runs by default) -- it returns the number of units of cluster cid; when out
 * is non-NULL it also writes unit i of that cluster as out[0..6] = tile
 * row, tile column, first K slice, end K slice, shared-tile flag, part
 * (1 leaves its fp32 partial, 0 adds the partial and finishes the tile) and
 * the partial-sum slot.  Returns GEMM_ERR_INVALID_ARG for a bad argument or
 * i out of range.
 */
GEMM_API int gemm_pair_schedule(int64_t tiles_m, int64_t tiles_n, int64_t group_m, int num_kb,
                                int ksub, int clusters, int stream_k, int cid, int i,
                                int64_t* out);

/*
 * gemm_cta_schedule: host-side view of how the single-CTA kernel deals its
 * work to `grid` CTAs (for tests; no device needed).  For a tiles_m x
 * tiles_n grid of tiles in the grouped order (group_m) and num_kb 64-wide K
 * slices: round-robin over the tiles x splits, or with stream_k != 0 one
 * contiguous run of (tile, K slice) iterations per CTA (grid at most
 * tiles_m * tiles_n * num_kb), a tile split over several CTAs being finished
 * by the CTA that holds its first K slice, after the other pieces (each the
 * first of its CTA's run) have left their fp32 partials.  Returns the number
 * of units of CTA `cta`; when out is non-NULL it also writes unit i as
 * out[0..8] = tile index, tile row, tile column, first K slice, end K slice,
 * pieces of the tile, this piece's rank in K order, the partial-sum slot it
 * writes (-1 for a whole tile and for the finishing piece) and the CTA that
 * the finishing CTA expects to hold this rank (-1 for a whole tile).
 * Returns GEMM_ERR_INVALID_ARG for a bad argument or i out of range.
 */
GEMM_API int gemm_cta_schedule(int64_t tiles_m, int64_t tiles_n, int64_t group_m, int num_kb,
                               int splits, int grid, int stream_k, int cta, int i, int64_t* out);

/*
 * gemm_decode_ring: host-side view of the shared-memory ring of the decode
 * kernel's bulk-copy form (for tests; no device needed).  For M rows
 * (1..4) of K elements and cpb columns per block it returns the number of
 * ring stages and writes the columns per stage to *cps and the dynamic
 * shared memory a block requests to *smem_bytes.  The form is taken only
 * when stages * cps >= cpb (every column has a slot: one round trip) or
 * stages >= 2 with cps = 8.  Returns GEMM_ERR_INVALID_ARG for M outside
 * 1..4, K <= 0, cpb outside 1..32 or a null output pointer.
 */
GEMM_API int gemm_decode_ring(int M, int64_t K, int cpb, int* cps, int64_t* smem_bytes);

/*
 * Test hooks (not for production use).
 * gemm_debug_set: flags bit 0 makes the load warp of the next gemm_run (the
 * copy thread, in the decode kernel's bulk-copy form) skip its first stage
 * fill, so that the consumer's bounded wait expires and the
 * kernel exits with GEMM_ERR_DEVICE_TIMEOUT; timeout_ns (0 = default, two
 * seconds) bounds every device-side wait of later runs.
 */
#define GEMM_DEBUG_SKIP_FIRST_FILL 1
GEMM_API int gemm_debug_set(gemm_handle_t h, int flags, uint64_t timeout_ns);

/*
 * Timeline hook (profiling and tests; not for production use): with a
 * non-null dev_buf (device memory of at least grid x GEMM_TRACE_EVENTS
 * uint64 values, owned by the caller), every later gemm_run whose plan runs
 * a tcgen05 kernel (single CTA or CTA pair) writes, per CTA c, global-timer stamps
 * (ns) at dev_buf[c * GEMM_TRACE_EVENTS + e] for the events e: 0 kernel
 * entry, 1 past the wait for the previous kernel in the stream, 2 first
 * operand loads issued, 3 first ring stage landed, 4 last accumulator
 * committed by the MMA thread, 5 last accumulator seen by the epilogue, 6
 * last tile stored, 7 past the final block barrier (0-2 stamped by thread
 * 0, 3-4 by the MMA thread, 5-7 by the first epilogue thread); with the
 * splits of a tile reduced within a cluster, 8 the other splits' sums of
 * the CTA's own column slices landed and 9 its sums of the other CTAs'
 * slices sent.  The single-CTA kernel also stamps, in its first unit's
 * epilogue, 10 when every epilogue warp is past the accumulator wait and
 * 11 + i when the slice at position i < 4 is done (without a K split the
 * slices go in pairs, both stamped when the pair is done).  In
 * the CTA-pair kernel the even CTA of each cluster also stamps 10 + 2i and
 * 11 + 2i when its MMA thread starts and commits its unit i (i < 11).
 * Stamps of CTAs without work, and events that do not apply, are not
 * defined.
 * A null dev_buf turns the hook off.  The grid is the "grid=" field of the
 * plan string.
 */
#define GEMM_TRACE_EVENTS 32
GEMM_API int gemm_trace_set(gemm_handle_t h, uint64_t* dev_buf);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */

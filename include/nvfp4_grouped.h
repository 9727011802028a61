/*
 * nvfp4_grouped.h -- C ABI of the GB300 (sm_103a) NVFP4 block-scaled grouped GEMM.
 *
 * For every group g with m, n > 0 the library computes
 *
 *     C_g[i][j] = fp16( sum_k e2m1(A_g[i][k]) * e4m3(SFA_g[i][k/16])
 *                             * e2m1(B_g[j][k]) * e4m3(SFB_g[j][k/16]) )
 *
 * on the tensor cores (tcgen05 block-scaled MMA, fp32 accumulation, one
 * round-to-nearest-even conversion to fp16). This is the problem of the
 * kernelindex.com "nvfp4 group gemm" submissions 506336, 385043 and 499344:
 * the entry point there takes per-group (a, b, c) tensors, per-group reordered
 * (sfa, sfb) scale tensors and per-group (m, n, k, l) sizes, and writes each c
 * in place (submission 499344, custom_kernel and its docstring; element types
 * in submission 506336's module-level kernel configuration).
 *
 * Conventions shared by all entry points
 * --------------------------------------
 *  - Every device pointer is a CUDA device address on the current device.
 *    Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy
 *    default stream), never synchronises, and keeps no pointer after it
 *    returns. The caller owns every buffer.
 *  - Return value: NVFP4_OK (0) or a negative nvfp4_status. Argument errors
 *    are detected on the host before anything is enqueued.
 *  - Thread safety: calls may come from several host threads; calls on the
 *    same stream are ordered by the stream.
 */
#ifndef NVFP4_GROUPED_H
#define NVFP4_GROUPED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *nvfp4_stream_t;

/* Per-group problem size, as in the submissions' problem_sizes list: (m, n, k, l).
 * l is the batch count of the group: l independent products of the same
 * shape (the submissions' benchmarks use l = 1, submission 499344 docstring;
 * their operand layouts carry l as the outermost mode, submission 506336,
 * where the per-group tensors are built). l == 0 makes the group empty. */
typedef struct nvfp4_problem_size {
    int32_t m, n, k, l;
} nvfp4_problem_size;

typedef enum nvfp4_status {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = -1, /* null array, negative size, null pointer in a non-empty group, too many groups */
    NVFP4_ERR_UNSUPPORTED = -2, /* k % 32 != 0 or n % 32 != 0 in a non-empty group, sizes too large */
    NVFP4_ERR_MISALIGNED = -3,  /* a pointer of a non-empty group is not 16-byte aligned */
    NVFP4_ERR_CUDA = -4,        /* a CUDA runtime/driver call or a launch failed */
    NVFP4_ERR_TIMEOUT = -5      /* a kernel's bounded wait ran out (reported by nvfp4_device_status) */
} nvfp4_status;

/* Largest group_count accepted by nvfp4_grouped_gemm. */
#define NVFP4_MAX_GROUPS 512
/* Most matrices one nvfp4_pack_scales_batched call packs (the SFA and SFB of
 * a call with NVFP4_MAX_GROUPS groups). */
#define NVFP4_PACK_MAX_BATCH 1024

/*
 * nvfp4_grouped_gemm -- the grouped block-scaled GEMM.
 *
 * problem_sizes, A, B, SFA, SFB, C: HOST arrays of group_count entries. The
 * pointer arrays hold DEVICE addresses (shown for l = 1; a group with l
 * batches stacks them batch-outermost: A [l][m][k/2], B [l][n][k/2],
 * C [l][m][n], SFA / SFB l consecutive atom blocks of nvfp4_scale_bytes(m, k)
 * / nvfp4_scale_bytes(n, k) bytes, batch b computed from batch b alone):
 *   A[g]   e2m1 codes, [m][k/2] bytes, K-major, two codes per byte (the even k
 *          in the low nibble), row stride k/2 bytes.
 *   B[g]   e2m1 codes, [n][k/2] bytes, same layout.
 *   SFA[g] e4m3fn scales of A in the reordered atom layout, nvfp4_scale_bytes(m, k)
 *          bytes: 512-byte atoms of 128 rows x 4 scale blocks, byte
 *          16*(r%32) + 4*((r/32)%4) + (kb%4) inside atom (r/128)*ceil(k/64) + kb/4
 *          (submission 385043, kernel body where the scale tensors are built);
 *          padding rows/blocks must hold 0x00 (nvfp4_pack_scales writes them).
 *          Scales must be non-negative and not NaN.
 *   SFB[g] e4m3fn scales of B, nvfp4_scale_bytes(n, k) bytes, same layout.
 *   C[g]   fp16, [m][n] row-major, written in full; nothing else is written.
 * Group rules: a group with m == 0, n == 0 or l == 0 is skipped and its
 * pointers are not read (they may be null); a group with k == 0 and m, n, l > 0
 * gets C = +0. Non-empty groups need k % 32 == 0, n % 32 == 0, l <= 65535,
 * l*m and l*n <= 2^31 - 1 and 16-byte aligned pointers (A, B, SFA, SFB may be
 * null when k == 0).
 * The library keeps a small device workspace per (device, stream), allocated
 * on the first call for that pair and reused in stream order.
 */
int nvfp4_grouped_gemm(int group_count, const nvfp4_problem_size *problem_sizes,
                       const void *const *A, const void *const *B,
                       const void *const *SFA, const void *const *SFB,
                       void *const *C, nvfp4_stream_t stream);

/*
 * nvfp4_grouped_gemm_batched -- several independent grouped problems in one
 * launch: problem p owns the group_counts[p] consecutive entries that follow
 * those of problems 0..p-1 in problem_sizes, A, B, SFA, SFB and C (HOST
 * arrays, layouts as in nvfp4_grouped_gemm). The result of every problem is
 * the one its own nvfp4_grouped_gemm call would give (within the parity
 * rule; bit-identical unless a K-split schedule is chosen), and all of them
 * come from one kernel launch over the sum of the group counts, which must
 * not exceed NVFP4_MAX_GROUPS. This is the merged launch of submission
 * 506336 (its host code that concatenates the group tables of one benchmark
 * call's problems into a single launch), offered as an entry point.
 * Errors: problem_count < 0, null group_counts, a negative count or a sum
 * above NVFP4_MAX_GROUPS give NVFP4_ERR_INVALID_ARG; the groups are checked
 * as in nvfp4_grouped_gemm.
 */
int nvfp4_grouped_gemm_batched(int problem_count, const int *group_counts,
                               const nvfp4_problem_size *problem_sizes,
                               const void *const *A, const void *const *B,
                               const void *const *SFA, const void *const *SFB,
                               void *const *C, nvfp4_stream_t stream);

/*
 * nvfp4_grouped_gemm_device -- nvfp4_grouped_gemm with the group table in
 * DEVICE memory, so that the sizes and pointers can come from an earlier
 * kernel (a mixture-of-experts router) without a host round trip, and so that
 * a CUDA graph captured once can be replayed with new sizes and pointers.
 * The submissions build problem_sizes and the pointer lists on the host and
 * copy them to the device before each launch (submission 506336, host code
 * that prepares the grouped launch); here the kernel reads the caller's
 * arrays directly.
 *
 *   group_count      HOST int, 0 <= group_count <= NVFP4_MAX_GROUPS: number of
 *                    entries of every array (entries may describe empty
 *                    groups, e.g. (0, 0, 0, 1) for an expert with no tokens).
 *   problem_sizes    DEVICE array of group_count nvfp4_problem_size, 16-byte
 *                    aligned.
 *   A, B, SFA, SFB, C  DEVICE arrays of group_count DEVICE addresses (8-byte
 *                    aligned arrays), same element layouts as
 *                    nvfp4_grouped_gemm.
 * The arrays are read by the kernel when it runs (in stream order), not when
 * the call returns; they must stay valid and unchanged until then.
 * Group rules are those of nvfp4_grouped_gemm plus m, n, k <= 2^24 and
 * l*m, l*n <= 2^30; they are
 * checked on the device: a group that breaks one is skipped (its C is not
 * written), the rest of the call completes, and the next nvfp4_device_status
 * on the stream reports NVFP4_ERR_INVALID_ARG. Only the host arguments are
 * checked before anything is enqueued (group_count range, null or misaligned
 * arrays).
 * Every call rewrites the TMA descriptors of all group_count entries and
 * launches one CTA per SM; the kernel derives the tile schedule itself.
 * Graph capture: the workspace of (device, stream) is allocated by the first
 * call on that pair, so make one call on the capturing stream before the
 * capture begins; the captured launch may then be replayed any number of
 * times (the arrays' contents may change between replays; their addresses
 * and group_count are fixed by the capture).
 */
int nvfp4_grouped_gemm_device(int group_count, const nvfp4_problem_size *problem_sizes,
                              const void *const *A, const void *const *B,
                              const void *const *SFA, const void *const *SFB,
                              void *const *C, nvfp4_stream_t stream);

/* Largest group_count accepted by nvfp4_grouped_gemm_noalloc. */
#define NVFP4_NOALLOC_MAX_GROUPS 64

/*
 * nvfp4_grouped_gemm_noalloc -- nvfp4_grouped_gemm without any device
 * allocation. The submissions have no counterpart: it exists for callers that
 * must not have the library allocate device memory, such as frameworks that
 * hand out every byte from their own pre-planned arena, and latency-critical
 * callers that cannot afford a cudaMalloc (which may synchronise the whole
 * device) in the middle of their work.
 *
 * Same arguments, layouts, results and error codes as nvfp4_grouped_gemm,
 * except:
 *  - at most NVFP4_NOALLOC_MAX_GROUPS (64) groups; more is rejected with
 *    NVFP4_ERR_INVALID_ARG before anything is enqueued;
 *  - the scratch (tile prefix sum, group table, TMA descriptors, status word;
 *    about 24 KiB) is one fixed array in the library's device memory, which
 *    every GPU that loads the library holds until the process exits. The call
 *    never calls cudaMalloc, cudaFree or any other allocating routine;
 *  - the array has no room for the fp32 partial tiles of the split-K
 *    schedule, so calls always run whole output tiles. Calls with fewer tiles
 *    than about one and a half waves of the GPU are then slower than through
 *    nvfp4_grouped_gemm (measured on GB300: the 8-group decode shape, m
 *    40..192, n 4096, k 7168, 47.6 us instead of 39.6 us for the same
 *    kernel). Results are the same within the fp16 rounding of a different
 *    summation order;
 *  - every call on a device shares that array and it keeps the previous
 *    call's contents (each call rewrites what it reads and clears its call
 *    counters first). Calls whose work overlaps on the GPU -- on different
 *    streams, or from different host threads without ordering -- race on it:
 *    issue them in one stream or otherwise serialise them;
 *  - the status word in the array collects the bits of every call on the
 *    device until nvfp4_device_status (any stream) reads and clears it;
 *  - the first call on a device sets that device up (looks up the array's
 *    device address, encodes the TMA descriptor templates, sets kernel
 *    attributes); make that first call before any stream capture begins.
 *    The address stays cached for the process: after cudaDeviceReset the
 *    entry point must not be used again.
 */
int nvfp4_grouped_gemm_noalloc(int group_count, const nvfp4_problem_size *problem_sizes,
                               const void *const *A, const void *const *B,
                               const void *const *SFA, const void *const *SFB,
                               void *const *C, nvfp4_stream_t stream);

/*
 * nvfp4_set_tile_n -- choose the BLOCK_N of the GEMM tile for later calls in
 * this process: 128 or 256, or 0 to restore the automatic choice (256, or
 * 128 if the NVFP4_TILE_N environment variable says so). Results do not
 * depend on it.
 * Returns NVFP4_OK or NVFP4_ERR_INVALID_ARG.
 */
int nvfp4_set_tile_n(int block_n);

/*
 * nvfp4_scale_bytes -- size of the reordered atom layout of a [rows][k/16]
 * scale matrix: ceil(rows/128)*128 * ceil(k/64)*4 bytes. Returns 0 for
 * rows <= 0 or k <= 0.
 */
size_t nvfp4_scale_bytes(int rows, int k);

/*
 * nvfp4_pack_scales -- reorder row-major scales into the atom layout.
 *   sf_rowmajor  DEVICE, [rows][k/16] e4m3fn codes, row stride k/16 bytes.
 *   sf_atoms     DEVICE, nvfp4_scale_bytes(rows, k) bytes; every byte is
 *                written (padding = 0x00). Must not overlap sf_rowmajor.
 * Requires rows >= 0, k >= 0, k % 16 == 0; rows == 0 or k == 0 is a no-op.
 */
int nvfp4_pack_scales(const void *sf_rowmajor, int rows, int k, void *sf_atoms,
                      nvfp4_stream_t stream);

/*
 * nvfp4_pack_scales_batched -- nvfp4_pack_scales for `count` matrices in one
 * kernel launch (e.g. the SFA and SFB of every group of a call), each matrix
 * packed exactly as nvfp4_pack_scales packs it.
 *   count        0 <= count <= NVFP4_PACK_MAX_BATCH.
 *   sf_rowmajor, rows, k, sf_atoms: HOST arrays of count entries; the
 *                pointers are DEVICE addresses with the layouts and sizes of
 *                nvfp4_pack_scales; entries with rows == 0 or k == 0 are
 *                skipped. No two entries may write overlapping bytes.
 * Every entry is checked before anything is enqueued: the first bad one
 * gives NVFP4_ERR_INVALID_ARG (count out of range, null arrays, negative
 * rows or k, null pointers), NVFP4_ERR_UNSUPPORTED (k % 16 != 0) or
 * NVFP4_ERR_MISALIGNED (sf_atoms not 16-byte aligned). NVFP4_ERR_CUDA if the
 * launch fails. Asynchronous on `stream`.
 */
int nvfp4_pack_scales_batched(int count, const void *const *sf_rowmajor, const int *rows, const int *k,
                              void *const *sf_atoms, nvfp4_stream_t stream);

/* Element types of nvfp4_quantize_pack's input. */
#define NVFP4_DTYPE_BF16 0
#define NVFP4_DTYPE_F16 1

/*
 * nvfp4_quantize_pack -- quantise an activation matrix to NVFP4 and write it in
 * the layouts nvfp4_grouped_gemm reads, in one pass over the input.
 *   x         DEVICE, [rows][k] bf16 (x_dtype NVFP4_DTYPE_BF16) or fp16
 *             (NVFP4_DTYPE_F16), row-major, row stride k elements.
 *   codes     DEVICE, [rows][k/2] bytes: e2m1 codes, two per byte, the even k
 *             in the low nibble (the A / B layout of nvfp4_grouped_gemm).
 *   sf_atoms  DEVICE, nvfp4_scale_bytes(rows, k) bytes: e4m3fn scales in the
 *             atom layout (every byte written, padding 0x00).
 * Per row and 16-element block: amax = max|x|; sf = e4m3fn(amax / 6), rounded
 * to nearest (ties to the even code) and saturating at 448; code =
 * e2m1(x / dec(sf)), rounded to nearest (ties to the even code), saturating
 * at 6, keeping the sign of x (a negative x that rounds to zero gives -0);
 * every code is +0 when dec(sf) == 0. This is the quantisation the
 * "nvfp4 group gemm" task states for its inputs; the submissions receive
 * their operands already in this form (submission 499344, custom_kernel
 * docstring). Inputs must be finite (codes for NaN or infinity are
 * unspecified).
 * Requires rows >= 0, k >= 0, k % 16 == 0, rows <= 65535 * 128 and 16-byte
 * aligned pointers; rows == 0 or k == 0 is a no-op. Errors are detected on the
 * host. The outputs must not overlap x.
 */
int nvfp4_quantize_pack(const void *x, int x_dtype, int rows, int k, void *codes, void *sf_atoms,
                        nvfp4_stream_t stream);

/*
 * nvfp4_device_status -- read and clear the device-side status words of the
 * (current device, stream) workspace and of the current device's
 * nvfp4_grouped_gemm_noalloc array. Synchronises `stream`. *status receives
 * NVFP4_OK; NVFP4_ERR_TIMEOUT if a kernel of an earlier call gave up a
 * bounded wait (its C is then incomplete); or NVFP4_ERR_INVALID_ARG if an
 * nvfp4_grouped_gemm_device call skipped a group that breaks the group rules.
 * Returns NVFP4_OK or NVFP4_ERR_CUDA.
 */
int nvfp4_device_status(nvfp4_stream_t stream, int *status);

/* Human-readable name of an nvfp4_status value (static string). */
const char *nvfp4_status_string(int status);

/* Detail of the last error returned on the calling host thread (static storage). */
const char *nvfp4_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GROUPED_H */

/*
 * wq4 — W4A16 mixed-input GEMM for NVIDIA GB300 (sm_103a), C ABI.
 *
 * Computes Y[M,N] = X[M,K] . dequant(Wq)[N,K]^T with X, the scales and Y in bf16 or fp16,
 * 4-bit weight codes, one scale (and zero point) per group of G consecutive K elements (G = 128
 * by default; or no scales) and fp32 accumulation.
 *
 * The problem statement follows "aphrodite-engine/kernels/quantization/machete/
 * machete_mainloop.cuh": its header comment (weights prepacked once, then Y = mm(X, B_prepacked);
 * the product computed as the transpose Y^t = W^t X^t so the narrow type is the MMA's A side),
 * get_conversion_mode (scale-only and scale-with-zero modes), Arguments (pointers, strides, group
 * size, zero pointer) and can_implement (the argument rules reproduced under "Errors" below).
 * The grouped variant follows "sm90_gemm_array_tma_warpspecialized_cooperative.hpp" (one GEMM per
 * group index L, all in one persistent launch).
 *
 * Conventions for every entry point:
 *  - Pointers named X, Wq, scales, zeros, Wp, Y and workspace are DEVICE pointers. Arrays of
 *    shapes and of per-problem pointers in the grouped call are HOST arrays.
 *  - The caller owns every buffer. The library allocates no device memory.
 *  - Calls that take a stream are asynchronous on it; NULL means the legacy default stream.
 *  - Arguments are checked before anything is launched; on a negative status nothing was
 *    launched and no buffer was touched.
 *  - dtype: WQ4_BF16 or WQ4_FP16; X, the scales and Y share it. qtype: WQ4_U4B8 (value =
 *    (code - 8) s), WQ4_U4_ZP (value = (code - z) s with a 4-bit zero point per group and row) or
 *    WQ4_U4_FZP (value = code s + zf with a float zero of the dtype per group and row, added after
 *    the scale: the scale-with-zero conversion of "machete_mainloop.cuh", transform_A_kblock;
 *    not with device-resident shapes or pointers).
 *  - group_size G: 64, or a multiple of 128 that divides K (G == K: one scale per row,
 *    channel-wise; "machete_mainloop.cuh", can_implement and load); other sizes give
 *    WQ4_ERR_UNSUPPORTED. N and K multiples of 128; M >= 0. The G passed to the GEMM calls must
 *    be the one the weight was prepacked with (the blob holds one scale set per 128-K record,
 *    two with G = 64).
 */
#ifndef WQ4_H_
#define WQ4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* wq4_stream_t;

enum {
    WQ4_OK = 0,
    WQ4_ERR_INVALID = -1,      /* bad shape, null pointer, zero pointer given/missing, bad enum */
    WQ4_ERR_ALIGN = -2,        /* a pointer is not 16-byte aligned (TMA rule) */
    WQ4_ERR_UNSUPPORTED = -3,  /* valid for the method, not built here (a group size that is not a
                                  multiple of 128 dividing K, N or K not multiples of 128, ...) */
    WQ4_ERR_WORKSPACE = -4,    /* workspace missing or smaller than the *_workspace_bytes answer */
    WQ4_ERR_CUDA = -5,         /* a CUDA runtime call failed (no device, launch failure, ...) */
    WQ4_ERR_TIMEOUT = -6,      /* a kernel's bounded pipeline wait ran out (see wq4_get_last_error) */
    WQ4_ERR_BOUNDS = -7        /* debug build only: a kernel's bounds check failed (wq4_last_violation) */
};
enum { WQ4_BF16 = 0, WQ4_FP16 = 1 };
enum { WQ4_U4B8 = 0, WQ4_U4_ZP = 1, WQ4_U4_FZP = 2 };

/* Library version (major * 10000 + minor * 100 + patch) and a text for a status code. */
int wq4_version(void);
const char* wq4_status_string(int status);

/* ------------------------------------------------------------------------------------------ *
 * Prepack ("machete_mainloop.cuh", header comment: weights reordered once into the layout the
 * mainloop consumes, so each thread fetches several MMAs' worth with one 128-bit load).
 * ------------------------------------------------------------------------------------------ */

/* Bytes of the prepacked blob for an N x K weight (256-byte header + one record per
 * 128-row x 128-K tile). Returns 0 if the shape is not supported. */
size_t wq4_prepacked_bytes(int N, int K, int group_size, int qtype);

/* Reorders a weight into the prepacked blob.
 *   Wq      [N][K/8] uint32, code of element k = 8j+i in bits [4i, 4i+4) of word j.
 *   scales  [K/G][N] dtype, N contiguous (one scale per group and row); NULL for a weight
 *           without scales (WQ4_U4B8 only: the value is code - 8, the direct conversion of
 *           "machete_mainloop.cuh", get_conversion_mode), stored as 1.0.
 *   zeros   WQ4_U4_ZP: [K/G][N/8] uint32, zero point of row n = 8j+i in bits [4i, 4i+4) of
 *           word j. WQ4_U4_FZP: [K/G][N] dtype, the float zero of each (group, row), N
 *           contiguous like the scales. Required for both (with scales); NULL for WQ4_U4B8.
 *   Wp_out  wq4_prepacked_bytes(...) bytes, 16-byte aligned; fully overwritten.
 * Integer work: the blob is a bit-exact permutation of the inputs. */
int wq4_prepack(const uint32_t* Wq, const void* scales, const void* zeros,
                int N, int K, int group_size, int dtype, int qtype,
                void* Wp_out, wq4_stream_t stream);

/* Exact inverse of wq4_prepack (a test and export aid), with the same G: group j of scales_out
 * [K/G][N] and zeros_out (wq4_prepack's zeros layout for the qtype) is read from its first 128-K
 * record. zeros_out must be NULL for U4B8; scales_out may be NULL (not written). */
int wq4_unprepack(const void* Wp, int N, int K, int group_size, int dtype, int qtype,
                  uint32_t* Wq_out, void* scales_out, void* zeros_out, wq4_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * GEMM ("machete_mainloop.cuh": transform_A_kblock defines the dequantised value (code - zero)
 * times the group's scale; mma/load define one scale row per group of K).
 * ------------------------------------------------------------------------------------------ */

/* Workspace bytes wq4_mm needs on the current device for this shape (partial sums of K-split
 * tiles and their arrival counters) under the current options; 0 when the call takes the
 * decode kernel (at most 32 tokens, where that kernel applies: WQ4_OPT_DECODE), which uses none
 * (workspace may then be NULL). The workspace must be
 * zero-filled once when allocated; every completed call leaves its counters at zero again.
 * Calls that may overlap on the GPU need separate workspaces. */
int wq4_workspace_bytes(int M, int N, int K, int group_size, size_t* bytes);

/* wq4_workspace_bytes for a given qtype. WQ4_U4_FZP on the tensor-core path (not the decode
 * kernel) adds a table of activation sums that a pre-pass writes on the stream before the GEMM
 * (per token and zero group of 128 K, or 64 with G = 64, split into a high and a low 16-bit
 * part): (M rounded up to the token tile) x 2 x (zero groups rounded up to 64) x 2 bytes after the
 * plan's own bytes (256-byte aligned). For the other qtypes the answer equals wq4_workspace_bytes. */
int wq4_workspace_bytes_ex(int M, int N, int K, int group_size, int qtype, size_t* bytes);

/* Y = X . dequant(Wp)^T.
 *   X   [M][K] dtype row-major, 16-byte aligned.
 *   Wp  blob from wq4_prepack with the same N, K, group_size, dtype and qtype.
 *   Y   [M][N] dtype row-major, fully overwritten (fp32 sums rounded to nearest even).
 *   workspace / workspace_bytes: see wq4_workspace_bytes.
 * M == 0 is a no-op. Results are identical from run to run (fixed reduction order). */
int wq4_mm(const void* X, const void* Wp, void* Y, int M, int N, int K, int group_size,
           int dtype, int qtype, void* workspace, size_t workspace_bytes, wq4_stream_t stream);

/* Y = alpha * (X . dequant(W)^T) + beta * C + bias, the epilogue with a source operand of the
 * pages' kernels ("sm90_gemm_array_tma_warpspecialized_cooperative.hpp": the epilogue loads C
 * and combines it with alpha and beta) plus a bias per output column:
 *   C     [M][N] dtype, row-major, 16-byte aligned; read only when beta != 0 (may then be NULL
 *         only if beta == 0); C may be Y itself (in place: every element is read, then written,
 *         by the same thread).
 *   bias  [N] dtype, 16-byte aligned, or NULL.
 * Computed in fp32 (alpha * acc, then + beta * C, then + bias) and rounded to dtype once.
 * Everything else as wq4_mm (same workspace rule, same plans). */
int wq4_mm_ex(const void* X, const void* Wp, void* Y, int M, int N, int K, int group_size,
              int dtype, int qtype, float alpha, const void* C, float beta, const void* bias,
              void* workspace, size_t workspace_bytes, wq4_stream_t stream);

/* Workspace bytes for wq4_grouped_mm with these P problems (host arrays of shapes); the same
 * zero-fill rule as wq4_workspace_bytes. */
int wq4_grouped_workspace_bytes(int P, const int* M, const int* N, const int* K, int group_size,
                                size_t* bytes);

/* The same for a weight format: float zeros (WQ4_U4_FZP) add the activation-sum tables of the
 * problems' zero steps (see wq4_workspace_bytes_ex); other formats as wq4_grouped_workspace_bytes. */
int wq4_grouped_workspace_bytes_ex(int P, const int* M, const int* N, const int* K, int group_size,
                                   int qtype, size_t* bytes);

/* P independent problems Y_p = X_p . dequant(Wp_p)^T in one launch (P <= 64).
 *   M, N, K            host arrays of P shapes; M[p] == 0 skips problem p (its pointers are
 *                      not dereferenced and may be NULL).
 *   X, Wp, Y           host arrays of P device pointers, per-problem layouts as in wq4_mm.
 * All problems share group_size, dtype and qtype. When every non-empty problem has at most 32
 * tokens (decode-sized experts), the problems' row blocks go through the decode kernel in one
 * launch, as wq4_mm does for one problem: no workspace (the workspace queries answer 0). */
int wq4_grouped_mm(int P, const int* M, const int* N, const int* K,
                   const void* const* X, const void* const* Wp, void* const* Y,
                   int group_size, int dtype, int qtype,
                   void* workspace, size_t workspace_bytes, wq4_stream_t stream);

/* Same computation as wq4_mm, for callers that cannot allocate device memory or hand the
 * library a buffer: code that must not call cudaMalloc (for instance inside a section where
 * allocation would stall or break a stream capture, or a plugin whose host runtime owns every
 * device allocation). There is no counterpart in the pages: it only changes where the K-split
 * scratch lives. Instead of a caller workspace it uses one fixed 24 MiB array in the library's
 * device memory (every GPU that loads the library holds it until the process exits).
 * Plans: calls that wq4_mm sends to the decode kernel go there too (no scratch). A GEMM plan
 * whose K-split scratch fits the array is wq4_mm's own; one that would need more (for example
 * 4096 tokens x N = 4096, whose 192-token tiles need 30 MB) keeps every tile whole instead.
 * Results: bit-identical to wq4_mm's under the same options when the plan is wq4_mm's; with
 * tiles kept whole, the same fp32 sums added in another order (equal within rounding, not bit
 * for bit). WQ4_ERR_WORKSPACE only when an option forces a split (WQ4_OPT_GRID,
 * WQ4_OPT_SPLIT_ALL) whose scratch exceeds the array.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress) with that device
 * current, whatever the shape; make that first call before any stream capture. The array is
 * shared by all calls on a device and keeps the last call's contents; each call that uses it
 * clears the part that must start at zero (an async memset on `stream`). Calls that overlap on
 * the GPU (other streams, or concurrently running graphs) race on the array and must be
 * serialised by the caller. Arguments and errors as wq4_mm. */
int wq4_mm_static_scratch(const void* X, const void* Wp, void* Y, int M, int N, int K, int group_size,
                          int dtype, int qtype, wq4_stream_t stream);

/* Grouped GEMM whose token counts are known only on the device (tokens routed to experts by a
 * kernel on the same stream): the grouped call of "sm90_gemm_array_tma_warpspecialized_cooperative.hpp"
 * with its problem shapes in device memory.
 *   M_dev   DEVICE array of P int token counts, read when the work starts (stream order);
 *           each is clamped to [0, M_cap[p]].
 *   M_cap   HOST array: rows that X[p] and Y[p] hold (the capacity of each problem's buffers).
 *   N, K, X, Wp, Y, group_size, dtype, qtype as in wq4_grouped_mm; X[p] is [M_cap[p]][K[p]] and
 *           only its first M_dev[p] rows matter; rows of Y[p] beyond M_dev[p] are not written.
 *   workspace  wq4_grouped_device_m_workspace_bytes(P) bytes, 16-byte aligned (the tile table
 *           a set-up kernel writes before the GEMM); no zero fill needed.
 * The plan (token tile, grid) is made for the capacities, with every tile whole. */
int wq4_grouped_device_m_workspace_bytes(int P, size_t* bytes);
int wq4_grouped_mm_device_m(int P, const int* M_dev, const int* M_cap, const int* N, const int* K,
                            const void* const* X, const void* const* Wp, void* const* Y,
                            int group_size, int dtype, int qtype,
                            void* workspace, size_t workspace_bytes, wq4_stream_t stream);

/* Grouped GEMM whose per-problem pointers live in device memory (written by a kernel on the same
 * stream, for example the expert buffers of a token router): the grouped call of
 * "sm90_gemm_array_tma_warpspecialized_cooperative.hpp" with its pointer arrays in device memory
 * and any number of problems up to 4096.
 *   M, N, K   HOST arrays of P shapes (the plan needs them); M[p] == 0 skips problem p (its
 *             pointers are not read).
 *   X_dev, Wp_dev, Y_dev   DEVICE arrays of P device pointers (8-byte aligned arrays), read when
 *             the work starts (stream order); per-problem layouts as in wq4_mm.
 *   group_size, dtype, qtype   shared by every problem; float zeros (WQ4_U4_FZP) are not
 *             supported here (WQ4_ERR_UNSUPPORTED).
 *   workspace  wq4_grouped_dev_ptrs_workspace_bytes(...) bytes, 128-byte aligned, zero-filled
 *             before its first use (the K-split counters come first and are left at zero by
 *             every call that completes; the rest, the problem table and one 128-byte activation
 *             tensor map per problem, is rewritten by every call). Calls that share a workspace
 *             must be in stream order.
 * A set-up kernel on `stream` reads the pointers, checks each non-empty problem's pointers (non-null,
 * 16-byte aligned) and blob header, writes its descriptor and its activation tensor map (encoded
 * on the host for its shape, the X address replaced on the device); then the GEMM runs the
 * plan wq4_grouped_mm would make for these shapes, reading the problems from the table. A problem
 * that fails the device-side check is skipped (its Y is not written) and wq4_get_last_error then
 * reports WQ4_ERR_INVALID; the other problems are computed. Host-side argument errors as
 * wq4_grouped_mm, plus WQ4_ERR_ALIGN for a pointer array not 8-byte aligned or a workspace not
 * 128-byte aligned. Results are bit-identical to wq4_grouped_mm's for the same problems. */
int wq4_grouped_dev_ptrs_workspace_bytes(int P, const int* M, const int* N, const int* K, int group_size,
                                         size_t* bytes);
int wq4_grouped_mm_dev_ptrs(int P, const int* M, const int* N, const int* K,
                            const void* const* X_dev, const void* const* Wp_dev, void* const* Y_dev,
                            int group_size, int dtype, int qtype,
                            void* workspace, size_t workspace_bytes, wq4_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * Errors and options.
 * ------------------------------------------------------------------------------------------ */

/* Synchronises the stream, then reports (and clears) what any wq4 kernel on the current device
 * recorded in the device status word: a failed bounds check of the debug build (WQ4_ERR_BOUNDS),
 * else a blob header that did not match its call (WQ4_ERR_INVALID), else a pipeline timeout
 * (WQ4_ERR_TIMEOUT); with nothing recorded, a pending CUDA error (WQ4_ERR_CUDA), else WQ4_OK. A
 * call whose waits ran out stops early and leaves its outputs undefined; the context stays
 * usable, but a workspace it used must be zero-filled again before the next call (its split
 * counters may be left non-zero). The status word is shared by every stream on the device and is
 * read, then cleared: a kernel still running on another stream may record between the two, and
 * that record is lost, so call it while no other wq4 work is in flight to see everything. */
int wq4_get_last_error(wq4_stream_t stream);

/* Bounds checks: 1 when this library is the debug build (libwq4_debug.so, compiled with
 * WQ4_DEBUG=1), 0 for the release build, whose kernels carry no checks. The debug build's
 * kernels check, before each use, every tiled tensor copy's innermost coordinate (a 16-byte
 * multiple, the box inside the tensor), every weight record's range inside its blob, every
 * scheduled tile against its problem's M, N and K groups, the K-split workspace slots and
 * counters, and every output column against N. A failed check never faults or waits: the copy
 * reads the tensor's origin (or the blob's first record) instead, a store or workspace access is
 * skipped, the CTA stops at its next pipeline wait, and wq4_get_last_error reports
 * WQ4_ERR_BOUNDS; the call's outputs are then undefined. */
int wq4_debug_checks(void);

/* The first violation that the last WQ4_ERR_BOUNDS report read back: record[0] = the check site
 * (1 tile, 2 activation tile copy, 3 activation sums, 4 weight record, 5 epilogue C copy,
 * 6 K-split partial slot, 7 K-split counter, 8 output column, 9 decode weight stage, 10 decode
 * activation piece, 11 problem index), record[1..3] = the offending coordinate or index, then two
 * values whose meaning depends on the site (listed with the sites in csrc/wq4_check.h). record
 * must hold 4 ints. Returns 1 and clears the saved violation if there was one, 0 (record zeroed)
 * otherwise, WQ4_ERR_INVALID for a null record. */
int wq4_last_violation(int* record);

/* Process-wide tuning and test options (not thread-safe; set before launching):
 *   WQ4_OPT_TOKEN_TILE      force the token tile (16, 64, 128, 160 or 192); 0 = automatic
 *   WQ4_OPT_GRID            force the number of persistent CTAs; 0 = automatic
 *   WQ4_OPT_SPLIT_ALL       1 = every tile goes through the K-split path (tests)
 *   WQ4_OPT_TIMEOUT_CYCLES  bound of every pipeline wait in SM clock cycles; 0 = default
 *   WQ4_OPT_TRACE           1 = print each dispatch decision to stderr
 *   WQ4_OPT_A_IN_SMEM       1 = stage the dequantised operand in shared memory instead of tensor
 *                           memory (both give the same result; for comparison)
 *   WQ4_OPT_CLUSTER         0 = automatic, -1 = never, 2..8 = force the cluster split: each tile's
 *                           K range split over a cluster of that many CTAs whose partial sums are
 *                           added through distributed shared memory
 *   WQ4_OPT_DECODE          0 = automatic, -1 = never, 1 = whenever the shape allows: wq4_mm with at
 *                           most 32 tokens uses a warp-level-MMA kernel that keeps whole weight rows
 *                           per CTA (no workspace)
 *   WQ4_OPT_PDL             0 = both kernels are launched with programmatic dependent launch (a
 *                           call's set-up overlaps the end of the previous kernel on the stream;
 *                           it touches global memory only after that kernel has completed);
 *                           -1 = plain stream order
 *   WQ4_OPT_TEST_STALL      1 = (tests of the failure path) every kernel makes one wait per CTA
 *                           on a barrier that nothing arrives on; it runs out after the
 *                           WQ4_OPT_TIMEOUT_CYCLES bound, the call stops early and
 *                           wq4_get_last_error reports WQ4_ERR_TIMEOUT. 0 = off
 *   WQ4_OPT_CONST_WEIGHTS   1 = the caller promises that no kernel still pending on the stream
 *                           writes a blob that a later call reads: the decode kernel then checks
 *                           the blob header and copies its first weights, and the tensor-core GEMM
 *                           (problems given on the host) its first ring of weight records, before
 *                           the kernel ahead has completed (activations, C and outputs keep stream
 *                           order). Results are undefined if the promise is broken. 0 = stream
 *                           order for every operand (default)
 *   WQ4_OPT_DECODE_DEPTH    weight ring slots of the decode kernel (one slot = one 16-row block x
 *                           1024 K); 0 = automatic, 2..16 = forced
 *   WQ4_OPT_DECODE_TRIGGER  0 = the decode kernel lets the next kernel on the stream start once its
 *                           activations have landed (default), 1 = at once
 *   WQ4_OPT_VERIFY_DEV_PTRS 1 = (tests) wq4_grouped_mm_dev_ptrs stops after its set-up kernels: it
 *                           synchronises the stream, reads back the activation tensor maps they
 *                           patched and compares each byte for byte with the map the host encoder
 *                           makes for the same address and row count; WQ4_OK when every map
 *                           matches, WQ4_ERR_UNSUPPORTED otherwise (the differing bytes printed
 *                           under WQ4_OPT_TRACE). The GEMM is not launched. 0 = off
 * Returns WQ4_ERR_INVALID for an unknown key or value. */
enum {
    WQ4_OPT_TOKEN_TILE = 1,
    WQ4_OPT_GRID = 2,
    WQ4_OPT_SPLIT_ALL = 3,
    WQ4_OPT_TIMEOUT_CYCLES = 4,
    WQ4_OPT_TRACE = 5,
    WQ4_OPT_A_IN_SMEM = 6,
    WQ4_OPT_CLUSTER = 7,
    WQ4_OPT_DECODE = 8,
    WQ4_OPT_PDL = 9,
    WQ4_OPT_TEST_STALL = 10,
    WQ4_OPT_CONST_WEIGHTS = 11,
    WQ4_OPT_DECODE_DEPTH = 12,
    WQ4_OPT_DECODE_TRIGGER = 13,
    WQ4_OPT_VERIFY_DEV_PTRS = 14
};
int wq4_set_option(int key, long long value);
long long wq4_get_option(int key);

#ifdef __cplusplus
}
#endif
#endif /* WQ4_H_ */

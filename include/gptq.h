/*
 * gptq.h - C ABI of the GB300 (sm_103a) GPTQ weight-only linear layer.
 *
 *     y[M, N] = x[M, K] . W^T,   W[n, k] = (code[k, n] - zero[g, n]) * scale[g, n],  g = g_idx[k]
 *
 * The operation and the checkpoint layout it consumes are the ones of
 *   - tensref.org "GPTQ packed checkpoint" (sections GptqLayer, QuantizeConfig, Reader and
 *     "Reject the file when": rules GPTQ-001 .. GPTQ-006), and
 *   - inference.shantanugoel.com ch. 39 "Quantized checkpoints", section "The format"
 *     (qweight int32 [K*bits/32, N], codes along K, low bits first; qzeros int32
 *     [G, N*bits/32], zeros along N, stored minus one; scales [G, N]; g_idx int32 [K]).
 * The same handle and GEMM serve the neighbouring formats of that chapter: gptq_v2 zero fields
 * and float32 scales (gptq_repack_ex), AutoAWQ GEMM checkpoints (section "AWQ",
 * gptq_repack_awq) and FP8 block-scaled W8A16 layers (section "FP8 checkpoints",
 * gptq_repack_fp8), with an optional bias (gptq_set_bias).
 * Weights stay packed from HBM until they reach registers or shared memory; the dense W is
 * never written to memory (mlinterviewnotes "Formats and kernels: FP8, INT8, INT4, Marlin,
 * Machete", opening section).
 *
 * Conventions for every entry point
 *   - Pointers named "device" must point to memory of the CUDA device that is current when the
 *     call is made; pointers named "host" must be host memory.  No pointer is retained after a
 *     call returns except inside a handle, which owns only memory it allocated itself.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Device
 *     work is enqueued on it and is stream-ordered with the caller's other work.
 *   - Every call returns a gptq_status_t.  Host-side argument checks happen before any device
 *     work is enqueued; a failed check leaves every output untouched.  gptq_last_error_message
 *     gives the text of the calling thread's last failure.  No call aborts, traps or asserts.
 *   - Element types: x, y and scales share one dtype (fp16 or bf16) per handle.  Accumulation is
 *     fp32; y is rounded to the dtype once, round-to-nearest-even.
 */
#ifndef GPTQ_GB300_H
#define GPTQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gptq_handle_s* gptq_handle_t;

typedef enum {
  GPTQ_OK = 0,
  GPTQ_ERR_INVALID_ARG = 1,   /* null pointer, negative size, handle/device mismatch         */
  GPTQ_ERR_UNSUPPORTED = 2,   /* bits not in {2,3,4,8} (GPTQ-001), dtype not fp16/bf16        */
  GPTQ_ERR_SHAPE = 3,         /* tensor shapes break GPTQ-002 / GPTQ-003 / GPTQ-004 (length)  */
  GPTQ_ERR_INVALID_GIDX = 4,  /* a g_idx value selects no scale/zero row (GPTQ-004)           */
  GPTQ_ERR_ALIGNMENT = 5,     /* a pointer is not aligned as documented below                */
  GPTQ_ERR_WORKSPACE = 6,     /* the call needs more workspace than gptq_reserve set up       */
  GPTQ_ERR_CUDA = 7,          /* a CUDA runtime call or kernel launch failed                  */
  GPTQ_ERR_DEVICE = 8,        /* the current device is not a compute capability 10.3 GPU     */
  GPTQ_ERR_TIMEOUT = 9        /* a bounded device-side wait gave up (the context stays usable)*/
} gptq_status_t;

typedef enum { GPTQ_FP16 = 0, GPTQ_BF16 = 1 } gptq_dtype_t;

/* Size limits of every entry point that builds a handle (UNSUPPORTED beyond them). */
#define GPTQ_MAX_K      131072   /* in_features  */
#define GPTQ_MAX_N      262144   /* out_features */
#define GPTQ_MAX_GROUPS 65536    /* G            */

/* Which kernel family gptq_gemm_path runs.  AUTO is what gptq_gemm does. */
typedef enum { GPTQ_PATH_AUTO = 0, GPTQ_PATH_SMALL_M = 1, GPTQ_PATH_LARGE_M = 2 } gptq_path_t;

/*
 * Shape rules of "Reject the file when" applied to declared tensor shapes, before any data is
 * touched.  Host only; safe without a GPU.
 *   bits                 GPTQ-001: must be 2, 3, 4 or 8                     (else UNSUPPORTED)
 *   qweight_rows/cols    GPTQ-002: qweight is [in_features/32*bits, out_features] and
 *                        in_features % 32 == 0; in_features = qweight_rows*32/bits  (else SHAPE)
 *   qzeros_rows/cols     GPTQ-003: qzeros_cols == out_features/32*bits; out_features must also be
 *                        a multiple of 32 so that the floor in that rule is exact   (else SHAPE)
 *                        qzeros_rows must equal G = ceil(in_features/group_size), or 1 when
 *                        group_size == -1 (a single group spans all of K)           (else SHAPE)
 *   scales_rows/cols     must be [G, out_features]                                  (else SHAPE)
 *   g_idx_len            GPTQ-004: must equal in_features, or be 0 without g_idx (else SHAPE)
 *   group_size           -1 or >= 1                                          (else INVALID_ARG)
 * On GPTQ_OK, *in_features and *out_features (if non-NULL) receive K and N.
 */
gptq_status_t gptq_check_shapes(int bits, int64_t qweight_rows, int64_t qweight_cols,
                                int64_t qzeros_rows, int64_t qzeros_cols,
                                int64_t scales_rows, int64_t scales_cols, int64_t g_idx_len,
                                int group_size, int* in_features, int* out_features);

/*
 * Build a runtime handle from one checkpoint layer (the "to_runtime" step of ch. 39, section
 * "The format": input columns are sorted by g_idx once at load time so groups become
 * contiguous, and activations are permuted to match at run time).
 *
 *   qweight  device, int32 [K*bits/32, N] row-major, codes along K, low bits first; for bits 3
 *            the 10 / split / 10 word layout (32 codes in 3 consecutive words).  4-byte aligned.
 *   qzeros   device, int32 [G, N*bits/32] row-major, zeros along N, each stored minus one
 *            (GPTQ-006: the zero used is stored + 1, with no wrap).  4-byte aligned.
 *   scales   device, dtype [G, N] row-major.  2-byte aligned.
 *   g_idx    device, int32 [K], or NULL for the sequential k / group_size.  4-byte aligned.
 *            Any values in [0, G) are accepted; each group's run in sorted order is padded to a
 *            multiple of 32 rows internally, so uneven groups cost bandwidth but stay exact.
 *   K, N     in_features and out_features: K % 32 == 0, N % 32 == 0, 32 <= K <= 131072 and
 *            32 <= N <= 262144 (GPTQ_MAX_K, GPTQ_MAX_N; UNSUPPORTED above them).
 *   bits     2, 3, 4 or 8.   group_size: -1 (one group) or >= 1; G = ceil(K/group_size).
 *   dtype    dtype of scales, and of x and y in every later gptq_gemm on this handle.
 *   stream   the copy/repack kernels run on it; the call synchronizes it once, at the end, to
 *            read back the g_idx check.  The checkpoint buffers may be freed or changed as soon
 *            as the call returns; the handle holds its own copy in its runtime layout.
 *   out      receives the handle (set to NULL on failure).
 * The handle allocates its runtime layout (about K*N*bits/8 bytes plus 6*G*N) and a workspace
 * for gptq_gemm calls with M <= 32; gptq_reserve enlarges the workspace.  The handle is
 * immutable: after any change to the weights, build a new one.
 * Errors: INVALID_ARG, UNSUPPORTED, SHAPE, ALIGNMENT, DEVICE, INVALID_GIDX, CUDA.
 */
gptq_status_t gptq_repack(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                          const int32_t* g_idx, int K, int N, int bits, int group_size,
                          gptq_dtype_t dtype, void* stream, gptq_handle_t* out);

/*
 * Make gptq_gemm calls with M <= max_M possible without any allocation inside gptq_gemm.
 * This is the caller-owned scratch contract of GPTQModel "Kernel Backends Reference", section
 * "Marlin and caller-owned scratch" (the scratch API and its property table): the workspace is
 * sized by a query-free reserve made before any graph capture, is owned by one stream at a time,
 * and a call never falls back to allocating when it is too small -- it fails (WORKSPACE) instead.
 * The page's scratch also holds reduction partials and a zeroed counter array; here the K splits
 * of both kernels keep their partials in the shared memory of a thread-block cluster, so the only
 * workspace is the permuted copy of x.  Only a handle whose g_idx order is not the identity
 * (act-order, or groups whose sizes are not multiples of 32) needs it above M = 32: max_M *
 * K_sorted activation elements.  Allocates (cudaMalloc) outside any stream capture; never shrinks;
 * the handle's device must be current.  Errors: INVALID_ARG, CUDA.
 */
gptq_status_t gptq_reserve(gptq_handle_t h, int max_M);

/*
 * Build a runtime handle from one FP8 block-scaled layer (inference.shantanugoel.com ch. 39,
 * section "FP8 checkpoints": float8_e4m3fn weights with one float32 factor per 128 x 128 block,
 * weight_scale_inv, which multiplies the stored values), for the W8A16 product:
 *   W[n, k] = e4m3(weight[n, k]) * scale_inv[n / 128][k / 128],   y = x . W^T.
 *   weight     device, float8_e4m3fn bytes [N, K] row-major (row n = output n).  Any alignment.
 *              NaN codes (0x7F, 0xFF) are not checked and give NaN outputs.
 *   scale_inv  device, float32 [ceil(N/128), ceil(K/128)] row-major.  4-byte aligned.
 *   K, N       K % 32 == 0, N % 32 == 0 (as gptq_repack).   dtype: x and y.
 * The weights are used exactly (every e4m3 number is an fp16 and a bf16 number); the products
 * accumulate in fp32 per 128-wide block of K and are multiplied by the block's factor in fp32.
 * The handle serves gptq_gemm, gptq_gemm_path, gptq_set_bias and the rest; gptq_get_info reports
 * fp8 = 1, bits = 8, group_size = 128; gptq_copy_runtime gives zeros for s_r and z_r, which an
 * FP8 handle does not keep.
 * Errors: INVALID_ARG, UNSUPPORTED (dtype), SHAPE, ALIGNMENT, DEVICE, CUDA.
 */
gptq_status_t gptq_repack_fp8(const void* weight, const float* scale_inv, int K, int N, gptq_dtype_t dtype,
                              void* stream, gptq_handle_t* out);

/* Flags of gptq_repack_ex. */
#define GPTQ_REPACK_ZEROS_V2    1u  /* qzeros fields hold the zero itself (the corrected gptq_v2
                                       layout named in ch. 39, "The format"), not zero - 1      */
#define GPTQ_REPACK_SCALES_FP32 2u  /* scales are float32 [G, N] (tensref.org GptqLayer allows the
                                       layer weight dtype; its Example stores F32): they are
                                       rounded once to `dtype`, to nearest even, at repack       */

/*
 * gptq_repack with format options.  flags = 0 is exactly gptq_repack.
 *   GPTQ_REPACK_ZEROS_V2     W[n, k] = (code - field) * scale; gptq_get_info reports
 *                            zero_offset = 0.  Fields 0 .. 2^bits - 1 are all valid zeros.
 *   GPTQ_REPACK_SCALES_FP32  `scales` is device float32 [G, N], 4-byte aligned; the kernels use
 *                            the rounded value, so y differs from a float32-scale product by at
 *                            most the scale rounding (2^-11 relative for fp16, 2^-9 for bf16,
 *                            per group).
 * Other arguments and errors as gptq_repack (INVALID_ARG also for unknown flag bits).
 */
gptq_status_t gptq_repack_ex(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                             const int32_t* g_idx, int K, int N, int bits, int group_size,
                             gptq_dtype_t dtype, unsigned flags, void* stream, gptq_handle_t* out);

/*
 * Attach the layer's bias (tensref.org GptqLayer: optional, [out_features], same dtype as the
 * scales): every later gptq_gemm / gptq_gemm_path on this handle computes y = x . W^T + bias,
 * the bias added in fp32 before the single rounding of y.
 *   bias       device, [N] of the handle's dtype (bias_fp32 = 0) or float32 (bias_fp32 = 1),
 *              2- or 4-byte aligned; copied (as float32) on `stream`, so it may be freed once
 *              that stream has passed this call.  NULL detaches the bias.
 * The first non-NULL call allocates N_padded float32 on the device; later calls reuse it.  Calls
 * captured in a CUDA graph before the first attach keep running without a bias.  Must not run
 * while a gptq_gemm on the handle is in flight on another stream.
 * Errors: INVALID_ARG, ALIGNMENT, CUDA.
 */
gptq_status_t gptq_set_bias(gptq_handle_t h, const void* bias, int bias_fp32, void* stream);

/*
 * Build a runtime handle from one AutoAWQ GEMM layer (inference.shantanugoel.com ch. 39
 * "Quantized checkpoints", section "AWQ": the pack_awq / unpack_awq / from_checkpoint
 * description).  The layer is 4-bit and has no g_idx; W[n, k] = (code[k, n] - zero[g, n]) *
 * scale[g, n] with g = k / group_size and the zero read as stored (no +1).
 *   qweight  device, int32 [K, N/8] row-major: eight 4-bit codes per word along the OUTPUT
 *            dimension, nibble j (bits 4j..4j+3) of word w holding output 8w + order[j],
 *            order = 0 2 4 6 1 3 5 7 (output 1 in bits 16-19).  4-byte aligned.
 *   qzeros   device, int32 [G, N/8] row-major, packed the same way; the field is the zero.
 *   scales   device, dtype [G, N] row-major (the format ships fp16; bf16 is accepted).  2-byte
 *            aligned.
 *   K, N, group_size, dtype, stream, out: as for gptq_repack (K % 32 == 0 and N % 32 == 0;
 *            G = ceil(K/group_size), or 1 for group_size == -1).
 * The handle is the same kind as gptq_repack's (sequential groups, so its sorted order is the
 * identity when group_size is a multiple of 32) and serves every other call; gptq_get_info
 * reports zero_offset = 0 for it.
 * Errors: INVALID_ARG, UNSUPPORTED (dtype), SHAPE, ALIGNMENT, DEVICE, CUDA.
 */
gptq_status_t gptq_repack_awq(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                              int K, int N, int group_size, gptq_dtype_t dtype, void* stream,
                              gptq_handle_t* out);

/*
 * y = x . W^T for the handle's layer, enqueued on `stream` (the spec GEMM of the weight-only
 * path: weights stream packed from HBM and are dequantised in registers, mlinterviewnotes "Formats
 * and kernels: FP8, INT8, INT4, Marlin, Machete", opening section and "Where the batch-size
 * crossover is"; the kernel family is chosen by M, as that page's M-bucketed dispatch describes).
 *   x   device, dtype [M, K] row-major (row stride K elements), 16-byte aligned.
 *   y   device, dtype [M, N] row-major (row stride N elements), 16-byte aligned; x and y must
 *       not overlap.
 *   M   >= 0.  M == 0 returns GPTQ_OK and launches nothing: an empty batch is a normal
 *       steady-state input (a data-parallel rank with no tokens still runs its layers), as the
 *       same page's discussion of SGLang's M-bucketing after the Machete section points out.
 * Never allocates and never synchronizes.  One handle may be used by one stream at a time
 * (calls on two streams must not overlap on the device: they share the handle's workspace,
 * GPTQModel "Kernel Backends Reference", scratch ownership: one device, host thread and stream).
 * After gptq_reserve(h, M) has returned, a call with that M may be captured in a CUDA graph.
 * Timeouts: if an earlier call on this handle gave up a bounded device-side wait (its output was
 * invalid), the kernel has recorded it in host-visible memory and this call returns
 * GPTQ_ERR_TIMEOUT without launching anything, until gptq_device_status clears the record.  The
 * record is read without synchronizing, so it shows the timeouts of kernels that have finished.
 * Errors: INVALID_ARG, ALIGNMENT, WORKSPACE (M above the reserved size on a path that needs
 * workspace), TIMEOUT, CUDA.
 */
gptq_status_t gptq_gemm(gptq_handle_t h, const void* x, void* y, int M, void* stream);

/* As gptq_gemm, with the kernel family forced (AUTO = gptq_gemm's choice).  Both families give
 * results within the same tolerance; this exists so each can be checked at any M. */
gptq_status_t gptq_gemm_path(gptq_handle_t h, const void* x, void* y, int M, gptq_path_t path,
                             void* stream);

/* Number of kernels one gptq_gemm_path call at this M launches (0 for M == 0), or -1 on a bad
 * argument.  Host only. */
int gptq_gemm_launches(gptq_handle_t h, int M, gptq_path_t path);

/* Number of K ranges a gptq_gemm_path call at this M is split into (1 = none): the large-M kernel
 * splits grids that would leave SMs idle or a last wave mostly empty, the ranges of an output tile
 * in one thread-block cluster; the small-M kernel splits layers with fewer 32-column tiles than SMs at M <= 8 when
 * each CTA's work shrinks enough, and layers whose x over all of K does not fit in shared memory at
 * M = 9 .. 16, with the K panels of a tile (or of a run of tiles) in one thread-block cluster
 * (partials exchanged in shared memory, no workspace).  -1 on a bad argument.  Host only. */
int gptq_gemm_k_splits(gptq_handle_t h, int M, gptq_path_t path);

/* Free the handle and everything it owns.  Waits for the device to finish using it
 * (cudaDeviceSynchronize on the handle's device).  NULL is accepted.  A handle is tied to the
 * buffers it was built from only through its own copy, so rebuilding after any change to the
 * weights means destroy + repack (GPTQModel "Kernel Backends Reference": do not reuse an initialised
 * native handle after replacing its buffers; invalidate handles on mutation, checklist item 5). */
gptq_status_t gptq_destroy(gptq_handle_t h);

/* Sizes of a handle's runtime layout. */
typedef struct {
  int K, N, bits, group_size, G;
  int K_sorted;     /* rows of the sorted, padded K order: a multiple of 128, >= K            */
  int N_padded;     /* N rounded up to a multiple of 256                                      */
  int identity;     /* 1 when the sorted order is k itself (no permutation, no padding)       */
  gptq_dtype_t dtype;
  int reserved_M;   /* largest M gptq_gemm accepts on every path without further reserve      */
  int zero_offset;  /* zero = stored zero field + zero_offset: 1 (GPTQ v1), 0 (gptq_v2, AWQ)     */
  int has_bias;     /* 1 while a bias is attached (gptq_set_bias)                              */
  int fp8;          /* 1 for a handle built by gptq_repack_fp8                                 */
  size_t weight_bytes;     /* runtime codes: K_sorted/128 * bits * N_padded * 16              */
  size_t device_bytes;     /* everything the handle holds on the device                      */
} gptq_info_t;

gptq_status_t gptq_get_info(gptq_handle_t h, gptq_info_t* info);

/*
 * Copy the runtime layout to host memory (synchronous), for checking the repack bit by bit.
 *   wr    host, info.weight_bytes bytes        perm  host, int32 [K_sorted]
 *   cgid  host, int32 [K_sorted/32]            s_r   host, dtype bits [G, N_padded]
 *   z_r   host, uint8 [G, N_padded]: the checkpoint's zero field (GPTQ: zero - 1; AWQ: the zero)
 * Any pointer may be NULL to skip that buffer.  Errors: INVALID_ARG, CUDA.
 */
gptq_status_t gptq_copy_runtime(gptq_handle_t h, void* wr, int32_t* perm, int32_t* cgid,
                                void* s_r, uint8_t* z_r);

/* GPTQ_ERR_TIMEOUT if a kernel launched with this handle gave up a bounded device-side wait (an
 * mbarrier wait that exceeded its time limit; the kernel then skipped its remaining work and the
 * outputs of that call are invalid) since the previous call of this function, else GPTQ_OK.  Clears
 * the record.  The record lives in mapped (host-visible) memory that the kernels write; this call
 * reads it without synchronizing anything, so synchronize the stream of the calls in question
 * first to include them.  Errors: INVALID_ARG. */
gptq_status_t gptq_device_status(gptq_handle_t h);

/*
 * Repack into caller-owned device buffers without allocating anything (no cudaMalloc, no
 * cudaFree, no allocating library call).  The pages have no counterpart of this call: it exists
 * for callers that cannot allocate device memory themselves at load time -- a server that carves
 * every weight out of one arena reserved up front, or a host framework that owns the device
 * allocator and forbids other allocations -- and that still want the runtime layout.
 *   qweight, qzeros, scales, g_idx, K, N, bits, group_size, dtype: as for gptq_repack.
 *   wr          device, wr_capacity bytes, 16-byte aligned: receives the packed codes.
 *   perm, cgid  device, int32 [kr_capacity] and [kr_capacity/32], 16-byte aligned.
 *   s_r, z_r    device, scale bits [G, N_padded] and stored zeros [G, N_padded], N_padded =
 *               roundup(N, 256).
 *   k_sorted    host, receives K_sorted (set before the capacity check, so a caller can retry).
 * The outputs are exactly what gptq_copy_runtime reports for a handle built from the same
 * checkpoint.  kr_capacity = roundup(K + 31*G, 128) and wr_capacity = kr_capacity/128*bits*
 * N_padded*16 always suffice.  Its scratch is a fixed array of 3*4096+8 int32 in device memory
 * that every GPU holds once the library is loaded, so a layer may have at most 4096 groups
 * (GPTQ_ERR_UNSUPPORTED above that).  Every call looks up that array's device address on the
 * current device (cudaGetSymbolAddress, which allocates nothing).  Every call on a device shares
 * the array, and the array stays in use until the call's work on `stream` has completed: the call
 * synchronizes `stream` once, to read the g_idx histogram, but the sort and pack kernels it
 * enqueues after that still read the array.  So a later call on another stream must first wait
 * for this call's stream (a stream synchronize or an event); calls that overlap on the GPU race.
 * Limits on K and N as gptq_repack (GPTQ_MAX_K, GPTQ_MAX_N).
 * Errors: INVALID_ARG, UNSUPPORTED, SHAPE, ALIGNMENT, DEVICE, INVALID_GIDX, WORKSPACE (output
 * buffers too small for the sorted K), CUDA.
 */
gptq_status_t gptq_repack_noalloc(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                                  const int32_t* g_idx, int K, int N, int bits, int group_size,
                                  gptq_dtype_t dtype, void* wr, size_t wr_capacity, int32_t* perm,
                                  int32_t* cgid, int kr_capacity, void* s_r, uint8_t* z_r,
                                  int* k_sorted, void* stream);

/* The launch plan gptq_gemm_path would use at this M (host only, no device work), for checking
 * which kernel variant a test or a benchmark actually exercises. */
typedef struct {
  int path;            /* GPTQ_PATH_SMALL_M or GPTQ_PATH_LARGE_M                               */
  int launches;        /* kernels per call (an activation gather or permute counts as one)     */
  int grid;            /* CTAs of the GEMM kernel (K split: clusters of k_splits CTAs)          */
  int threads;         /* threads per CTA                                                       */
  int smem_bytes;      /* dynamic shared memory per CTA                                         */
  int consumer_warps;  /* small-M: warps that dequantise and multiply; large-M: 4 dequantisers  */
  int m_tiles;         /* small-M: 8-row m-tiles (1, 2, 4); large-M: x rows per tile (64..256)  */
  int act_order_in_kernel; /* small-M: 1 when x is permuted in shared memory (no pre-pass)      */
  int k_splits;        /* CTAs that share one output tile's K (1 = no split)                    */
  int k_panels;        /* small-M: K panels x is staged in (1 = all of K at once)               */
  int stages;          /* weight ring depth                                                     */
  int row_passes;      /* small-M: 2 when the call runs as two launches over row slices of x and
                          y (the first 16 rows, then the rest), 1 otherwise; the fields above then
                          describe the first pass, and `launches` counts both                  */
} gptq_plan_t;

/* Errors: INVALID_ARG (bad handle, M < 1, unknown path, M above the small-M kernel's 32 rows),
 * UNSUPPORTED (no plan fits this layer). */
gptq_status_t gptq_gemm_plan(gptq_handle_t h, int M, gptq_path_t path, gptq_plan_t* plan);

/* Test hook for the error path of the bounded waits; not for production use.  While `on` is 1,
 * the small-M kernel's copy producer issues no copy at all, so nothing is ever in flight and every
 * consumer wait runs into its limit, which is `wait_limit_ns` (e.g. 1000000 for 1 ms) instead of the
 * normal 2 s.  The call's output is then invalid and the handle records GPTQ_ERR_TIMEOUT (see
 * gptq_gemm and gptq_device_status).  on = 0 restores normal operation and the 2 s limit.
 * Errors: INVALID_ARG. */
gptq_status_t gptq_set_test_stall(gptq_handle_t h, int on, uint64_t wait_limit_ns);

/* Static text for a status: the name of the code.  Together with gptq_last_error_message, which
 * names the violated rule, this is the "fail rather than silently fall back" error contract of
 * GPTQModel "Kernel Backends Reference" (scratch property table: invalid buffers fail) and of
 * tensref.org "GPTQ packed checkpoint", section "Reject the file when". */
const char* gptq_status_string(gptq_status_t s);

/* Text of the calling thread's most recent failure ("" if none).  Valid until the next call. */
const char* gptq_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* GPTQ_GB300_H */

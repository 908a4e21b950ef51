// Host side of the C ABI: argument checks (the reject rules of tensref.org "GPTQ packed
// checkpoint", section "Reject the file when"), handle lifecycle, and the per-call M dispatch.
#include "internal.cuh"

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <new>
#include <string>

namespace gptq {

namespace {
thread_local std::string g_last_error;
constexpr int kMaxK = GPTQ_MAX_K;        // in_features limit (index arithmetic and repack cost)
constexpr int kMaxN = GPTQ_MAX_N;        // out_features limit
constexpr int kMaxGroups = GPTQ_MAX_GROUPS;
// Largest M routed to the small-M (mma.sync weight-streaming) kernel by gptq_gemm.  Up to M = 16
// the layer is HBM-bound on GB300 (ridge M* = P * 4.125 / (16 * BW) ~ 72 for 4-bit group 128) and
// the swap-AB mma.sync kernel keeps every SM streaming weights.  With four m-tiles it also beats
// the tcgen05 kernel up to M = 28 (measured: 22 vs 28 us at M = 24 on a 4096 x 14336 layer, 84 vs
// 110 us on 8192 x 28672); above that its x panels shrink to four blocks and it falls behind, unless
// the call runs as two passes of at most 16 rows (auto_path).
constexpr int kSmallMMax = 28;
}  // namespace

gptq_status_t fail(gptq_status_t s, const std::string& msg) {
  g_last_error = std::string(gptq_status_string(s)) + ": " + msg;
  return s;
}

gptq_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(GPTQ_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

gptq_status_t build_runtime(Handle& h, const void* qweight, const int32_t* qzeros, const void* scales,
                            const int32_t* g_idx, int fmt, bool scales_fp32, cudaStream_t st);

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static void free_handle(Handle* h) {
  if (!h) return;
  cudaFree(h->wr);
  cudaFree(h->perm);
  cudaFree(h->cgid);
  cudaFree(h->s_r);
  cudaFree(h->z_r);
  cudaFree(h->zst);
  cudaFree(h->xp);
  cudaFree(h->bias);
  cudaFree(h->scale_inv);
  if (h->err_host) cudaFreeHost(const_cast<int32_t*>(h->err_host));
  delete h;
}

static gptq_status_t check_device(int* dev_out, int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0, sms = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(GPTQ_ERR_DEVICE, "this library is built for sm_103a (compute capability 10.3); device " +
                                     std::to_string(dev) + " is " + std::to_string(major) + "." + std::to_string(minor));
  *dev_out = dev;
  *sms_out = sms;
  return GPTQ_OK;
}

// Rows of the first of the small-M kernel's passes at M (M when the call is one pass).  At M = 17 .. 32
// the kernel stages x per K panel when x of M rows over all of K does not fit its shared memory.
// With four or more panels, on a layer with at least one 32-column tile per SM, two launches over
// row slices -- the first 16 rows (two m-tiles: x staged once, or split across a cluster), then
// the rest -- take less time: 70B gate layer M = 24 104.1 -> 74.7 us, M = 28 111.7 -> 90.7 us;
// decode layer M = 28 28.6 -> 22.6 us.  With fewer tiles than SMs the second launch's fixed cost
// wins (K = N = 4096, 8-bit, M = 28: 14.8 vs 18.7 us), and at three panels neither does (decode
// layer M = 17: 20.3 vs 25.6 us).  Every row's result is its own sum either way, within the same
// tolerance; the summation order differs between the plans.
static int small_first_rows(const Handle& h, int M) {
  if (M <= 16 || M > small_m_max()) return M;
  const int64_t key = ((int64_t)0x7f << 32) | (uint32_t)M;   // cached beside the launch plans
  {
    std::lock_guard<std::mutex> lock(h.plan_mu);
    auto it = h.plans.find(key);
    if (it != h.plans.end()) return (int)it->second[0];
  }
  gptq_plan_t p{};
  const int m1 = (small_m_plan_info(h, M, &p) && p.k_panels >= 4 && (h.N + 31) / 32 >= h.sm_count) ? 16 : M;
  std::lock_guard<std::mutex> lock(h.plan_mu);
  h.plans[key] = std::vector<int64_t>{m1};
  return m1;
}

// GPTQ_PATH_AUTO: the small-M kernel up to kSmallMMax rows, and up to its 32 rows where it runs as
// two passes (70B gate layer M = 32: 91 us in two passes against 95.7 us on the large-M kernel;
// decode layer: ~22.8 against 29.2 us); the large-M kernel above.
static gptq_path_t auto_path(const Handle& h, int M) {
  if (!large_m_available() || M <= kSmallMMax) return GPTQ_PATH_SMALL_M;
  return (M <= small_m_max() && small_first_rows(h, M) < M) ? GPTQ_PATH_SMALL_M : GPTQ_PATH_LARGE_M;
}

static int small_launches_total(const Handle& h, int M) {
  const int m1 = small_first_rows(h, M);
  return small_m_launches(h, m1) + (m1 < M ? small_m_launches(h, M - m1) : 0);
}

static gptq_status_t gemm_impl(gptq_handle_t hh, const void* x, void* y, int M, gptq_path_t path, void* stream) {
  if (!hh) return fail(GPTQ_ERR_INVALID_ARG, "handle is NULL");
  const Handle& h = *reinterpret_cast<const Handle*>(hh);
  if (M < 0) return fail(GPTQ_ERR_INVALID_ARG, "M must be >= 0");
  if (path != GPTQ_PATH_AUTO && path != GPTQ_PATH_SMALL_M && path != GPTQ_PATH_LARGE_M)
    return fail(GPTQ_ERR_INVALID_ARG, "unknown path");
  if (M == 0) return GPTQ_OK;   // an empty batch is a normal input: nothing to launch
  if (!x || !y) return fail(GPTQ_ERR_INVALID_ARG, "x and y must be device pointers");
  if (!aligned(x, 16) || !aligned(y, 16)) return fail(GPTQ_ERR_ALIGNMENT, "x and y must be 16-byte aligned");
  const size_t es = 2;
  const char* xb = static_cast<const char*>(x);
  const char* yb = static_cast<const char*>(y);
  if (xb < yb + (size_t)M * h.N * es && yb < xb + (size_t)M * h.K * es)
    return fail(GPTQ_ERR_INVALID_ARG, "x and y overlap");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h.device)
    return fail(GPTQ_ERR_INVALID_ARG, "handle belongs to device " + std::to_string(h.device) +
                                          " but device " + std::to_string(dev) + " is current");
  if (*h.err_host != DEV_ERR_NONE)
    return fail(GPTQ_ERR_TIMEOUT, "an earlier call on this handle gave up a bounded device-side wait and its output "
                                  "was invalid; gptq_device_status clears the record");
  if (path == GPTQ_PATH_AUTO) path = auto_path(h, M);
  if (path == GPTQ_PATH_LARGE_M && !large_m_available())
    return fail(GPTQ_ERR_UNSUPPORTED, "the large-M kernel is not part of this build");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (path == GPTQ_PATH_LARGE_M) {
    if (!h.identity && M > h.reserved_M)
      return fail(GPTQ_ERR_WORKSPACE, "M = " + std::to_string(M) + " needs gptq_reserve(h, M): the handle's g_idx "
                                      "order is not the identity and only M <= " + std::to_string(h.reserved_M) + " is reserved");
    e = launch_gemm_large(h, x, y, M, st);
  } else {
    if (M > small_m_max())
      return fail(GPTQ_ERR_INVALID_ARG, "M = " + std::to_string(M) + " is above the small-M kernel's " +
                                            std::to_string(small_m_max()) + " rows");
    const int m1 = small_first_rows(h, M);
    // a pass that gathers x into the workspace needs its rows reserved
    for (const int r : {m1, M - m1})
      if (r > 0 && !h.identity && r > h.reserved_M && small_m_launches(h, r) == 2)
        return fail(GPTQ_ERR_WORKSPACE, "M = " + std::to_string(M) + " needs gptq_reserve(h, " + std::to_string(r) +
                                        "): the handle's g_idx order is not the identity and only M <= " +
                                        std::to_string(h.reserved_M) + " is reserved");
    e = launch_gemm_small(h, x, y, m1, st);
    if (e == cudaSuccess && m1 < M)
      e = launch_gemm_small(h, xb + (size_t)m1 * h.K * es, static_cast<char*>(y) + (size_t)m1 * h.N * es, M - m1, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "gptq_gemm launch");
  return GPTQ_OK;
}

}  // namespace gptq

using namespace gptq;

extern "C" {

const char* gptq_status_string(gptq_status_t s) {
  switch (s) {
    case GPTQ_OK: return "GPTQ_OK";
    case GPTQ_ERR_INVALID_ARG: return "GPTQ_ERR_INVALID_ARG";
    case GPTQ_ERR_UNSUPPORTED: return "GPTQ_ERR_UNSUPPORTED";
    case GPTQ_ERR_SHAPE: return "GPTQ_ERR_SHAPE";
    case GPTQ_ERR_INVALID_GIDX: return "GPTQ_ERR_INVALID_GIDX";
    case GPTQ_ERR_ALIGNMENT: return "GPTQ_ERR_ALIGNMENT";
    case GPTQ_ERR_WORKSPACE: return "GPTQ_ERR_WORKSPACE";
    case GPTQ_ERR_CUDA: return "GPTQ_ERR_CUDA";
    case GPTQ_ERR_DEVICE: return "GPTQ_ERR_DEVICE";
    case GPTQ_ERR_TIMEOUT: return "GPTQ_ERR_TIMEOUT";
  }
  return "GPTQ_ERR_UNKNOWN";
}

const char* gptq_last_error_message(void) { return g_last_error.c_str(); }

gptq_status_t gptq_check_shapes(int bits, int64_t qweight_rows, int64_t qweight_cols, int64_t qzeros_rows,
                                int64_t qzeros_cols, int64_t scales_rows, int64_t scales_cols, int64_t g_idx_len,
                                int group_size, int* in_features, int* out_features) {
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8)
    return fail(GPTQ_ERR_UNSUPPORTED, "GPTQ-001: bits must be 2, 3, 4 or 8, got " + std::to_string(bits));
  if (group_size != -1 && group_size < 1)
    return fail(GPTQ_ERR_INVALID_ARG, "group_size must be -1 or >= 1, got " + std::to_string(group_size));
  if (qweight_rows <= 0 || qweight_cols <= 0 || (qweight_rows * 32) % bits != 0)
    return fail(GPTQ_ERR_SHAPE, "GPTQ-002: qweight rows must be in_features // 32 * bits");
  const int64_t K = qweight_rows * 32 / bits, N = qweight_cols;
  if (K % 32 != 0) return fail(GPTQ_ERR_SHAPE, "GPTQ-002: in_features must be divisible by 32");
  if (N % 32 != 0) return fail(GPTQ_ERR_SHAPE, "GPTQ-003: out_features must be a multiple of 32 (qzeros width N/32*bits)");
  if (qzeros_cols != N / 32 * bits)
    return fail(GPTQ_ERR_SHAPE, "GPTQ-003: qzeros.shape[1] must be out_features // 32 * bits = " + std::to_string(N / 32 * bits));
  const int64_t G = group_size == -1 ? 1 : (K + group_size - 1) / group_size;
  if (qzeros_rows != G)
    return fail(GPTQ_ERR_SHAPE, "qzeros.shape[0] must be ceil(in_features / group_size) = " + std::to_string(G));
  if (scales_rows != G || scales_cols != N)
    return fail(GPTQ_ERR_SHAPE, "scales must be [ceil(in_features / group_size), out_features]");
  if (g_idx_len != 0 && g_idx_len != K)
    return fail(GPTQ_ERR_SHAPE, "GPTQ-004: g_idx length must equal in_features = " + std::to_string(K));
  if (K > kMaxK || N > kMaxN || G > kMaxGroups)
    return fail(GPTQ_ERR_UNSUPPORTED, "layer too large for this build (K <= " + std::to_string(kMaxK) + ", N <= " + std::to_string(kMaxN) + ", groups <= " + std::to_string(kMaxGroups) + ")");
  if (in_features) *in_features = (int)K;
  if (out_features) *out_features = (int)N;
  return GPTQ_OK;
}

}  // extern "C"

namespace gptq {
// Argument checks shared by both checkpoint formats, then the handle and its runtime layout.
static gptq_status_t reserve_impl(Handle& h, int max_M);

static gptq_status_t repack_impl(const void* qweight, const int32_t* qzeros, const void* scales,
                                 const int32_t* g_idx, int K, int N, int bits, int group_size, gptq_dtype_t dtype,
                                 int fmt, unsigned flags, void* stream, gptq_handle_t* out) {
  if (!out) return fail(GPTQ_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  const bool fp8 = fmt == kFmtFp8;
  if (!qweight || (!qzeros && !fp8) || !scales)
    return fail(GPTQ_ERR_INVALID_ARG, fp8 ? "weight and scale_inv are required" : "qweight, qzeros and scales are required");
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8)
    return fail(GPTQ_ERR_UNSUPPORTED, "GPTQ-001: bits must be 2, 3, 4 or 8, got " + std::to_string(bits));
  if (dtype != GPTQ_FP16 && dtype != GPTQ_BF16) return fail(GPTQ_ERR_UNSUPPORTED, "dtype must be GPTQ_FP16 or GPTQ_BF16");
  if (group_size != -1 && group_size < 1)
    return fail(GPTQ_ERR_INVALID_ARG, "group_size must be -1 or >= 1, got " + std::to_string(group_size));
  if (K < 32 || K % 32 != 0) return fail(GPTQ_ERR_SHAPE, "GPTQ-002: in_features must be a positive multiple of 32");
  if (N < 32 || N % 32 != 0) return fail(GPTQ_ERR_SHAPE, "GPTQ-003: out_features must be a positive multiple of 32");
  const int G = group_size == -1 ? 1 : (K + group_size - 1) / group_size;
  if (K > kMaxK || N > kMaxN || G > kMaxGroups)
    return fail(GPTQ_ERR_UNSUPPORTED, "layer too large for this build (K <= " + std::to_string(kMaxK) + ", N <= " + std::to_string(kMaxN) + ", groups <= " + std::to_string(kMaxGroups) + ")");
  if (flags & ~(unsigned)(GPTQ_REPACK_ZEROS_V2 | GPTQ_REPACK_SCALES_FP32))
    return fail(GPTQ_ERR_INVALID_ARG, "unknown repack flag bits");
  const bool sf32 = (flags & GPTQ_REPACK_SCALES_FP32) != 0;
  if (fp8 ? !aligned(scales, 4)
          : (!aligned(qweight, 4) || !aligned(qzeros, 4) || !aligned(scales, sf32 ? 4 : 2) || (g_idx && !aligned(g_idx, 4))))
    return fail(GPTQ_ERR_ALIGNMENT, fp8 ? "scale_inv needs 4-byte alignment"
                                        : "qweight, qzeros, g_idx need 4-byte and scales 2-byte (float32: 4-byte) alignment");
  int dev = 0, sms = 0;
  gptq_status_t s = check_device(&dev, &sms);
  if (s != GPTQ_OK) return s;
  Handle* h = new (std::nothrow) Handle();
  if (!h) return fail(GPTQ_ERR_INVALID_ARG, "out of host memory");
  h->device = dev;
  h->sm_count = sms;
  h->K = K; h->N = N; h->bits = bits; h->group_size = group_size; h->G = G;
  h->Np = (N + 255) / 256 * 256;
  h->dtype = dtype;
  h->zoff = (fmt != kFmtGptq || (flags & GPTQ_REPACK_ZEROS_V2)) ? 0 : 1;
  h->fp8 = fp8 ? 1 : 0;
  h->kb = (K + 127) / 128;
  void* eh = nullptr;
  cudaError_t ce = cudaHostAlloc(&eh, sizeof(int32_t), cudaHostAllocMapped);
  if (ce != cudaSuccess) { free_handle(h); return cuda_fail(ce, "cudaHostAlloc(error word)"); }
  h->err_host = static_cast<volatile int32_t*>(eh);
  *h->err_host = DEV_ERR_NONE;
  ce = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->err), eh, 0);
  if (ce != cudaSuccess) { free_handle(h); return cuda_fail(ce, "cudaHostGetDevicePointer(error word)"); }
  s = build_runtime(*h, qweight, qzeros, scales, g_idx, fmt, sf32, static_cast<cudaStream_t>(stream));
  if (s != GPTQ_OK) { free_handle(h); return s; }
  h->reserved_M = 0;
  s = reserve_impl(*h, 32);     // the permuted-x workspace for M <= 32
  if (s != GPTQ_OK) { free_handle(h); return s; }
  *out = reinterpret_cast<gptq_handle_t>(h);
  return GPTQ_OK;
}
}  // namespace gptq

extern "C" {

gptq_status_t gptq_repack(const int32_t* qweight, const int32_t* qzeros, const void* scales, const int32_t* g_idx,
                          int K, int N, int bits, int group_size, gptq_dtype_t dtype, void* stream,
                          gptq_handle_t* out) {
  return repack_impl(qweight, qzeros, scales, g_idx, K, N, bits, group_size, dtype, kFmtGptq, 0u, stream, out);
}

gptq_status_t gptq_repack_ex(const int32_t* qweight, const int32_t* qzeros, const void* scales, const int32_t* g_idx,
                             int K, int N, int bits, int group_size, gptq_dtype_t dtype, unsigned flags, void* stream,
                             gptq_handle_t* out) {
  return repack_impl(qweight, qzeros, scales, g_idx, K, N, bits, group_size, dtype, kFmtGptq, flags, stream, out);
}

gptq_status_t gptq_set_bias(gptq_handle_t hh, const void* bias, int bias_fp32, void* stream) {
  if (!hh) return fail(GPTQ_ERR_INVALID_ARG, "handle is NULL");
  Handle& h = *reinterpret_cast<Handle*>(hh);
  if (bias_fp32 != 0 && bias_fp32 != 1) return fail(GPTQ_ERR_INVALID_ARG, "bias_fp32 must be 0 or 1");
  if (!bias) {
    h.has_bias = 0;
    return GPTQ_OK;
  }
  if (!aligned(bias, bias_fp32 ? 4 : 2)) return fail(GPTQ_ERR_ALIGNMENT, "bias needs 2-byte (float32: 4-byte) alignment");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h.device)
    return fail(GPTQ_ERR_INVALID_ARG, "handle belongs to device " + std::to_string(h.device) + " but device " +
                                          std::to_string(dev) + " is current");
  if (!h.bias && (e = cudaMalloc(&h.bias, sizeof(float) * (size_t)h.Np)) != cudaSuccess) {
    h.bias = nullptr;
    return cuda_fail(e, "cudaMalloc(bias)");
  }
  const int kind = bias_fp32 ? 2 : (h.dtype == GPTQ_BF16 ? 1 : 0);
  if ((e = launch_bias_f32(bias, kind, h.N, h.Np, h.bias, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "bias conversion launch");
  h.has_bias = 1;
  return GPTQ_OK;
}

gptq_status_t gptq_repack_awq(const int32_t* qweight, const int32_t* qzeros, const void* scales, int K, int N,
                              int group_size, gptq_dtype_t dtype, void* stream, gptq_handle_t* out) {
  return repack_impl(qweight, qzeros, scales, nullptr, K, N, 4, group_size, dtype, kFmtAwq, 0u, stream, out);
}

gptq_status_t gptq_repack_fp8(const void* weight, const float* scale_inv, int K, int N, gptq_dtype_t dtype,
                              void* stream, gptq_handle_t* out) {
  return repack_impl(weight, nullptr, scale_inv, nullptr, K, N, 8, 128, dtype, kFmtFp8, 0u, stream, out);
}

}  // extern "C"

namespace gptq {
// Workspace for calls with M <= max_M: the permuted-x copy (handles whose sorted order is not the
// identity).  The K splits of both kernels exchange their partials in shared memory across a
// thread-block cluster and need none.
static gptq_status_t reserve_impl(Handle& h, int max_M) {
  if (max_M > h.reserved_M && !h.identity) {
    const size_t bytes = (size_t)max_M * h.Kr * 2;
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(gptq_reserve workspace)");
    cudaFree(h.xp);
    h.xp = p;
    h.xp_bytes = bytes;
  }
  if (max_M > h.reserved_M) h.reserved_M = max_M;
  return GPTQ_OK;
}
}  // namespace gptq

extern "C" {

gptq_status_t gptq_reserve(gptq_handle_t hh, int max_M) {
  if (!hh) return fail(GPTQ_ERR_INVALID_ARG, "handle is NULL");
  if (max_M < 0) return fail(GPTQ_ERR_INVALID_ARG, "max_M must be >= 0");
  Handle& h = *reinterpret_cast<Handle*>(hh);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h.device)
    return fail(GPTQ_ERR_INVALID_ARG, "handle belongs to device " + std::to_string(h.device) + " but device " +
                                          std::to_string(dev) + " is current");
  return reserve_impl(h, max_M);
}

gptq_status_t gptq_gemm(gptq_handle_t h, const void* x, void* y, int M, void* stream) {
  return gemm_impl(h, x, y, M, GPTQ_PATH_AUTO, stream);
}

gptq_status_t gptq_gemm_path(gptq_handle_t h, const void* x, void* y, int M, gptq_path_t path, void* stream) {
  return gemm_impl(h, x, y, M, path, stream);
}

int gptq_gemm_launches(gptq_handle_t hh, int M, gptq_path_t path) {
  if (!hh || M < 0) return -1;
  const Handle& h = *reinterpret_cast<const Handle*>(hh);
  if (M == 0) return 0;
  if (path == GPTQ_PATH_AUTO) path = auto_path(h, M);
  return path == GPTQ_PATH_LARGE_M ? large_m_launches(h, M) : small_launches_total(h, M);
}

int gptq_gemm_k_splits(gptq_handle_t hh, int M, gptq_path_t path) {
  if (!hh || M < 0) return -1;
  if (path != GPTQ_PATH_AUTO && path != GPTQ_PATH_SMALL_M && path != GPTQ_PATH_LARGE_M) return -1;
  const Handle& h = *reinterpret_cast<const Handle*>(hh);
  if (path == GPTQ_PATH_AUTO) path = auto_path(h, M);
  return path == GPTQ_PATH_LARGE_M ? large_split(h, M) : small_m_k_splits(h, small_first_rows(h, M));
}

gptq_status_t gptq_destroy(gptq_handle_t hh) {
  if (!hh) return GPTQ_OK;
  Handle* h = reinterpret_cast<Handle*>(hh);
  const int dev = h->device;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != dev) cudaSetDevice(dev);
  cudaError_t e = cudaDeviceSynchronize();
  free_handle(h);
  if (cur >= 0 && cur != dev) cudaSetDevice(cur);
  if (e != cudaSuccess) return cuda_fail(e, "gptq_destroy: cudaDeviceSynchronize");
  return GPTQ_OK;
}

gptq_status_t gptq_device_status(gptq_handle_t hh) {
  if (!hh) return fail(GPTQ_ERR_INVALID_ARG, "handle is NULL");
  Handle& h = *reinterpret_cast<Handle*>(hh);
  const int32_t word = *h.err_host;
  if (word != DEV_ERR_NONE) *h.err_host = DEV_ERR_NONE;
  if (word == DEV_ERR_TIMEOUT)
    return fail(GPTQ_ERR_TIMEOUT, "a kernel gave up a bounded wait on an mbarrier; that call's output is invalid");
  return GPTQ_OK;
}

gptq_status_t gptq_get_info(gptq_handle_t hh, gptq_info_t* info) {
  if (!hh || !info) return fail(GPTQ_ERR_INVALID_ARG, "handle and info are required");
  const Handle& h = *reinterpret_cast<const Handle*>(hh);
  info->K = h.K; info->N = h.N; info->bits = h.bits; info->group_size = h.group_size; info->G = h.G;
  info->K_sorted = h.Kr; info->N_padded = h.Np; info->identity = h.identity; info->dtype = h.dtype;
  info->reserved_M = h.reserved_M;
  info->zero_offset = h.zoff;
  info->has_bias = h.has_bias;
  info->fp8 = h.fp8;
  info->weight_bytes = h.wr_bytes();
  info->device_bytes = h.wr_bytes() + sizeof(int32_t) * (size_t)h.Kr + sizeof(int32_t) * (size_t)(h.Kr / 32) +
                       (size_t)h.G * h.Np * (h.fp8 ? 3 : 6) + h.xp_bytes + (h.bias ? sizeof(float) * (size_t)h.Np : 0) +
                       (h.scale_inv ? sizeof(float) * (size_t)((h.N + 127) / 128) * h.kb : 0);
  return GPTQ_OK;
}

gptq_status_t gptq_copy_runtime(gptq_handle_t hh, void* wr, int32_t* perm, int32_t* cgid, void* s_r, uint8_t* z_r) {
  if (!hh) return fail(GPTQ_ERR_INVALID_ARG, "handle is NULL");
  const Handle& h = *reinterpret_cast<const Handle*>(hh);
  cudaError_t e = cudaSuccess;
  if (wr && (e = cudaMemcpy(wr, h.wr, h.wr_bytes(), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "copy wr");
  if (perm && (e = cudaMemcpy(perm, h.perm, sizeof(int32_t) * h.Kr, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "copy perm");
  if (cgid && (e = cudaMemcpy(cgid, h.cgid, sizeof(int32_t) * (h.Kr / 32), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "copy cgid");
  // an FP8 handle keeps no per-column scales or zeros: those outputs read as zeros
  if (s_r && !h.s_r) std::memset(s_r, 0, 2 * (size_t)h.G * h.Np);
  if (z_r && !h.z_r) std::memset(z_r, 0, (size_t)h.G * h.Np);
  if (s_r && h.s_r && (e = cudaMemcpy(s_r, h.s_r, 2 * (size_t)h.G * h.Np, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "copy s_r");
  if (z_r && h.z_r && (e = cudaMemcpy(z_r, h.z_r, (size_t)h.G * h.Np, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "copy z_r");
  return GPTQ_OK;
}

}  // extern "C"

extern "C" {

gptq_status_t gptq_gemm_plan(gptq_handle_t hh, int M, gptq_path_t path, gptq_plan_t* plan) {
  if (!hh || !plan) return fail(GPTQ_ERR_INVALID_ARG, "handle and plan are required");
  if (M < 1) return fail(GPTQ_ERR_INVALID_ARG, "M must be >= 1");
  if (path != GPTQ_PATH_AUTO && path != GPTQ_PATH_SMALL_M && path != GPTQ_PATH_LARGE_M)
    return fail(GPTQ_ERR_INVALID_ARG, "unknown path");
  const Handle& h = *reinterpret_cast<const Handle*>(hh);
  if (path == GPTQ_PATH_AUTO) path = auto_path(h, M);
  std::memset(plan, 0, sizeof(*plan));
  plan->path = path;
  if (path == GPTQ_PATH_SMALL_M) {
    if (M > small_m_max())
      return fail(GPTQ_ERR_INVALID_ARG, "M = " + std::to_string(M) + " is above the small-M kernel's " +
                                            std::to_string(small_m_max()) + " rows");
    const int m1 = small_first_rows(h, M);
    if (!small_m_plan_info(h, m1, plan)) return fail(GPTQ_ERR_UNSUPPORTED, "no small-M plan fits this layer");
    plan->launches = small_launches_total(h, M);
    plan->row_passes = m1 < M ? 2 : 1;
  } else if (!large_m_plan_info(h, M, plan)) {
    return fail(GPTQ_ERR_UNSUPPORTED, "no large-M plan fits this layer");
  } else {
    plan->row_passes = 1;
  }
  return GPTQ_OK;
}

gptq_status_t gptq_set_test_stall(gptq_handle_t hh, int on, uint64_t wait_limit_ns) {
  if (!hh) return fail(GPTQ_ERR_INVALID_ARG, "handle is NULL");
  if (on != 0 && on != 1) return fail(GPTQ_ERR_INVALID_ARG, "on must be 0 or 1");
  if (on && (wait_limit_ns < 1000 || wait_limit_ns > 2000000000ull))
    return fail(GPTQ_ERR_INVALID_ARG, "wait_limit_ns must lie in [1 us, 2 s]");
  Handle& h = *reinterpret_cast<Handle*>(hh);
  h.test_stall = on;
  h.wait_ns = on ? wait_limit_ns : 2000000000ull;
  return GPTQ_OK;
}

}  // extern "C"

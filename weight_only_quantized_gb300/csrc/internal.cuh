// Internal declarations shared by the translation units of the GPTQ library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <atomic>
#include <cstdint>
#include <cstddef>
#include <mutex>
#include <string>
#include <unordered_map>
#include <type_traits>
#include <vector>

#include "../../include/gptq.h"

namespace gptq {

// Runtime handle: the checkpoint re-laid for the kernels (see repack.cu for the layout).
struct Handle {
  int device = 0;
  int K = 0, N = 0, bits = 0, group_size = 0, G = 0;
  int Kr = 0;          // rows of the sorted, padded K order (multiple of 128)
  int Np = 0;          // N padded to a multiple of 256
  int identity = 0;    // sorted order == k and Kr == K
  gptq_dtype_t dtype = GPTQ_FP16;
  int sm_count = 0;
  // runtime layout
  uint8_t* wr = nullptr;     // codes: [Kr/128][bits vectors][Np][16 B]
  int32_t* perm = nullptr;   // [Kr], -1 for pad rows
  int32_t* cgid = nullptr;   // [Kr/32] group of each 32-row chunk
  uint16_t* s_r = nullptr;   // [G][Np] scale bits
  uint8_t* z_r = nullptr;    // [G][Np] stored zero field (GPTQ: zero - 1; AWQ: the zero itself)
  int zoff = 1;              // zero = stored field + zoff: 1 for GPTQ v1 fields, 0 for gptq_v2 and AWQ
  float* bias = nullptr;     // [Np] float32 bias added to y (pad columns 0), allocated by gptq_set_bias
  // FP8 block-scaled layers (codes are e4m3 bytes; no zeros; s_r and z_r are not allocated)
  int fp8 = 0;
  float* scale_inv = nullptr;   // [ceil(N/128)][kb] float32, one factor per 128 x 128 block
  int kb = 0;                   // ceil(K/128)
  int has_bias = 0;          // 1: the GEMM kernels add bias
  uint8_t* zst = nullptr;    // [Np/32][G][96]: per 32-column tile and group, 32 stored zeros then
                             // 32 scales, column c at position (c % 8) * 4 + c / 8 (small-M path)
  std::vector<int32_t> cgid_host;   // host copy of cgid (split planning)
  CUtensorMap wr_map;               // wr as uint64 [Kr/128 * bits rows][2 Np]: one box = kSmallBlocksPerBox
                                    // blocks of one 32-column tile (small-M path)
  // Error word in mapped, pinned host memory: the kernels store DEV_ERR_TIMEOUT into it when a
  // bounded wait gives up, and the host reads it without synchronizing (err is the device view of
  // err_host).
  int32_t* err = nullptr;
  volatile int32_t* err_host = nullptr;
  // Limit of every bounded wait of the small-M kernel, and the test hook that makes its producer
  // issue nothing (gptq_set_test_stall).
  uint64_t wait_ns = 2000000000ull;
  int test_stall = 0;
  // workspace
  int reserved_M = 0;
  void* xp = nullptr;        // [reserved_M][Kr] activations in sorted order (large-M path)
  size_t xp_bytes = 0;
  size_t wr_bytes() const { return (size_t)Kr / 128 * bits * Np * 16; }
  // Launch plans by (path, M): computed once, so a call costs one kernel launch on the host.
  mutable std::mutex plan_mu;
  mutable std::unordered_map<int64_t, std::vector<int64_t>> plans;
  // Thread-block clusters of S = 2 .. 8 whole-SM CTAs that the GPU holds at once (index S; 0: not
  // queried yet, -1: none).  The SMs pair up by TPC and group by GPC, so a cluster size that does
  // not divide a GPC's SMs leaves some of them idle.
  mutable std::atomic<int> clusters_fit[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
};

// 128-row blocks fetched by one TMA box of the small-M kernel.
constexpr int kSmallBlocksPerBox = 4;

// Column position inside a 32-column group of the runtime codes: vector v of a block stores the
// 16-byte word of column c (c = n % 32) at position (c + code_col_rot(bits, v)) % 32.  With
// these rotations, the lanes of a quarter warp that read different vectors of the same columns
// land on different shared-memory banks when a block is copied densely.
__host__ __device__ __forceinline__ int code_col_rot(int bits, int v) {
  return bits == 4 ? 2 * v : bits == 8 ? 2 * (v >> 1) : (bits == 2 || v < 2) ? 4 * v : 0;
}
__host__ __device__ __forceinline__ int code_col_pos(int bits, int v, int n) {
  return (n & ~31) | (((n & 31) + code_col_rot(bits, v)) & 31);
}

// FP8 layers: the runtime layout keeps a pair's two e4m3 bytes side by side in one 16-bit half of a
// lane word (the even k in the low byte).  One conversion gives the exact fp16 pair; for bf16 the
// fp16 bits move into bf16 position as the value times 2^-112 (every e4m3 number is a normal fp16,
// 2^-9 .. 448, whose low seven mantissa bits are zero, so the shifted fields are exact and never
// subnormal), the sign is put back, and one exact multiply by 2^112 restores the value.
template <typename T>
__device__ __forceinline__ uint32_t fp8_pair(uint32_t word, int half) {
  uint32_t d;
  if (half == 0) asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.rn.f16x2.e4m3x2 %0, lo; }" : "=r"(d) : "r"(word));
  else asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.rn.f16x2.e4m3x2 %0, hi; }" : "=r"(d) : "r"(word));
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    uint32_t t;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(t) : "r"(d >> 3), "r"(0x0FFF0FFFu), "r"(d & 0x80008000u));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(0x77807780u));   // 2^112 in both halves
  }
  return d;
}

// cuTensorMapEncodeTiled from the driver (nullptr if unavailable).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// Status with message, recorded per thread.
gptq_status_t fail(gptq_status_t s, const std::string& msg);
gptq_status_t cuda_fail(cudaError_t e, const char* what);

// ---- kernels launched from the host code (defined in the .cu files) ----

// Checkpoint formats the repack reads.
enum Format { kFmtGptq = 0, kFmtAwq = 1, kFmtFp8 = 2 };

// bias[n] -> float32 [Np] (kind 0 fp16, 1 bf16, 2 float32; pad columns 0), enqueued on st.
cudaError_t launch_bias_f32(const void* src, int kind, int N, int Np, float* dst, cudaStream_t st);

// Large-M K split: ranges for M given the workspace on hand (1 = none); the workspace bytes a split
// may take at most.
int large_split(const Handle& h, int M);
// Thread-block clusters of S CTAs with a whole SM each that the GPU runs at once (S = 1 .. 8); 0 when
// none fits, or the query failed (no split of that size is then planned).
int whole_sm_clusters(const Handle& h, int S);

// Small-M path: persistent bulk-copy-fed mma.sync (swap-AB) kernel (plus an x gather when not identity).
int small_m_launches(const Handle& h, int M);
int small_m_max();   // largest M the small-M kernel covers (four m-tiles of 8 rows)
int small_m_k_splits(const Handle& h, int M);   // K panels the small-M kernel splits a call into (1 = none)
cudaError_t launch_gemm_small(const Handle& h, const void* x, void* y, int M, cudaStream_t st);
cudaError_t launch_gemm_small_bf16(const Handle& h, const void* x, void* y, int M, cudaStream_t st);   // bf16 layers
bool small_m_plan_info(const Handle& h, int M, gptq_plan_t* out);   // false: no plan fits

// Large-M path: tcgen05 / TMEM / TMA kernel (plus an x-permute pre-pass when not identity).
bool large_m_available();
int large_m_launches(const Handle& h, int M);
cudaError_t launch_gemm_large(const Handle& h, const void* x, void* y, int M, cudaStream_t st);
bool large_m_plan_info(const Handle& h, int M, gptq_plan_t* out);   // false: no plan fits

// ---- device helpers ----
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Device error codes written to Handle::err (0 = none).
enum : int32_t { DEV_ERR_NONE = 0, DEV_ERR_TIMEOUT = 1 };
// Record a timeout in the handle's error word, which lives in mapped host memory: a plain
// system-visible store (every writer stores the same value), then a fence so the host sees it.
__device__ __forceinline__ void report_timeout(int32_t* err) {
  *reinterpret_cast<volatile int32_t*>(err) = DEV_ERR_TIMEOUT;
  __threadfence_system();
}

// ---- mbarrier and bulk-copy helpers (sm_90+ PTX) ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete; give up after limit_ns (returns false).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}
// The same bounded wait as one asm block whose only output is the limit: on a timeout it sets
// limit_ns to 0, so every later wait polls once and falls through.  A thread that issues
// tcgen05.mma uses this form: when a branch or an operand between two MMAs depends on a value
// read from shared memory (a wait result, a flag), the MMA issue rate drops by 2.5-4x on sm_103a
// (measured); a wait whose result feeds only the next wait's limit keeps the full rate.
__device__ __forceinline__ void mbar_wait_poison(uint32_t bar, uint32_t parity, uint64_t& limit_ns) {
  asm volatile("{\n\t.reg .pred p;\n\t.reg .u64 t0, t1;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "@p bra WP_END;\n\t"
               "mov.u64 t0, %%globaltimer;\n\t"
               "WP_LOOP:\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "@p bra WP_END;\n\t"
               "mov.u64 t1, %%globaltimer;\n\t"
               "sub.u64 t1, t1, t0;\n\t"
               "setp.lt.u64 p, t1, %0;\n\t"
               "@p bra WP_LOOP;\n\t"
               "mov.u64 %0, 0;\n\t"
               "WP_END:\n\t}"
               : "+l"(limit_ns) : "r"(bar), "r"(parity) : "memory");
}
// Bulk copy global -> this CTA's shared memory, completing tx bytes on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

}  // namespace gptq

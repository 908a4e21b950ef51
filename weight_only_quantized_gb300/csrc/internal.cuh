// Internal declarations shared by the translation units of the GPTQ library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstddef>
#include <mutex>
#include <string>
#include <unordered_map>
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
  uint8_t* z_r = nullptr;    // [G][Np] stored zero (zero - 1)
  std::vector<int32_t> cgid_host;   // host copy of cgid (split planning)
  int32_t* err = nullptr;    // device error word: kernels set it when a bounded wait gives up
  // workspace
  int reserved_M = 0;
  void* xp = nullptr;        // [reserved_M][Kr] activations in sorted order (large-M path)
  size_t xp_bytes = 0;
  size_t wr_bytes() const { return (size_t)Kr / 128 * bits * Np * 16; }
  // Launch plans by (path, M): computed once, so a call costs one kernel launch on the host.
  mutable std::mutex plan_mu;
  mutable std::unordered_map<int64_t, std::vector<int64_t>> plans;
};

// Status with message, recorded per thread.
gptq_status_t fail(gptq_status_t s, const std::string& msg);
gptq_status_t cuda_fail(cudaError_t e, const char* what);

// ---- kernels launched from the host code (defined in the .cu files) ----

// Small-M path: mma.sync (swap-AB) kernel with split-K reduced inside a thread-block cluster.
int small_m_launches(const Handle& h, int M);
cudaError_t launch_gemm_small(const Handle& h, const void* x, void* y, int M, cudaStream_t st);

// Large-M path: tcgen05 / TMEM / TMA kernel (plus an x-permute pre-pass when not identity).
bool large_m_available();
int large_m_launches(const Handle& h, int M);
cudaError_t launch_gemm_large(const Handle& h, const void* x, void* y, int M, cudaStream_t st);

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

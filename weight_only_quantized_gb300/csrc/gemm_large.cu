// Large-M GEMM (prefill): tcgen05.mma with per-group partial sums in tensor memory.
//
// mlinterviewnotes "Formats and kernels: FP8, INT8, INT4, Marlin, Machete": above the ridge
// M* (section "Where the batch-size crossover is") the layer is tensor-core bound; the weight
// format is not on the tensor-core menu, so the kernel converts in the mainloop, and a scale that
// varies along K must take part inside the k reduction (section on the LOP3 dequant and the scale).
//
// Exact operands, scale in fp32.  Rounding every dequantised weight (code - zero) * scale to bf16
// before the MMA costs up to 2^-9 relative per weight, and bf16 rounding of y alone already costs
// up to 2^-8 |y|; together they exceed a 4e-3 * max|y| budget.  So the MMA multiplies x by the
// exact integers (code - zero), accumulates each group's partial sum in fp32 in tensor memory,
// and the group scale multiplies that partial sum in fp32 -- the same arithmetic as the small-M
// kernel, inside the k reduction.
//
// Design on sm_103a, one CTA per tile of 128 output features x 256 rows of x (swap-AB: D[n][m]):
//  * warp 0: producer.  cp.async.bulk copies of the packed 128-row blocks of the tile's 128
//    columns, and TMA (cp.async.bulk.tensor.2d, SWIZZLE_128B) loads of 256 x 64 x tiles, each into
//    a ring tracked by mbarriers.
//  * warps 2..3: dequantisers.  Thread d owns weight rows n0 + d and n0 + d + 64: one LOP3 per code pair makes
//    magic + code, one packed subtract of (magic + zero) leaves the exact integer code - zero, and
//    the row is written in the UMMA K-major SWIZZLE_128B layout (16-byte chunk j of row r at chunk
//    j ^ (r % 8) of its 128-byte row), then a generic-to-async proxy fence and an arrive.
//  * warp 1: allocates all 512 TMEM columns (two 256-column partial-sum buffers); one thread issues
//    tcgen05.mma.cta_group::1.kind::f16 (M = 128 weight rows, N = 256 x rows, K = 16), two per
//    32-row chunk, restarting the accumulator at each group and committing the buffer when the
//    group ends.
//  * warps 4..19: sixteen scaler warps, four per TMEM lane quarter, 64 columns each.  Per group:
//    tcgen05.ld the partial sums, S += scale[g][n] * P in registers, release the buffer.  At the end
//    they round S to the output type and store y.
// Act-order handles first gather x into the handle's workspace in sorted k order (one extra launch).
// Every wait is bounded; a timeout sets the handle's error word and the CTA drains and exits.
#include "internal.cuh"

#include <cuda.h>
#include <type_traits>

namespace gptq {
namespace {

constexpr int BN = 128, BMX = 256, HK = 64;   // weight rows (MMA M), x rows (MMA N), k per stage
constexpr int kDqWarps = 2, kScWarps = 16;
constexpr int kWarpsL = 2 + kDqWarps + kScWarps;
constexpr int kThreadsL = kWarpsL * 32;         // 640: up to 96 registers a thread, so the scalers' sums stay in registers
constexpr int PS = 2, XS = 3, WS = 3;
constexpr int X_BYTES = BMX * HK * 2;           // 32 KB
constexpr int W_BYTES = BN * HK * 2;            // 16 KB
constexpr int kTmemCols = 512;                  // two partial-sum buffers of 256 columns
template <int BITS> constexpr int PK_BYTES = BN * 16 * BITS;  // one 128-row block of 128 columns

template <typename T> struct MagicL;
template <> struct MagicL<__half> { static constexpr uint32_t bits = 0x6400u; };
template <> struct MagicL<__nv_bfloat16> { static constexpr uint32_t bits = 0x4300u; };
template <typename T, int BITS> constexpr bool kF32Path = BITS == 8 && std::is_same<T, __nv_bfloat16>::value;

// Shared-memory carve-up from a 1024-byte-aligned base.
template <int BITS> struct LargeSmem {
  static constexpr int x = 0;
  static constexpr int w = x + XS * X_BYTES;
  static constexpr int pk = w + WS * W_BYTES;
  static constexpr int bars = pk + PS * PK_BYTES<BITS>;
  static constexpr int nbars = 2 * XS + 2 * WS + 2 * PS + 4;
  static constexpr int tmem_slot = bars + nbars * 8;
  static constexpr int cg = tmem_slot + 16;       // int32 chunk groups of the whole K follow
};

struct LargeArgs {
  const uint8_t* wr; const int32_t* cgid; const uint16_t* s_r; const uint8_t* z_r;
  void* y; int32_t* err;
  int M, N, Np, Kr, G;
};

__device__ __forceinline__ uint32_t and_or_l(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
template <typename T> __device__ __forceinline__ uint32_t sub2l(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t sub2l<__half>(uint32_t a, uint32_t b) {
  uint32_t d; asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b)); return d;
}
template <> __device__ __forceinline__ uint32_t sub2l<__nv_bfloat16>(uint32_t a, uint32_t b) {
  uint32_t d; asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b)); return d;
}
template <typename T> __device__ __forceinline__ uint16_t to_bits(float v);
template <> __device__ __forceinline__ uint16_t to_bits<__half>(float v) { return __half_as_ushort(__float2half_rn(v)); }
template <> __device__ __forceinline__ uint16_t to_bits<__nv_bfloat16>(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
template <typename T> __device__ __forceinline__ float scale_f(uint16_t b);
template <> __device__ __forceinline__ float scale_f<__half>(uint16_t b) { return __half2float(__ushort_as_half(b)); }
template <> __device__ __forceinline__ float scale_f<__nv_bfloat16>(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Words of one lane (t = 0..3) of one column from a packed stage laid out [vector][column][16 B].
template <int BITS> struct Words { uint32_t w[BITS]; };
template <int BITS>
__device__ __forceinline__ void stage_words(Words<BITS>& o, const uint8_t* stage, int d, int t) {
  if constexpr (BITS == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(stage + ((size_t)t * BN + d) * 16);
    o.w[0] = v.x; o.w[1] = v.y; o.w[2] = v.z; o.w[3] = v.w;
  } else if constexpr (BITS == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(stage + ((size_t)(t >> 1) * BN + d) * 16 + 8 * (t & 1));
    o.w[0] = v.x; o.w[1] = v.y;
  } else if constexpr (BITS == 8) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(stage + ((size_t)(2 * t) * BN + d) * 16);
    const uint4 v1 = *reinterpret_cast<const uint4*>(stage + ((size_t)(2 * t + 1) * BN + d) * 16);
    o.w[0] = v0.x; o.w[1] = v0.y; o.w[2] = v0.z; o.w[3] = v0.w;
    o.w[4] = v1.x; o.w[5] = v1.y; o.w[6] = v1.z; o.w[7] = v1.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(stage + ((size_t)(t >> 1) * BN + d) * 16 + 8 * (t & 1));
    o.w[0] = v.x; o.w[1] = v.y;
    o.w[2] = *reinterpret_cast<const uint32_t*>(stage + ((size_t)2 * BN + d) * 16 + 4 * t);
  }
}

// Exact code - zero of pair p of a lane, both halves (zq: prepared zero).
template <typename T, int BITS>
__device__ __forceinline__ uint32_t code_minus_zero(const Words<BITS>& lw, int p, uint32_t zq) {
  if constexpr (kF32Path<T, BITS>) {
    const uint32_t codes = (lw.w[p / 2] >> (8 * (p % 2))) & 0x00FF00FFu;
    const float zf = __uint_as_float(zq);
    const float lo = __uint_as_float(0x4B000000u | (codes & 0xFFFFu)) - zf;   // exact integers, |v| <= 256
    const float hi = __uint_as_float(0x4B000000u | (codes >> 16)) - zf;
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
  } else {
    constexpr uint32_t M2 = MagicL<T>::bits * 0x00010001u;
    uint32_t v;
    if constexpr (BITS == 3) {
      const uint32_t lo = and_or_l(lw.w[p / 8] >> (2 * (p % 8)), 0x00030003u, M2);
      const uint32_t hi = p <= 2 ? (lw.w[2] << (2 - p)) : (lw.w[2] >> (p - 2));
      v = and_or_l(hi, 0x00040004u, lo);
    } else {
      constexpr int F = 16 / BITS;
      constexpr uint32_t mask = ((1u << BITS) - 1u) * 0x00010001u;
      v = and_or_l(lw.w[p / F] >> (BITS * (p % F)), mask, M2);
    }
    return sub2l<T>(v, zq);
  }
}

template <typename T, int BITS>
__device__ __forceinline__ uint32_t prep_zero_l(uint32_t stored) {
  const uint32_t z = stored + 1u;
  if constexpr (kF32Path<T, BITS>) return __float_as_uint(8388608.0f + (float)z);
  else return (MagicL<T>::bits + z) * 0x00010001u;
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
               :: "r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar) : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}

// 8 consecutive fp32 columns of this warp's TMEM lane quarter.
__device__ __forceinline__ void tmem_ld8(uint32_t addr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(addr));
}

template <typename T, int BITS>
__global__ void __launch_bounds__(kThreadsL, 1) k_gemm_large(const LargeArgs a, const __grid_constant__ CUtensorMap tmap_x) {
  using S = LargeSmem<BITS>;
  constexpr int PKB = PK_BYTES<BITS>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m0 = blockIdx.x * BMX, n0 = blockIdx.y * BN;
  const int nblocks = a.Kr / 128;
  const int nhalf = 2 * nblocks, nchunks = a.Kr / 32;

  const uint32_t xs_s = base_s + S::x, ws_s = base_s + S::w;
  uint8_t* pk = base + S::pk;
  const uint32_t bar = base_s + S::bars;
  auto x_full = [&](int i) { return bar + 8 * i; };
  auto x_empty = [&](int i) { return bar + 8 * (XS + i); };
  auto w_full = [&](int i) { return bar + 8 * (2 * XS + i); };
  auto w_empty = [&](int i) { return bar + 8 * (2 * XS + WS + i); };
  auto pk_full = [&](int i) { return bar + 8 * (2 * XS + 2 * WS + i); };
  auto pk_empty = [&](int i) { return bar + 8 * (2 * XS + 2 * WS + PS + i); };
  auto p_full = [&](int b) { return bar + 8 * (2 * XS + 2 * WS + 2 * PS + b); };
  auto p_empty = [&](int b) { return bar + 8 * (2 * XS + 2 * WS + 2 * PS + 2 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + S::tmem_slot);
  int32_t* cg = reinterpret_cast<int32_t*>(base + S::cg);
  // a 32-row chunk c ends its group when the next chunk has another group (or c is the last)
  auto group_ends = [&](int c) { return c + 1 == nchunks || cg[c + 1] != cg[c]; };

  if (tid == 0) {
    for (int i = 0; i < XS; ++i) { mbar_init(x_full(i), 1); mbar_init(x_empty(i), 1); }
    for (int i = 0; i < WS; ++i) { mbar_init(w_full(i), kDqWarps); mbar_init(w_empty(i), 1); }
    for (int i = 0; i < PS; ++i) { mbar_init(pk_full(i), 1); mbar_init(pk_empty(i), kDqWarps); }
    for (int b = 0; b < 2; ++b) { mbar_init(p_full(b), 1); mbar_init(p_empty(b), kScWarps); }
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int i = tid; i < nchunks; i += kThreadsL) cg[i] = __ldg(&a.cgid[i]);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  bool ok = true;
  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int pk_issued = 0, x_issued = 0;
      for (int blk = 0; blk < nblocks && ok; ++blk) {
        const int ps = blk % PS;
        if (blk >= PS && !mbar_wait(pk_empty(ps), ((blk / PS) - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(pk_full(ps), PKB);
        const uint8_t* src = a.wr + ((size_t)blk * BITS * a.Np + n0) * 16;
#pragma unroll
        for (int v = 0; v < BITS; ++v)
          bulk_g2s(smem_u32(pk + ps * PKB + v * BN * 16), src + (size_t)v * a.Np * 16, BN * 16, pk_full(ps));
        ++pk_issued;
        if (blk == 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // x may come from the previous grid
        for (int h = 0; h < 2; ++h) {
          const int i = 2 * blk + h, xs = i % XS;
          if (i >= XS && !mbar_wait(x_empty(xs), ((i / XS) - 1) & 1)) { ok = false; break; }
          mbar_arrive_expect_tx(x_full(xs), X_BYTES);
          tma_load_2d(xs_s + xs * X_BYTES, &tmap_x, i * HK, m0, x_full(xs));
          ++x_issued;
        }
      }
      // every issued copy must land before the CTA may exit
      for (int b = pk_issued > PS ? pk_issued - PS : 0; b < pk_issued; ++b)
        if (!mbar_wait(pk_full(b % PS), (b / PS) & 1)) ok = false;
      for (int i = x_issued > XS ? x_issued - XS : 0; i < x_issued; ++i)
        if (!mbar_wait(x_full(i % XS), (i / XS) & 1)) ok = false;
      if (!ok) atomicExch(a.err, DEV_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
      constexpr uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(BMX >> 3) << 17) | ((uint32_t)(BN >> 4) << 24);
      int gi = 0;                 // groups started so far; buffer gi % 2, its use gi / 2
      bool fresh = true;          // next MMA starts a group
      for (int i = 0; i < nhalf && ok; ++i) {
        const int xs = i % XS, ws = i % WS;
        if (!mbar_wait(x_full(xs), (i / XS) & 1) || !mbar_wait(w_full(ws), (i / WS) & 1)) { ok = false; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint64_t ad = smem_desc_sw128(ws_s + ws * W_BYTES);     // A: weights, 128 rows
        const uint64_t bd = smem_desc_sw128(xs_s + xs * X_BYTES);     // B: x, 256 rows
        for (int cc = 0; cc < 2 && ok; ++cc) {
          const int c = 2 * i + cc;
          const int b = gi & 1;
          if (fresh && gi >= 2 && !mbar_wait(p_empty(b), ((gi >> 1) - 1) & 1)) { ok = false; break; }
          if (fresh) asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t d = tmem + (uint32_t)(b * 256);
          umma_f16(d, ad + 2 * (2 * cc), bd + 2 * (2 * cc), idesc, fresh ? 0u : 1u);
          umma_f16(d, ad + 2 * (2 * cc + 1), bd + 2 * (2 * cc + 1), idesc, 1u);
          fresh = false;
          if (group_ends(c)) {
            umma_commit(p_full(b));
            ++gi;
            fresh = true;
          }
        }
        umma_commit(x_empty(xs));
        umma_commit(w_empty(ws));
      }
      if (!ok) atomicExch(a.err, DEV_ERR_TIMEOUT);
    }
  } else if (warp < 2 + kDqWarps) {
    // ---------------- dequantisers: thread d owns weight rows n0 + d + 64 r, r = 0, 1 ----------------
    const int d0 = tid - 64;
    uint32_t zq[2][4];
    auto load_zeros = [&](int blk, uint32_t (&z)[2][4]) {
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          z[r][c] = prep_zero_l<T, BITS>(__ldg(&a.z_r[(size_t)cg[blk * 4 + c] * a.Np + n0 + d0 + 64 * r]));
    };
    if (nblocks > 0) load_zeros(0, zq);
    for (int blk = 0; blk < nblocks && ok; ++blk) {
      const int ps = blk % PS;
      if (!mbar_wait(pk_full(ps), (blk / PS) & 1)) { ok = false; break; }
      const uint8_t* stage = pk + ps * PKB;
      uint32_t zn[2][4];
      if (blk + 1 < nblocks) load_zeros(blk + 1, zn);     // next block's zeros, ahead of use
      for (int h = 0; h < 2; ++h) {
        const int i = 2 * blk + h, ws = i % WS;
        if (i >= WS && !mbar_wait(w_empty(ws), ((i / WS) - 1) & 1)) { ok = false; break; }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int d = d0 + 64 * r;
          Words<BITS> lw[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) stage_words<BITS>(lw[t], stage, d, t);
          uint8_t* row = base + S::w + ws * W_BYTES + d * 128;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * h + cc;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint4 o;
              o.x = code_minus_zero<T, BITS>(lw[t], 4 * c + 0, zq[r][c]);
              o.y = code_minus_zero<T, BITS>(lw[t], 4 * c + 1, zq[r][c]);
              o.z = code_minus_zero<T, BITS>(lw[t], 4 * c + 2, zq[r][c]);
              o.w = code_minus_zero<T, BITS>(lw[t], 4 * c + 3, zq[r][c]);
              const int j = 4 * cc + t;                       // 16-byte chunk (8 k) inside the 64-k row
              *reinterpret_cast<uint4*>(row + ((j ^ (d & 7)) << 4)) = o;
            }
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(w_full(ws));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(pk_empty(ps));           // both halves of this block are written
      if (blk + 1 < nblocks) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) zq[r][c] = zn[r][c];
      }
    }
    if (!ok) atomicExch(a.err, DEV_ERR_TIMEOUT);
  } else {
    // ---------------- scalers: S += scale * P per group, then y ----------------
    const int sw = warp - (2 + kDqWarps);
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int cs = sw >> 2;                   // 64-column slice of the 256 x rows
    const int nrow = 32 * q + lane;           // weight row of this thread inside the tile
    const int n = n0 + nrow;
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
    int gi = 0;
    float sc_next = 0.f;
    int c_next = 0;
    // the scale of the group that starts at chunk c
    auto scale_at = [&](int c) { return scale_f<T>(__ldg(&a.s_r[(size_t)cg[c] * a.Np + n])); };
    if (nchunks > 0) sc_next = scale_at(0);
    for (int c = 0; c < nchunks && ok; ++c) {
      if (!group_ends(c)) continue;
      const float sc = sc_next;
      c_next = c + 1;
      if (c_next < nchunks) sc_next = scale_at(c_next);     // next group's scale, ahead of use
      const int b = gi & 1;
      if (!mbar_wait(p_full(b), (gi >> 1) & 1)) { ok = false; break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * 256 + 64 * cs);
#pragma unroll
      for (int part = 0; part < 8; ++part) {
        uint32_t r[8];
        tmem_ld8(taddr + 8 * part, r);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[8 * part + j] = fmaf(sc, __uint_as_float(r[j]), acc[8 * part + j]);
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(p_empty(b));
      ++gi;
    }
    if (!ok) atomicExch(a.err, DEV_ERR_TIMEOUT);
    // y[m][n] for the 64 x rows of this slice: lanes are consecutive n, so each store is 64 bytes
    uint16_t* y = static_cast<uint16_t*>(a.y);
    if (n < a.N) {
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int m = m0 + 64 * cs + j;
        if (m < a.M) y[(size_t)m * a.N + n] = to_bits<T>(acc[j]);
      }
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// x_p[m][j] = x[m][perm[j]] (0 for pad rows): activations in sorted k order for the TMA loads.
__global__ void k_permute_x(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, uint16_t* __restrict__ xp,
                            int M, int K, int Kr) {
  for (int m = blockIdx.y; m < M; m += gridDim.y)
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < Kr; j += gridDim.x * blockDim.x) {
      const int k = __ldg(&perm[j]);
      xp[(size_t)m * Kr + j] = k >= 0 ? x[(size_t)m * K + k] : (uint16_t)0;
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

template <int BITS> size_t large_smem_bytes(int Kr) { return 1024 + LargeSmem<BITS>::cg + (size_t)(Kr / 32) * 4; }

template <typename T, int BITS>
cudaError_t launch_tb(const Handle& h, const CUtensorMap& map, void* y, int M, cudaStream_t st) {
  const size_t smem = large_smem_bytes<BITS>(h.Kr);
  auto kern = k_gemm_large<T, BITS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  LargeArgs args{h.wr, h.cgid, h.s_r, h.z_r, y, h.err, M, h.N, h.Np, h.Kr, h.G};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + BMX - 1) / BMX, h.Np / BN, 1);     // consecutive CTAs share a weight tile
  cfg.blockDim = dim3(kThreadsL);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args, map);
}

template <typename T>
cudaError_t launch_t(const Handle& h, const CUtensorMap& map, void* y, int M, cudaStream_t st) {
  switch (h.bits) {
    case 2: return launch_tb<T, 2>(h, map, y, M, st);
    case 3: return launch_tb<T, 3>(h, map, y, M, st);
    case 4: return launch_tb<T, 4>(h, map, y, M, st);
    default: return launch_tb<T, 8>(h, map, y, M, st);
  }
}

}  // namespace

bool large_m_available() { return true; }

int large_m_launches(const Handle& h, int M) { return M > 0 ? (h.identity ? 1 : 2) : 0; }

cudaError_t launch_gemm_large(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  if (large_smem_bytes<8>(h.Kr) > 227 * 1024) return cudaErrorInvalidConfiguration;
  const void* src = x;
  int kdim = h.K;
  if (!h.identity) {
    dim3 grid((h.Kr + 255) / 256 < 64 ? (h.Kr + 255) / 256 : 64, M < 65535 ? M : 65535);
    k_permute_x<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(x), h.perm, static_cast<uint16_t*>(h.xp), M, h.K, h.Kr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    src = h.xp;
    kdim = h.Kr;
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)kdim, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)kdim * 2};
  const cuuint32_t box[2] = {HK, BMX};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = h.dtype == GPTQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (enc(&map, dt, 2, const_cast<void*>(src), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (h.dtype == GPTQ_BF16) return launch_t<__nv_bfloat16>(h, map, y, M, st);
  return launch_t<__half>(h, map, y, M, st);
}

}  // namespace gptq

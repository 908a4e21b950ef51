// Small-M GEMM (decode, M <= 16): weight streaming at HBM speed.
//
// mlinterviewnotes "Formats and kernels: FP8, INT8, INT4, Marlin, Machete": at small M "only the
// weight bytes matter" (opening section); the quantised weight only pays if it stays packed
// until the registers that feed the tensor core; a group scale cannot be hoisted out of the k
// reduction (section on the LOP3 dequant and the scale); for tiny M the lever is many CTAs
// streaming weights at once, and the skinny operand goes in the MMA's N slot (swap-AB, section
// "Where the batch-size crossover is" and the M-bucketed dispatch discussion).
//
// Design on sm_103a (each point measured on GB300):
//  * Programmatic dependent launch.  A CTA first lets the next grid on the stream launch, starts
//    its weight stream (weights belong to the handle and never depend on earlier work), and only
//    then waits (griddepcontrol.wait) for the previous grid before it reads x or writes y.  Back to
//    back, a 29 MB read kernel drops from 8.2 us to 4.2 us this way.
//  * A CTA owns NCW x 32 output features and, normally, all of K: its eight warps are NCW column
//    warps times 8/NCW k-groups, each k-group a contiguous slice of the 128-row blocks.  Partial
//    sums of the k-groups meet once in shared memory at the end.  Only when x for the whole K
//    would not fit in shared memory is K split across the CTAs of a thread-block cluster, reduced
//    through distributed shared memory in fixed rank order.  No workspace, no atomics.
//  * Every lane streams its own lane words with cp.async into a private slot of its warp's
//    shared-memory ring (STAGES blocks deep): no registers held by loads in flight, no barriers.
//  * mma.sync.m16n8k16 with swap-AB: A = weights (16 output features x 16 k), B = x^T (16 k x 8
//    batch rows), fp32 accumulators.
//  * Conversion: one LOP3 puts two codes into the mantissas of a magic fp16 (1024) or bf16 (128)
//    pair (exactly magic + code), one packed subtract of (magic + zero) leaves the exact integer
//    code - zero; the LOP3 (and the shift for fields above the low one) runs on the integer pipe,
//    the subtract on the fp16 pipe.  8-bit codes with bf16 go through the 2^23 fp32 magic because
//    bf16 holds 128 + q exactly only for q < 128.  The group scale multiplies each group's fp32
//    partial sum; the runtime layout keeps every MMA step inside one 32-row chunk, hence inside one
//    group.
#include "internal.cuh"

#include <algorithm>
#include <type_traits>

namespace gptq {
namespace {

constexpr int kMaxSplit = 8;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kXsBudget = 48 * 1024;       // shared memory for staged x before K is split over a cluster

template <typename T> struct Magic;
template <> struct Magic<__half> { static constexpr uint32_t bits = 0x6400u; };
template <> struct Magic<__nv_bfloat16> { static constexpr uint32_t bits = 0x4300u; };

template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);
template <> __device__ __forceinline__ void mma16816<__half>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <> __device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T> __device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b);
template <> __device__ __forceinline__ uint32_t sub2<__half>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <> __device__ __forceinline__ uint32_t sub2<__nv_bfloat16>(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) { return pack_f16x2(lo, hi); }
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) { return pack_bf16x2(lo, hi); }

template <typename T> __device__ __forceinline__ float to_float(uint32_t b);
template <> __device__ __forceinline__ float to_float<__half>(uint32_t b) { return __half2float(__ushort_as_half((uint16_t)b)); }
template <> __device__ __forceinline__ float to_float<__nv_bfloat16>(uint32_t b) { return __uint_as_float(b << 16); }

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 8-bit codes with bf16 activations go through fp32; every other case uses the fp16/bf16 magic.
template <typename T, int BITS> constexpr bool kViaF32 = BITS == 8 && std::is_same<T, __nv_bfloat16>::value;

// Zero point (stored + 1) in the form code_minus_zero subtracts.
template <typename T, int BITS>
__device__ __forceinline__ uint32_t prep_zero(uint32_t stored) {
  const uint32_t z = stored + 1u;
  if constexpr (kViaF32<T, BITS>) return __float_as_uint(8388608.0f + (float)z);   // 2^23 + z, exact
  else return (Magic<T>::bits + z) * 0x00010001u;                                   // magic + z, both halves
}

// Lane words of one (block, column) for this lane: BITS words (bits 3: 2 words of the 2-bit plane
// then 1 word of the 1-bit plane).
template <int BITS> struct LaneWords { uint32_t w[BITS]; };

// (code - zero) of pair p of this lane as a T2 register (low half = even k of the pair), exact.
template <typename T, int BITS>
__device__ __forceinline__ uint32_t operand(const LaneWords<BITS>& lw, int p, uint32_t zq) {
  constexpr uint32_t M2 = Magic<T>::bits * 0x00010001u;
  if constexpr (BITS == 3) {
    const uint32_t lo = and_or(lw.w[p / 8] >> (2 * (p % 8)), 0x00030003u, M2);
    const uint32_t hi = p <= 2 ? (lw.w[2] << (2 - p)) : (lw.w[2] >> (p - 2));
    return sub2<T>(and_or(hi, 0x00040004u, lo), zq);
  } else if constexpr (kViaF32<T, BITS>) {
    const uint32_t codes = (lw.w[p / 2] >> (8 * (p % 2))) & 0x00FF00FFu;
    const float zf = __uint_as_float(zq);
    const float lo = __uint_as_float(0x4B000000u | (codes & 0xFFFFu)) - zf;
    const float hi = __uint_as_float(0x4B000000u | (codes >> 16)) - zf;
    return pack_bf16x2(lo, hi);
  } else {
    constexpr int F = 16 / BITS;
    constexpr uint32_t mask = ((1u << BITS) - 1u) * 0x00010001u;
    return sub2<T>(and_or(lw.w[p / F] >> (BITS * (p % F)), mask, M2), zq);
  }
}

// ---- per-lane cp.async ring ----
// A slot holds one block for one warp: [row idx 0..3][lane][bytes of that row], plane after plane
// for bits 3, so every lane reads and writes 16-, 8- or 4-byte words at a 16-, 8- or 4-byte stride.
template <int BITS> __host__ __device__ constexpr int slot_bytes() { return 4 * 32 * BITS * 4; }
template <int BITS> __host__ __device__ constexpr int ring_stages() { return BITS == 8 ? 2 : BITS == 2 ? 6 : 3; }

template <int N>
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src) {
  if constexpr (N == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" :: "r"(dst), "l"(src), "n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Issue this lane's copies of block B, rows n[idx] (idx = 2 * tile + r), into slot base `dst`.
template <int BITS>
__device__ __forceinline__ void issue_block(uint32_t dst, const uint8_t* __restrict__ wr, long B, int Np,
                                            const int (&n)[4], int t, int lane) {
#pragma unroll
  for (int idx = 0; idx < 4; ++idx) {
    if constexpr (BITS == 4) {
      cp_async<16>(dst + (idx * 32 + lane) * 16, wr + (((size_t)B * 4 + t) * Np + n[idx]) * 16);
    } else if constexpr (BITS == 2) {
      cp_async<8>(dst + (idx * 32 + lane) * 8, wr + (((size_t)B * 2 + (t >> 1)) * Np + n[idx]) * 16 + 8 * (t & 1));
    } else if constexpr (BITS == 8) {
      cp_async<16>(dst + ((2 * idx) * 32 + lane) * 16, wr + (((size_t)B * 8 + 2 * t) * Np + n[idx]) * 16);
      cp_async<16>(dst + ((2 * idx + 1) * 32 + lane) * 16, wr + (((size_t)B * 8 + 2 * t + 1) * Np + n[idx]) * 16);
    } else {
      cp_async<8>(dst + (idx * 32 + lane) * 8, wr + (((size_t)B * 3 + (t >> 1)) * Np + n[idx]) * 16 + 8 * (t & 1));
      cp_async<4>(dst + 1024 + (idx * 32 + lane) * 4, wr + (((size_t)B * 3 + 2) * Np + n[idx]) * 16 + 4 * t);
    }
  }
}

template <int BITS>
__device__ __forceinline__ void read_block(LaneWords<BITS> (&lw)[4], const uint8_t* slot, int lane) {
#pragma unroll
  for (int idx = 0; idx < 4; ++idx) {
    if constexpr (BITS == 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(slot + (idx * 32 + lane) * 16);
      lw[idx].w[0] = v.x; lw[idx].w[1] = v.y; lw[idx].w[2] = v.z; lw[idx].w[3] = v.w;
    } else if constexpr (BITS == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(slot + (idx * 32 + lane) * 8);
      lw[idx].w[0] = v.x; lw[idx].w[1] = v.y;
    } else if constexpr (BITS == 8) {
      const uint4 v0 = *reinterpret_cast<const uint4*>(slot + ((2 * idx) * 32 + lane) * 16);
      const uint4 v1 = *reinterpret_cast<const uint4*>(slot + ((2 * idx + 1) * 32 + lane) * 16);
      lw[idx].w[0] = v0.x; lw[idx].w[1] = v0.y; lw[idx].w[2] = v0.z; lw[idx].w[3] = v0.w;
      lw[idx].w[4] = v1.x; lw[idx].w[5] = v1.y; lw[idx].w[6] = v1.z; lw[idx].w[7] = v1.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(slot + (idx * 32 + lane) * 8);
      lw[idx].w[0] = v.x; lw[idx].w[1] = v.y;
      lw[idx].w[2] = *reinterpret_cast<const uint32_t*>(slot + 1024 + (idx * 32 + lane) * 4);
    }
  }
}

// Parameters of one launch.
struct SmallArgs {
  const uint8_t* wr; const int32_t* perm; const int32_t* cgid; const uint16_t* s_r; const uint8_t* z_r;
  const void* x; void* y; int32_t* err;
  int M, N, Np, K, Kr, G, identity, bps, splits, span_max;
  int g_first[kMaxSplit];    // first group of each split's k-range
};

__host__ __device__ inline int round16(int b) { return (b + 15) / 16 * 16; }

// Shared-memory carve-up of one CTA (byte offsets), shared by the kernel and the planner.
struct SmallSmem { int ring, xs, zs, cg, bgrp, red, total; };
__host__ __device__ inline SmallSmem small_smem(int slot_b, int stages, int bps, int mrows, int span_max,
                                               int ncol, int kg, int mt8) {
  SmallSmem o;
  o.ring = 0;
  o.xs = o.ring + kWarps * stages * slot_b;
  o.zs = o.xs + bps * 8 * mrows * 4 * 8;
  o.cg = o.zs + span_max * ncol * 8;
  o.bgrp = o.cg + round16(4 * bps * 4);
  o.red = o.bgrp + round16(bps * 4);
  o.total = o.red + kg * mt8 * 8 * (ncol + 4) * 4;
  return o;
}

template <typename T, int BITS, int MT8, int NCW>
__global__ void __launch_bounds__(kThreads) k_gemm_small(const SmallArgs a) {
  constexpr int KG = kWarps / NCW;
  constexpr int NCOL = NCW * 32;
  constexpr int STAGES = ring_stages<BITS>();
  constexpr int SLOT = slot_bytes<BITS>();
  constexpr int RS = NCOL + 4;
  extern __shared__ __align__(128) uint8_t smem[];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int cw = warp % NCW, kg = warp / NCW;
  const int n_cta = blockIdx.x * NCOL;
  const int m0 = blockIdx.z * (MT8 * 8);
  const int Mr = min(a.M - m0, MT8 * 8);          // x rows this CTA stages and stores
  const int NB = a.Kr / 128;
  const int blk0 = blockIdx.y * a.bps;
  const int nblk = max(0, min(NB, blk0 + a.bps) - blk0);
  const int bpw = (nblk + KG - 1) / KG;            // blocks per k-group
  const int jb0 = kg * bpw;                        // this warp's first CTA-local block
  const int nmine = max(0, min(nblk, jb0 + bpw) - jb0);
  const int g_first = a.g_first[blockIdx.y];

  const SmallSmem L = small_smem(SLOT, STAGES, a.bps, Mr, a.span_max, NCOL, KG, MT8);
  uint8_t* ring = smem + L.ring + (size_t)warp * STAGES * SLOT;
  const uint32_t ring_s = smem_u32(ring);
  uint2* xs = reinterpret_cast<uint2*>(smem + L.xs);        // [bl][s][m < Mr][t]: 4 sorted k of x row m
  uint2* zsm = reinterpret_cast<uint2*>(smem + L.zs);       // [span_max][NCOL] (prepared zero, scale bits)
  int32_t* cg = reinterpret_cast<int32_t*>(smem + L.cg);    // [4*bps] group of each chunk
  int32_t* bgrp = reinterpret_cast<int32_t*>(smem + L.bgrp);  // [bps] group of a block, -1 if it has several
  float* red = reinterpret_cast<float*>(smem + L.red);      // [KG][MT8*8][RS]

  // Let the next grid on the stream launch now; it waits for this one before touching our outputs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Rows of this lane: tile i (16 output features), r = 0/1 -> + 8; idx = 2 i + r.
  int nrow[4];
#pragma unroll
  for (int idx = 0; idx < 4; ++idx) nrow[idx] = n_cta + cw * 32 + 16 * (idx >> 1) + 8 * (idx & 1) + g;

  // Start the weight stream (handle-owned data: no dependency on the previous grid).
#pragma unroll
  for (int j = 0; j < STAGES - 1; ++j) {
    if (j < nmine) issue_block<BITS>(ring_s + j * SLOT, a.wr, blk0 + jb0 + j, a.Np, nrow, t, lane);
    cp_async_commit();
  }

  // Handle-owned tables.
  for (int i = tid; i < 4 * nblk; i += kThreads) cg[i] = __ldg(&a.cgid[4 * blk0 + i]);
  for (int i = tid; i < a.span_max * NCOL; i += kThreads) {
    const int gg = g_first + i / NCOL;
    uint2 v = make_uint2(0u, 0u);
    if (gg < a.G) {
      const size_t o = (size_t)gg * a.Np + n_cta + (i % NCOL);
      v = make_uint2(prep_zero<T, BITS>(__ldg(&a.z_r[o])), __ldg(&a.s_r[o]));
    }
    zsm[i] = v;
  }

  // x may be the previous grid's output.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  {
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    const int nq = nblk * 32 * Mr;
    for (int i0 = tid; i0 < nq; i0 += 4 * kThreads) {
      uint2 v[4];
      int dst[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kThreads;
        dst[u] = -1;
        if (i < nq) {
          const int m = i % Mr, q = (i / Mr) & 31, bl = i / (Mr * 32);
          const int j = 128 * (blk0 + bl) + 4 * q;
          const uint16_t* xr = static_cast<const uint16_t*>(x) + (size_t)(m0 + m) * a.K;
          if (a.identity) {
            v[u] = *reinterpret_cast<const uint2*>(xr + j);
          } else {
            const int4 kk = __ldg(reinterpret_cast<const int4*>(a.perm + j));
            const uint32_t e0 = kk.x >= 0 ? xr[kk.x] : 0u, e1 = kk.y >= 0 ? xr[kk.y] : 0u;
            const uint32_t e2 = kk.z >= 0 ? xr[kk.z] : 0u, e3 = kk.w >= 0 ? xr[kk.w] : 0u;
            v[u] = make_uint2(e0 | (e1 << 16), e2 | (e3 << 16));
          }
          const int s = 2 * (q >> 3) + (q & 1), tt = (q & 7) >> 1;
          dst[u] = ((bl * 8 + s) * Mr + m) * 4 + tt;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (dst[u] >= 0) xs[dst[u]] = v[u];
    }
  }
  __syncthreads();
  for (int bl = tid; bl < nblk; bl += kThreads) bgrp[bl] = cg[4 * bl] == cg[4 * bl + 3] ? cg[4 * bl] : -1;
  __syncthreads();

  // ---------------- main loop ----------------
  float acc[2][MT8][4], part[2][MT8][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int mt = 0; mt < MT8; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) { acc[i][mt][q] = 0.f; part[i][mt][q] = 0.f; }
  uint32_t zq[4];
  float sc[4];
  int cur = -1;
  const int col0 = cw * 32 + g;          // CTA-local column of idx 0; idx adds 16 (idx >> 1) + 8 (idx & 1)
  auto load_group = [&](int gg) {
    const int li = gg - g_first;
#pragma unroll
    for (int idx = 0; idx < 4; ++idx) {
      const int c = col0 + 16 * (idx >> 1) + 8 * (idx & 1);
      uint2 v;
      if (li < a.span_max) {
        v = zsm[li * NCOL + c];
      } else {
        const size_t o = (size_t)gg * a.Np + n_cta + c;
        v = make_uint2(prep_zero<T, BITS>(__ldg(&a.z_r[o])), __ldg(&a.s_r[o]));
      }
      zq[idx] = v.x;
      sc[idx] = to_float<T>(v.y);
    }
  };
  auto flush = [&]() {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int mt = 0; mt < MT8; ++mt) {
        acc[i][mt][0] = fmaf(sc[2 * i], part[i][mt][0], acc[i][mt][0]);
        acc[i][mt][1] = fmaf(sc[2 * i], part[i][mt][1], acc[i][mt][1]);
        acc[i][mt][2] = fmaf(sc[2 * i + 1], part[i][mt][2], acc[i][mt][2]);
        acc[i][mt][3] = fmaf(sc[2 * i + 1], part[i][mt][3], acc[i][mt][3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) part[i][mt][q] = 0.f;
      }
  };
  bool mval[MT8];
#pragma unroll
  for (int mt = 0; mt < MT8; ++mt) mval[mt] = 8 * mt + g < Mr;
  const int xlane = g * 4 + t;

  for (int j = 0; j < nmine; ++j) {
    cp_async_wait<STAGES - 2>();                     // block j has landed in this lane's slot
    LaneWords<BITS> lw[4];
    read_block<BITS>(lw, ring + (j % STAGES) * SLOT, lane);
    // refill the slot read in the previous iteration
    const int jn = j + STAGES - 1;
    if (jn < nmine) issue_block<BITS>(ring_s + (jn % STAGES) * SLOT, a.wr, blk0 + jb0 + jn, a.Np, nrow, t, lane);
    cp_async_commit();

    const int bl = jb0 + j;
    const int gb = bgrp[bl];
    if (gb >= 0 && gb != cur) {
      if (cur >= 0) flush();
      cur = gb;
      load_group(gb);
    }
    const uint2* xb = xs + (size_t)bl * 8 * Mr * 4;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (gb < 0 && (s & 1) == 0) {
        const int gg = cg[bl * 4 + (s >> 1)];
        if (gg != cur) {
          if (cur >= 0) flush();
          cur = gg;
          load_group(gg);
        }
      }
      uint2 xv[MT8];
#pragma unroll
      for (int mt = 0; mt < MT8; ++mt)
        xv[mt] = mval[mt] ? xb[s * Mr * 4 + mt * 32 + xlane] : make_uint2(0u, 0u);
      const int p0 = 4 * (s >> 1) + 2 * (s & 1);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t af[4];
        af[0] = operand<T, BITS>(lw[2 * i], p0, zq[2 * i]);
        af[1] = operand<T, BITS>(lw[2 * i + 1], p0, zq[2 * i + 1]);
        af[2] = operand<T, BITS>(lw[2 * i], p0 + 1, zq[2 * i]);
        af[3] = operand<T, BITS>(lw[2 * i + 1], p0 + 1, zq[2 * i + 1]);
#pragma unroll
        for (int mt = 0; mt < MT8; ++mt) mma16816<T>(part[i][mt], af, xv[mt].x, xv[mt].y);
      }
    }
  }
  cp_async_wait<0>();
  if (cur >= 0) flush();

  // ---- k-group partial tiles meet in shared memory: red[kg][m][n] ----
  {
    float* rk = red + (size_t)kg * MT8 * 8 * RS;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int mt = 0; mt < MT8; ++mt) {
        const int nl = cw * 32 + 16 * i + g;
        const int ml = 8 * mt + 2 * t;
        rk[ml * RS + nl] = acc[i][mt][0];
        rk[(ml + 1) * RS + nl] = acc[i][mt][1];
        rk[ml * RS + nl + 8] = acc[i][mt][2];
        rk[(ml + 1) * RS + nl + 8] = acc[i][mt][3];
      }
  }
  __syncthreads();
  T* y = static_cast<T*>(a.y);
  const int S = a.splits;
  if (S == 1) {
    for (int i = tid; i < Mr * (NCOL / 4); i += kThreads) {
      const int ml = i / (NCOL / 4), cl = 4 * (i % (NCOL / 4));
      float4 sum = *reinterpret_cast<const float4*>(&red[ml * RS + cl]);
#pragma unroll
      for (int k = 1; k < KG; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(&red[(size_t)k * MT8 * 8 * RS + ml * RS + cl]);
        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
      }
      const int n = n_cta + cl;
      if (n < a.N) {   // N % 32 == 0: a group of 4 columns is all in or all out
        uint2 o;
        o.x = pack2<T>(sum.x, sum.y);
        o.y = pack2<T>(sum.z, sum.w);
        *reinterpret_cast<uint2*>(y + (size_t)(m0 + ml) * a.N + n) = o;
      }
    }
    return;
  }
  // ---- K split over the cluster: fold the k-groups, then ranks in fixed order ----
  for (int i = tid; i < Mr * NCOL; i += kThreads) {
    const int ml = i / NCOL, nl = i % NCOL;
    float v = red[ml * RS + nl];
#pragma unroll
    for (int k = 1; k < KG; ++k) v += red[(size_t)k * MT8 * 8 * RS + ml * RS + nl];
    red[ml * RS + nl] = v;
  }
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  const int cols = NCOL / S, c0 = (int)rank * cols;
  for (int i = tid; i < Mr * (cols / 4); i += kThreads) {
    const int ml = i / (cols / 4), cl = c0 + 4 * (i % (cols / 4));
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t local = smem_u32(&red[ml * RS + cl]);
    for (int sp = 0; sp < S; ++sp) {
      float4 v;
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(sp));
      asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote));
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    const int n = n_cta + cl;
    if (n < a.N) {
      uint2 o;
      o.x = pack2<T>(sum.x, sum.y);
      o.y = pack2<T>(sum.z, sum.w);
      *reinterpret_cast<uint2*>(y + (size_t)(m0 + ml) * a.N + n) = o;
    }
  }
  // keep this CTA's shared memory alive until every rank has read it
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct SmallPlan { int ncw, splits, bps, mtiles, ntiles, span_max; size_t smem; int g_first[kMaxSplit]; };

template <typename T, int BITS, int MT8, int NCW>
int occupancy(int smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemm_small<T, BITS, MT8, NCW>, kThreads, smem) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// Group span of each split: cgid ascends, so the groups of chunks [c0, c1) lie in
// [cgid[c0], cgid[c1-1]].  Returns the largest span (capped at the chunk count) and fills g_first.
int split_spans(const Handle& h, int bps, int S, int* g_first) {
  const int NB = h.Kr / 128;
  int best = 1;
  for (int sp = 0; sp < kMaxSplit; ++sp) g_first[sp] = 0;
  for (int sp = 0; sp < S; ++sp) {
    const int b0 = sp * bps;
    if (b0 >= NB) continue;
    const int c0 = 4 * b0, c1 = 4 * std::min(NB, b0 + bps);
    g_first[sp] = h.cgid_host[c0];
    best = std::max(best, h.cgid_host[c1 - 1] - h.cgid_host[c0] + 1);
  }
  return std::min(best, 4 * bps);
}

template <typename T, int BITS, int MT8, int NCW>
void consider(const Handle& h, int M, SmallPlan& best, long& best_cost) {
  constexpr int KG = kWarps / NCW, NCOL = NCW * 32;
  const int NB = h.Kr / 128;
  const int mtiles = (M + MT8 * 8 - 1) / (MT8 * 8);
  const int mrows = std::min(M, MT8 * 8);
  const int ntiles = h.Np / NCOL;
  for (int S = 1; S <= kMaxSplit && S <= NB; S *= 2) {
    const int bps = (NB + S - 1) / S;
    if (S > 1 && bps * 128 * mrows * 2 <= kXsBudget / 2) break;   // split K only to make x fit
    if (bps * 128 * mrows * 2 > kXsBudget && S < kMaxSplit && S < NB) continue;
    int gf[kMaxSplit];
    const int span = split_spans(h, bps, S, gf);
    const SmallSmem L = small_smem(slot_bytes<BITS>(), ring_stages<BITS>(), bps, mrows, span, NCOL, KG, MT8);
    if (L.total > 227 * 1024) continue;
    const int R = occupancy<T, BITS, MT8, NCW>(L.total);
    const long ctas = (long)ntiles * S * mtiles;
    const long per_sm = (ctas + h.sm_count - 1) / h.sm_count;     // CTAs on the busiest SM
    const long waves = (ctas + (long)R * h.sm_count - 1) / ((long)R * h.sm_count);
    const int bpw = (bps + KG - 1) / KG;
    // cost: weight bytes the busiest SM streams (blocks x columns), one wave preferred; a small charge
    // for long per-warp chains and for cluster splits
    const long cost = per_sm * bps * NCW * 64 + (waves - 1) * 100000000L + (long)bpw + 8L * (S - 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best.ncw = NCW; best.splits = S; best.bps = bps; best.mtiles = mtiles; best.ntiles = ntiles;
      best.span_max = span; best.smem = L.total;
      std::copy(gf, gf + kMaxSplit, best.g_first);
    }
  }
}

template <typename T, int BITS, int MT8, int NCW>
cudaError_t launch_kernel(const Handle& h, const SmallPlan& p, const void* x, void* y, int M, cudaStream_t st) {
  auto kern = k_gemm_small<T, BITS, MT8, NCW>;
  SmallArgs args{h.wr, h.perm, h.cgid, h.s_r, h.z_r, x, y, h.err, M, h.N, h.Np, h.K, h.Kr, h.G, h.identity,
                 p.bps, p.splits, p.span_max, {}};
  std::copy(p.g_first, p.g_first + kMaxSplit, args.g_first);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ntiles, p.splits, p.mtiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = p.splits;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.splits > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

template <typename T, int BITS, int MT8>
cudaError_t launch_t(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  SmallPlan p{};
  {
    std::lock_guard<std::mutex> lock(h.plan_mu);
    const int64_t key = ((int64_t)GPTQ_PATH_SMALL_M << 32) | (uint32_t)M;
    auto it = h.plans.find(key);
    if (it == h.plans.end()) {
      long best_cost = -1;
      consider<T, BITS, MT8, 1>(h, M, p, best_cost);
      consider<T, BITS, MT8, 2>(h, M, p, best_cost);
      consider<T, BITS, MT8, 4>(h, M, p, best_cost);
      if (best_cost < 0) return cudaErrorInvalidConfiguration;
      // every plan fits 227 KB; allow the kernels that much dynamic shared memory
      for (cudaError_t e : {cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024),
                            cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024),
                            cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)})
        if (e != cudaSuccess) return e;
      std::vector<int64_t> v = {p.ncw, p.splits, p.bps, p.mtiles, p.ntiles, p.span_max, (int64_t)p.smem};
      v.insert(v.end(), p.g_first, p.g_first + kMaxSplit);
      h.plans[key] = v;
    } else {
      const auto& v = it->second;
      p.ncw = (int)v[0]; p.splits = (int)v[1]; p.bps = (int)v[2]; p.mtiles = (int)v[3]; p.ntiles = (int)v[4];
      p.span_max = (int)v[5]; p.smem = (size_t)v[6];
      for (int i = 0; i < kMaxSplit; ++i) p.g_first[i] = (int)v[7 + i];
    }
  }
  switch (p.ncw) {
    case 1: return launch_kernel<T, BITS, MT8, 1>(h, p, x, y, M, st);
    case 2: return launch_kernel<T, BITS, MT8, 2>(h, p, x, y, M, st);
    default: return launch_kernel<T, BITS, MT8, 4>(h, p, x, y, M, st);
  }
}

template <typename T, int BITS>
cudaError_t launch_bits(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  return M <= 8 ? launch_t<T, BITS, 1>(h, x, y, M, st) : launch_t<T, BITS, 2>(h, x, y, M, st);
}

template <typename T>
cudaError_t launch_dtype(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  switch (h.bits) {
    case 2: return launch_bits<T, 2>(h, x, y, M, st);
    case 3: return launch_bits<T, 3>(h, x, y, M, st);
    case 4: return launch_bits<T, 4>(h, x, y, M, st);
    default: return launch_bits<T, 8>(h, x, y, M, st);
  }
}

}  // namespace

int small_m_launches(const Handle&, int M) { return M > 0 ? 1 : 0; }

cudaError_t launch_gemm_small(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  if (h.dtype == GPTQ_BF16) return launch_dtype<__nv_bfloat16>(h, x, y, M, st);
  return launch_dtype<__half>(h, x, y, M, st);
}

}  // namespace gptq

// Small-M GEMM (decode, M <= 16): weight streaming at HBM speed.
//
// mlinterviewnotes "Formats and kernels: FP8, INT8, INT4, Marlin, Machete": at small M "only the
// weight bytes matter" (opening section), the quantised weight only pays if it stays packed
// until the registers that feed the tensor core, and the group scale cannot be hoisted out of
// the k reduction (section on the LOP3 dequant and the scale).  For tiny M the lever is many
// CTAs streaming weights at once with deep K (section "Where the batch-size crossover is" and the
// tile-table discussion) and the skinny operand goes in the MMA's N slot (swap-AB).
//
// Design on sm_103a:
//  * mma.sync.m16n8k16 with swap-AB: A = dequantised weights (16 output features x 16 k),
//    B = x^T (16 k x 8 batch rows), fp32 accumulators in registers.  One A fragment row needs
//    4 codes per lane per step; the runtime layout stores exactly those codes per lane.
//  * Packed words are read once, straight from HBM with 128-bit non-allocating loads, STAGES
//    blocks of 128 k ahead in registers.
//  * Conversion: a mask-and-or of two codes into the mantissas of a magic fp16 (1024) or bf16
//    (128) pair, one packed subtract of (magic + zero) -> the exact integer (code - zero).
//    8-bit codes with bf16 go through fp32 (2^23 magic) because bf16 holds 128 + q exactly only
//    for q < 128.  The group scale multiplies the fp32 partial sum of each group (exact operands,
//    one fp32 rounding per group), because the runtime layout makes every MMA step lie inside
//    one 32-row chunk, hence one group.
//  * Split-K across the CTAs of a thread-block cluster (up to 8), reduced through distributed
//    shared memory in fixed rank order: no workspace, no atomics, deterministic.
#include "internal.cuh"

#include <algorithm>
#include <type_traits>

namespace gptq {
namespace {

constexpr int kMaxSplit = 8;

template <typename T> struct Magic;
template <> struct Magic<__half> { static constexpr uint32_t base = 0x6400u; };         // 1024.0
template <> struct Magic<__nv_bfloat16> { static constexpr uint32_t base = 0x4300u; };  // 128.0

template <typename T>
__device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b);
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

template <typename T> __device__ __forceinline__ float to_float(uint16_t b);
template <> __device__ __forceinline__ float to_float<__half>(uint16_t b) { return __half2float(__ushort_as_half(b)); }
template <> __device__ __forceinline__ float to_float<__nv_bfloat16>(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Lane words of one (block, column) for this lane: BITS words (bits 3: 2 words of the 2-bit plane
// then 1 word of the 1-bit plane).
template <int BITS> struct LaneWords { uint32_t w[BITS]; };

template <int BITS>
__device__ __forceinline__ void load_lane_words(LaneWords<BITS>& lw, const uint8_t* __restrict__ wr, long B, int Np, int n, int t) {
  if constexpr (BITS == 4) {
    uint4 v = ldg_stream_v4(wr + (((size_t)B * 4 + t) * Np + n) * 16);
    lw.w[0] = v.x; lw.w[1] = v.y; lw.w[2] = v.z; lw.w[3] = v.w;
  } else if constexpr (BITS == 2) {
    uint2 v = ldg_stream_v2(wr + (((size_t)B * 2 + (t >> 1)) * Np + n) * 16 + 8 * (t & 1));
    lw.w[0] = v.x; lw.w[1] = v.y;
  } else if constexpr (BITS == 8) {
    uint4 v0 = ldg_stream_v4(wr + (((size_t)B * 8 + 2 * t) * Np + n) * 16);
    uint4 v1 = ldg_stream_v4(wr + (((size_t)B * 8 + 2 * t + 1) * Np + n) * 16);
    lw.w[0] = v0.x; lw.w[1] = v0.y; lw.w[2] = v0.z; lw.w[3] = v0.w;
    lw.w[4] = v1.x; lw.w[5] = v1.y; lw.w[6] = v1.z; lw.w[7] = v1.w;
  } else {  // 3
    uint2 v = ldg_stream_v2(wr + (((size_t)B * 3 + (t >> 1)) * Np + n) * 16 + 8 * (t & 1));
    lw.w[0] = v.x; lw.w[1] = v.y;
    lw.w[2] = ldg_stream_u32(wr + (((size_t)B * 3 + 2) * Np + n) * 16 + 4 * t);
  }
}

// Codes of pair p of this lane, one code per 16-bit half (low half = even k of the pair).
template <int BITS>
__device__ __forceinline__ uint32_t pair_codes(const LaneWords<BITS>& lw, int p) {
  if constexpr (BITS == 3) {
    uint32_t lo = (lw.w[p / 8] >> (2 * (p % 8))) & 0x00030003u;
    uint32_t hi = ((lw.w[2] >> p) & 0x00010001u) << 2;
    return lo | hi;
  } else {
    constexpr int F = 16 / BITS;
    constexpr uint32_t mask = ((1u << BITS) - 1u) * 0x00010001u;
    return (lw.w[p / F] >> (BITS * (p % F))) & mask;
  }
}

// (code - zero) for both halves, as a T2 register.  zq: zero prepared by prep_zero.
template <typename T, int BITS>
__device__ __forceinline__ uint32_t code_minus_zero(uint32_t codes, uint32_t zq) {
  if constexpr (BITS == 8 && std::is_same<T, __nv_bfloat16>::value) {
    const float zf = __uint_as_float(zq);
    float lo = __uint_as_float(0x4B000000u | (codes & 0xFFFFu)) - zf;
    float hi = __uint_as_float(0x4B000000u | (codes >> 16)) - zf;
    return pack_bf16x2(lo, hi);
  } else {
    return sub2<T>(codes | (Magic<T>::base * 0x00010001u), zq);
  }
}

// Zero point (stored + 1) in the form code_minus_zero subtracts.
template <typename T, int BITS>
__device__ __forceinline__ uint32_t prep_zero(uint32_t stored) {
  const uint32_t z = stored + 1u;
  if constexpr (BITS == 8 && std::is_same<T, __nv_bfloat16>::value) {
    return __float_as_uint(8388608.0f + (float)z);      // 2^23 + z, exact
  } else {
    return (Magic<T>::base + z) * 0x00010001u;          // magic + z in both halves, exact
  }
}

template <int MT8>
struct XSlot { uint32_t v[2 * MT8]; };

// Parameters of one launch.
struct SmallArgs {
  const uint8_t* wr; const int32_t* perm; const int32_t* cgid; const uint16_t* s_r; const uint8_t* z_r;
  const void* x; void* y;
  int M, N, Np, K, Kr, identity, bps, splits;
};

template <typename T, int BITS, int MT8, int NWARP, int STAGES>
__global__ void __launch_bounds__(NWARP * 32) k_gemm_small(const SmallArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int n_cta = blockIdx.x * (NWARP * 32);
  const int split = blockIdx.y;
  const int m0 = blockIdx.z * (MT8 * 8);
  const int NB = a.Kr / 128;
  const int blk0 = split * a.bps;
  const int blk1 = min(NB, blk0 + a.bps);
  const int nblk = max(0, blk1 - blk0);

  XSlot<MT8>* xs = reinterpret_cast<XSlot<MT8>*>(smem);                 // [bps][8][32]
  int32_t* cg = reinterpret_cast<int32_t*>(smem + (size_t)a.bps * 8 * 32 * sizeof(XSlot<MT8>));
  float* red = reinterpret_cast<float*>(cg + a.bps * 4);                 // [MT8*8][NWARP*32 + 4]
  constexpr int RS = NWARP * 32 + 4;

  // rows of this lane: tile i covers 16 output features; lane holds rows g and g + 8.
  const int nrow0 = n_cta + warp * 32 + g;       // tile 0: nrow0, nrow0 + 8; tile 1: +16, +24

  // ---- prologue: start the weight stream before staging x ----
  LaneWords<BITS> wb[STAGES][2][2];
#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st)
    if (st < nblk) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int r = 0; r < 2; ++r) load_lane_words<BITS>(wb[st][i][r], a.wr, blk0 + st, a.Np, nrow0 + 16 * i + 8 * r, t);
    }

  // ---- stage x fragments (gathered through perm) and chunk groups ----
  {
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    const int nslots = nblk * 8 * 32 * 2 * MT8;
    uint32_t* xw = reinterpret_cast<uint32_t*>(xs);
    for (int i = threadIdx.x; i < nslots; i += NWARP * 32) {
      // slot order: [bl][s][lane][mt][wsel]
      const int wsel = i & 1, mt = (i >> 1) % MT8;
      const int rest = (i >> 1) / MT8;
      const int ln = rest & 31, s = (rest >> 5) & 7, bl = rest >> 8;
      const int m = m0 + 8 * mt + (ln >> 2);
      const int P = 128 * (blk0 + bl) + 32 * (s >> 1) + 8 * (ln & 3) + 4 * (s & 1) + 2 * wsel;
      uint32_t v = 0;
      if (m < a.M) {
        if (a.identity) {
          v = __ldg(reinterpret_cast<const uint32_t*>(x + (size_t)m * a.K + P));
        } else {
          const int k0 = __ldg(&a.perm[P]), k1 = __ldg(&a.perm[P + 1]);
          const uint32_t lo = k0 >= 0 ? __ldg(x + (size_t)m * a.K + k0) : 0u;
          const uint32_t hi = k1 >= 0 ? __ldg(x + (size_t)m * a.K + k1) : 0u;
          v = lo | (hi << 16);
        }
      }
      xw[i] = v;
    }
    for (int i = threadIdx.x; i < nblk * 4; i += NWARP * 32) cg[i] = __ldg(&a.cgid[blk0 * 4 + i]);
  }
  __syncthreads();

  float acc[2][MT8][4], part[2][MT8][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int mt = 0; mt < MT8; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) { acc[i][mt][q] = 0.f; part[i][mt][q] = 0.f; }

  int cur_g = nblk > 0 ? cg[0] : 0;
  uint32_t zq[2][2];
  float sc[2][2];
  auto load_group = [&](int gg) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const size_t o = (size_t)gg * a.Np + nrow0 + 16 * i + 8 * r;
        zq[i][r] = prep_zero<T, BITS>(__ldg(&a.z_r[o]));
        sc[i][r] = to_float<T>(__ldg(&a.s_r[o]));
      }
  };
  auto flush = [&]() {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int mt = 0; mt < MT8; ++mt) {
        acc[i][mt][0] = fmaf(sc[i][0], part[i][mt][0], acc[i][mt][0]);
        acc[i][mt][1] = fmaf(sc[i][0], part[i][mt][1], acc[i][mt][1]);
        acc[i][mt][2] = fmaf(sc[i][1], part[i][mt][2], acc[i][mt][2]);
        acc[i][mt][3] = fmaf(sc[i][1], part[i][mt][3], acc[i][mt][3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) part[i][mt][q] = 0.f;
      }
  };
  if (nblk > 0) load_group(cur_g);

  // ---- main loop over 128-row blocks ----
  for (int bb = 0; bb < nblk; bb += STAGES) {
#pragma unroll
    for (int st = 0; st < STAGES; ++st) {
      const int bl = bb + st;
      if (bl < nblk) {
        const int nb = bl + STAGES - 1;
        if (nb < nblk) {
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int r = 0; r < 2; ++r)
              load_lane_words<BITS>(wb[(st + STAGES - 1) % STAGES][i][r], a.wr, blk0 + nb, a.Np, nrow0 + 16 * i + 8 * r, t);
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          if ((s & 1) == 0) {
            const int gg = cg[bl * 4 + (s >> 1)];
            if (gg != cur_g) { flush(); cur_g = gg; load_group(gg); }
          }
          const XSlot<MT8> xv = xs[(bl * 8 + s) * 32 + lane];
          const int p0 = 4 * (s >> 1) + 2 * (s & 1);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            uint32_t af[4];
            af[0] = code_minus_zero<T, BITS>(pair_codes<BITS>(wb[st][i][0], p0), zq[i][0]);
            af[1] = code_minus_zero<T, BITS>(pair_codes<BITS>(wb[st][i][1], p0), zq[i][1]);
            af[2] = code_minus_zero<T, BITS>(pair_codes<BITS>(wb[st][i][0], p0 + 1), zq[i][0]);
            af[3] = code_minus_zero<T, BITS>(pair_codes<BITS>(wb[st][i][1], p0 + 1), zq[i][1]);
#pragma unroll
            for (int mt = 0; mt < MT8; ++mt) mma16816<T>(part[i][mt], af, xv.v[2 * mt], xv.v[2 * mt + 1]);
          }
        }
      }
    }
  }
  flush();

  // ---- per-CTA partial tile into shared memory: red[m][n] ----
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int mt = 0; mt < MT8; ++mt) {
      const int nl = warp * 32 + 16 * i + g;
      const int ml = 8 * mt + 2 * t;
      red[ml * RS + nl] = acc[i][mt][0];
      red[(ml + 1) * RS + nl] = acc[i][mt][1];
      red[ml * RS + nl + 8] = acc[i][mt][2];
      red[(ml + 1) * RS + nl + 8] = acc[i][mt][3];
    }

  // ---- split-K reduction across the cluster (fixed rank order) and the store of y ----
  const int S = a.splits;
  uint32_t rank = 0;
  if (S > 1) {
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  } else {
    __syncthreads();
  }
  constexpr int NCOL = NWARP * 32;
  const int cols = NCOL / S;            // columns this CTA reduces and stores
  const int c0 = (int)rank * cols;
  const int groups = (MT8 * 8) * (cols / 4);
  T* y = static_cast<T*>(a.y);
  for (int i = threadIdx.x; i < groups; i += NWARP * 32) {
    const int ml = i / (cols / 4);
    const int cl = c0 + 4 * (i % (cols / 4));
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t local = smem_u32(&red[ml * RS + cl]);
    for (int s = 0; s < S; ++s) {
      float4 v;
      if (S > 1) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(s));
        asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote));
      } else {
        v = *reinterpret_cast<const float4*>(&red[ml * RS + cl]);
      }
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    const int m = m0 + ml, n = n_cta + cl;
    if (m < a.M && n < a.N) {     // N % 32 == 0, so a group of 4 columns is all in or all out
      uint2 o;
      o.x = pack2<T>(sum.x, sum.y);
      o.y = pack2<T>(sum.z, sum.w);
      *reinterpret_cast<uint2*>(y + (size_t)m * a.N + n) = o;
    }
  }
  if (S > 1) {
    // keep this CTA's shared memory alive until every rank has read it
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
}

struct SmallPlan { int nwarp, mt8, splits, bps, mtiles, ntiles; size_t smem; };

SmallPlan plan_small(const Handle& h, int M) {
  SmallPlan p{};
  p.mt8 = M <= 8 ? 1 : 2;
  p.mtiles = (M + p.mt8 * 8 - 1) / (p.mt8 * 8);
  const int NB = h.Kr / 128;
  const int target = 2 * h.sm_count;
  const int bps_max = p.mt8 == 1 ? 32 : 16;
  p.nwarp = 8;
  p.ntiles = h.Np / 256;
  if (p.ntiles * p.mtiles * kMaxSplit < target) { p.nwarp = 4; p.ntiles = h.Np / 128; }
  p.splits = 1;
  while (p.splits < kMaxSplit && p.splits < NB &&
         (p.ntiles * p.mtiles * p.splits < target || (NB + p.splits - 1) / p.splits > bps_max))
    p.splits *= 2;
  p.bps = (NB + p.splits - 1) / p.splits;
  const size_t xs = (size_t)p.bps * 8 * 32 * 8 * p.mt8;
  p.smem = xs + (size_t)p.bps * 4 * 4 + (size_t)p.mt8 * 8 * (p.nwarp * 32 + 4) * 4;
  return p;
}

template <typename T, int BITS, int MT8, int NWARP>
cudaError_t launch_t(const SmallPlan& p, const SmallArgs& args, cudaStream_t st) {
  constexpr int STAGES = BITS == 8 ? 2 : 3;
  auto kern = k_gemm_small<T, BITS, MT8, NWARP, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ntiles, p.splits, p.mtiles);
  cfg.blockDim = dim3(NWARP * 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = p.splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

template <typename T, int BITS>
cudaError_t launch_bits(const SmallPlan& p, const SmallArgs& args, cudaStream_t st) {
  if (p.mt8 == 1) return p.nwarp == 8 ? launch_t<T, BITS, 1, 8>(p, args, st) : launch_t<T, BITS, 1, 4>(p, args, st);
  return p.nwarp == 8 ? launch_t<T, BITS, 2, 8>(p, args, st) : launch_t<T, BITS, 2, 4>(p, args, st);
}

template <typename T>
cudaError_t launch_dtype(const SmallPlan& p, const SmallArgs& args, int bits, cudaStream_t st) {
  switch (bits) {
    case 2: return launch_bits<T, 2>(p, args, st);
    case 3: return launch_bits<T, 3>(p, args, st);
    case 4: return launch_bits<T, 4>(p, args, st);
    default: return launch_bits<T, 8>(p, args, st);
  }
}

}  // namespace

int small_m_launches(const Handle&, int M) { return M > 0 ? 1 : 0; }

cudaError_t launch_gemm_small(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  const SmallPlan p = plan_small(h, M);
  SmallArgs args{h.wr, h.perm, h.cgid, h.s_r, h.z_r, x, y, M, h.N, h.Np, h.K, h.Kr, h.identity, p.bps, p.splits};
  if (h.dtype == GPTQ_BF16) return launch_dtype<__nv_bfloat16>(p, args, h.bits, st);
  return launch_dtype<__half>(p, args, h.bits, st);
}

}  // namespace gptq

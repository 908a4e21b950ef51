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
// Design on sm_103a, one CTA per tile of 128 output features x BMX rows of x (swap-AB: D[n][m];
// BMX = 64, 128 or 256, the smallest that covers M, so a mid-size M does not pay for 256 rows):
//  * warp 0: x producer, TMA (cp.async.bulk.tensor.2d, SWIZZLE_128B) loads of BMX x 64 x tiles;
//    warp 2: code producer, cp.async.bulk copies of each packed 128-row block of the tile's 128
//    columns plus the stored zeros of its four chunks; each into a ring tracked by mbarriers.
//  * warps 4..7: dequantisers, one per SM sub-partition.  Thread d owns weight row n0 + d: one LOP3
//    per code pair makes magic + code, one packed subtract of (magic + zero) leaves the exact
//    integer code - zero, and the row is written in the UMMA K-major SWIZZLE_128B layout (16-byte
//    chunk j of row r at chunk j ^ (r % 8) of its 128-byte row), then a generic-to-async proxy
//    fence and an arrive.
//  * warp 1: allocates all 512 TMEM columns (512 / BMX partial-sum buffers of BMX columns); the warp runs
//    the schedule and one elected lane issues tcgen05.mma.cta_group::1.kind::f16 (M = 128 weight
//    rows, N = BMX x rows, K = 16), two per 32-row chunk, restarting the accumulator at each group
//    and committing the buffer when the group ends.
//  * warps 8..15: eight scaler warps, two per TMEM lane quarter, BMX / 2 columns each.  Per group:
//    tcgen05.ld the partial sums (16 columns in flight while the previous 16 are used),
//    S += scale[g][n] * P in registers, release the buffer.  At the end they round S to the output
//    type and store y.  setmaxnreg gives them 184 registers a thread and the other warps 72.
// Act-order handles first gather x into the handle's workspace in sorted k order (one extra launch).
// FP8 block-scaled layers (template FP8): the dequantisers convert e4m3 pairs (fp8_pair) with no
// zero, and the scalers multiply by the CTA's 128 x 128 block factor.
// K split (grids that would leave SMs idle): blockIdx.z takes a range of 128-row blocks, the
// ranges of a tile form one thread-block cluster, each CTA leaves its fp32 partial in its own
// shared memory, and CTA z sums the z-th slice of the tile's rows over all ranges in range order
// (distributed shared memory reads) and stores y.  A very long K narrows the x tile until the tables fit.
// Every wait is bounded; a timeout sets the handle's error word and the CTA drains and exits.
#include "internal.cuh"

#include <cuda.h>
#include <type_traits>

namespace gptq {
namespace {

constexpr int BN = 128, HK = 64;   // weight rows (MMA M), k per stage; x rows per tile (MMA N): BMX
// Four warpgroups: {x producer, MMA issuer, code producer, spare}, four dequantisers (one per SM sub-partition),
// and eight scalers (two per TMEM lane quarter, BMX / 2 fp32 sums a thread).  setmaxnreg moves
// registers from the first two warpgroups to the scalers: 2 x 128 x (72 + 184) = 65536.
constexpr int kDqWarps = 4, kScWarps = 8;
constexpr int kDqWarp0 = 4, kScWarp0 = 8;
constexpr int kThreadsL = 512;
constexpr int kRegsLaunch = 128, kRegsLight = 72, kRegsScaler = 184;
static_assert(2 * 128 * (kRegsLight + kRegsScaler) <= kThreadsL * kRegsLaunch, "register split exceeds the launch");
// Ring depths.  A weight stage passes dequantisers -> proxy fence -> MMA issue -> tcgen05 commit
// before it is free again, a round trip of a few thousand cycles; with a small x tile the MMA
// of a stage is short, so the weight ring must be deeper to keep that round trip off the critical
// path.  x stages are small then, and four cover the TMA load latency.
template <int BITS, int BMX> constexpr int XS = BMX <= 128 ? 4 : (BITS == 8 ? 3 : 4);
template <int BMX> constexpr int WS = BMX == 256 ? 3 : 4;
template <int BMX> constexpr int X_BYTES = BMX * HK * 2;   // 32 KB at BMX = 256
constexpr int W_BYTES = BN * HK * 2;            // 16 KB
// Partial-sum buffers in tensor memory: all 512 columns, BMX each.  The MMA can run NPB - 1 groups
// ahead of the scalers, so the commit -> scaler -> release round trip of one buffer is hidden
// behind the other buffers when the x tile is narrow.
template <int BMX> constexpr int NPB = 512 / BMX;          // 8, 4 or 2
constexpr int kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
template <int BITS> constexpr int PK_BYTES = BN * 16 * BITS;  // one 128-row block of 128 columns
// A packed stage: the block's codes, then the stored zero of each of its four 32-row chunks for the
// tile's 128 columns (copied by the producer, so the dequant warps never wait on global loads).
template <int BITS> constexpr int PKS_BYTES = PK_BYTES<BITS> + 4 * BN;
// packed stages in the code ring: the bytes in flight per SM must cover the HBM latency
template <int BITS, int BMX> constexpr int PSB = BMX == 256 ? (BITS == 8 ? 3 : 4) : (BITS == 8 ? 4 : 8);

template <typename T> struct MagicL;
template <> struct MagicL<__half> { static constexpr uint32_t bits = 0x6400u; };
template <> struct MagicL<__nv_bfloat16> { static constexpr uint32_t bits = 0x4300u; };
template <typename T, int BITS> constexpr bool kF32Path = BITS == 8 && std::is_same<T, __nv_bfloat16>::value;

// Shared-memory carve-up from a 1024-byte-aligned base.
template <int BITS, int BMX> struct LargeSmem {
  static constexpr int x = 0;
  static constexpr int w = x + XS<BITS, BMX> * X_BYTES<BMX>;
  static constexpr int pk = w + WS<BMX> * W_BYTES;
  static constexpr int bars = pk + PSB<BITS, BMX> * PKS_BYTES<BITS>;
  static constexpr int nbars = 2 * XS<BITS, BMX> + 2 * WS<BMX> + 2 * PSB<BITS, BMX> + 2 * NPB<BMX> + 1;
  static constexpr int tmem_slot = bars + nbars * 8;
  static constexpr int cg = tmem_slot + 16;       // int32 group of every 32-row chunk, then one
                                                  // uint32 group-end mask per 32 chunks
};

struct LargeArgs {
  const uint8_t* wr; const int32_t* cgid; const uint16_t* s_r; const uint8_t* z_r;
  void* y; int32_t* err;
  int M, N, Np, Kr, G;
  int zoff;         // zero = stored byte + zoff (1: GPTQ v1 fields; 0: gptq_v2, AWQ)
  const float* bias;   // [Np] float32 added to y, or nullptr
  const float* scale_inv;   // FP8 layers: [ceil(N/128)][kb] block factors
  int kb;
  // K split: CTA z of a tile takes 128-row blocks [NB z / split, NB (z + 1) / split); the tile's
  // CTAs form one thread-block cluster and sum their fp32 partials in shared memory, in z order
  int split;
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

// Words of one lane (t = 0..3) of one column.
template <int BITS> struct Words { uint32_t w[BITS]; };

// The words of lane t that chunks 2h and 2h + 1 of a 128-row block use (other entries untouched):
// 4-bit: word c of vector t; 2-bit: word c/2; 8-bit: words 2c, 2c+1 (vector 2t + h); 3-bit: word
// c/2 of the 2-bit plane and the lane's word of the 1-bit plane.
template <int BITS>
__device__ __forceinline__ void half_words(Words<BITS>& o, const uint8_t* stage, int d, int t, int h) {
  // a stage holds, per vector, the 128 columns of the tile: column d of vector v at code_col_pos
  auto at = [&](int v) { return stage + ((size_t)v * BN + code_col_pos(BITS, v, d)) * 16; };
  if constexpr (BITS == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(at(t) + 8 * h);
    o.w[2 * h] = v.x; o.w[2 * h + 1] = v.y;
  } else if constexpr (BITS == 2) {
    o.w[h] = *reinterpret_cast<const uint32_t*>(at(t >> 1) + 8 * (t & 1) + 4 * h);
  } else if constexpr (BITS == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(at(2 * t + h));
    o.w[4 * h] = v.x; o.w[4 * h + 1] = v.y; o.w[4 * h + 2] = v.z; o.w[4 * h + 3] = v.w;
  } else {
    o.w[h] = *reinterpret_cast<const uint32_t*>(at(t >> 1) + 8 * (t & 1) + 4 * h);
    o.w[2] = *reinterpret_cast<const uint32_t*>(at(2) + 4 * t);
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

// Zero = stored byte + zoff (1 for GPTQ fields, stored minus one; 0 for AWQ fields).
template <typename T, int BITS>
__device__ __forceinline__ uint32_t prep_zero_l(uint32_t stored, uint32_t zoff) {
  const uint32_t z = stored + zoff;
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

// Commit only when pred != 0 (a predicated instruction, no branch).
__device__ __forceinline__ void umma_commit_if(uint32_t bar, uint32_t pred) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
               "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
               :: "r"(bar), "r"(pred) : "memory");
}
// tcgen05.mma issued only by the lane with go != 0.
__device__ __forceinline__ void umma_f16_if(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc, uint32_t go) {
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
               "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(go) : "memory");
}
// 1 in exactly one lane of the (converged) warp.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred;
}

// 16 consecutive fp32 columns of this warp's TMEM lane quarter; the wait names the registers so
// no use of them can be scheduled above it.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(addr));
}
// Wait for every tcgen05.ld of this thread; the registers of the loads are named by the
// reg_after_wait calls that follow, so no use of them is scheduled above the wait.
__device__ __forceinline__ void tmem_wait_all() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void reg_after_wait(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :: "memory");
}
// Thread-block cluster helpers (the K split).
__device__ __forceinline__ void cluster_sync_l() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// 16 bytes of CTA `rank`'s shared memory at the same offset as the local address `smem_addr`.
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t smem_addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(d) : "memory");
  return v;
}

template <typename T, int BITS, int BMX, bool FP8>
__global__ void __launch_bounds__(kThreadsL, 1) k_gemm_large(const LargeArgs a, const __grid_constant__ CUtensorMap tmap_x) {
  static_assert(BMX == 64 || BMX == 128 || BMX == 256, "MMA N: a multiple of 16 up to 256; TMEM: a power of two");
  static_assert(!FP8 || BITS == 8, "FP8 layers use the 8-bit layout");
  static_assert((size_t)BMX * BN * 4 <= (size_t)LargeSmem<BITS, BMX>::bars, "K-split partial below the barriers");
  using S = LargeSmem<BITS, BMX>;
  constexpr int XB = X_BYTES<BMX>;
  constexpr int XS = gptq::XS<BITS, BMX>;
  constexpr int WS = gptq::WS<BMX>;
  constexpr int kCols = kTmemCols;
  constexpr int NP_ = NPB<BMX>;
  constexpr int kDq = kDqWarps, kSc = kScWarps, kSc0 = kScWarp0;
  constexpr int HC = BMX / 2;                 // x rows (TMEM columns) per scaler warp
  constexpr int PKB = PKS_BYTES<BITS>;
  constexpr int PS = PSB<BITS, BMX>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m0 = blockIdx.x * BMX, n0 = blockIdx.y * BN;
  // this CTA's K range: blocks [kb0, kb1) of 128 sorted rows (all of K without a split)
  const int z = blockIdx.z;
  const int kb0 = (int)(((long)(a.Kr / 128) * z) / a.split);
  const int kb1 = (int)(((long)(a.Kr / 128) * (z + 1)) / a.split);
  const int nblocks = kb1 - kb0;
  const int nhalf = 2 * nblocks, nchunks = 4 * nblocks;
  const int c0 = 4 * kb0;                     // first chunk of the range

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
  auto p_empty = [&](int b) { return bar + 8 * (2 * XS + 2 * WS + 2 * PS + NP_ + b); };
  const uint32_t mma_done = bar + 8 * (2 * XS + 2 * WS + 2 * PS + 2 * NP_);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + S::tmem_slot);
  int32_t* cg = reinterpret_cast<int32_t*>(base + S::cg);
  uint32_t* gmask = reinterpret_cast<uint32_t*>(base + S::cg + 4 * nchunks);
  const int nwin = (nchunks + 31) / 32;

  if (tid == 0) {
    for (int i = 0; i < XS; ++i) { mbar_init(x_full(i), 1); mbar_init(x_empty(i), 1); }
    for (int i = 0; i < WS; ++i) { mbar_init(w_full(i), kDq); mbar_init(w_empty(i), 1); }
    for (int i = 0; i < PS; ++i) { mbar_init(pk_full(i), 1); mbar_init(pk_empty(i), kDq); }
    for (int b = 0; b < NP_; ++b) { mbar_init(p_full(b), 1); mbar_init(p_empty(b), kSc); }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(kCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  for (int i = tid; i < nchunks; i += kThreadsL) cg[i] = __ldg(&a.cgid[c0 + i]);
  __syncthreads();
  // bit j of gmask[w]: chunk 32 w + j of the range is the last chunk of its group inside the range
  // (the MMA issuer's schedule); the range's last chunk always closes one (from the shared copy:
  // one global round trip fewer before the pipeline starts)
  for (int w0 = 32 * warp; w0 < nchunks; w0 += kThreadsL) {
    const int c = w0 + lane;
    const bool end = c < nchunks && (c + 1 == nchunks || cg[c + 1] != cg[c]);
    const uint32_t m = __ballot_sync(0xffffffffu, end);
    if (lane == 0) gmask[w0 / 32] = m;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  bool ok = true;
  if (warp >= kSc0) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kRegsScaler));
    // ---------------- scalers: S += scale * P per group, then y ----------------
    const int sw = warp - kSc0;
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int hs = sw >> 2;                   // half of the BMX x rows
    const int nrow = 32 * q + lane;           // weight row of this thread inside the tile
    const int n = n0 + nrow;
    float acc[HC];
#pragma unroll
    for (int j = 0; j < HC; ++j) acc[j] = 0.f;
    // Scales of the next kSq groups in flight: each CTA reads its own columns' scales once, from
    // HBM, so a load issued only one group ahead left every group waiting for it.  The groups are
    // visited in order of their last chunk, walking the group-end mask.
    constexpr int kSq = 8;
    int ew = 0;                               // mask word of the next group end not yet prefetched
    uint32_t ebits = nwin > 0 ? gmask[0] : 0u;
    auto next_end = [&]() -> int {            // chunk that ends the next group, -1 after the last
      while (ebits == 0u) {
        if (++ew >= nwin) return -1;
        ebits = gmask[ew];
      }
      const int j = __ffs(ebits) - 1;
      ebits &= ebits - 1u;
      return 32 * ew + j;
    };
    // (FP8: the CTA's 128 rows are one scale block; a block past N has no factor and stores nothing)
    auto scale_of_end = [&](int e) {
      if constexpr (FP8) return (e >= 0 && n0 < a.N) ? __ldg(&a.scale_inv[(size_t)(n0 / BN) * a.kb + cg[e]]) : 0.f;
      else return e >= 0 ? scale_f<T>(__ldg(&a.s_r[(size_t)cg[e] * a.Np + n])) : 0.f;
    };
    int ng = 0;                               // groups in K
    for (int w = 0; w < nwin; ++w) ng += __popc(gmask[w]);
    float sq[kSq];
#pragma unroll
    for (int j = 0; j < kSq; ++j) sq[j] = scale_of_end(next_end());
    // GB groups per pass: their buffers are waited for, all their columns loaded back to back and
    // waited for once, then released together (one tcgen05.ld round trip per pass, not per group;
    // the MMA runs NP_ groups ahead, so it still has GB buffers to fill meanwhile)
    // (BMX = 64: four groups of 32 columns, 128 registers of loads; wider tiles: one group, 64
    // columns per round, as the accumulators themselves take 64 or 128 registers)
    constexpr int GB = BMX == 64 ? 4 : 1;
    constexpr int RC = BMX == 64 ? HC : 64;          // columns of one group per load round
    static_assert(kSq % GB == 0 && NP_ >= 2 * GB, "scaler batching");
    for (int g0 = 0; g0 < ng && ok; g0 += kSq) {
#pragma unroll
      for (int jb = 0; jb < kSq; jb += GB) {
        const int gb0 = g0 + jb;
        if (gb0 >= ng || !ok) break;
#pragma unroll
        for (int j = 0; j < GB; ++j) {
          const int gi = gb0 + j;
          if (gi < ng && ok && !mbar_wait(p_full(gi & (NP_ - 1)), (gi / NP_) & 1)) ok = false;
        }
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
        for (int r0 = 0; r0 < HC; r0 += RC) {
          uint32_t rv[GB][RC / 16][16];
#pragma unroll
          for (int j = 0; j < GB; ++j) {
            const int b = (gb0 + j) & (NP_ - 1);
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BMX + HC * hs + r0);
            if (gb0 + j < ng)
#pragma unroll
              for (int k = 0; k < RC / 16; ++k) tmem_ld16(taddr + 16 * k, rv[j][k]);
          }
          tmem_wait_all();
#pragma unroll
          for (int j = 0; j < GB; ++j)
#pragma unroll
            for (int k = 0; k < RC / 16; ++k) reg_after_wait(rv[j][k]);
#pragma unroll
          for (int j = 0; j < GB; ++j) {
            if (gb0 + j < ng) {
              const float sc = sq[jb + j];
#pragma unroll
              for (int k = 0; k < RC / 16; ++k)
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                  acc[r0 + 16 * k + jj] = fmaf(sc, __uint_as_float(rv[j][k][jj]), acc[r0 + 16 * k + jj]);
            }
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int j = 0; j < GB; ++j) {
          const int gi = gb0 + j;
          if (gi < ng) {
            if (lane == 0) mbar_arrive(p_empty(gi & (NP_ - 1)));
            sq[jb + j] = scale_of_end(next_end());      // group gi + kSq
          }
        }
      }
    }
    if (!ok) report_timeout(a.err);
    uint16_t* y = static_cast<uint16_t*>(a.y);
    if (a.split > 1) {
      // This K range's partial goes into the CTA's own shared memory, [x row][weight row] fp32, over
      // the x ring and what follows it (idle now: every MMA that read them has completed, and every
      // copy into them was consumed).  The K ranges of a tile are the CTAs of one cluster
      // (1 x 1 x split).  Once every partial is in place, CTA z sums the z-th slice of the tile's x
      // rows over all ranges, in order of z (the same sum whichever CTA adds it), reading the other
      // CTAs' shared memory, and stores y; a second cluster barrier keeps every CTA until no other
      // still reads its partial.  Every thread of every CTA passes both barriers (the other warps at
      // the end of their roles), after a timeout too.
      float* part = reinterpret_cast<float*>(base);
#pragma unroll
      for (int j = 0; j < HC; ++j) part[(HC * hs + j) * BN + nrow] = acc[j];
      cluster_sync_l();
      const int rows = min(BMX, a.M - m0), S = a.split;
      const int r0 = rows * z / S, r1 = rows * (z + 1) / S;
      for (int i = 32 * sw + lane; i < (r1 - r0) * (BN / 4); i += 32 * kSc) {
        const int m = r0 + i / (BN / 4), nn = 4 * (i % (BN / 4));
        const uint32_t off = base_s + (uint32_t)((m * BN + nn) * 4);
        float4 t = ld_cluster_f4(off, 0);
        for (int zz = 1; zz < S; ++zz) {
          const float4 v = ld_cluster_f4(off, (uint32_t)zz);
          t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
        }
        const int gn = n0 + nn;
        if (gn < a.N) {
          if (a.bias) {
            const float4 bb = __ldg(reinterpret_cast<const float4*>(a.bias + gn));
            t.x += bb.x; t.y += bb.y; t.z += bb.z; t.w += bb.w;
          }
          uint2 o;
          o.x = (uint32_t)to_bits<T>(t.x) | ((uint32_t)to_bits<T>(t.y) << 16);
          o.y = (uint32_t)to_bits<T>(t.z) | ((uint32_t)to_bits<T>(t.w) << 16);
          *reinterpret_cast<uint2*>(y + (size_t)(m0 + m) * a.N + gn) = o;
        }
      }
      cluster_sync_l();
    } else if (n < a.N) {
      // y[m][n] for the HC x rows of this half: lanes are consecutive n, so each store is 64 bytes
      if (a.bias) {
        const float b = __ldg(a.bias + n);
#pragma unroll
        for (int j = 0; j < HC; ++j) acc[j] += b;
      }
#pragma unroll
      for (int j = 0; j < HC; ++j) {
        const int m = m0 + HC * hs + j;
        if (m < a.M) y[(size_t)m * a.N + n] = to_bits<T>(acc[j]);
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsLight));
    if (warp == 0) {
      // ---------------- x producer: TMA tiles of x ----------------
      if (lane == 0) {
        int x_issued = 0;
        asm volatile("griddepcontrol.wait;" ::: "memory");   // x may come from the previous grid
        for (int i = 0; i < nhalf && ok; ++i) {
          const int xs = i % XS;
          if (i >= XS && !mbar_wait(x_empty(xs), ((i / XS) - 1) & 1)) { ok = false; break; }
          mbar_arrive_expect_tx(x_full(xs), XB);
          tma_load_2d(xs_s + xs * XB, &tmap_x, (2 * kb0 + i) * HK, m0, x_full(xs));
          ++x_issued;
        }
        // every issued copy must land before the CTA may exit
        for (int i = x_issued > XS ? x_issued - XS : 0; i < x_issued; ++i)
          if (!mbar_wait(x_full(i % XS), (i / XS) & 1)) ok = false;
        if (!ok) report_timeout(a.err);
      }
    } else if (warp == 2) {
      // ---------------- packed-code producer: codes and stored zeros of each block ----------------
      // (its own warp, so the code ring runs ahead of the x ring; handle-owned data, no wait on
      // the previous grid)
      if (lane == 0) {
        int pk_issued = 0;
        for (int blk = 0; blk < nblocks && ok; ++blk) {
          const int ps = blk % PS;
          if (blk >= PS && !mbar_wait(pk_empty(ps), ((blk / PS) - 1) & 1)) { ok = false; break; }
          mbar_arrive_expect_tx(pk_full(ps), FP8 ? (uint32_t)PK_BYTES<BITS> : (uint32_t)PKB);   // FP8: no zeros
          const uint8_t* src = a.wr + ((size_t)(kb0 + blk) * BITS * a.Np + n0) * 16;
  #pragma unroll
          for (int v = 0; v < BITS; ++v)
            bulk_g2s(smem_u32(pk + ps * PKB + v * BN * 16), src + (size_t)v * a.Np * 16, BN * 16, pk_full(ps));
  #pragma unroll
          for (int c = 0; c < (FP8 ? 0 : 4); ++c)     // stored zeros of the block's chunks, 128 columns each
            bulk_g2s(smem_u32(pk + ps * PKB + PK_BYTES<BITS> + c * BN), a.z_r + (size_t)cg[4 * blk + c] * a.Np + n0,
                     BN, pk_full(ps));
          ++pk_issued;
        }
        for (int b = pk_issued > PS ? pk_issued - PS : 0; b < pk_issued; ++b)
          if (!mbar_wait(pk_full(b % PS), (b / PS) & 1)) ok = false;
        if (!ok) report_timeout(a.err);
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      // The whole warp runs the schedule and every lane waits; one elected lane issues the MMAs and
      // commits as predicated instructions.  Group boundaries come from a register copy of gmask
      // (loaded one 32-chunk window ahead) and the waits only poison the limit, so nothing between
      // two MMAs depends on a shared-memory value.  Measured on sm_103a: this keeps tcgen05.mma at
      // its full rate, where the same loop run by lane 0 alone lost ~40%.
      {
        constexpr uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
        constexpr uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(BMX >> 3) << 17) | ((uint32_t)(BN >> 4) << 24);
        const uint32_t me = elect_one();
        uint64_t limit = kWaitLimitNs;
        uint32_t cur = gmask[0];
        uint32_t nxt = nwin > 1 ? gmask[1] : 0u;
        int gi = 0;                 // groups started so far; buffer gi % 2, its use gi / 2
        uint32_t fresh = 1;         // next MMA starts a group
        int xs = 0, ws = 0;
        uint32_t xph = 0, wph = 0;
        for (int i = 0; i < nhalf; ++i) {
          mbar_wait_poison(x_full(xs), xph, limit);
          mbar_wait_poison(w_full(ws), wph, limit);
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint64_t ad = smem_desc_sw128(ws_s + ws * W_BYTES);     // A: weights, 128 rows
          const uint64_t bd = smem_desc_sw128(xs_s + xs * XB);          // B: x, BMX rows
  #pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * i + cc;
            if ((c & 31) == 0 && c > 0) {
              cur = nxt;
              nxt = (c >> 5) + 1 < nwin ? gmask[(c >> 5) + 1] : 0u;
            }
            const int b = gi & (NP_ - 1);
            if (fresh && gi >= NP_) {
              mbar_wait_poison(p_empty(b), ((gi / NP_) - 1) & 1, limit);
              asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            }
            const uint32_t d = tmem + (uint32_t)(b * BMX);
            umma_f16_if(d, ad + 4 * cc, bd + 4 * cc, idesc, fresh ^ 1u, me);
            umma_f16_if(d, ad + 4 * cc + 2, bd + 4 * cc + 2, idesc, 1u, me);
            const uint32_t end = (cur >> (c & 31)) & 1u;
            umma_commit_if(p_full(b), end & me);
            gi += (int)end;
            fresh = end;
          }
          umma_commit_if(x_empty(xs), me);
          umma_commit_if(w_empty(ws), me);
          if (++xs == XS) { xs = 0; xph ^= 1u; }
          if (++ws == WS) { ws = 0; wph ^= 1u; }
        }
        // every MMA must have landed before tensor memory is released
        // (after a timeout the issued MMAs still complete -- they only read shared memory -- so the
        // drain takes a fresh limit: tensor memory must never be freed under an MMA in flight)
        umma_commit_if(mma_done, me);
        uint64_t drain = kWaitLimitNs;
        mbar_wait_poison(mma_done, 0, drain);
        if ((limit == 0 || drain == 0) && me) report_timeout(a.err);
      }
    } else if (warp >= kDqWarp0 && warp < kDqWarp0 + kDq) {
      // ---------------- dequantisers: thread owns weight row n0 + nrow ----------------
      const int nrow = 32 * (warp - kDqWarp0) + lane;
      const uint32_t zoff = (uint32_t)a.zoff;
      uint32_t zq[4];
      for (int blk = 0; blk < nblocks && ok; ++blk) {
        const int ps = blk % PS;
        if (!mbar_wait(pk_full(ps), (blk / PS) & 1)) { ok = false; break; }
        const uint8_t* stage = pk + ps * PKB;
        if constexpr (!FP8) {
  #pragma unroll
          for (int c = 0; c < 4; ++c) zq[c] = prep_zero_l<T, BITS>(stage[PK_BYTES<BITS> + c * BN + nrow], zoff);
        }
        for (int h = 0; h < 2; ++h) {
          const int i = 2 * blk + h, ws = i % WS;
          if (i >= WS && !mbar_wait(w_empty(ws), ((i / WS) - 1) & 1)) { ok = false; break; }
          Words<BITS> lw[4] = {};
  #pragma unroll
          for (int t = 0; t < 4; ++t) half_words<BITS>(lw[t], stage, nrow, t, h);
          uint8_t* row = base + S::w + ws * W_BYTES + nrow * 128;
  #pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * h + cc;
  #pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint4 o;
              if constexpr (FP8) {   // pairs 4c .. 4c + 3: words 2c, 2c + 1, halves 0 and 1
                o.x = fp8_pair<T>(lw[t].w[2 * c], 0);
                o.y = fp8_pair<T>(lw[t].w[2 * c], 1);
                o.z = fp8_pair<T>(lw[t].w[2 * c + 1], 0);
                o.w = fp8_pair<T>(lw[t].w[2 * c + 1], 1);
              } else {
                o.x = code_minus_zero<T, BITS>(lw[t], 4 * c + 0, zq[c]);
                o.y = code_minus_zero<T, BITS>(lw[t], 4 * c + 1, zq[c]);
                o.z = code_minus_zero<T, BITS>(lw[t], 4 * c + 2, zq[c]);
                o.w = code_minus_zero<T, BITS>(lw[t], 4 * c + 3, zq[c]);
              }
              const int j = 4 * cc + t;                         // 16-byte chunk (8 k) inside the 64-k row
              *reinterpret_cast<uint4*>(row + ((j ^ (nrow & 7)) << 4)) = o;
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(w_full(ws));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(pk_empty(ps));           // both halves of this block are written
      }
      if (!ok) report_timeout(a.err);
    }
    if (a.split > 1) {   // the cluster's two barriers around the scalers' reduction of the partials
      cluster_sync_l();
      cluster_sync_l();
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kCols) : "memory");
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

template <int BITS, int BMX> size_t large_smem_bytes(int Kr) {
  return 1024 + LargeSmem<BITS, BMX>::cg + (size_t)(Kr / 32) * 4 + (size_t)((Kr / 32 + 31) / 32) * 4;
}

// x rows per tile: the smallest of 64, 128, 256 that covers M (and 256 above it)
inline int bmx_for(int M) { return M <= 64 ? 64 : M <= 128 ? 128 : 256; }

template <int BITS> size_t smem_at(int bmx, int Kr) {
  return bmx == 64 ? large_smem_bytes<BITS, 64>(Kr) : bmx == 128 ? large_smem_bytes<BITS, 128>(Kr)
                                                                  : large_smem_bytes<BITS, 256>(Kr);
}
inline size_t smem_bits(int bits, int bmx, int Kr) {
  return bits == 2 ? smem_at<2>(bmx, Kr) : bits == 3 ? smem_at<3>(bmx, Kr) : bits == 4 ? smem_at<4>(bmx, Kr)
                                                                                    : smem_at<8>(bmx, Kr);
}
// The x tile used at M: bmx_for(M), narrowed while the chunk tables of a very long K leave its
// rings no room (the narrower tiles have smaller x rings); 0 if even 64 rows do not fit.
inline int large_bmx(const Handle& h, int M) {
  int bmx = bmx_for(M);
  while (bmx > 64 && smem_bits(h.bits, bmx, h.Kr) > 227 * 1024) bmx /= 2;
  return smem_bits(h.bits, bmx, h.Kr) <= 227 * 1024 ? bmx : 0;
}

}  // namespace

// K split of the large-M kernel at M: the number of ranges s (1 .. 8, each of at least 8 blocks)
// with the smallest estimated time waves(s) * (t0 + t_k / s + t_red(s)), where waves(s) =
// ceil(tiles / clusters of s CTAs that run at once), t_k is one CTA's pass over all of K (~700 / 800
// / 950 cycles per 64-k stage at 64 / 128 / 256 x rows, at 1.9 GHz), t0 ~3 us a CTA's fixed start
// and drain, and t_red the cluster's reduction (two cluster barriers, ~0.8 us, and each CTA's read of
// one slice from every range, ~150 GB/s).  A grid with fewer tiles than SMs, or a mostly empty last
// wave, gains.  No workspace: the partials stay in the cluster's shared memory.
int large_split(const Handle& h, int M) {
  const int bmx = M > 0 ? large_bmx(h, M) : 0;
  if (bmx == 0) return 1;
  const long tiles = (long)((M + bmx - 1) / bmx) * (h.Np / BN);
  const int nb = h.Kr / 128;
  const double stage_cycles = bmx == 64 ? 700.0 : bmx == 128 ? 800.0 : 950.0;
  const double t_k = (h.Kr / 64) * stage_cycles / 1.9e3;          // us
  const double t0 = 3.0;
  auto cost = [&](int s) {
    const long slots = s > 1 ? whole_sm_clusters(h, s) : h.sm_count;
    const double waves = (double)((tiles + slots - 1) / slots);
    const double red = s > 1 ? 0.8 + (double)std::min(M, bmx) * BN * 4 / 150e3 : 0.0;
    return waves * (t0 + t_k / s + red);
  };
  int best = 1;
  double best_cost = cost(1);
  for (int s = 2; s <= 8 && nb / s >= 8; ++s) {
    if (whole_sm_clusters(h, s) < 1) continue;   // no cluster of s CTAs fits the GPU
    if (cost(s) < best_cost * 0.95) {
      best = s;
      best_cost = cost(s);
    }
  }
  return best;
}

namespace {

template <typename T, int BITS, int BMX, bool FP8>
cudaError_t launch_tbm(const Handle& h, const CUtensorMap& map, void* y, int M, cudaStream_t st) {
  const size_t smem = large_smem_bytes<BITS, BMX>(h.Kr);
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  auto kern = k_gemm_large<T, BITS, BMX, FP8>;
  // setmaxnreg redistributes the registers the block is launched with; a launch with fewer than
  // kRegsLaunch a thread could never satisfy the scalers' increase, so refuse it.
  static const int regs = [&] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.numRegs : -1;
  }();   // one per instantiation
  if (regs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int split = large_split(h, M);
  LargeArgs args{h.wr, h.cgid, h.s_r, h.z_r, y, h.err, M, h.N, h.Np, h.Kr, h.G, h.zoff, h.has_bias ? h.bias : nullptr,
                 h.scale_inv, h.kb, split};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + BMX - 1) / BMX, h.Np / BN, split);  // consecutive CTAs share a weight tile
  cfg.blockDim = dim3(kThreadsL);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;   // K split: a tile's ranges form one cluster
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = (unsigned)split;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, args, map);
}

template <typename T, int BITS, bool FP8 = false>
cudaError_t launch_tb(const Handle& h, const CUtensorMap& map, void* y, int M, cudaStream_t st) {
  switch (large_bmx(h, M)) {
    case 64: return launch_tbm<T, BITS, 64, FP8>(h, map, y, M, st);
    case 128: return launch_tbm<T, BITS, 128, FP8>(h, map, y, M, st);
    default: return launch_tbm<T, BITS, 256, FP8>(h, map, y, M, st);
  }
}

template <typename T>
cudaError_t launch_t(const Handle& h, const CUtensorMap& map, void* y, int M, cudaStream_t st) {
  if (h.fp8) return launch_tb<T, 8, true>(h, map, y, M, st);
  switch (h.bits) {
    case 2: return launch_tb<T, 2>(h, map, y, M, st);
    case 3: return launch_tb<T, 3>(h, map, y, M, st);
    case 4: return launch_tb<T, 4>(h, map, y, M, st);
    default: return launch_tb<T, 8>(h, map, y, M, st);
  }
}

}  // namespace

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

bool large_m_available() { return true; }

int large_m_launches(const Handle& h, int M) { return M > 0 ? (h.identity ? 1 : 2) : 0; }

bool large_m_plan_info(const Handle& h, int M, gptq_plan_t* out) {
  const int bmx = M > 0 ? large_bmx(h, M) : 0;
  if (bmx == 0) return false;
  const int split = large_split(h, M);
  out->path = GPTQ_PATH_LARGE_M;
  out->launches = large_m_launches(h, M);
  out->grid = (M + bmx - 1) / bmx * (h.Np / BN) * split;
  out->threads = kThreadsL;
  out->smem_bytes = (int)smem_bits(h.fp8 ? 8 : h.bits, bmx, h.Kr);
  out->consumer_warps = kDqWarps;
  out->m_tiles = bmx;
  out->act_order_in_kernel = 0;
  out->k_splits = split;
  out->k_panels = 1;
  out->stages = bmx == 256 ? 3 : 4;
  return true;
}

cudaError_t launch_gemm_large(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  const int bmx = large_bmx(h, M);
  if (bmx == 0) return cudaErrorInvalidConfiguration;
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
  const cuuint32_t box[2] = {HK, (cuuint32_t)bmx};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = h.dtype == GPTQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (enc(&map, dt, 2, const_cast<void*>(src), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (h.dtype == GPTQ_BF16) return launch_t<__nv_bfloat16>(h, map, y, M, st);
  return launch_t<__half>(h, map, y, M, st);
}

}  // namespace gptq

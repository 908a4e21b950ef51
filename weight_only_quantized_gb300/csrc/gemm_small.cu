// Small-M GEMM (decode, M <= 32): a persistent weight stream at HBM speed.
//
// mlinterviewnotes "Formats and kernels: FP8, INT8, INT4, Marlin, Machete": at small M the
// call time is set by the bytes of the packed weights (opening section); the quantised weight only
// pays if it stays packed until the registers that feed the tensor core; a group scale cannot be
// hoisted out of the k reduction (section on the LOP3 dequant and the scale); for tiny M the lever
// is every SM streaming weights at once, with the skinny operand in the MMA's N slot (swap-AB,
// section "Where the batch-size crossover is" and the M-bucketed dispatch discussion).
//
// Design on sm_103a:
//  * One CTA per SM, each owning a balanced run of 32-column tiles.  For every tile it streams
//    the 128-row blocks of packed codes, four blocks per 2-D TMA box (8 KB at 4 bits; smaller
//    copies were issue-bound), into a ring of stages several tens of KB deep, with an evict-first
//    L2 policy.  One producer warp issues the copies; 8 or 16 consumer warps take the blocks of a
//    tile round robin.
//  * Programmatic dependent launch: the producer starts the weight stream (handle-owned data),
//    and only then waits (griddepcontrol.wait) for the previous grid before it copies x; the
//    consumers write y only after x has arrived.  A short CTA needs at most half an SM, so the
//    next call's CTAs start streaming while this call finishes.
//  * x is staged per K-panel (all of K when it fits) by bulk copies into rows 64 bytes apart
//    modulo 128, so a lane's fragment loads meet no other lane on their banks.  With act-order,
//    x is put in sorted k order by the consumers from a copy of the caller's rows (M <= 2) or by
//    a small gather kernel into the handle's workspace.
//  * Zeros and scales come from a tile-major copy of the runtime layout (per tile and group 32
//    zero bytes and 32 scales, permuted so that the four columns of a lane are adjacent): one
//    bulk copy per tile and panel, then two shared loads per lane per block.
//  * mma.sync.m16n8k16 with swap-AB: A = weights (16 output features x 16 k), B = x^T (16 k x 8
//    batch rows), fp32 accumulators.  The codes go in as the exact values magic + code (one LOP3
//    per pair of codes; fp16 1024 + q, bf16 128 + q) and the zero comes out once per block in fp32
//    against the sum of x; the group scale multiplies that fp32 partial sum.  8-bit codes with bf16
//    go through the 2^23 fp32 magic, because bf16 holds 128 + q exactly only for q < 128.
//  * FP8 block-scaled layers (template FP8): the e4m3 bytes of a pair sit side by side in the
//    layout, one cvt.rn.f16x2.e4m3x2 makes the operand (plus an exact shift and multiply for bf16),
//    no zero fold, and the 128 x 128 block's factor multiplies the partial sum.
//  * Very long K (template XS false): when the per-block x-sum table does not fit shared memory the
//    planner takes 8 consumer warps, smaller K panels and recomputes the x sums for every tile.
//  * K split (template SPLIT), for layers with fewer 32-column tiles than SMs at M <= 8 and for
//    layers whose x over all of K does not fit shared memory at M = 9 .. 16: the CTAs of a
//    thread-block cluster take the K panels of a tile (or of a run of tiles), each stages x of its
//    panel once, and the first CTA adds up the others' tile sums, sent into its shared memory by
//    st.async.
//  * Every wait is bounded; a timeout sets the handle's error word, and the CTA drains its copies
//    and exits.
// This file is compiled twice: as itself (fp16 layers, the plan queries and the cluster count) and,
// through gemm_small_bf16.cu with GPTQ_SMALL_BF16_UNIT, for bf16 layers, so that the two halves of
// the kernel instantiations build in parallel.
#include "internal.cuh"

#include <algorithm>
#include <cstring>
#include <type_traits>

namespace gptq {
namespace {

// Consumer warps CW: 16 when a CTA streams a long run of tiles (the dequant chains are
// latency-bound and more warps hide more), 8 when the CTA is short and should leave room on the SM
// for the next call's CTA, and 8 at M > 8 (twice the accumulators).  Plus one producer warp.
template <int CW> __host__ __device__ constexpr int threads_of() { return (CW + 1) * 32; }
constexpr int kTileN = 32;                   // output features per tile
constexpr int kZsRow = 96;                   // bytes of one (tile, group) row of zst
constexpr int kSmemHalf = 110 * 1024;        // two CTAs (consecutive calls) share an SM
constexpr int kSmemFull = 227 * 1024;
constexpr int kXSmall = 24 * 1024;           // x for all of K up to this size: half an SM
constexpr int kXSingle = 136 * 1024;         // up to this size: x staged once, a whole SM
constexpr int kXPanel = 64 * 1024;           // otherwise per K-panel of this size, double buffered
constexpr uint64_t kWaitNs = 2000000000ull;

template <typename T> struct Magic;
template <> struct Magic<__half> { static constexpr uint32_t bits = 0x6400u; };
template <> struct Magic<__nv_bfloat16> { static constexpr uint32_t bits = 0x4300u; };

// One stage = kSmallBlocksPerBox 128-row blocks of one 32-column tile, copied densely by a single
// TMA box: block u's vector v (32 columns) at (u * BITS + v) * 512, column order rotated per
// vector by the runtime layout so that the consumers' reads are free of bank conflicts.  Boxes of
// one block (2 KB at 4 bits) left the stream limited by copies in flight; four blocks are 8 KB.
constexpr int kSPB = kSmallBlocksPerBox;
template <int BITS> __host__ __device__ constexpr int stage_bytes() { return kSPB * BITS * 512; }

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

// D = A * B (no accumulator input): the first MMA of a block's partial sums.
template <typename T>
__device__ __forceinline__ void mma16816_z(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  if constexpr (std::is_same<T, __half>::value)
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
                 : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  else
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
                 : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
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

// 1 in exactly one lane of the (converged) warp.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred;
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 8-bit codes with bf16 activations go through fp32; every other case uses the fp16/bf16 magic.
template <typename T, int BITS> constexpr bool kViaF32 = BITS == 8 && std::is_same<T, __nv_bfloat16>::value;

// Zero point (stored + zoff) in the form operand() subtracts: 2^23 + z as fp32 bits, exact.
template <typename T, int BITS>
__device__ __forceinline__ uint32_t prep_zero(uint32_t stored, uint32_t zoff) {
  static_assert(kViaF32<T, BITS>, "the subtract form serves 8-bit codes with bf16 only");
  return __float_as_uint(8388608.0f + (float)(stored + zoff));
}

// Codes go into the MMA as the exact values magic + code (bf16 128 + q, fp16 1024 + q) and the
// zero is taken out once per group in fp32: sum_k x (q - z) = sum_k x (magic + q) - (magic + z) sum_k x,
// with sum_k x from one extra MMA against an all-ones operand.  Products stay exact; the
// subtraction cancels at most ~11 of fp32's 24 bits, far inside the 4e-3 relative budget, and the
// per-pair packed subtract (half-rate fp16 pipe) disappears.  Not for 8-bit codes with bf16, whose
// 128 + q is not exact.
template <typename T, int BITS> constexpr bool kFoldZero = !kViaF32<T, BITS>;
template <typename T> constexpr float kMagicF = std::is_same<T, __nv_bfloat16>::value ? 128.0f : 1024.0f;
template <typename T> constexpr uint32_t kOnes2 = std::is_same<T, __nv_bfloat16>::value ? 0x3F803F80u : 0x3C003C00u;

// Lane words of one (block, column) for this lane: BITS words (bits 3: 2 words of the 2-bit plane
// then 1 word of the 1-bit plane).
template <int BITS> struct LaneWords { uint32_t w[BITS]; };

// (code - zero) of pair p of this lane as a bf16x2 register (low half = even k of the pair), exact:
// 8-bit codes with bf16 (128 + q is not exact in bf16, so the fold-zero form does not apply); the
// codes become 2^23 + q in fp32, the zero comes off there, and the integer rounds exactly to bf16.
template <typename T, int BITS>
__device__ __forceinline__ uint32_t operand(const LaneWords<BITS>& lw, int p, uint32_t zq) {
  static_assert(kViaF32<T, BITS>, "the subtract form serves 8-bit codes with bf16 only");
  const uint32_t codes = (lw.w[p / 2] >> (8 * (p % 2))) & 0x00FF00FFu;
  const float zf = __uint_as_float(zq);
  const float lo = __uint_as_float(0x4B000000u | (codes & 0xFFFFu)) - zf;
  const float hi = __uint_as_float(0x4B000000u | (codes >> 16)) - zf;
  return pack_bf16x2(lo, hi);
}

// magic + code of pair p (both halves), exact (the kFoldZero form).
template <typename T, int BITS>
__device__ __forceinline__ uint32_t operand_raw(const LaneWords<BITS>& lw, int p) {
  constexpr uint32_t M2 = Magic<T>::bits * 0x00010001u;
  if constexpr (BITS == 4 && std::is_same<T, __half>::value) {
    // fp16 holds 10 mantissa bits, so the odd nibbles need no shift: masked in place they read as
    // 1024 + 16 q, and one exact fma (x 1/16 + 960) makes 1024 + q; one shift by 8 serves the
    // upper two nibbles.  Per word one shift instead of three (the integer pipe is the busy one).
    const uint32_t w = (p % 4) < 2 ? lw.w[p / 4] : (lw.w[p / 4] >> 8);
    if ((p % 2) == 0) return and_or(w, 0x000F000Fu, M2);
    const uint32_t v = and_or(w, 0x00F000F0u, M2);
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(v), "r"(0x2C002C00u), "r"(0x63806380u));
    return d;
  } else if constexpr (BITS == 3) {
    const uint32_t lo = and_or(lw.w[p / 8] >> (2 * (p % 8)), 0x00030003u, M2);
    const uint32_t hi = p <= 2 ? (lw.w[2] << (2 - p)) : (lw.w[2] >> (p - 2));
    return and_or(hi, 0x00040004u, lo);
  } else {
    constexpr int F = 16 / BITS;
    constexpr uint32_t mask = ((1u << BITS) - 1u) * 0x00010001u;
    return and_or(lw.w[p / F] >> (BITS * (p % F)), mask, M2);
  }
}

// Byte offsets, inside one block of a stage, of this lane's words: vector v of column c sits at
// v * 512 + 16 * code_col_pos(c).  Lane (g, t) owns columns g + 8 idx, idx = 0..3, and lane t's
// words (4-bit: vector t; 8-bit: vectors 2t, 2t+1; 2-bit: half t%2 of vector t/2; 3-bit: that,
// plus word t of the 1-bit-plane vector 2).  Lane constants, computed once.
template <int BITS> struct LaneOffsets { int o[4]; int o2[4]; };
template <int BITS>
__device__ __forceinline__ LaneOffsets<BITS> lane_offsets(int g, int t) {
  LaneOffsets<BITS> L;
  auto at = [&](int v, int c) { return v * 512 + code_col_pos(BITS, v, c) * 16; };
#pragma unroll
  for (int idx = 0; idx < 4; ++idx) {
    const int c = g + 8 * idx;
    if constexpr (BITS == 4) { L.o[idx] = at(t, c); L.o2[idx] = 0; }
    else if constexpr (BITS == 8) { L.o[idx] = at(2 * t, c); L.o2[idx] = at(2 * t + 1, c); }
    else if constexpr (BITS == 2) { L.o[idx] = at(t >> 1, c) + 8 * (t & 1); L.o2[idx] = 0; }
    else { L.o[idx] = at(t >> 1, c) + 8 * (t & 1); L.o2[idx] = at(2, c) + 4 * t; }
  }
  return L;
}
template <int BITS>
__device__ __forceinline__ void read_block(LaneWords<BITS> (&lw)[4], const uint8_t* blk, const LaneOffsets<BITS>& L) {
#pragma unroll
  for (int idx = 0; idx < 4; ++idx) {
    if constexpr (BITS == 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(blk + L.o[idx]);
      lw[idx].w[0] = v.x; lw[idx].w[1] = v.y; lw[idx].w[2] = v.z; lw[idx].w[3] = v.w;
    } else if constexpr (BITS == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(blk + L.o[idx]);
      lw[idx].w[0] = v.x; lw[idx].w[1] = v.y;
    } else if constexpr (BITS == 8) {
      const uint4 v0 = *reinterpret_cast<const uint4*>(blk + L.o[idx]);
      const uint4 v1 = *reinterpret_cast<const uint4*>(blk + L.o2[idx]);
      lw[idx].w[0] = v0.x; lw[idx].w[1] = v0.y; lw[idx].w[2] = v0.z; lw[idx].w[3] = v0.w;
      lw[idx].w[4] = v1.x; lw[idx].w[5] = v1.y; lw[idx].w[6] = v1.z; lw[idx].w[7] = v1.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(blk + L.o[idx]);
      lw[idx].w[0] = v.x; lw[idx].w[1] = v.y;
      lw[idx].w[2] = *reinterpret_cast<const uint32_t*>(blk + L.o2[idx]);
    }
  }
}

// One 2-D TMA box (global -> this CTA's shared memory), completing its bytes on an mbarrier, with
// an L2 cache policy (the weight stream is read once per call: evict first, so that it does not
// push the activations, tables and outputs that the next calls reuse out of L2).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar,
                                            uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
               :: "r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar), "l"(policy) : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Launch parameters (one plan per handle and M, cached on the host).
struct SmallArgs {
  const uint8_t* wr; const int32_t* cgid; const uint8_t* zst;
  const uint16_t* x; void* y; int32_t* err;
  int ldx;          // row stride of x (elements): K for the caller's x, Kr for the gathered copy
  int M, N, Np, Kr, G;
  int ntiles;       // 32-column tiles holding at least one column < N
  int pb;           // 128-row blocks per K-panel
  int npanel;
  int single;       // 1: one panel covers K, x is staged once per CTA
  int lg_rd;        // log2 of the stages in the weight ring (a power of two: slot and phase by mask and shift)
  int span_max;     // rows of a zero/scale table (groups of one panel)
  int x_row;        // bytes of one staged x row: pb * 256 + 64 (rows 64 bytes apart mod 128)
  int o_x, o_zs, o_red, o_cg, o_bar;   // shared-memory offsets; the ring starts at 0
  int o_xs;         // x sums of the single-group blocks [NB][8 MT8] (fp32)
  // act-order with x staged once and M <= 2: the producer copies the caller's x rows and perm
  // into shared memory and the consumers permute x there (no pre-pass launch)
  const int32_t* perm;
  int gather;
  int o_pm;         // int32 [Kr] copy of perm (-1: pad row)
  int o_raw;        // the caller's x rows, [M][K] as given
  int cg_async;     // 1: the producer bulk-copies the chunk-group table (CTAs that own a whole SM, whose
                    // start is not hidden behind the previous call); 0: every thread loads it at start
  int zoff;         // zero = stored byte + zoff (1: GPTQ v1 fields, stored minus one; 0: gptq_v2, AWQ)
  const float* bias;   // [Np] float32 added to y, or nullptr
  uint64_t wait_ns; // limit of every bounded wait
  int stall;        // test hook: the producer issues no copy, so every wait runs into its limit
  int o_recv;       // SPLIT: two receive slots in the first CTA of a cluster for the other CTAs'
                    // tile sums, [2][panels - 1][M][32] floats, then its own sums [2][M][32]
};

// Thread-block cluster helpers (the K-split kernels).
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// The shared::cluster address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_addr), "r"(rank));
  return d;
}
// Arrive on an mbarrier of another CTA of the cluster, relaxed: no fence.  The caller issues it after
// a barrier of the CTA's threads that read the slot being freed, and bar.sync completes their
// shared-memory loads (their values are bound before it), so the other CTA's next writes into the
// slot cannot reach a read.  A release arrive at cluster scope cost ~0.5 us per tile here.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
// Bounded parity wait on this CTA's mbarrier for a phase that another CTA of the cluster completes
// (acquire at cluster scope).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(r) : "r"(bar), "r"(parity) : "memory");
  return r != 0u;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cluster(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}
// 16 bytes into another CTA's shared memory, completing on that CTA's mbarrier.
__device__ __forceinline__ void st_async_f4(uint32_t dst, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               :: "r"(dst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar) : "memory");
}

template <int CW>
__device__ __forceinline__ void named_sync_consumers() {
  asm volatile("bar.sync 1, %0;" :: "n"(CW * 32) : "memory");
}

// XS: the x sums of the CTA's first tile are kept (a table of NB * 8 * MT8 floats) for its later
// tiles; false only in the layouts for very long K, where shared memory cannot hold the table.
// SPLIT: the CTA walks one K panel (blockIdx.y) of each tile of its run, x of that panel staged
// once; the panels form a thread-block cluster, and the first CTA adds up the others' sums.
template <typename T, int BITS, int MT8, int CW, bool GATHER, bool FP8, bool XS = true, bool SPLIT = false>
__global__ void __launch_bounds__(threads_of<CW>(), (CW == 8 && MT8 == 1) ? 2 : 1) k_gemm_small(const SmallArgs a, const __grid_constant__ CUtensorMap wmap) {
  static_assert(!FP8 || (BITS == 8 && !GATHER), "FP8 layers: 8-bit layout, x staged without gather");
  // the zero fold applies to integer codes; FP8 weights are their own values
  constexpr bool kFZ = kFoldZero<T, BITS> && !FP8;
  constexpr int kCW = CW;
  constexpr int kThreadsS = threads_of<CW>();
  constexpr int SB = stage_bytes<BITS>();
  constexpr int RS = kTileN + 4;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // TMA boxes land on 128-byte boundaries
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NB = a.Kr / 128;
  // Tile runs of ntiles / grid or one more; the first (ntiles % grid) CTAs take the longer runs.
  // A CTA that needs a whole SM starts only when the previous call's CTA there has left, and CTAs
  // start in index order as SMs free up, so the CTAs that start last have the shorter runs (the
  // 70B gate layer at M = 1: 27.5 -> 26.5 us against runs spread evenly over the indices; kept as
  // plain register arithmetic, since this kernel sits at its register limit).
  const int t_base = a.ntiles / (int)gridDim.x, t_extra = a.ntiles % (int)gridDim.x;
  const int T0 = (int)blockIdx.x * t_base + min((int)blockIdx.x, t_extra);
  const int T1 = T0 + t_base + ((int)blockIdx.x < t_extra ? 1 : 0);
  const int lg = a.lg_rd, rd = 1 << lg;

  uint8_t* ring = smem;
  uint8_t* xreg = smem + a.o_x;
  uint8_t* zsreg = smem + a.o_zs;
  float* red = reinterpret_cast<float*>(smem + a.o_red);
  float* xsb = reinterpret_cast<float*>(smem + a.o_xs);
  int32_t* cg = reinterpret_cast<int32_t*>(smem + a.o_cg);
  const uint32_t bar0 = smem_u32(smem + a.o_bar);
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (rd + i); };
  auto hfull = [&](int i) { return bar0 + 8u * (2 * rd + i); };
  auto hempty = [&](int i) { return bar0 + 8u * (2 * rd + 2 + i); };
  const uint32_t cgfull = bar0 + 8u * (2 * rd + 4);   // the chunk-group table has landed
  // SPLIT: receive slot s of the first CTA is full (the other CTAs' sums of one tile have landed),
  // and, in every other CTA, slot s of the first CTA is free again
  auto rbar = [&](int s) { return bar0 + 8u * (2 * rd + 5 + s); };
  auto sfree = [&](int s) { return bar0 + 8u * (2 * rd + 7 + s); };
  // K panels this CTA walks: all of them, or (SPLIT) the one of blockIdx.y
  const int p_lo = SPLIT ? (int)blockIdx.y : 0;
  const int p_hi = SPLIT ? (int)blockIdx.y + 1 : a.npanel;
  const int32_t* pm = reinterpret_cast<const int32_t*>(smem + a.o_pm);
  uint8_t* rawx = smem + a.o_raw;
  const int zs_bytes = a.span_max * kZsRow;
  const int x_bytes = a.M * a.x_row;

  // Let the next grid on the stream launch; it waits for this one before touching our outputs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int i = 0; i < rd; ++i) { mbar_init(full(i), 1); mbar_init(empty(i), kSPB); }
    for (int i = 0; i < 2; ++i) { mbar_init(hfull(i), 1); mbar_init(hempty(i), kCW); }
    mbar_init(cgfull, 1);
    if constexpr (SPLIT && MT8 == 1) {
      // the first CTA of the cluster expects the other panels' sums of its tile
      mbar_init(rbar(0), 1);
      if (blockIdx.y == 0) mbar_arrive_expect_tx(rbar(0), (gridDim.y - 1) * (uint32_t)a.M * kTileN * 4u);
    } else if constexpr (SPLIT) {
      // the first CTA of the cluster expects the other panels' sums of its first two tiles (one
      // slot each) and re-arms a slot when it has added it up
      for (int sl = 0; sl < 2; ++sl) { mbar_init(rbar(sl), 1); mbar_init(sfree(sl), 1); }
      if (blockIdx.y == 0)
        for (int sl = 0; sl < 2 && sl < T1 - T0; ++sl)
          mbar_arrive_expect_tx(rbar(sl), (gridDim.y - 1) * (uint32_t)a.M * kTileN * 4u);
    }
    fence_mbar_init();
  }
  // A CTA that owns a whole SM starts only when the previous call's CTA there has left, so its
  // chunk-group table comes in by one bulk copy from the producer (below) and the weight stream
  // starts without a global round trip first; a half-SM CTA starts beside the previous call's and
  // loads the table directly.
  if (!a.cg_async)
    for (int i = tid; i < NB * 4; i += kThreadsS) cg[i] = __ldg(&a.cgid[i]);
  __syncthreads();
  // every thread of the cluster arrives once here (after the barrier inits, which the release
  // publishes to the cluster) and waits once before it exits or touches another CTA's memory
  if constexpr (SPLIT) cluster_arrive();

  // Blocks of panel p, and the first group a panel touches (cgid ascends in the sorted order).
  auto panel_blocks = [&](int p) { return min(NB, (p + 1) * a.pb) - p * a.pb; };

  if (warp == kCW) {
    // ---------------- producer ----------------
    // The whole warp runs the schedule and waits; one elected lane issues.  Nothing between two
    // copies branches on a shared-memory value: the waits only poison the limit (an early-exit
    // branch on a wait result made each issue wait for the previous copy, ~4x slower here).
    uint32_t go = elect_one();
    if (a.stall) go = 0u;
    const uint64_t stream_policy = l2_evict_first();
    uint64_t limit = a.wait_ns;
    bool waited = false;            // griddepcontrol.wait done (x may be the previous grid's output)
    int s_issued = 0;               // weight stages issued
    int q = 0;                      // segments (tile, panel) started
    int s_sent = 0, q_sent = 0;     // stages and segment headers actually issued
    if (a.cg_async && go) {         // handle data, independent of the previous grid
      mbar_arrive_expect_tx(cgfull, (uint32_t)NB * 16u);
      bulk_g2s(smem_u32(cg), a.cgid, (uint32_t)NB * 16u, cgfull);
    }
    const bool cg_sent = a.cg_async && go != 0;

    for (int ti = T0; ti < T1; ++ti) {
      for (int p = p_lo; p < p_hi; ++p, ++q) {
        const int nb = panel_blocks(p);
        const int hs = q & 1;
        if (q >= 2) mbar_wait_poison(hempty(hs), ((q >> 1) - 1) & 1, limit);
        go &= limit != 0 ? 1u : 0u;   // after a timeout nothing more is issued
        const int nst = (nb + kSPB - 1) / kSPB;
        int j = 0;
        auto issue_stage = [&](int l) {
          const int s = s_issued;
          const int slot = s & (rd - 1);
          if (s >= rd) mbar_wait_poison(empty(slot), (uint32_t)(((s >> lg) - 1) & 1), limit);
          go &= limit != 0 ? 1u : 0u;
          if (go) {
            mbar_arrive_expect_tx(full(slot), (uint32_t)SB);
            // box: the kSPB * BITS vector rows from block p * pb + kSPB * l on, tile ti's 512 bytes
            // (64 uint64) of each; rows past the last block read as zero
            tma_load_2d(smem_u32(ring + (size_t)slot * SB), &wmap, ti * 64, (p * a.pb + kSPB * l) * BITS, full(slot),
                        stream_policy);
          }
          s_sent += go ? 1 : 0;
          ++s_issued;
        };
        if (q == 0) {
          // weights of the first segment (up to 4 stages) need neither the table nor the previous
          // grid: they go out first
          const int pre = min(nst, min(rd, 4));
          for (; j < pre; ++j) issue_stage(j);
          if (a.cg_async) mbar_wait_poison(cgfull, 0u, limit);
          go &= limit != 0 ? 1u : 0u;
        }
        const int gf = cg[4 * p * a.pb], gl = cg[4 * (p * a.pb + nb) - 1];
        const bool load_x = !a.single || q == 0;
        const uint32_t zs_tx = (uint32_t)(gl - gf + 1) * kZsRow;
        // x bytes: the staged rows, or (gathering) perm and the caller's rows as given
        const uint32_t x_tx = !load_x ? 0u : GATHER ? (uint32_t)a.Kr * 4u + (uint32_t)a.M * a.ldx * 2u
                                                    : (uint32_t)a.M * nb * 256u;
        if (go) {
          mbar_arrive_expect_tx(hfull(hs), zs_tx + x_tx);
          bulk_g2s(smem_u32(zsreg + hs * zs_bytes), a.zst + ((size_t)ti * a.G + gf) * kZsRow, zs_tx, hfull(hs));
          if (GATHER && load_x)     // handle data, before the wait on the previous grid
            bulk_g2s(smem_u32(pm), a.perm, (uint32_t)a.Kr * 4u, hfull(hs));
        }
        q_sent += go ? 1 : 0;
        if (load_x) {
          // x waits for the previous grid
          if (!waited) { asm volatile("griddepcontrol.wait;" ::: "memory"); waited = true; }
          if (go) {
            if constexpr (GATHER) {
              for (int m = 0; m < a.M; ++m)
                bulk_g2s(smem_u32(rawx + (size_t)m * a.ldx * 2), a.x + (size_t)m * a.ldx, (uint32_t)a.ldx * 2u, hfull(hs));
            } else {
              uint8_t* xd = xreg + (a.single ? 0 : hs * x_bytes);
              for (int m = 0; m < a.M; ++m)
                bulk_g2s(smem_u32(xd + m * a.x_row), a.x + (size_t)m * a.ldx + (size_t)p * a.pb * 128,
                         (uint32_t)nb * 256u, hfull(hs));
            }
          }
        }
        for (; j < nst; ++j) issue_stage(j);
      }
    }
    // every copy issued must land before the CTA may exit.  Issue stops at the first timeout, so
    // the issued stages are the first s_sent (headers: q_sent), none overwriting an unconsumed
    // slot; the drain gets a fresh limit since the copies are reads of valid addresses.
    uint64_t drain = kWaitNs;
    const int first = s_sent > rd ? s_sent - rd : 0;
    for (int s = first; s < s_sent; ++s) mbar_wait_poison(full(s & (rd - 1)), (uint32_t)((s >> lg) & 1), drain);
    for (int qq = q_sent > 2 ? q_sent - 2 : 0; qq < q_sent; ++qq)
      mbar_wait_poison(hfull(qq & 1), (uint32_t)((qq >> 1) & 1), drain);
    if (cg_sent) mbar_wait_poison(cgfull, 0u, drain);
    if ((limit == 0 || drain == 0) && lane == 0) report_timeout(a.err);
    if constexpr (SPLIT) {
      cluster_wait();
      if constexpr (MT8 > 1)   // runs of tiles (one tile per cluster at M <= 8)
        if (T1 - T0 > 1) { cluster_arrive(); cluster_wait(); }   // the cluster's closing barrier
    }
    return;
  }

  // ---------------- consumers ----------------
  // Stages are dealt round robin over the eight warps across segments (stage s to warp s % 8).
  // Each warp keeps the current group's prepared zeros and scales and its partial sums, and folds
  // the partial sums into the total (times the scale) only when the group changes.
  const int g = lane >> 2, t = lane & 3;
  const LaneOffsets<BITS> LO = lane_offsets<BITS>(g, t);
  bool ok = true;
  bool waited = false;
  float acc[2][MT8][4], part[2][MT8][4];
  float xsp[MT8][4];               // kFoldZero: sum of x over the group so far (c0: column 2t, c1: 2t + 1)
  bool mval[MT8];
#pragma unroll
  for (int mt = 0; mt < MT8; ++mt) mval[mt] = 8 * mt + g < a.M;
  // this lane's x fragments: row 8 mt + g (row 0 when that row is absent), k offset 8 t inside
  // each 32-row chunk (the runtime layout's k order: lane t of 16-k step ks holds sorted rows
  // 4q .. 4q + 3, q = 8 (ks / 2) + 2 t + ks % 2)
  int xoff[MT8];
#pragma unroll
  for (int mt = 0; mt < MT8; ++mt) xoff[mt] = (mval[mt] ? 8 * mt + g : 0) * a.x_row + 16 * t;
  uint32_t zq[4];                  // prepared zero (the subtract form)
  float zc[4];                     // magic + zero in fp32 (the kFoldZero form)
  const float zsub = 8388608.0f - kMagicF<T> - (float)a.zoff;   // 2^23 + stored -> magic + zero
  float sc[4];
  // x sums of this lane's two batch columns (8 mt + 2t and + 1) over the chunks being folded
  float2 xsv[MT8];
  auto flush = [&](const bool rezero) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int mt = 0; mt < MT8; ++mt) {
        if constexpr (kFZ) {
          acc[i][mt][0] = fmaf(sc[2 * i], fmaf(-zc[2 * i], xsv[mt].x, part[i][mt][0]), acc[i][mt][0]);
          acc[i][mt][1] = fmaf(sc[2 * i], fmaf(-zc[2 * i], xsv[mt].y, part[i][mt][1]), acc[i][mt][1]);
          acc[i][mt][2] = fmaf(sc[2 * i + 1], fmaf(-zc[2 * i + 1], xsv[mt].x, part[i][mt][2]), acc[i][mt][2]);
          acc[i][mt][3] = fmaf(sc[2 * i + 1], fmaf(-zc[2 * i + 1], xsv[mt].y, part[i][mt][3]), acc[i][mt][3]);
        } else {
          acc[i][mt][0] = fmaf(sc[2 * i], part[i][mt][0], acc[i][mt][0]);
          acc[i][mt][1] = fmaf(sc[2 * i], part[i][mt][1], acc[i][mt][1]);
          acc[i][mt][2] = fmaf(sc[2 * i + 1], part[i][mt][2], acc[i][mt][2]);
          acc[i][mt][3] = fmaf(sc[2 * i + 1], part[i][mt][3], acc[i][mt][3]);
        }
        if (rezero)
#pragma unroll
          for (int r = 0; r < 4; ++r) part[i][mt][r] = 0.f;
      }
    if (rezero)
#pragma unroll
      for (int mt = 0; mt < MT8; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) xsp[mt][r] = 0.f;
  };
  if (a.cg_async && !mbar_wait(cgfull, 0u, a.wait_ns)) ok = false;   // the chunk-group table (no block runs without it)
  int s_base = 0;
  int q = 0;
  for (int ti = T0; ti < T1; ++ti) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int mt = 0; mt < MT8; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) { acc[i][mt][r] = 0.f; part[i][mt][r] = 0.f; xsp[mt][r] = 0.f; }
    for (int p = p_lo; p < p_hi; ++p, ++q) {
      const int nb = panel_blocks(p);
      const int hs = q & 1;
      if (ok && !mbar_wait(hfull(hs), (uint32_t)((q >> 1) & 1), a.wait_ns)) ok = false;
      if (GATHER && q == 0) {
        // x[m][perm[j]] from the copied rows into the staged rows (only after the copy of perm has
        // landed: after a timeout the indices would be garbage).  One warp per 128-row block, lane l
        // on the block's sorted rows 4l .. 4l + 3 (one 16-byte load of perm, one 8-byte store per x
        // row); the warp also sums the block's x per batch row into the x-sum table, so that no tile
        // needs the all-ones MMAs (columns of absent batch rows read row 0, as the fragments do).
        if (ok) {
          const int b0p = SPLIT ? p * a.pb : 0;     // blocks of this CTA's rows: all, or its panel's
          const int nbp = SPLIT ? nb : NB;
          const uint16_t* rx = reinterpret_cast<const uint16_t*>(rawx);
          for (int bl = warp; bl < nbp; bl += kCW) {
            const int b = b0p + bl;
            const int4 kk = *reinterpret_cast<const int4*>(pm + 128 * b + 4 * lane);
            float srow[2] = {0.f, 0.f};
            for (int m = 0; m < a.M; ++m) {
              const uint16_t* xr = rx + (size_t)m * a.ldx;
              const uint32_t v0 = kk.x >= 0 ? xr[kk.x] : 0u, v1 = kk.y >= 0 ? xr[kk.y] : 0u;
              const uint32_t v2 = kk.z >= 0 ? xr[kk.z] : 0u, v3 = kk.w >= 0 ? xr[kk.w] : 0u;
              *reinterpret_cast<uint2*>(xreg + m * a.x_row + 256 * bl + 8 * lane) =
                  make_uint2(v0 | (v1 << 16), v2 | (v3 << 16));
              float sm = (to_float<T>(v0) + to_float<T>(v1)) + (to_float<T>(v2) + to_float<T>(v3));
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
              srow[m & 1] = sm;
            }
            if (XS && lane < 8 * MT8) xsb[(size_t)b * (8 * MT8) + lane] = (lane == 1 && a.M == 2) ? srow[1] : srow[0];
          }
        }
        named_sync_consumers<kCW>();      // every consumer's share of x is in place
      }
      const uint8_t* xb = xreg + (a.single ? 0 : hs * x_bytes);
      const uint8_t* zs = zsreg + hs * zs_bytes;
      const int gf = cg[4 * p * a.pb];
      int cur = -1;                    // group whose zeros and scales are loaded
      const int nst = (nb + kSPB - 1) / kSPB;
      // block slot bs = kSPB * js + u of stage js goes to warp (kSPB * (s_base + js) + u) % kCW;
      // every slot's owner releases it once, also past the last block (the stage's empty barrier
      // counts kSPB arrivals)
      // The block loop in two compiled forms: during the CTA's first tile the x sums of the
      // single-group blocks come from the all-ones MMAs and are kept in a table; later tiles read
      // them (x is the same for every tile) and skip those MMAs.
      auto run_blocks = [&](auto reuse_tag) {
        constexpr bool kReuse = decltype(reuse_tag)::value && kFZ;
        for (int bs = (warp - kSPB * s_base) & (kCW - 1); bs < kSPB * nst && ok; bs += kCW) {
          const int js = bs / kSPB, u = bs % kSPB;
          const int s = s_base + js;
          const int slot = s & (rd - 1);
          const int lb = bs;
          const int b = p * a.pb + lb;
          // The block's groups and the zeros and scales of its first group are read before the
          // wait for its codes: they do not depend on the stage, so their load latency overlaps the
          // wait and the code loads.
          int g0 = 0, g3 = 0;
          uint32_t zw0 = 0;
          uint2 sw0 = make_uint2(0u, 0u);
          if (lb < nb) {
            g0 = cg[4 * b];
            g3 = cg[4 * b + 3];
            const uint8_t* zrow = zs + (g0 - gf) * kZsRow;
            zw0 = *reinterpret_cast<const uint32_t*>(zrow + 4 * g);
            sw0 = *reinterpret_cast<const uint2*>(zrow + 32 + 8 * g);
          }
          if (!mbar_wait(full(slot), (uint32_t)((s >> lg) & 1), a.wait_ns)) { ok = false; break; }
          if (lb >= nb) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(slot));
            continue;
          }
          {
            LaneWords<BITS> lw[4];
            read_block<BITS>(lw, ring + (size_t)slot * SB + u * BITS * 512, LO);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(slot));       // this block's words are in registers
            const uint8_t* xblk = xb + lb * 256;
            auto set_group = [&](const int gq, const uint32_t zw, const uint2 sw) {
              cur = gq;
#pragma unroll
              for (int idx = 0; idx < 4; ++idx) {
                if constexpr (FP8) {
                  // the block's float32 factor, one for all 32 columns of the tile, in every zero slot
                  (void)sw;
                  sc[idx] = __uint_as_float(zw);
                  continue;
                } else if constexpr (kFZ) {
                  // magic + stored zero + zoff in fp32: one byte permute builds 2^23 + stored (exact),
                  // one add moves it (exact: integers below 2^24)
                  zc[idx] = __uint_as_float(__byte_perm(zw, 0x4B000000u, 0x7440u + idx)) - zsub;
                } else {
                  zq[idx] = prep_zero<T, BITS>((zw >> (8 * idx)) & 0xFFu, (uint32_t)a.zoff);
                }
              }
              if constexpr (!FP8) {
                sc[0] = to_float<T>(sw.x & 0xFFFFu); sc[1] = to_float<T>(sw.x >> 16);
                sc[2] = to_float<T>(sw.y & 0xFFFFu); sc[3] = to_float<T>(sw.y >> 16);
              }
            };
            auto load_group = [&](const int gq) {
              const uint8_t* zrow = zs + (gq - gf) * kZsRow;
              set_group(gq, *reinterpret_cast<const uint32_t*>(zrow + 4 * g), *reinterpret_cast<const uint2*>(zrow + 32 + 8 * g));
            };
            auto chunk_mma = [&](const int c, const bool first, auto ones_tag) {
              constexpr bool kOnes = decltype(ones_tag)::value;
              // both 16-k steps of the chunk: one 16-byte load per m-tile (lanes of absent rows read
              // row 0; their columns of the product are never stored)
              uint4 xv[MT8];
#pragma unroll
              for (int mt = 0; mt < MT8; ++mt) xv[mt] = *reinterpret_cast<const uint4*>(xblk + xoff[mt] + 64 * c);
#pragma unroll
              for (int s2 = 0; s2 < 2; ++s2) {
                const int p0 = 4 * c + 2 * s2;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  uint32_t af[4];
                  if constexpr (FP8) {
                    af[0] = fp8_pair<T>(lw[2 * i].w[p0 / 2], p0 % 2);
                    af[1] = fp8_pair<T>(lw[2 * i + 1].w[p0 / 2], p0 % 2);
                    af[2] = fp8_pair<T>(lw[2 * i].w[(p0 + 1) / 2], (p0 + 1) % 2);
                    af[3] = fp8_pair<T>(lw[2 * i + 1].w[(p0 + 1) / 2], (p0 + 1) % 2);
                  } else if constexpr (kFZ) {
                    af[0] = operand_raw<T, BITS>(lw[2 * i], p0);
                    af[1] = operand_raw<T, BITS>(lw[2 * i + 1], p0);
                    af[2] = operand_raw<T, BITS>(lw[2 * i], p0 + 1);
                    af[3] = operand_raw<T, BITS>(lw[2 * i + 1], p0 + 1);
                  } else {
                    af[0] = operand<T, BITS>(lw[2 * i], p0, zq[2 * i]);
                    af[1] = operand<T, BITS>(lw[2 * i + 1], p0, zq[2 * i + 1]);
                    af[2] = operand<T, BITS>(lw[2 * i], p0 + 1, zq[2 * i]);
                    af[3] = operand<T, BITS>(lw[2 * i + 1], p0 + 1, zq[2 * i + 1]);
                  }
#pragma unroll
                  for (int mt = 0; mt < MT8; ++mt) {
                    if (first && s2 == 0) mma16816_z<T>(part[i][mt], af, xv[mt].x, xv[mt].y);
                    else mma16816<T>(part[i][mt], af, s2 ? xv[mt].z : xv[mt].x, s2 ? xv[mt].w : xv[mt].y);
                  }
                }
                if constexpr (kFZ && kOnes) {
                  const uint32_t ones[4] = {kOnes2<T>, kOnes2<T>, kOnes2<T>, kOnes2<T>};
#pragma unroll
                  for (int mt = 0; mt < MT8; ++mt) {
                    if (first && s2 == 0) mma16816_z<T>(xsp[mt], ones, xv[mt].x, xv[mt].y);
                    else mma16816<T>(xsp[mt], ones, s2 ? xv[mt].z : xv[mt].x, s2 ? xv[mt].w : xv[mt].y);
                  }
                }
              }
            };
            // Every block's partial sums are folded into the total at the block's end (per block or
            // per group change, the sum of scaled partials is the same), so no state crosses blocks.
            if (g0 == g3) {
              // one group for the whole block (cgid ascends): no branch between the chunks; the first
              // MMA starts the partial sums from zero
              if (g0 != cur) set_group(g0, zw0, sw0);
              if constexpr (kReuse) {
                // x sums of this block from the table written during the CTA's first tile (read
                // before the MMAs, so that the load is off the way to the flush)
#pragma unroll
                for (int mt = 0; mt < MT8; ++mt)
                  xsv[mt] = *reinterpret_cast<const float2*>(xsb + (size_t)b * (8 * MT8) + 8 * mt + 2 * t);
#pragma unroll
                for (int c = 0; c < 4; ++c) chunk_mma(c, c == 0, std::false_type{});
              } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) chunk_mma(c, c == 0, std::true_type{});
#pragma unroll
                for (int mt = 0; mt < MT8; ++mt) {
                  xsv[mt] = make_float2(xsp[mt][0], xsp[mt][1]);
                  if (kFZ && XS && g == 0)
                    *reinterpret_cast<float2*>(xsb + (size_t)b * (8 * MT8) + 8 * mt + 2 * t) = xsv[mt];
                }
              }
              flush(false);
            } else {
              bool pending = false;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int gq = cg[4 * b + c];
                if (gq != cur) {
                  if (pending) {
#pragma unroll
                    for (int mt = 0; mt < MT8; ++mt) xsv[mt] = make_float2(xsp[mt][0], xsp[mt][1]);
                    flush(false);
                  }
                  load_group(gq);
                  pending = false;
                }
                chunk_mma(c, !pending, std::true_type{});
                pending = true;
              }
#pragma unroll
              for (int mt = 0; mt < MT8; ++mt) xsv[mt] = make_float2(xsp[mt][0], xsp[mt][1]);
              flush(false);
            }
          }
        }
      };
      if constexpr (XS && GATHER) run_blocks(std::true_type{});   // the permute wrote the x-sum table
      else if (XS && ti > T0) run_blocks(std::true_type{});
      else run_blocks(std::false_type{});
      s_base += nst;
      __syncwarp();
      if (lane == 0) mbar_arrive(hempty(hs));
    }
    // ---- the eight warps' partial tiles meet in shared memory: red[w][m][n] ----
    named_sync_consumers<kCW>();               // the previous tile's sums have been read
    {
      float* rw = red + (size_t)warp * MT8 * 8 * RS;
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int mt = 0; mt < MT8; ++mt) {
          const int nl = 16 * i + g;
          const int ml = 8 * mt + 2 * t;
          rw[ml * RS + nl] = acc[i][mt][0];
          rw[(ml + 1) * RS + nl] = acc[i][mt][1];
          rw[ml * RS + nl + 8] = acc[i][mt][2];
          rw[(ml + 1) * RS + nl + 8] = acc[i][mt][3];
        }
    }
    named_sync_consumers<kCW>();
    if (!waited) { asm volatile("griddepcontrol.wait;" ::: "memory"); waited = true; }
    T* y = static_cast<T*>(a.y);
    // the CTA's sum of the tile: the warps' totals in warp order, per four columns
    auto tile_sum = [&](const int ml, const int cl) {
      float4 sum = *reinterpret_cast<const float4*>(&red[ml * RS + cl]);
#pragma unroll
      for (int w = 1; w < kCW; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(&red[(size_t)w * MT8 * 8 * RS + ml * RS + cl]);
        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
      }
      return sum;
    };
    auto store_y = [&](const int ml, const int n, float4 sum) {
      if (a.bias) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(a.bias + n));
        sum.x += b.x; sum.y += b.y; sum.z += b.z; sum.w += b.w;
      }
      uint2 o;
      o.x = pack2<T>(sum.x, sum.y);
      o.y = pack2<T>(sum.z, sum.w);
      *reinterpret_cast<uint2*>(y + (size_t)ml * a.N + n) = o;
    };
    if constexpr (SPLIT && MT8 == 1) {
      // M <= 8: one tile per cluster.  Every CTA but the first sends its sum of the tile into the
      // first one's shared memory (st.async, completing on the first CTA's receive barrier) and is
      // done; the first adds the partials in panel order (its own, then ranks 1, 2, ...) and stores
      // y.  One cluster-wide barrier (passed long before, at the CTAs' start) orders the sends
      // after the receive barrier's init; the receive is bounded.
      cluster_wait();
      const int rank = (int)blockIdx.y;
      const uint32_t recv = smem_u32(smem + a.o_recv);
      if (rank != 0) {
        const uint32_t dst = cluster_map(recv, 0), dbar = cluster_map(rbar(0), 0);
        for (int i = tid; i < a.M * (kTileN / 4); i += kCW * 32) {
          const int ml = i / (kTileN / 4), cl = 4 * (i % (kTileN / 4));
          st_async_f4(dst + (uint32_t)((((rank - 1) * a.M + ml) * kTileN + cl) * 4), tile_sum(ml, cl), dbar);
        }
      } else {
        // always waited for (after a timeout too, with the drain's limit): the other CTAs write
        // into this CTA's shared memory, so it must not exit while their sends are in flight
        if (!mbar_wait(rbar(0), 0u, ok ? a.wait_ns : kWaitNs)) ok = false;
        const float* rv = reinterpret_cast<const float*>(smem + a.o_recv);
        for (int i = tid; i < a.M * (kTileN / 4); i += kCW * 32) {
          const int ml = i / (kTileN / 4), cl = 4 * (i % (kTileN / 4));
          float4 sum = tile_sum(ml, cl);
          for (int r = 1; r < (int)gridDim.y; ++r) {
            const float4 v = *reinterpret_cast<const float4*>(rv + ((r - 1) * a.M + ml) * kTileN + cl);
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
          }
          if (ok) store_y(ml, ti * kTileN + cl, sum);   // a tile's 32 columns are all below N
        }
      }
    } else if constexpr (SPLIT) {
      // M = 9 .. 16: the K panels of the run's tiles are the CTAs of one cluster.  Every CTA but
      // the first sends its sum of each tile into one of two receive slots in the first CTA's
      // shared memory (st.async, completing on that slot's receive barrier).  The first CTA keeps
      // its own sum and adds tile i up (its own, then ranks 1, 2, ... in order) after its own sum
      // of tile i + 1, so that the exchange is off its way; then it re-arms the slot and arrives on
      // the other CTAs' slot-free barriers, which they wait for before they send tile i + 2 into
      // it.  The cluster barrier passed at the first tile orders every send and remote arrive
      // after the barriers' init; every wait is bounded.
      static_assert(MT8 * 8 * (kTileN / 4) < kCW * 32, "one tile sum float4 per thread, the last thread free");
      const int it = ti - T0, run = T1 - T0, slot = it & 1;
      const int rank = (int)blockIdx.y, nsend = (int)gridDim.y - 1;
      const int per = a.M * kTileN;                 // floats of one tile sum
      float* recv = reinterpret_cast<float*>(smem + a.o_recv);
      float* own = recv + 2 * nsend * per;
      if (it == 0) cluster_wait();
      if (rank != 0) {
        if (it >= 2 && !mbar_wait_cluster(sfree(slot), (uint32_t)(((it >> 1) - 1) & 1), ok ? a.wait_ns : kWaitNs))
          ok = false;
        // (sent after a timeout too: the first CTA counts on every send of every tile)
        const uint32_t dst = cluster_map(smem_u32(recv + (slot * nsend + rank - 1) * per), 0);
        const uint32_t dbar = cluster_map(rbar(slot), 0);
        for (int i = tid; i < a.M * (kTileN / 4); i += kCW * 32) {
          const int ml = i / (kTileN / 4), cl = 4 * (i % (kTileN / 4));
          st_async_f4(dst + (uint32_t)((ml * kTileN + cl) * 4), tile_sum(ml, cl), dbar);
        }
      } else {
        for (int i = tid; i < a.M * (kTileN / 4); i += kCW * 32) {
          const int ml = i / (kTileN / 4), cl = 4 * (i % (kTileN / 4));
          *reinterpret_cast<float4*>(own + slot * per + ml * kTileN + cl) = tile_sum(ml, cl);
        }
        auto finish = [&](const int j) {
          const int sj = j & 1;
          // always waited for (after a timeout too, with the drain's limit): the other CTAs write
          // into this CTA's shared memory, so it must not exit while their sends are in flight
          if (!mbar_wait(rbar(sj), (uint32_t)((j >> 1) & 1), ok ? a.wait_ns : kWaitNs)) ok = false;
          // one float4 of the tile per thread, in the first half of the consumer threads (each
          // reads back only the own sum it wrote itself)
          const bool mine = tid < a.M * (kTileN / 4);
          const int ml = tid / (kTileN / 4), cl = 4 * (tid % (kTileN / 4));
          float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
          if (mine) {
            sum = *reinterpret_cast<const float4*>(own + sj * per + ml * kTileN + cl);
            for (int r = 0; r < nsend; ++r) {
              const float4 v = *reinterpret_cast<const float4*>(recv + (sj * nsend + r) * per + ml * kTileN + cl);
              sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
          }
          if (j + 2 < run) {
            named_sync_consumers<kCW>();             // every consumer has read slot sj
            // The last consumer thread frees the slot: it stores no y (from thread 0, with the y
            // stores before it, the arrive held warp 0 ~1 us per tile, and every warp then waited
            // for warp 0 at the next tile).
            if (tid == kCW * 32 - 1) {
              mbar_arrive_expect_tx(rbar(sj), (uint32_t)(nsend * per) * 4u);
              for (int r = 1; r <= nsend; ++r) mbar_arrive_remote(cluster_map(sfree(sj), (uint32_t)r));
            }
          }
          if (mine && ok) store_y(ml, (T0 + j) * kTileN + cl, sum);   // a tile's 32 columns are all below N
        };
        if (it >= 1) finish(it - 1);
        if (it == run - 1) finish(it);
      }
    } else {
      for (int i = tid; i < a.M * (kTileN / 4); i += kCW * 32) {
        const int ml = i / (kTileN / 4), cl = 4 * (i % (kTileN / 4));
        float4 sum = *reinterpret_cast<const float4*>(&red[ml * RS + cl]);
#pragma unroll
        for (int w = 1; w < kCW; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(&red[(size_t)w * MT8 * 8 * RS + ml * RS + cl]);
          sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
        }
        const int n = ti * kTileN + cl;
        if (n < a.N) {   // N % 32 == 0: a group of 4 columns is all in or all out
          if (a.bias) {
            const float4 b = __ldg(reinterpret_cast<const float4*>(a.bias + n));
            sum.x += b.x; sum.y += b.y; sum.z += b.z; sum.w += b.w;
          }
          uint2 o;
          o.x = pack2<T>(sum.x, sum.y);
          o.y = pack2<T>(sum.z, sum.w);
          *reinterpret_cast<uint2*>(y + (size_t)ml * a.N + n) = o;
        }
      }
    }
  }
  if constexpr (SPLIT && MT8 > 1)
    if (T1 - T0 > 1) { cluster_arrive(); cluster_wait(); }   // the cluster's closing barrier
  if (!ok) report_timeout(a.err);
}

// xp[m][j] = x[m][perm[j]] (0 for pad rows): activations in sorted k order for the bulk copies.
__global__ void k_gather_x(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, uint16_t* __restrict__ xp,
                           int M, int K, int Kr) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");    // x may be the previous grid's output
  const long total = (long)M * Kr;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int m = (int)(i / Kr), j = (int)(i % Kr);
    const int k = __ldg(&perm[j]);
    xp[i] = k >= 0 ? x[(size_t)m * K + k] : (uint16_t)0;
  }
}

// Host plan: ints only, cached per handle and M.
struct SmallPlan {
  int grid, ntiles, pb, npanel, single, lg_rd, span_max, x_row, o_x, o_zs, o_red, o_cg, o_xs, o_bar, smem, cw,
      gather, o_pm, o_raw, cg_async, xs_on, split, o_recv;
};

// K split for layers with fewer 32-column tiles than SMs (M <= 8): the largest of 2, 4, 8 K panels
// whose CTAs (one per tile and panel, a whole SM each; a tile's panels form one cluster) all run
// at once, with at least two stages per panel; 1 = no split.  The split costs about a
// microsecond (cluster launch and the partials' exchange) and saves ~0.06 us per 128-row block a
// CTA no longer walks, so it is taken only when it saves at least 20 blocks per CTA (measured:
// K = 4096 in two panels was 0.6 us slower, K = 8192 in two 0.3 us faster).
//
// M = 9 .. 16 (two m-tiles), when x over all of K is too large to stage once: the fewest of 2, 4, 8
// K panels whose x fits, each CTA of a cluster walking its panel of every tile of the cluster's
// run, so x is staged once per CTA instead of once per tile and panel (the 70B gate layer at
// M = 16: 67.9 us with x staged per panel; the same per-CTA work with x staged once, 38.9 us).
int split_panels(const Handle& h, int M) {
  const int NB = h.Kr / 128;
  const int ntiles = (h.N + kTileN - 1) / kTileN;
  if (M > 8) {
    if (M > 16 || M * (NB * 256 + 64) <= kXSingle) return 1;
    for (int sp = 2; sp <= 8; sp *= 2) {
      const int pb = ((NB + sp - 1) / sp + kSPB - 1) / kSPB * kSPB;
      if (pb < 2 * kSPB || (NB + pb - 1) / pb != sp) return 1;
      if (M * (pb * 256 + 64) <= kXSingle) return sp;
    }
    return 1;
  }
  int best = 1;
  for (int sp = 2; sp <= 8; sp *= 2) {
    if (ntiles > whole_sm_clusters(h, sp)) break;
    const int pb = ((NB + sp - 1) / sp + kSPB - 1) / kSPB * kSPB;
    if (pb < 2 * kSPB || (NB + pb - 1) / pb != sp) break;
    best = sp;
  }
  if (best > 1 && NB * (best - 1) < 20 * best) best = 1;
  return best;
}

// Layout for codes of `bits` bits and MT8 m-tiles; with_gather adds the perm copy.
// level 0: the preferred layout; level >= 1 (when that does not fit, e.g. K of 64 Ki and more, whose
// per-group header and per-block tables grow with K): 8 consumer warps, no x-sum table, and K
// panels of at most NB >> (level - 1) blocks.
// split > 1: clusters of `split` CTAs, one per K panel, over runs of tiles (x of one panel staged
// once).
bool plan_layout(const Handle& h, int M, int bits, int mt8, bool with_gather, SmallPlan& p, int level = 0,
                 int split = 1) {
  const int NB = h.Kr / 128;
  p.ntiles = (h.N + kTileN - 1) / kTileN;
  p.grid = split > 1 ? std::min(p.ntiles, whole_sm_clusters(h, split)) : std::min(p.ntiles, h.sm_count);
  if (p.grid < 1) return false;   // no cluster of this size fits the GPU
  p.split = split;
  const int pb_split = ((NB + split - 1) / split + kSPB - 1) / kSPB * kSPB;
  // K-panel: all of K when x fits, else as many blocks as kXPanel holds (x double buffered)
  const int x_all = M * ((split > 1 ? pb_split : NB) * 256 + 64);
  int target = kSmemFull;
  // A short CTA (x small, at most three tiles) takes half an SM and 8 consumer warps, so the next
  // call's CTA can start streaming beside it; a long one takes the whole SM, a deeper ring and
  // (at M <= 8) 16 consumer warps.
  // Measured: the half-SM shape wins only when the runs are nearly even (decode layer, 448 tiles on
  // 152 CTAs: 8.9 vs 9.3 us at M = 1).  A CTA with a single tile, or runs where more than an eighth
  // of the CTAs have one tile less, take the whole SM: 16 warps finish sooner than 8 beside the next
  // call's CTA (K = 4096, N = 11008: 8.5 -> 7.9 us; K = N = 4096: 13-29 % faster).
  const int tiles_per_cta = (p.ntiles + p.grid - 1) / p.grid;
  const bool short_cta = split == 1 && x_all <= kXSmall && tiles_per_cta >= 2 && tiles_per_cta <= 3 &&
                         p.ntiles >= tiles_per_cta * p.grid - p.grid / 8;
  p.cw = (mt8 == 1 && !short_cta && level == 0) ? 16 : 8;
  // the split kernels: 16 consumer warps for one m-tile, 8 for two
  if (split > 1 && (mt8 > 2 || p.cw != (mt8 == 1 ? 16 : 8))) return false;
  p.xs_on = level == 0 ? 1 : 0;
  if (split > 1) {
    // one tile and one K panel per CTA, x of the panel staged once
    if (level != 0 || x_all > kXSingle || (NB + pb_split - 1) / pb_split != split) return false;
    p.single = 1;
    p.pb = pb_split;
  } else if (level == 0 && x_all <= kXSingle) {
    p.single = 1;
    p.pb = NB;
    if (short_cta) target = kSmemHalf;
  } else if (level == 0) {
    p.single = 0;
    p.pb = std::max(kSPB, (kXPanel / M - 64) / 256 / kSPB * kSPB);
  } else {
    const int cap = std::max(kSPB, (NB >> (level - 1)) / kSPB * kSPB);
    p.pb = std::min(cap, std::max(kSPB, (kXPanel / M - 64) / 256 / kSPB * kSPB));
    p.single = p.pb >= NB ? 1 : 0;
    if (p.single) p.pb = NB;
  }
  p.gather = (with_gather && p.single) ? 1 : 0;
  p.npanel = (NB + p.pb - 1) / p.pb;
  p.span_max = 1;
  for (int q = 0; q < p.npanel; ++q) {
    const int b0 = q * p.pb, b1 = std::min(NB, b0 + p.pb);
    p.span_max = std::max(p.span_max, h.cgid_host[4 * b1 - 1] - h.cgid_host[4 * b0] + 1);
  }
  p.x_row = p.pb * 256 + 64;
  const int x_bytes = (p.single ? 1 : 2) * M * p.x_row;
  const int zs_bytes = 2 * p.span_max * kZsRow;
  const int red_bytes = p.cw * mt8 * 8 * (kTileN + 4) * 4;
  const int cg_bytes = (NB * 4 * 4 + 15) / 16 * 16;
  const int xs_bytes = p.xs_on ? NB * 8 * mt8 * 4 : 0;   // x sums per block, reused by the later tiles
  const int pm_bytes = p.gather ? h.Kr * 4 : 0;
  const int raw_bytes = p.gather ? M * h.K * 2 : 0;
  // the cluster's partial sums: two receive slots of the other CTAs' sums and two of the CTA's own
  const int recv_bytes = split > 1 ? 2 * split * M * kTileN * 4 : 0;
  const int fixed = x_bytes + zs_bytes + red_bytes + cg_bytes + xs_bytes + pm_bytes + raw_bytes + recv_bytes + 9 * 8 + 16;
  const int SB = kSPB * bits * 512;
  int budget = target - fixed - 128;
  int rd = budget / (SB + 16);
  if (rd < 4) {   // large tables: take up to a whole SM's shared memory
    target = kSmemFull;
    budget = kSmemFull - fixed - 128;
    rd = budget / (SB + 16);
  }
  p.cg_async = target == kSmemFull ? 1 : 0;
  if (rd < 2) return false;
  rd = std::min(rd, 128);
  p.lg_rd = 0;
  while ((2 << p.lg_rd) <= rd) ++p.lg_rd;     // largest power of two <= rd
  const int rdp = 1 << p.lg_rd;
  // A consumer warp's consecutive stages are cw / kSPB apart.  A parity wait on a slot tells apart
  // only the slot's current and previous phase, and that previous phase must be one the waiting
  // warp has consumed itself: the ring depth must be a multiple of that distance (then the slot's
  // previous stage is the warp's own earlier one, complete), which for the power-of-two rings and
  // 8 or 16 consumer warps means at least that many stages.  (A ring that is not a multiple --
  // 12 warps, 3 stages apart, on a 4-stage ring -- let a warp wait on a slot whose previous stage,
  // taken by other warps, was still in flight, and read it as its own: bulk copies can complete
  // out of order.)
  if (rdp * kSPB < p.cw || rdp % (p.cw / kSPB) != 0) return false;
  p.o_x = rdp * SB;
  p.o_zs = p.o_x + (x_bytes + 15) / 16 * 16;
  p.o_red = p.o_zs + zs_bytes;
  p.o_cg = p.o_red + red_bytes;
  p.o_xs = p.o_cg + cg_bytes;
  p.o_pm = p.o_xs + xs_bytes;
  p.o_raw = p.o_pm + pm_bytes;
  p.o_recv = p.o_raw + raw_bytes;
  p.o_bar = p.o_recv + recv_bytes;
  p.smem = p.o_bar + (2 * rdp + 9) * 8 + 128;     // + alignment slack of the base
  return p.smem <= 227 * 1024;
}

// The plan: act-order handles gather x in the GEMM kernel at M <= 2 when x is staged once and the
// weight ring keeps at least eight stages; otherwise a pre-pass gathers x into the workspace.
bool make_plan(const Handle& h, int M, SmallPlan& p) {
  const int mt8 = M <= 8 ? 1 : M <= 16 ? 2 : 4;
  const int split = split_panels(h, M);
  if (split > 1) {
    if (!h.identity && !h.fp8 && M <= 2 && plan_layout(h, M, h.bits, mt8, true, p, 0, split) && p.gather && p.lg_rd >= 3)
      return true;
    if (plan_layout(h, M, h.bits, mt8, false, p, 0, split)) return true;
  }
  if (!h.identity && !h.fp8 && M <= 2 && plan_layout(h, M, h.bits, mt8, true, p) && p.gather && p.lg_rd >= 3) return true;
  for (int level = 0; level <= 12; ++level)
    if (plan_layout(h, M, h.bits, mt8, false, p, level)) return true;
  return false;
}

template <typename T, int BITS, int MT8, bool FP8>
cudaError_t launch_t(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  SmallPlan p{};
  {
    std::lock_guard<std::mutex> lock(h.plan_mu);
    const int64_t key = ((int64_t)GPTQ_PATH_SMALL_M << 32) | (uint32_t)M;
    auto it = h.plans.find(key);
    if (it == h.plans.end()) {
      if (!make_plan(h, M, p)) return cudaErrorInvalidConfiguration;
      cudaError_t e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 8, false, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 8, false, FP8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if constexpr (MT8 == 1) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 16, false, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if constexpr (!FP8) {
          if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 8, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
          if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 16, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
          if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 16, true, false, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        }
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 16, false, FP8, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      }
      if constexpr (MT8 == 2)
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_small<T, BITS, MT8, 8, false, FP8, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      std::vector<int64_t> v((sizeof(SmallPlan) + 7) / 8, 0);
      std::memcpy(v.data(), &p, sizeof(SmallPlan));
      h.plans[key] = v;
    } else {
      std::memcpy(&p, it->second.data(), sizeof(SmallPlan));
    }
  }
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  int ldx = h.K;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;   // K split: a tile's panels form one cluster
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = (unsigned)p.split;
  attr[1].val.clusterDim.z = 1;
  if (!h.identity && !p.gather) {
    cudaLaunchConfig_t gcfg = {};
    const long total = (long)M * h.Kr;
    gcfg.gridDim = dim3((unsigned)std::min<long>((total + 255) / 256, 2L * h.sm_count));
    gcfg.blockDim = dim3(256);
    gcfg.stream = st;
    gcfg.attrs = attr;
    gcfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&gcfg, k_gather_x, static_cast<const uint16_t*>(x), (const int32_t*)h.perm,
                                       static_cast<uint16_t*>(h.xp), M, h.K, h.Kr);
    if (e != cudaSuccess) return e;
    xs = static_cast<const uint16_t*>(h.xp);
    ldx = h.Kr;
  }
  SmallArgs args{h.wr, h.cgid, h.zst, xs, y, h.err, ldx, M, h.N, h.Np, h.Kr, h.G,
                 p.ntiles, p.pb, p.npanel, p.single, p.lg_rd, p.span_max, p.x_row,
                 p.o_x, p.o_zs, p.o_red, p.o_cg, p.o_bar, p.o_xs, h.perm, p.gather, p.o_pm, p.o_raw, p.cg_async,
                 h.zoff, h.has_bias ? h.bias : nullptr, h.wait_ns, h.test_stall, p.o_recv};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid, p.split);
  cfg.blockDim = dim3(p.cw == 16 ? threads_of<16>() : threads_of<8>());
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = p.split > 1 ? 2 : 1;
  if (!p.xs_on)   // the long-K layouts: 8 consumer warps, no gather, no x-sum table
    return cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 8, false, FP8, false>, args, h.wr_map);
  if constexpr (MT8 == 1) {
    if (p.split > 1) {   // K split (planned only with 16 consumer warps and the x-sum table)
      // block size must match the kernel, and this kernel ends one tile per cluster
      if (p.cw != 16 || !p.xs_on || p.grid != p.ntiles) return cudaErrorInvalidConfiguration;
      if constexpr (!FP8)
        if (p.gather) return cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 16, true, false, true, true>, args, h.wr_map);
      return cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 16, false, FP8, true, true>, args, h.wr_map);
    }
    if constexpr (!FP8) {
      if (p.gather)
        return p.cw == 16 ? cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 16, true, false>, args, h.wr_map)
                          : cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 8, true, false>, args, h.wr_map);
    }
    if (p.cw == 16) return cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 16, false, FP8>, args, h.wr_map);
  } else if constexpr (MT8 == 2) {
    if (p.split > 1) {   // K split at two m-tiles: 8 consumer warps, x staged by the gather pre-pass
      if (p.cw != 8 || p.gather) return cudaErrorInvalidConfiguration;
      return cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 8, false, FP8, true, true>, args, h.wr_map);
    }
  }
  if (p.split > 1 || p.cw != 8) return cudaErrorInvalidConfiguration;   // no kernel built for that plan
  return cudaLaunchKernelEx(&cfg, k_gemm_small<T, BITS, MT8, 8, false, FP8>, args, h.wr_map);
}

template <typename T, int BITS, bool FP8 = false>
cudaError_t launch_bits(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  if (M <= 8) return launch_t<T, BITS, 1, FP8>(h, x, y, M, st);
  if (M <= 16) return launch_t<T, BITS, 2, FP8>(h, x, y, M, st);
  if (M <= 32) return launch_t<T, BITS, 4, FP8>(h, x, y, M, st);
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dtype(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  if (h.fp8) return launch_bits<T, 8, true>(h, x, y, M, st);
  switch (h.bits) {
    case 2: return launch_bits<T, 2>(h, x, y, M, st);
    case 3: return launch_bits<T, 3>(h, x, y, M, st);
    case 4: return launch_bits<T, 4>(h, x, y, M, st);
    default: return launch_bits<T, 8>(h, x, y, M, st);
  }
}

}  // namespace

#ifndef GPTQ_SMALL_BF16_UNIT
// Clusters of S CTAs that take a whole SM each and that the GPU runs at once (also used by the
// large-M kernel's K split: both kernels run one CTA per SM).  One kernel built for clusters answers
// for all of them: at one CTA per SM the count depends only on the cluster size and on how the SMs
// are grouped.
int whole_sm_clusters(const Handle& h, int S) {
  if (S <= 1 || S > 8) return S == 1 ? h.sm_count : 0;
  const int idx = S;
  int n = h.clusters_fit[idx].load(std::memory_order_relaxed);
  if (n != 0) return n > 0 ? n : 0;   // -1: queried, none fit
  auto fn = k_gemm_small<__half, 4, 2, 8, false, false, true, true>;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = (unsigned)S;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, (unsigned)S);
  cfg.blockDim = dim3(threads_of<8>());
  cfg.dynamicSmemBytes = kSmemFull;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemFull) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;   // unknown: no split of this size is planned
  }
  n = std::max(0, std::min(n, h.sm_count / S));
  h.clusters_fit[idx].store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n;
}
#endif

#ifndef GPTQ_SMALL_BF16_UNIT
int small_m_max() { return 32; }

bool small_m_plan_info(const Handle& h, int M, gptq_plan_t* out) {
  SmallPlan p{};
  if (M < 1 || M > 32 || !make_plan(h, M, p)) return false;
  out->path = GPTQ_PATH_SMALL_M;
  out->launches = (h.identity || p.gather) ? 1 : 2;
  out->grid = p.grid;
  out->threads = p.cw == 16 ? threads_of<16>() : threads_of<8>();
  out->smem_bytes = p.smem;
  out->consumer_warps = p.cw;
  out->m_tiles = M <= 8 ? 1 : M <= 16 ? 2 : 4;
  out->act_order_in_kernel = p.gather;
  out->k_splits = p.split;
  out->k_panels = p.npanel;
  out->stages = 1 << p.lg_rd;
  return true;
}

int small_m_k_splits(const Handle& h, int M) {
  SmallPlan p{};
  return (M >= 1 && M <= 32 && make_plan(h, M, p)) ? p.split : 1;
}

int small_m_launches(const Handle& h, int M) {
  if (M <= 0) return 0;
  if (h.identity) return 1;
  SmallPlan p{};
  return (make_plan(h, M, p) && p.gather) ? 1 : 2;
}

cudaError_t launch_gemm_small(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  if (h.dtype == GPTQ_BF16) return launch_gemm_small_bf16(h, x, y, M, st);
  return launch_dtype<__half>(h, x, y, M, st);
}
#else
cudaError_t launch_gemm_small_bf16(const Handle& h, const void* x, void* y, int M, cudaStream_t st) {
  return launch_dtype<__nv_bfloat16>(h, x, y, M, st);
}
#endif

}  // namespace gptq

// Repack: checkpoint layout -> the kernel-private runtime layout (runs once per layer, at load).
//
// The checkpoint is the AutoGPTQ "cuda" pack (tensref.org "GPTQ packed checkpoint", sections
// GptqLayer and Reader).  The runtime layout follows the loader of inference.shantanugoel.com
// ch. 39 "Quantized checkpoints", section "The format": input columns are sorted by g_idx once,
// so that groups become contiguous, and x is permuted to match at run time.
//
// Runtime layout (every kernel reads exactly this):
//  * Sorted, padded K.  Each group's run of input features (ascending k inside the group) is
//    padded to a multiple of 32 rows; the total is padded to Kr, a multiple of 128.  perm[j]
//    is the input feature of sorted row j, or -1 for a pad row (its activation is 0).
//    cgid[c] is the group of the 32-row chunk c; chunks after the last real row take the last
//    real chunk's group.
//  * N padded to Np (multiple of 256); pad columns hold code 0, stored zero 0, scale 0.
//  * Codes: in blocks of 128 sorted rows.  Inside block B, row r = j % 128 has chunk c = r/32,
//    lane t = (r%32)/8 and e = r%8; it is element e%2 ("half" h) of pair p = 4c + e/2 of lane t.
//    A plane of bp bits per code holds F = 16/bp fields in each 16-bit half of a word; pair p
//    lives in lane word jw = p/F, field f = p%F, at bit 16h + bp*f.  Lane t owns words
//    q = t*bp .. t*bp + bp-1; word q sits in 16-byte vector q/4, slot q%4.  Vectors of one
//    (block, column) are stored [B][vector][column][16 bytes], plane after plane; inside each
//    group of 32 columns, vector V keeps column c at position (c + rot(V)) % 32 with rot = 2V
//    (4-bit), 2 (V / 2) (8-bit), 4V (2-bit, and the 2-bit plane of 3-bit), 0 (3-bit 1-bit plane),
//    so that lanes reading different vectors of a densely copied block use different banks.
//    bits 2/4/8 use one plane (bp = bits); bits 3 uses a 2-bit plane (code & 3) followed by a
//    1-bit plane (code >> 2), in the spirit of GPTQModel's planar packing (fields never
//    straddle words), a layout chosen for the decoder, not a checkpoint format.
//    Why: the two 16-bit halves of a word give the two bf16/fp16 lanes of one register after a
//    single mask-and-or with a magic exponent, and lane t's pairs are exactly the k indices an
//    mma.sync m16n8k16 A-fragment row needs after a fixed relabelling of k, while a whole
//    128-row block of one column is 16*bits contiguous-by-vector bytes for the large-M loader.
//  * s_r[g][n]: scale bits; z_r[g][n]: the checkpoint's zero field as one byte (GPTQ: zero - 1;
//    AutoAWQ: the zero itself); the handle's zoff (1 or 0) turns the field into the zero.
//
// AutoAWQ GEMM checkpoints (4-bit, codes packed along the output dimension, no g_idx) go through
// the same kernels: only the reading of a code and of a zero field differs (awq_code).
#include "internal.cuh"

#include <vector>

namespace gptq {
namespace {

// Code k of a packed column: the column's words read as one little-endian bit string, code k at
// bits [bits*k, bits*k + bits).  For bits 2/4/8 that is "word k / (32/bits), shifted by
// bits*(k % (32/bits))" (the Reader); for bits 3 it is the 10 / split / 10 word layout, where
// codes 10 and 21 of each 32 straddle a word boundary.
__device__ __forceinline__ uint32_t column_code(const int32_t* __restrict__ words, long stride, long k, int bits) {
  long bit = (long)bits * k;
  long row = bit >> 5;
  int sh = (int)(bit & 31);
  uint32_t v = (uint32_t)__ldg(&words[row * stride]) >> sh;
  if (sh + bits > 32) v |= (uint32_t)__ldg(&words[(row + 1) * stride]) << (32 - sh);
  return v & ((1u << bits) - 1u);
}

// Code of output column n in one row of an AutoAWQ GEMM tensor (inference.shantanugoel.com ch. 39,
// section "AWQ"): 4-bit fields packed eight to a word along the output dimension, nibble j of word
// n / 8 holding column 8 (n / 8) + order[j] with order = 0 2 4 6 1 3 5 7.  Column o = n % 8 is
// therefore nibble o / 2 for even o and 4 + o / 2 for odd o.
__device__ __forceinline__ uint32_t awq_code(const int32_t* __restrict__ row, int n) {
  const int o = n & 7;
  return ((uint32_t)__ldg(&row[n >> 3]) >> (4 * ((o >> 1) + 4 * (o & 1)))) & 0xFu;
}

__device__ __forceinline__ int group_of(const int32_t* __restrict__ g_idx, int k, int group_size) {
  if (g_idx) return __ldg(&g_idx[k]);
  return group_size == -1 ? 0 : k / group_size;
}

// meta[] slots written by k_histogram
enum { M_BAD_GIDX = 0, M_NONDECR = 1, M_KS = 2, M_KR = 3, M_LAST_G = 4, M_ALL32 = 5, M_BAD_K = 6, M_N = 8 };

// One block: histogram of g_idx, range check, padded exclusive scan of the group runs.
__global__ void k_histogram(const int32_t* __restrict__ g_idx, int K, int G, int group_size,
                            int32_t* __restrict__ cnt, int32_t* __restrict__ off, int32_t* __restrict__ meta) {
  __shared__ int s_bad, s_nondecr, s_last, s_all32, s_bad_k;
  __shared__ long s_carry;
  __shared__ int s_warp[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) { s_bad = 0; s_nondecr = 1; s_last = -1; s_all32 = 1; s_bad_k = -1; s_carry = 0; }
  for (int g = tid; g < G; g += nt) cnt[g] = 0;
  __syncthreads();
  for (int k = tid; k < K; k += nt) {
    int g = group_of(g_idx, k, group_size);
    if (g < 0 || g >= G) {
      atomicExch(&s_bad, 1);
      atomicMax(&s_bad_k, k);
      continue;
    }
    atomicAdd(&cnt[g], 1);
    atomicMax(&s_last, g);
    if (k > 0 && group_of(g_idx, k - 1, group_size) > g) atomicExch(&s_nondecr, 0);
  }
  __syncthreads();
  // exclusive scan of roundup(cnt, 32), 1024 groups at a time
  for (int base = 0; base < G; base += nt) {
    int g = base + tid;
    int c = g < G ? cnt[g] : 0;
    if (c % 32) atomicExch(&s_all32, 0);
    int v = (c + 31) / 32 * 32;
    // inclusive scan inside the warp
    int lane = tid & 31, w = tid >> 5;
    int x = v;
    for (int d = 1; d < 32; d <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    if (w == 0) {
      int nw = nt / 32;
      int y = lane < nw ? s_warp[lane] : 0;
      for (int d = 1; d < 32; d <<= 1) {
        int z = __shfl_up_sync(0xffffffffu, y, d);
        if (lane >= d) y += z;
      }
      if (lane < nw) s_warp[lane] = y;       // inclusive scan of warp totals
    }
    __syncthreads();
    long before = s_carry + (w > 0 ? s_warp[w - 1] : 0) + (x - v);
    if (g < G) off[g] = (int32_t)before;
    __syncthreads();
    if (tid == nt - 1) s_carry += s_warp[nt / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) {
    long Ks = s_carry;
    meta[M_BAD_GIDX] = s_bad;
    meta[M_NONDECR] = s_nondecr;
    meta[M_KS] = (int32_t)Ks;
    meta[M_KR] = (int32_t)((Ks + 127) / 128 * 128);
    meta[M_LAST_G] = s_last;
    meta[M_ALL32] = s_all32;
    meta[M_BAD_K] = s_bad_k;
  }
}

// One warp: stable scatter of every k to its sorted row.  32 consecutive k at a time; lanes that
// share a group take consecutive slots in ascending k (rank = earlier peers in the warp).
__global__ void k_scatter_perm(const int32_t* __restrict__ g_idx, int K, int group_size,
                               const int32_t* __restrict__ off, int32_t* __restrict__ cursor,
                               int32_t* __restrict__ perm) {
  const int lane = threadIdx.x;
  for (int base = 0; base < K; base += 32) {
    const int k = base + lane;                  // K % 32 == 0: every lane has a k
    const int g = group_of(g_idx, k, group_size);
    const unsigned peers = __match_any_sync(0xffffffffu, g);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    const int b = *(volatile int32_t*)&cursor[g];
    perm[off[g] + b + rank] = k;
    __syncwarp();
    if (lane == leader) *(volatile int32_t*)&cursor[g] = b + __popc(peers);
    __syncwarp();
  }
}

// One thread per group: pad rows of its run, chunk group ids, and the trailing pad chunks.
__global__ void k_pads(int G, int Ks, int Kr, int last_g, const int32_t* __restrict__ cnt,
                       const int32_t* __restrict__ off, int32_t* __restrict__ perm, int32_t* __restrict__ cgid) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  const int c = cnt[g], j0 = off[g], run = (c + 31) / 32 * 32;
  for (int j = j0 + c; j < j0 + run; ++j) perm[j] = -1;
  for (int ch = j0 / 32; ch < (j0 + run) / 32; ++ch) cgid[ch] = g;
  if (g == last_g) {
    for (int j = Ks; j < Kr; ++j) perm[j] = -1;
    for (int ch = Ks / 32; ch < Kr / 32; ++ch) cgid[ch] = g;
  }
}

// One thread per (block B, vector V, column n): assembles that 16-byte vector.  fmt: kFmtGptq reads
// qweight as the GPTQ [K*bits/32, N] tensor, kFmtAwq as an AutoAWQ [K, N/8] one (4-bit), kFmtFp8 as
// e4m3 bytes [N, K] (8-bit), whose pairs keep their two bytes side by side in one 16-bit half (pair
// p in half p % 2, the even k in the low byte) so that one e4m3x2 conversion makes an operand.
__global__ void k_pack_codes(const void* __restrict__ qweight_v, const int32_t* __restrict__ perm, int K,
                             int N, int Np, int bits, int nBV, int fmt, uint8_t* __restrict__ wr) {
  const int32_t* qweight = static_cast<const int32_t*>(qweight_v);
  const uint8_t* w8 = static_cast<const uint8_t*>(qweight_v);
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= Np) return;
  for (int by = blockIdx.y; by < nBV; by += gridDim.y) {
  const int B = by / bits, V = by % bits;
  int bp, v, plane;
  if (bits == 3) { plane = V < 2 ? 0 : 1; bp = plane == 0 ? 2 : 1; v = plane == 0 ? V : 0; }
  else { plane = 0; bp = bits; v = V; }
  const int F = 16 / bp;
  uint32_t out[4];
#pragma unroll 1
  for (int w = 0; w < 4; ++w) {
    const int q = 4 * v + w, t = q / bp, jw = q % bp;
    uint32_t word = 0;
    for (int h = 0; h < 2; ++h)
      for (int f = 0; f < F; ++f) {
        const int p = jw * F + f, c = p / 4, e = 2 * (p % 4) + h;
        const int jj = 128 * B + 32 * c + 8 * t + e;
        const int k = __ldg(&perm[jj]);
        uint32_t code = 0u;
        if (k >= 0 && n < N)
          code = fmt == kFmtFp8 ? (uint32_t)__ldg(&w8[(long)n * K + k])
               : fmt == kFmtAwq ? awq_code(qweight + (long)k * (N / 8), n) : column_code(qweight + n, N, k, bits);
        uint32_t val = bits == 3 ? (plane == 0 ? (code & 3u) : (code >> 2)) : code;
        word |= val << (fmt == kFmtFp8 ? 16 * f + 8 * h : 16 * h + bp * f);
      }
    out[w] = word;
  }
  uint4* dst = reinterpret_cast<uint4*>(wr + (((size_t)B * bits + V) * Np + code_col_pos(bits, V, n)) * 16);
  *dst = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// One thread per (group, column): scale bits and stored zero field (awq: qzeros is an AutoAWQ
// [G, N/8] tensor, whose field is the zero itself).  sf32: scales are float32, rounded here to the
// handle's dtype (round to nearest even; bf16 when to_bf16) -- the type the layer computes in.
__global__ void k_pack_sz(const int32_t* __restrict__ qzeros, const void* __restrict__ scales,
                          int N, int Np, int bits, int G, int awq, int sf32, int to_bf16,
                          uint16_t* __restrict__ s_r, uint8_t* __restrict__ z_r) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= Np) return;
  const long wpr = (long)N * bits / 32;
  for (int g = blockIdx.y; g < G; g += gridDim.y) {
  uint16_t s = 0;
  uint8_t z = 0;
  if (n < N) {
    if (sf32) {
      const float f = __ldg(static_cast<const float*>(scales) + (long)g * N + n);
      s = to_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f)) : __half_as_ushort(__float2half_rn(f));
    } else {
      s = __ldg(static_cast<const uint16_t*>(scales) + (long)g * N + n);
    }
    z = (uint8_t)(awq ? awq_code(qzeros + (long)g * (N / 8), n) : column_code(qzeros + (long)g * wpr, 1, n, bits));
  }
  s_r[(long)g * Np + n] = s;
  z_r[(long)g * Np + n] = z;
  }
}

// zst[(T * G + g) * 96 + pos] = z_r[g][32 T + c] and, as 16-bit words after the 32 zero bytes,
// s_r[g][32 T + c], with pos = (c % 8) * 4 + c / 8: the four columns c = g8 + 8 j that one lane of
// the small-M kernel owns are adjacent.  One warp per (tile, group row range).
__global__ void k_pack_zst(const uint16_t* __restrict__ s_r, const uint8_t* __restrict__ z_r, int Np, int G,
                           uint8_t* __restrict__ zst) {
  const int c = threadIdx.x & 31;
  const int T = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (T >= Np / 32) return;
  const int pos = (c % 8) * 4 + c / 8;
  const long n = 32L * T + c;
  for (int g = blockIdx.y; g < G; g += gridDim.y) {
    uint8_t* row = zst + ((long)T * G + g) * 96;
    row[pos] = z_r[(long)g * Np + n];
    reinterpret_cast<uint16_t*>(row + 32)[pos] = s_r[(long)g * Np + n];
  }
}

// FP8 layers: every (32-column tile T, group g) row of zst carries the block's float32 factor
// scale_inv[32 T / 128][g] in each of its eight 4-byte zero slots (the slot lane group g8 of the
// small-M kernel reads), and zeros elsewhere; tiles past N get 0.
__global__ void k_pack_zst_fp8(const float* __restrict__ scale_inv, int kb, int N, int Np, int G,
                               uint8_t* __restrict__ zst) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;      // one thread per (T, g) row
  if (i >= (Np / 32) * G) return;
  const int T = i / G, g = i % G;
  const float s = 32 * T < N ? __ldg(&scale_inv[(long)(32 * T / 128) * kb + g]) : 0.0f;
  uint32_t* row = reinterpret_cast<uint32_t*>(zst + (size_t)i * 96);
  for (int w = 0; w < 8; ++w) row[w] = __float_as_uint(s);
  for (int w = 8; w < 24; ++w) row[w] = 0u;
}

// bias[n] as float32 (0 for the pad columns n >= N): kind 0 fp16 bits, 1 bf16 bits, 2 float32.
__global__ void k_bias_f32(const void* __restrict__ src, int kind, int N, int Np, float* __restrict__ dst) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= Np) return;
  float v = 0.0f;
  if (n < N) {
    if (kind == 2) v = __ldg(static_cast<const float*>(src) + n);
    else {
      const uint16_t b = __ldg(static_cast<const uint16_t*>(src) + n);
      v = kind == 1 ? __bfloat162float(__ushort_as_bfloat16(b)) : __half2float(__ushort_as_half(b));
    }
  }
  dst[n] = v;
}

}  // namespace

cudaError_t launch_bias_f32(const void* src, int kind, int N, int Np, float* dst, cudaStream_t st) {
  k_bias_f32<<<(Np + 255) / 256, 256, 0, st>>>(src, kind, N, Np, dst);
  return cudaGetLastError();
}

gptq_status_t build_runtime(Handle& h, const void* qweight, const int32_t* qzeros, const void* scales,
                            const int32_t* g_idx, int fmt, bool scales_fp32, cudaStream_t st) {
  const int K = h.K, N = h.N, G = h.G;
  int32_t* tmp = nullptr;   // cnt[G] | off[G] | cursor[G] | meta[M_N]
  cudaError_t e = cudaMalloc(&tmp, sizeof(int32_t) * ((size_t)3 * G + M_N));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(repack scratch)");
  int32_t* cnt = tmp;
  int32_t* off = tmp + G;
  int32_t* cursor = tmp + 2 * (size_t)G;
  int32_t* meta = tmp + 3 * (size_t)G;
  int32_t meta_h[M_N] = {};
  auto cleanup = [&]() { cudaFree(tmp); };

  k_histogram<<<1, 1024, 0, st>>>(g_idx, K, G, h.group_size, cnt, off, meta);
  if ((e = cudaGetLastError()) != cudaSuccess) { cleanup(); return cuda_fail(e, "histogram launch"); }
  if ((e = cudaMemcpyAsync(meta_h, meta, sizeof(meta_h), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess) {
    cleanup();
    return cuda_fail(e, "repack: reading the g_idx histogram");
  }
  if (meta_h[M_BAD_GIDX]) {
    cleanup();
    return fail(GPTQ_ERR_INVALID_GIDX, "GPTQ-004: g_idx[" + std::to_string(meta_h[M_BAD_K]) +
                                           "] selects no scale/zero row (valid groups are 0.." + std::to_string(G - 1) + ")");
  }
  h.Kr = meta_h[M_KR];
  h.identity = meta_h[M_NONDECR] && meta_h[M_ALL32] && h.Kr == K;
  const int Ks = meta_h[M_KS], last_g = meta_h[M_LAST_G];

  size_t wr_b = h.wr_bytes();
  const bool fp8 = fmt == kFmtFp8;
  const size_t nsc = fp8 ? (size_t)((N + 127) / 128) * h.kb : 0;
  if ((e = cudaMalloc(&h.wr, wr_b)) != cudaSuccess || (e = cudaMalloc(&h.perm, sizeof(int32_t) * h.Kr)) != cudaSuccess ||
      (e = cudaMalloc(&h.cgid, sizeof(int32_t) * (h.Kr / 32))) != cudaSuccess ||
      (!fp8 && (e = cudaMalloc(&h.s_r, sizeof(uint16_t) * (size_t)G * h.Np)) != cudaSuccess) ||
      (!fp8 && (e = cudaMalloc(&h.z_r, (size_t)G * h.Np)) != cudaSuccess) ||
      (fp8 && (e = cudaMalloc(&h.scale_inv, sizeof(float) * nsc)) != cudaSuccess) ||
      (e = cudaMalloc(&h.zst, (size_t)G * h.Np * 3)) != cudaSuccess) {
    cleanup();
    return cuda_fail(e, "cudaMalloc(runtime layout)");
  }
  {
    // the small-M kernel's view of wr: uint64 [Kr/128 * bits rows][2 Np], one box = four blocks
    // of one 32-column tile (4 * bits rows of 512 bytes)
    EncodeTiledFn enc = encode_fn();
    const cuuint64_t dims[2] = {(cuuint64_t)h.Np * 2, (cuuint64_t)(h.Kr / 128) * h.bits};
    const cuuint64_t strides[1] = {(cuuint64_t)h.Np * 16};
    const cuuint32_t box[2] = {64, (cuuint32_t)(kSmallBlocksPerBox * h.bits)};
    const cuuint32_t estr[2] = {1, 1};
    if (!enc || enc(&h.wr_map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, h.wr, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      cleanup();
      return fail(GPTQ_ERR_CUDA, "cuTensorMapEncodeTiled(runtime codes) failed");
    }
  }
  if ((e = cudaMemsetAsync(cursor, 0, sizeof(int32_t) * G, st)) != cudaSuccess) { cleanup(); return cuda_fail(e, "memset"); }
  k_scatter_perm<<<1, 32, 0, st>>>(g_idx, K, h.group_size, off, cursor, h.perm);
  k_pads<<<(G + 127) / 128, 128, 0, st>>>(G, Ks, h.Kr, last_g, cnt, off, h.perm, h.cgid);
  const int nBV = (h.Kr / 128) * h.bits;
  dim3 gc(h.Np / 256, nBV < 65535 ? nBV : 65535);
  k_pack_codes<<<gc, 256, 0, st>>>(qweight, h.perm, K, N, h.Np, h.bits, nBV, fmt, h.wr);
  if (fp8) {
    if ((e = cudaMemcpyAsync(h.scale_inv, scales, sizeof(float) * nsc, cudaMemcpyDeviceToDevice, st)) != cudaSuccess) {
      cleanup();
      return cuda_fail(e, "copy scale_inv");
    }
    const int rows = (h.Np / 32) * G;
    k_pack_zst_fp8<<<(rows + 255) / 256, 256, 0, st>>>(static_cast<const float*>(scales), h.kb, N, h.Np, G, h.zst);
  } else {
    dim3 gs(h.Np / 256, G < 65535 ? G : 65535);
    k_pack_sz<<<gs, 256, 0, st>>>(qzeros, scales, N, h.Np, h.bits, G, fmt == kFmtAwq ? 1 : 0, scales_fp32 ? 1 : 0,
                                  h.dtype == GPTQ_BF16 ? 1 : 0, h.s_r, h.z_r);
    dim3 gz(h.Np / 32 / 8, G < 65535 ? G : 65535);
    k_pack_zst<<<gz, 256, 0, st>>>(h.s_r, h.z_r, h.Np, G, h.zst);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) { cleanup(); return cuda_fail(e, "repack launch"); }
  h.cgid_host.resize(h.Kr / 32);
  if ((e = cudaMemcpyAsync(h.cgid_host.data(), h.cgid, sizeof(int32_t) * (h.Kr / 32), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess) {
    cleanup();
    return cuda_fail(e, "repack");
  }
  cleanup();
  return GPTQ_OK;
}

// ---------------------------------------------------------------------------------------------
// Allocation-free repack (gptq_repack_noalloc).  Its only scratch, the per-group counts, offsets
// and cursors of the sort plus a few flags, lives in this file-scope device array, which every
// device that loads the library holds until the process exits.  In host code the array's name is
// a host-side stand-in, so every call looks up its device address on the current device with
// cudaGetSymbolAddress (cheap next to the stream synchronize the call makes anyway, and never stale
// after the context is torn down and created again) and passes that address to the kernels.  All
// calls on a device share the array: the counts are cleared by k_histogram and the cursors by a
// memset on every call, and the array is in use until the call's kernels on its stream have
// finished, so calls that overlap on the same GPU (for example on two streams) race on it.
constexpr int kNoallocMaxGroups = 4096;
static __device__ __align__(256) int32_t g_noalloc_scratch[3 * kNoallocMaxGroups + M_N];

}  // namespace gptq

extern "C" gptq_status_t gptq_repack_noalloc(const int32_t* qweight, const int32_t* qzeros, const void* scales,
                                             const int32_t* g_idx, int K, int N, int bits, int group_size,
                                             gptq_dtype_t dtype, void* wr, size_t wr_capacity, int32_t* perm,
                                             int32_t* cgid, int kr_capacity, void* s_r, uint8_t* z_r,
                                             int* k_sorted, void* stream) {
  using namespace gptq;
  if (k_sorted) *k_sorted = 0;
  if (!qweight || !qzeros || !scales || !wr || !perm || !cgid || !s_r || !z_r || !k_sorted)
    return fail(GPTQ_ERR_INVALID_ARG, "gptq_repack_noalloc: every input and output buffer is required");
  if (bits != 2 && bits != 3 && bits != 4 && bits != 8)
    return fail(GPTQ_ERR_UNSUPPORTED, "GPTQ-001: bits must be 2, 3, 4 or 8, got " + std::to_string(bits));
  if (dtype != GPTQ_FP16 && dtype != GPTQ_BF16) return fail(GPTQ_ERR_UNSUPPORTED, "dtype must be GPTQ_FP16 or GPTQ_BF16");
  if (group_size != -1 && group_size < 1) return fail(GPTQ_ERR_INVALID_ARG, "group_size must be -1 or >= 1");
  if (K < 32 || K % 32 != 0) return fail(GPTQ_ERR_SHAPE, "GPTQ-002: in_features must be a positive multiple of 32");
  if (N < 32 || N % 32 != 0) return fail(GPTQ_ERR_SHAPE, "GPTQ-003: out_features must be a positive multiple of 32");
  if (K > GPTQ_MAX_K || N > GPTQ_MAX_N)
    return fail(GPTQ_ERR_UNSUPPORTED, "layer too large for this build (K <= " + std::to_string(GPTQ_MAX_K) +
                                          ", N <= " + std::to_string(GPTQ_MAX_N) + ")");
  const int G = group_size == -1 ? 1 : (K + group_size - 1) / group_size;
  if (G > kNoallocMaxGroups)
    return fail(GPTQ_ERR_UNSUPPORTED, "gptq_repack_noalloc: at most " + std::to_string(kNoallocMaxGroups) +
                                          " groups (its fixed scratch); this layer has " + std::to_string(G));
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(wr) | reinterpret_cast<uintptr_t>(perm) | reinterpret_cast<uintptr_t>(cgid);
  if ((a16 & 15) || (reinterpret_cast<uintptr_t>(qweight) & 3) || (reinterpret_cast<uintptr_t>(qzeros) & 3) ||
      (reinterpret_cast<uintptr_t>(scales) & 1) || (reinterpret_cast<uintptr_t>(s_r) & 1) ||
      (g_idx && (reinterpret_cast<uintptr_t>(g_idx) & 3)))
    return fail(GPTQ_ERR_ALIGNMENT, "wr, perm and cgid need 16-byte alignment; qweight, qzeros, g_idx 4; scales, s_r 2");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3) return fail(GPTQ_ERR_DEVICE, "this library is built for sm_103a (compute capability 10.3)");
  int32_t* scratch = nullptr;
  if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&scratch), g_noalloc_scratch)) != cudaSuccess)
    return cuda_fail(e, "cudaGetSymbolAddress(repack scratch)");
  int32_t* cnt = scratch;
  int32_t* off = scratch + G;
  int32_t* cursor = scratch + 2 * G;
  int32_t* meta = scratch + 3 * kNoallocMaxGroups;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int Np = (N + 255) / 256 * 256;

  int32_t meta_h[M_N] = {};
  k_histogram<<<1, 1024, 0, st>>>(g_idx, K, G, group_size, cnt, off, meta);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "histogram launch");
  if ((e = cudaMemcpyAsync(meta_h, meta, sizeof(meta_h), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return cuda_fail(e, "repack: reading the g_idx histogram");
  if (meta_h[M_BAD_GIDX])
    return fail(GPTQ_ERR_INVALID_GIDX, "GPTQ-004: g_idx[" + std::to_string(meta_h[M_BAD_K]) + "] selects no scale/zero row");
  const int Kr = meta_h[M_KR], Ks = meta_h[M_KS], last_g = meta_h[M_LAST_G];
  *k_sorted = Kr;
  const size_t wr_b = (size_t)Kr / 128 * bits * Np * 16;
  if (Kr > kr_capacity || wr_b > wr_capacity)
    return fail(GPTQ_ERR_WORKSPACE, "gptq_repack_noalloc: the sorted K is " + std::to_string(Kr) + " rows (" +
                                        std::to_string(wr_b) + " code bytes); the output buffers are smaller");
  if ((e = cudaMemsetAsync(cursor, 0, sizeof(int32_t) * G, st)) != cudaSuccess) return cuda_fail(e, "memset");
  k_scatter_perm<<<1, 32, 0, st>>>(g_idx, K, group_size, off, cursor, perm);
  k_pads<<<(G + 127) / 128, 128, 0, st>>>(G, Ks, Kr, last_g, cnt, off, perm, cgid);
  const int nBV = (Kr / 128) * bits;
  dim3 gc(Np / 256, nBV < 65535 ? nBV : 65535);
  k_pack_codes<<<gc, 256, 0, st>>>(qweight, perm, K, N, Np, bits, nBV, kFmtGptq, static_cast<uint8_t*>(wr));
  dim3 gs(Np / 256, G < 65535 ? G : 65535);
  k_pack_sz<<<gs, 256, 0, st>>>(qzeros, scales, N, Np, bits, G, 0, 0, 0, static_cast<uint16_t*>(s_r), z_r);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "repack launch");
  return GPTQ_OK;
}

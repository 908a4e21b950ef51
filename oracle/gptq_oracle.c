/*
 * CPU oracle for the GPTQ weight-only linear layer  y = x . dequant(qweight, qzeros, scales, g_idx)^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA library, and the CUDA library never calls it.
 *
 * Everything here is a plain loop written from the pages' statement of the format:
 *   [P4] inference.shantanugoel.com, ch. 39 "Quantized checkpoints", section "The format"
 *        (qweight int32 [in/8, out], eight 4-bit codes along the INPUT dimension per int32,
 *         low bits first; qzeros along the OUTPUT dimension, stored minus one;
 *         W[o,i] = scales[g_idx[i],o] * (q[i,o] - (qzeros[g_idx[i],o] + 1))),
 *        and its pack_gptq / unpack_gptq description.
 *   [P5] tensref.org "GPTQ packed checkpoint", sections GptqLayer, QuantizeConfig, Reader,
 *        "Reject the file when" (GPTQ-001 .. GPTQ-006).
 *
 * Precision.  The Reader dequantises in float32 ((code - zero) as float times scale as
 * float); the product of a <= 9-bit integer and an fp16/bf16 scale is exact in float32,
 * so W is exact.  The matrix product is not fixed by the pages; it is accumulated here in
 * double, in ascending original k, one accumulator per output, with -ffp-contract=off.
 *
 * Readings of points the pages leave open (each also listed in the design notes):
 *   - 3-bit words: the Reader gives unpacking only as the inverse of pack()'s 10 / split / 10 loop.
 *     Reading: 32 consecutive codes share 3 consecutive words; codes 0-9 sit at bits 3j of
 *     word 0, code 10 has bits 0-1 at word-0 bits 30-31 and bit 2 at word-1 bit 0, codes
 *     11-20 at word-1 bits 1+3(j-11), code 21 has bit 0 at word-1 bit 31 and bits 1-2 at
 *     word-2 bits 0-1, codes 22-31 at word-2 bits 2+3(j-22).  Zeros use the same scheme
 *     along N.  Compatibility with external 3-bit files: parity unpinned.
 *   - zeros: z = stored + 1 with no wrap (GPTQ-006), so z is in [1, 2^bits].
 *   - group_size = -1: one group, g_idx = 0 for every k.  g_idx = NULL means k // group_size.
 *
 * Runtime layout (oracle_runtime_layout) is this library's own kernel-private format: the
 * kernel-side layout that the GPTQModel "Kernel Backends Reference" page keeps apart from the
 * checkpoint layout.  Its definition is written out in that function's comment.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

enum { DT_FP16 = 0, DT_BF16 = 1 };

/* ---- scalar decoders for the activation / scale types (IEEE 754 binary16, bfloat16) ---- */

static float fp16_to_float(uint16_t h) {
  /* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
  uint32_t sign = (uint32_t)(h >> 15) & 1u;
  uint32_t expo = (uint32_t)(h >> 10) & 0x1Fu;
  uint32_t frac = (uint32_t)h & 0x3FFu;
  float mag;
  if (expo == 0) {
    mag = (float)frac * (1.0f / 16777216.0f);           /* subnormal: frac * 2^-24 */
  } else if (expo == 31) {
    union { uint32_t u; float f; } v;
    v.u = 0x7F800000u | (frac << 13);                   /* inf or nan */
    mag = v.f;
  } else {
    union { uint32_t u; float f; } v;
    v.u = ((expo - 15 + 127) << 23) | (frac << 13);
    mag = v.f;
  }
  return sign ? -mag : mag;
}

static float bf16_to_float(uint16_t h) {
  union { uint32_t u; float f; } v;
  v.u = (uint32_t)h << 16;                              /* bfloat16 is the top half of binary32 */
  return v.f;
}

static float half_bits_to_float(uint16_t h, int dtype) {
  return dtype == DT_BF16 ? bf16_to_float(h) : fp16_to_float(h);
}

float oracle_half_to_float(uint16_t h, int dtype) { return half_bits_to_float(h, dtype); }

/*
 * float32 -> binary16 / bfloat16 bits, round to nearest, ties to even (IEEE 754), written from the
 * formats' definitions with integers only.  Used where the library takes float32 scales ([P5]
 * GptqLayer: scales are float16 "or the layer weight dtype"; its Example file stores F32 scales):
 * a layer that computes in fp16/bf16 uses its scales in that type, so they are rounded once.
 *   value = S * 2^E exactly (S the 24-bit significand); the target keeps mb fraction bits, its
 *   smallest quantum is 2^qmin (qmin = 1 - bias - mb, the subnormal spacing), and a value whose
 *   rounded exponent field reaches all ones is infinity.
 */
static uint16_t round_fp32_bits(uint32_t u, int mb, int eb, int bias) {
  const uint32_t sign = (u >> 31) << (mb + eb);
  const uint32_t expo = (u >> 23) & 0xFFu, frac = u & 0x7FFFFFu;
  const uint32_t inf = ((1u << eb) - 1u) << mb;
  if (expo == 0xFFu) return (uint16_t)(sign | inf | (frac ? 1u << (mb - 1) : 0u));   /* nan / inf */
  uint64_t S = expo ? (frac | 0x800000u) : frac;
  int E = expo ? (int)expo - 127 - 23 : -149;
  if (S == 0) return (uint16_t)sign;
  int top = 63;
  while (!((S >> top) & 1u)) --top;                    /* floor(log2 S) */
  const int qmin = 1 - bias - mb;
  int q = top + E - mb;                                 /* quantum that keeps mb fraction bits */
  if (q < qmin) q = qmin;
  uint64_t m;
  const int shift = q - E;
  if (shift <= 0) {
    m = S << -shift;
  } else if (shift > 40) {
    m = 0;                                              /* below half the smallest quantum */
  } else {
    m = S >> shift;
    const uint64_t rem = S & ((1ull << shift) - 1u), half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (m & 1u))) ++m;
  }
  if (m >> (mb + 1)) { m >>= 1; ++q; }                  /* rounding carried into a new binade */
  if (m < (1ull << mb)) return (uint16_t)(sign | (uint32_t)m);   /* subnormal (q == qmin) or zero */
  const int biased = q + mb + bias;
  if (biased >= (1 << eb) - 1) return (uint16_t)(sign | inf);
  return (uint16_t)(sign | ((uint32_t)biased << mb) | (uint32_t)(m - (1ull << mb)));
}

/* n float32 values (as bits) -> dtype bits: DT_FP16 binary16, DT_BF16 bfloat16. */
int oracle_round_fp32(const uint32_t* in, long n, int dtype, uint16_t* out) {
  if (dtype != DT_FP16 && dtype != DT_BF16) return 1;
  for (long i = 0; i < n; ++i)
    out[i] = dtype == DT_FP16 ? round_fp32_bits(in[i], 10, 5, 15) : round_fp32_bits(in[i], 7, 8, 127);
  return 0;
}

/* ---- unpacking codes along one axis ---- */

/*
 * Code number i of a packed column, where the column is the sequence of int32 words
 * words[0], words[stride], words[2*stride], ... (qweight packs along K with stride N;
 * qzeros packs along N with stride 1).
 * bits 2/4/8: the Reader's loop: word row i / pack, field (i % pack), shift bits*(i%pack),
 *             mask (1 << bits) - 1, words read as unsigned (two's complement, [P4] as_int32).
 * bits 3:     the 10 / split / 10 reading above.
 */
static uint32_t code_at(const int32_t* words, long stride, long i, int bits) {
  if (bits == 2 || bits == 4 || bits == 8) {
    long pack = 32 / bits;
    uint32_t w = (uint32_t)words[(i / pack) * stride];
    return (w >> (bits * (i % pack))) & ((1u << bits) - 1u);
  }
  /* bits == 3 */
  long grp = i / 32, j = i % 32;
  uint32_t w0 = (uint32_t)words[(grp * 3 + 0) * stride];
  uint32_t w1 = (uint32_t)words[(grp * 3 + 1) * stride];
  uint32_t w2 = (uint32_t)words[(grp * 3 + 2) * stride];
  if (j < 10) return (w0 >> (3 * j)) & 7u;
  if (j == 10) return ((w0 >> 30) & 3u) | ((w1 & 1u) << 2);
  if (j < 21) return (w1 >> (1 + 3 * (j - 11))) & 7u;
  if (j == 21) return ((w1 >> 31) & 1u) | ((w2 & 3u) << 1);
  return (w2 >> (2 + 3 * (j - 22))) & 7u;
}

/* Inverse of code_at: OR code v into position i (the words must start zeroed). */
static void put_code(int32_t* words, long stride, long i, int bits, uint32_t v) {
  v &= (1u << bits) - 1u;
  if (bits == 2 || bits == 4 || bits == 8) {
    long pack = 32 / bits;
    uint32_t* w = (uint32_t*)&words[(i / pack) * stride];
    *w |= v << (bits * (i % pack));
    return;
  }
  long grp = i / 32, j = i % 32;
  uint32_t* w0 = (uint32_t*)&words[(grp * 3 + 0) * stride];
  uint32_t* w1 = (uint32_t*)&words[(grp * 3 + 1) * stride];
  uint32_t* w2 = (uint32_t*)&words[(grp * 3 + 2) * stride];
  if (j < 10) { *w0 |= v << (3 * j); return; }
  if (j == 10) { *w0 |= (v & 3u) << 30; *w1 |= (v >> 2) & 1u; return; }
  if (j < 21) { *w1 |= v << (1 + 3 * (j - 11)); return; }
  if (j == 21) { *w1 |= (v & 1u) << 31; *w2 |= (v >> 1) & 3u; return; }
  *w2 |= v << (2 + 3 * (j - 22));
}

static int bits_ok(int bits) { return bits == 2 || bits == 3 || bits == 4 || bits == 8; }

/* qweight int32 [K*bits/32, N] -> codes uint8 [K][N] ([P5] Reader; [P4] unpack_gptq). */
int oracle_unpack_codes(const int32_t* qweight, int K, int N, int bits, uint8_t* codes) {
  if (!bits_ok(bits) || K % 32 || N <= 0) return ORACLE_EINVAL;
  for (long k = 0; k < K; ++k)
    for (long n = 0; n < N; ++n)
      codes[k * N + n] = (uint8_t)code_at(qweight + n, N, k, bits);
  return ORACLE_OK;
}

/* codes uint8 [K][N] -> qweight int32 [K*bits/32, N] ([P4] pack_gptq, generalised to bits). */
int oracle_pack_codes(const uint8_t* codes, int K, int N, int bits, int32_t* qweight) {
  if (!bits_ok(bits) || K % 32 || N <= 0) return ORACLE_EINVAL;
  memset(qweight, 0, sizeof(int32_t) * (size_t)K * bits / 32 * N);
  for (long k = 0; k < K; ++k)
    for (long n = 0; n < N; ++n)
      put_code(qweight + n, N, k, bits, codes[k * N + n]);
  return ORACLE_OK;
}

/* qzeros int32 [G, N*bits/32] -> zero points int32 [G][N], z = stored + 1 (GPTQ-006). */
int oracle_unpack_zeros(const int32_t* qzeros, int G, int N, int bits, int32_t* z) {
  if (!bits_ok(bits) || N % 32 || G <= 0) return ORACLE_EINVAL;
  long wpr = (long)N * bits / 32;
  for (long g = 0; g < G; ++g)
    for (long n = 0; n < N; ++n)
      z[g * N + n] = (int32_t)code_at(qzeros + g * wpr, 1, n, bits) + 1;
  return ORACLE_OK;
}

/* zero points [G][N] -> qzeros, storing (z - 1) masked to bits ([P4] pack_gptq). */
int oracle_pack_zeros(const int32_t* z, int G, int N, int bits, int32_t* qzeros) {
  if (!bits_ok(bits) || N % 32 || G <= 0) return ORACLE_EINVAL;
  long wpr = (long)N * bits / 32;
  memset(qzeros, 0, sizeof(int32_t) * (size_t)G * wpr);
  for (long g = 0; g < G; ++g)
    for (long n = 0; n < N; ++n)
      put_code(qzeros + g * wpr, 1, n, bits, (uint32_t)(z[g * N + n] - 1));
  return ORACLE_OK;
}

/* Number of groups: ceil(K / group_size), or 1 when group_size == -1 ([P5] GptqLayer, QuantizeConfig). */
int oracle_num_groups(int K, int group_size) {
  if (group_size == -1) return 1;
  if (group_size <= 0) return -1;
  return (K + group_size - 1) / group_size;
}

static int group_of(const int32_t* g_idx, long k, int group_size) {
  if (g_idx) return g_idx[k];
  return group_size == -1 ? 0 : (int)(k / group_size);
}

/*
 * One dequantised weight row n (all K inputs), float32, per the Reader:
 *   W[n, k] = (float(code[k, n]) - float(z[g, n])) * float(scales[g, n]),  g = g_idx[k],
 * z = stored field + zoff: zoff 1 for the AutoGPTQ (v1) fields stored minus one ([P4] "The
 * format"), 0 for the corrected gptq_v2 fields that hold the zero itself (same section; [P1]
 * keeps the v1/v2 interpretation apart).
 */
static void dequant_row(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                        const int32_t* g_idx, int K, int N, int bits, int group_size, uint32_t zoff, long n,
                        float* row) {
  long wpr = (long)N * bits / 32;
  for (long k = 0; k < K; ++k) {
    int g = group_of(g_idx, k, group_size);
    float q = (float)code_at(qweight + n, N, k, bits);
    float z = (float)(code_at(qzeros + (long)g * wpr, 1, n, bits) + zoff);
    float s = half_bits_to_float(scales[(long)g * N + n], dtype);
    row[k] = (q - z) * s;
  }
}

static int check_gidx(const int32_t* g_idx, int K, int G) {
  if (!g_idx) return ORACLE_OK;
  for (long k = 0; k < K; ++k)
    if (g_idx[k] < 0 || g_idx[k] >= G) return ORACLE_EINVAL;
  return ORACLE_OK;
}

/* Dense W float32 [N][K] (the Reader's output, [out_features, in_features]); zoff as dequant_row. */
int oracle_dequant_ex(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                      const int32_t* g_idx, int K, int N, int bits, int group_size, int zoff, float* W) {
  int G = oracle_num_groups(K, group_size);
  if (!bits_ok(bits) || K % 32 || N % 32 || G <= 0 || check_gidx(g_idx, K, G)) return ORACLE_EINVAL;
  if (!g_idx && group_size != -1 && group_size > K) return ORACLE_EINVAL;
  if (zoff != 0 && zoff != 1) return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
  for (long n = 0; n < N; ++n)
    dequant_row(qweight, qzeros, scales, dtype, g_idx, K, N, bits, group_size, (uint32_t)zoff, n, W + n * (long)K);
  return ORACLE_OK;
}

int oracle_dequant(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                   const int32_t* g_idx, int K, int N, int bits, int group_size, float* W) {
  return oracle_dequant_ex(qweight, qzeros, scales, dtype, g_idx, K, N, bits, group_size, 1, W);
}

/*
 * y[r][c] = sum_k x[rows[r]][k] * W[cols[c]][k] (+ bias[cols[c]]), over the sampled rows and columns.
 * x: [M][K] fp16/bf16 bits.  The weight row W[n] is dequantised once per sampled column, then
 * dotted with each sampled x row in ascending k, accumulating in double; the bias ([P5]
 * GptqLayer: optional, [out_features], same dtype as scales) is added to the double sum.
 * zoff as dequant_row.  bias: NULL, or N values of bias_kind 0 (fp16 bits), 1 (bf16 bits) or
 * 2 (float32).
 */
int oracle_linear_ex(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                     const int32_t* g_idx, int K, int N, int bits, int group_size, int zoff, const void* bias,
                     int bias_kind, const uint16_t* x, int M, const int32_t* rows, int nrows, const int32_t* cols,
                     int ncols, double* y) {
  int G = oracle_num_groups(K, group_size);
  if (!bits_ok(bits) || K % 32 || N % 32 || G <= 0 || check_gidx(g_idx, K, G)) return ORACLE_EINVAL;
  if ((zoff != 0 && zoff != 1) || bias_kind < 0 || bias_kind > 2) return ORACLE_EINVAL;
  for (int r = 0; r < nrows; ++r) if (rows[r] < 0 || rows[r] >= M) return ORACLE_EINVAL;
  for (int c = 0; c < ncols; ++c) if (cols[c] < 0 || cols[c] >= N) return ORACLE_EINVAL;
  float* xf = (float*)malloc(sizeof(float) * (size_t)nrows * K);
  if (!xf) return ORACLE_EINVAL;
  for (long r = 0; r < nrows; ++r)
    for (long k = 0; k < K; ++k) xf[r * K + k] = half_bits_to_float(x[(long)rows[r] * K + k], dtype);
  int fail = 0;
#pragma omp parallel
  {
    float* row = (float*)malloc(sizeof(float) * (size_t)K);
    if (!row) {
#pragma omp atomic write
      fail = 1;
    } else {
#pragma omp for schedule(static)
      for (long c = 0; c < ncols; ++c) {
        dequant_row(qweight, qzeros, scales, dtype, g_idx, K, N, bits, group_size, (uint32_t)zoff, cols[c], row);
        double b = 0.0;
        if (bias) {
          const long n = cols[c];
          b = bias_kind == 2 ? (double)((const float*)bias)[n]
                             : (double)half_bits_to_float(((const uint16_t*)bias)[n], bias_kind == 1 ? DT_BF16 : DT_FP16);
        }
        for (long r = 0; r < nrows; ++r) {
          double acc = 0.0;
          const float* xr = xf + r * K;
          for (long k = 0; k < K; ++k) acc += (double)xr[k] * (double)row[k];
          y[r * ncols + c] = bias ? acc + b : acc;
        }
      }
      free(row);
    }
  }
  free(xf);
  return fail ? ORACLE_EINVAL : ORACLE_OK;
}

int oracle_linear(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                  const int32_t* g_idx, int K, int N, int bits, int group_size,
                  const uint16_t* x, int M, const int32_t* rows, int nrows, const int32_t* cols, int ncols,
                  double* y) {
  return oracle_linear_ex(qweight, qzeros, scales, dtype, g_idx, K, N, bits, group_size, 1, NULL, 0, x, M, rows,
                          nrows, cols, ncols, y);
}

/* Thread count the parallel loops above use (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Thread count for the parallel loops that follow (a measurement setting; no arithmetic changes). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * Reject rules of [P5] "Reject the file when", as far as shapes and values decide them.
 * Returns 0 when accepted, else the rule number (1..4) that rejects:
 *   GPTQ-001 bits in {2,3,4,8};
 *   GPTQ-002 qweight.shape == [in_features // 32 * bits, out_features] and in_features % 32 == 0;
 *   GPTQ-003 qzeros.shape[1] == out_features // 32 * bits;
 *   GPTQ-004 len(g_idx) == in_features and each index selects a scale/zero row.
 * in_features is taken from g_idx's length when g_idx is given, else from qweight's rows.
 * The scale/zero row count is qzeros.shape[0]; scales must be [that, out_features].
 * GPTQ-005 (checkpoint_format marlin) and GPTQ-006 (add 1 to zeros) are not shape rules.
 */
int oracle_check_rules(int bits, int qw_rows, int qw_cols, int qz_rows, int qz_cols,
                       int sc_rows, int sc_cols, int in_features, const int32_t* g_idx, int gidx_len) {
  if (!bits_ok(bits)) return 1;
  int out_f = qw_cols;
  if (in_features % 32 != 0 || qw_rows != in_features / 32 * bits) return 2;
  if (qz_cols != out_f / 32 * bits) return 3;
  if (sc_rows != qz_rows || sc_cols != out_f) return 3;
  if (g_idx) {
    if (gidx_len != in_features) return 4;
    for (int k = 0; k < gidx_len; ++k)
      if (g_idx[k] < 0 || g_idx[k] >= qz_rows) return 4;
  }
  return 0;
}

/*
 * The runtime layout (this library's kernel-private format), written out as plain loops.
 *
 * Inputs: the checkpoint tensors and (K, N, bits, group_size).  G = number of groups.
 * 1. Sorted, padded K.  cnt[g] = #{k : g_idx[k] == g}; each group's run is padded to
 *    P[g] = roundup(cnt[g], 32); off[g] = sum of P over earlier groups; Ks = sum P;
 *    Kr = roundup(Ks, 128).  perm[j] (j < Kr) lists, for g = 0..G-1, the k with g_idx[k] == g
 *    in ascending k at j = off[g] + 0..cnt[g]-1; every other j is -1 (a pad row, x = 0).
 *    cgid[c] (c < Kr/32) is the group owning sorted rows 32c..32c+31; chunks at or past Ks
 *    take the group of chunk Ks/32 - 1.  [P4] "to_runtime sorts the input columns by g_idx
 *    once at load time, so that groups become contiguous".
 * 2. N is padded to Np = roundup(N, 256); pad columns hold code 0, stored zero 0, scale 0.
 * 3. Codes of sorted row j, column n: code = q[perm[j]][n], or 0 for a pad row or column.
 *    Planes: bits 2/4/8 -> one plane of width bp = bits holding the code; bits 3 -> plane 0
 *    of width 2 holding code & 3 and plane 1 of width 1 holding code >> 2.
 * 4. Within a block of 128 sorted rows (B = j / 128), let r = j % 128, c = r / 32 (chunk),
 *    t = (r % 32) / 8 (lane), e = r % 8.  Pair p = 4c + e/2, half h = e % 2.  In a plane of
 *    width bp a word holds F = 16/bp fields per 16-bit half; the value goes to word
 *    jw = p / F, field f = p % F, bit 16h + bp*f.  The lane's words are numbered
 *    q = t*bp + jw (bp words per lane, 4*bp per (block, column)); vector v = q / 4, word
 *    q % 4 inside the 16-byte vector.  Vectors of plane 0 come first, then plane 1.
 *    Byte offset of the word: ((B*bits + V) * Np + pos(V, n)) * 16 + 4 * (q % 4), with
 *    V = vbase + v, vbase the number of vectors of earlier planes (0, or 2 for 3-bit plane 1),
 *    and pos(V, n) = 32*(n/32) + (n%32 + rot(V)) % 32: inside each group of 32 columns the
 *    column order of vector V is rotated by rot(V) = 2V for 4-bit, 2*(V/2) for 8-bit, 4V for
 *    2-bit and for the 2-bit plane of 3-bit, 0 for the 1-bit plane of 3-bit.
 * 5. S_r[g][n] (n < Np): the scale bits, 0 for pad columns.  Z_r[g][n]: the stored zero
 *    (z - 1) as one byte, 0 for pad columns.
 * Sizes: wr = Kr/128 * bits * Np * 16 bytes; perm Kr int32; cgid Kr/32 int32; S_r, Z_r G*Np.
 * The caller sizes the outputs with oracle_runtime_dims first.
 */
int oracle_runtime_dims(const int32_t* g_idx, int K, int N, int group_size, int* Kr_out, int* Np_out) {
  int G = oracle_num_groups(K, group_size);
  if (G <= 0 || K % 32 || N % 32 || check_gidx(g_idx, K, G)) return ORACLE_EINVAL;
  long Ks = 0;
  for (int g = 0; g < G; ++g) {
    long cnt = 0;
    for (long k = 0; k < K; ++k) cnt += group_of(g_idx, k, group_size) == g;
    Ks += (cnt + 31) / 32 * 32;
  }
  *Kr_out = (int)((Ks + 127) / 128 * 128);
  *Np_out = (N + 255) / 256 * 256;
  return ORACLE_OK;
}

/* Column rotation of vector V inside a group of 32 columns (step 4 above). */
static long column_rotation(int bits, long V) {
  if (bits == 4) return 2 * V;
  if (bits == 8) return 2 * (V / 2);
  if (bits == 2) return 4 * V;
  return V < 2 ? 4 * V : 0;   /* 3-bit: 2-bit plane vectors 0, 1; 1-bit plane vector 2 */
}

int oracle_runtime_layout(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                          const int32_t* g_idx, int K, int N, int bits, int group_size,
                          uint8_t* wr, int32_t* perm, int32_t* cgid, uint16_t* s_r, uint8_t* z_r) {
  int G = oracle_num_groups(K, group_size);
  int Kr, Np;
  if (!bits_ok(bits) || oracle_runtime_dims(g_idx, K, N, group_size, &Kr, &Np)) return ORACLE_EINVAL;
  /* 1. sorted, padded K */
  long j = 0;
  for (long c = 0; c < Kr / 32; ++c) cgid[c] = -1;
  for (long i = 0; i < Kr; ++i) perm[i] = -1;
  for (int g = 0; g < G; ++g) {
    long start = j;
    for (long k = 0; k < K; ++k)
      if (group_of(g_idx, k, group_size) == g) perm[j++] = (int32_t)k;
    j = start + (j - start + 31) / 32 * 32;
    for (long c = start / 32; c < j / 32; ++c) cgid[c] = g;
  }
  for (long c = j / 32; c < Kr / 32; ++c) cgid[c] = cgid[j / 32 - 1];
  /* 3.-4. codes into plane words */
  memset(wr, 0, (size_t)Kr / 128 * bits * Np * 16);
  int nplanes = bits == 3 ? 2 : 1;
  for (long jj = 0; jj < Kr; ++jj) {
    long B = jj / 128, r = jj % 128, c = r / 32, t = (r % 32) / 8, e = r % 8;
    long p = 4 * c + e / 2, h = e % 2;
    for (long n = 0; n < Np; ++n) {
      uint32_t code = 0;
      if (perm[jj] >= 0 && n < N) code = code_at(qweight + n, N, perm[jj], bits);
      long vbase = 0;
      for (int pl = 0; pl < nplanes; ++pl) {
        int bp = bits == 3 ? (pl == 0 ? 2 : 1) : bits;
        uint32_t val = bits == 3 ? (pl == 0 ? (code & 3u) : (code >> 2)) : code;
        long F = 16 / bp, jw = p / F, f = p % F;
        long q = t * bp + jw, v = q / 4;
        long V = vbase + v;
        long pos = n / 32 * 32 + (n % 32 + column_rotation(bits, V)) % 32;
        size_t off = ((size_t)(B * bits + V) * Np + pos) * 16 + 4 * (q % 4);
        uint32_t* word = (uint32_t*)(wr + off);
        *word |= val << (16 * h + bp * f);
        vbase += bp;
      }
    }
  }
  /* 5. scales and stored zeros per (group, column) */
  long wpr = (long)N * bits / 32;
  for (long g = 0; g < G; ++g)
    for (long n = 0; n < Np; ++n) {
      s_r[g * Np + n] = n < N ? scales[g * N + n] : 0;
      z_r[g * Np + n] = n < N ? (uint8_t)code_at(qzeros + g * wpr, 1, n, bits) : 0;
    }
  return ORACLE_OK;
}

/*
 * AutoAWQ GEMM checkpoints, [P4] ch. 39, section "AWQ" (its pack_awq / unpack_awq /
 * from_checkpoint description): 4-bit codes, eight to an int32 word along the OUTPUT
 * dimension in the interleaved order 0 2 4 6 1 3 5 7 -- nibble j (bits 4j..4j+3) of word w
 * holds output column 8w + order[j], so output 1 sits in bits 16-19.  qweight is [K, N/8],
 * qzeros [G, N/8] packed the same way, scales [G, N]; from_checkpoint builds the offset as
 * -zero * scale with the stored zero itself (no +1), and groups are consecutive runs of
 * group_size input rows (the format carries no g_idx):
 *   W[n, k] = (q[k, n] - z[g, n]) * scales[g, n],  g = k // group_size.
 */
static const int awq_order[8] = {0, 2, 4, 6, 1, 3, 5, 7};

/* Nibble of word row[n / 8] that holds output column n. */
static uint32_t awq_code(const int32_t* row, long n) {
  int o = (int)(n % 8), j = 0;
  while (awq_order[j] != o) ++j;
  return ((uint32_t)row[n / 8] >> (4 * j)) & 0xFu;
}

/* packed int32 [rows, N/8] -> codes uint8 [rows][N] */
int oracle_awq_unpack(const int32_t* packed, int rows, int N, uint8_t* out) {
  if (rows <= 0 || N <= 0 || N % 8) return ORACLE_EINVAL;
  for (long r = 0; r < rows; ++r)
    for (long n = 0; n < N; ++n) out[r * N + n] = (uint8_t)awq_code(packed + r * (N / 8), n);
  return ORACLE_OK;
}

/* codes uint8 [rows][N] (values 0..15) -> packed int32 [rows, N/8], the inverse of oracle_awq_unpack */
int oracle_awq_pack(const uint8_t* codes, int rows, int N, int32_t* packed) {
  if (rows <= 0 || N <= 0 || N % 8) return ORACLE_EINVAL;
  for (long r = 0; r < rows; ++r)
    for (long w = 0; w < N / 8; ++w) {
      uint32_t word = 0;
      for (int j = 0; j < 8; ++j) word |= ((uint32_t)codes[r * N + 8 * w + awq_order[j]] & 0xFu) << (4 * j);
      packed[r * (N / 8) + w] = (int32_t)word;
    }
  return ORACLE_OK;
}

static void awq_dequant_row(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                            int K, int N, int group_size, long n, float* row) {
  for (long k = 0; k < K; ++k) {
    long g = group_size == -1 ? 0 : k / group_size;
    float q = (float)awq_code(qweight + k * (N / 8), n);
    float z = (float)awq_code(qzeros + g * (N / 8), n);
    float s = half_bits_to_float(scales[g * N + n], dtype);
    row[k] = (q - z) * s;
  }
}

static int awq_shape_ok(int K, int N, int group_size) {
  if (K <= 0 || K % 32 || N <= 0 || N % 32) return 0;
  if (group_size != -1 && (group_size <= 0 || group_size > K)) return 0;
  return 1;
}

/* Dense W float32 [N][K] of an AWQ checkpoint. */
int oracle_awq_dequant(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                       int K, int N, int group_size, float* W) {
  if (!awq_shape_ok(K, N, group_size)) return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
  for (long n = 0; n < N; ++n) awq_dequant_row(qweight, qzeros, scales, dtype, K, N, group_size, n, W + n * (long)K);
  return ORACLE_OK;
}

/* y[r][c] = sum_k x[rows[r]][k] * W[cols[c]][k] for an AWQ checkpoint, as oracle_linear. */
int oracle_awq_linear(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales, int dtype,
                      int K, int N, int group_size, const uint16_t* x, int M, const int32_t* rows, int nrows,
                      const int32_t* cols, int ncols, double* y) {
  if (!awq_shape_ok(K, N, group_size)) return ORACLE_EINVAL;
  for (int r = 0; r < nrows; ++r) if (rows[r] < 0 || rows[r] >= M) return ORACLE_EINVAL;
  for (int c = 0; c < ncols; ++c) if (cols[c] < 0 || cols[c] >= N) return ORACLE_EINVAL;
  float* xf = (float*)malloc(sizeof(float) * (size_t)nrows * K);
  if (!xf) return ORACLE_EINVAL;
  for (long r = 0; r < nrows; ++r)
    for (long k = 0; k < K; ++k) xf[r * K + k] = half_bits_to_float(x[(long)rows[r] * K + k], dtype);
  int fail = 0;
#pragma omp parallel
  {
    float* row = (float*)malloc(sizeof(float) * (size_t)K);
    if (!row) {
#pragma omp atomic write
      fail = 1;
    } else {
#pragma omp for schedule(static)
      for (long c = 0; c < ncols; ++c) {
        awq_dequant_row(qweight, qzeros, scales, dtype, K, N, group_size, cols[c], row);
        for (long r = 0; r < nrows; ++r) {
          double acc = 0.0;
          const float* xr = xf + r * K;
          for (long k = 0; k < K; ++k) acc += (double)xr[k] * (double)row[k];
          y[r * ncols + c] = acc;
        }
      }
      free(row);
    }
  }
  free(xf);
  return fail ? ORACLE_EINVAL : ORACLE_OK;
}

/*
 * The same codes and zero fields in GPTQ packing (codes along K, zero fields along N), for the
 * runtime-layout comparison: the zero field carries the AWQ zero itself, which a handle built
 * from an AWQ checkpoint reads with a zero offset of 0 (GPTQ fields read with offset 1).
 * qweight_gptq int32 [K/8, N]; qzeros_gptq int32 [G, N/8].
 */
int oracle_awq_to_gptq_fields(const int32_t* qweight, const int32_t* qzeros, int K, int N, int group_size,
                              int32_t* qweight_gptq, int32_t* qzeros_gptq) {
  if (!awq_shape_ok(K, N, group_size)) return ORACLE_EINVAL;
  int G = oracle_num_groups(K, group_size);
  memset(qweight_gptq, 0, sizeof(int32_t) * (size_t)K / 8 * N);
  memset(qzeros_gptq, 0, sizeof(int32_t) * (size_t)G * (N / 8));
  for (long k = 0; k < K; ++k)
    for (long n = 0; n < N; ++n) put_code(qweight_gptq + n, N, k, 4, awq_code(qweight + k * (N / 8), n));
  for (long g = 0; g < G; ++g)
    for (long n = 0; n < N; ++n) put_code(qzeros_gptq + g * (N / 8), 1, n, 4, awq_code(qzeros + g * (N / 8), n));
  return ORACLE_OK;
}

/*
 * FP8 block-scaled checkpoints, [P4] ch. 39, section "FP8 checkpoints" (its quantize_blocks /
 * dequantize_blocks description and the W8A16 kernel that widens the FP8 tiles and multiplies by
 * the block's factor): weight float8_e4m3fn [N, K] (one byte per weight, row n holds input
 * features 0..K-1), scale_inv float32 [ceil(N/128), ceil(K/128)], one factor per 128 x 128 block
 * that multiplies the stored values:
 *   W[n, k] = e4m3(weight[n, k]) * scale_inv[n / 128][k / 128]   (float32 product)
 * E4M3 ("fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
 * (m * 2^-9); no infinities; exponent 15 with mantissa 7 is NaN; the largest value is 448.
 */
static float e4m3_value(uint8_t b) {
  const int sgn = b >> 7, e = (b >> 3) & 15, m = b & 7;
  float v;
  if (e == 15 && m == 7) {
    union { uint32_t u; float f; } q;
    q.u = 0x7FC00000u;
    return q.f;
  }
  if (e == 0) v = (float)m / 512.0f;                    /* m * 2^-9 */
  else {
    v = 1.0f + (float)m / 8.0f;
    for (int i = 7; i < e; ++i) v *= 2.0f;              /* times 2^(e - 7), exact */
    for (int i = e; i < 7; ++i) v *= 0.5f;
  }
  return sgn ? -v : v;
}

int oracle_e4m3_to_float(const uint8_t* in, long n, float* out) {
  for (long i = 0; i < n; ++i) out[i] = e4m3_value(in[i]);
  return ORACLE_OK;
}

static int fp8_shape_ok(int K, int N) { return K > 0 && N > 0 && K % 32 == 0 && N % 32 == 0; }

static void fp8_dequant_row(const uint8_t* weight, const float* scale_inv, int K, int N, long n, float* row) {
  const long kb = (K + 127) / 128;
  for (long k = 0; k < K; ++k) row[k] = e4m3_value(weight[n * K + k]) * scale_inv[(n / 128) * kb + k / 128];
}

/* Dense W float32 [N][K] of an FP8 block-scaled layer. */
int oracle_fp8_dequant(const uint8_t* weight, const float* scale_inv, int K, int N, float* W) {
  if (!fp8_shape_ok(K, N)) return ORACLE_EINVAL;
#pragma omp parallel for schedule(static)
  for (long n = 0; n < N; ++n) fp8_dequant_row(weight, scale_inv, K, N, n, W + n * (long)K);
  return ORACLE_OK;
}

/* y[r][c] = sum_k x[rows[r]][k] * W[cols[c]][k] in double, as oracle_linear. */
int oracle_fp8_linear(const uint8_t* weight, const float* scale_inv, int dtype, int K, int N, const uint16_t* x,
                      int M, const int32_t* rows, int nrows, const int32_t* cols, int ncols, double* y) {
  if (!fp8_shape_ok(K, N)) return ORACLE_EINVAL;
  for (int r = 0; r < nrows; ++r) if (rows[r] < 0 || rows[r] >= M) return ORACLE_EINVAL;
  for (int c = 0; c < ncols; ++c) if (cols[c] < 0 || cols[c] >= N) return ORACLE_EINVAL;
  float* xf = (float*)malloc(sizeof(float) * (size_t)nrows * K);
  if (!xf) return ORACLE_EINVAL;
  for (long r = 0; r < nrows; ++r)
    for (long k = 0; k < K; ++k) xf[r * K + k] = half_bits_to_float(x[(long)rows[r] * K + k], dtype);
  int fail = 0;
#pragma omp parallel
  {
    float* row = (float*)malloc(sizeof(float) * (size_t)K);
    if (!row) {
#pragma omp atomic write
      fail = 1;
    } else {
#pragma omp for schedule(static)
      for (long c = 0; c < ncols; ++c) {
        fp8_dequant_row(weight, scale_inv, K, N, cols[c], row);
        for (long r = 0; r < nrows; ++r) {
          double acc = 0.0;
          const float* xr = xf + r * K;
          for (long k = 0; k < K; ++k) acc += (double)xr[k] * (double)row[k];
          y[r * ncols + c] = acc;
        }
      }
      free(row);
    }
  }
  free(xf);
  return fail ? ORACLE_EINVAL : ORACLE_OK;
}

/*
 * Runtime layout of an FP8 layer (this library's kernel-private format): the 8-bit layout of
 * oracle_runtime_layout with sequential groups of 128 input features (one per scale block), except
 * that the two bytes of a pair sit next to each other -- pair p of a lane word lives in its 16-bit
 * half p % 2, the even k in the low byte -- so that one e4m3x2 conversion yields both halves of
 * an MMA operand register.  wr, perm and cgid as in oracle_runtime_layout (sized by
 * oracle_runtime_dims(NULL, K, N, 128)).
 */
int oracle_runtime_layout_fp8(const uint8_t* weight, int K, int N, uint8_t* wr, int32_t* perm, int32_t* cgid) {
  int Kr, Np;
  if (!fp8_shape_ok(K, N) || oracle_runtime_dims(NULL, K, N, 128, &Kr, &Np)) return ORACLE_EINVAL;
  const int G = oracle_num_groups(K, 128);
  long j = 0;
  for (long c = 0; c < Kr / 32; ++c) cgid[c] = -1;
  for (long i = 0; i < Kr; ++i) perm[i] = -1;
  for (int g = 0; g < G; ++g) {
    long start = j;
    for (long k = 128L * g; k < K && k < 128L * (g + 1); ++k) perm[j++] = (int32_t)k;
    j = start + (j - start + 31) / 32 * 32;
    for (long c = start / 32; c < j / 32; ++c) cgid[c] = g;
  }
  for (long c = j / 32; c < Kr / 32; ++c) cgid[c] = cgid[j / 32 - 1];
  memset(wr, 0, (size_t)Kr / 128 * 8 * Np * 16);
  for (long jj = 0; jj < Kr; ++jj) {
    long B = jj / 128, r = jj % 128, c = r / 32, t = (r % 32) / 8, e = r % 8;
    long p = 4 * c + e / 2, h = e % 2;
    long jw = p / 2, f = p % 2;
    long q = t * 8 + jw, V = q / 4;
    for (long n = 0; n < Np; ++n) {
      uint32_t b = (perm[jj] >= 0 && n < N) ? weight[n * K + perm[jj]] : 0u;
      long pos = n / 32 * 32 + (n % 32 + column_rotation(8, V)) % 32;
      uint32_t* word = (uint32_t*)(wr + ((size_t)(B * 8 + V) * Np + pos) * 16 + 4 * (q % 4));
      *word |= b << (16 * f + 8 * h);
    }
  }
  return ORACLE_OK;
}

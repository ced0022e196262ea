/*
 * fp4q_oracle.c - plain, slow, scalar CPU restatement of the FP4 communication codec.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this file:
 * only the tests, the smoke check of the package entry module and the CPU-baseline leg of
 * the benchmark use it. It shares no code, header, table or constant with the CUDA
 * library; every constant below is written out again from the method's definition.
 *
 * Sources (web pages on the method):
 *   [P1] "FP4Quant: Efficient 4-Bit Communication Compression for Model-Parallel LLM
 *        Training" (shd-paper.top), English abstract and the method section's technical
 *        framework: micro-grouped dual-scale FP4 quantization, warp-cooperative FP4
 *        packing, hybrid two-level FWHT.
 *   [P3] "4-bit compression speeds up LLM training by 56 percent with minimal accuracy
 *        loss" (zot.news), lead paragraph ("tiny clusters of values share scaling
 *        factors", "packed two per byte", "a fast transform keeps errors low") and
 *        "Read it as" (the AllReduce of tensor parallelism is what is compressed).
 *   [P4] "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"
 *        (gist.science), technical summary, problem statement: FP4 elements are E2M1, and
 *        the microscaled MXFP4 format scales blocks of 32 elements.
 * The pages give no numbers. The numbers used here (block 256, FWHT as 16 x 16 in Sylvester
 * order, group 16 or 32, E4M3 group scale x FP32 block scale with 2688 = 6 * 448, ties to
 * even, the -0 code, the all-zero guard, the payload layout) are the build's stated
 * readings of those passages; each is listed with its reason in the design notes.
 *
 * Arithmetic: every floating-point step is one FP32 operation rounded to nearest, in the
 * order written, compiled with -ffp-contract=off and without fast-math. The method's
 * scales are FP32 by definition, and each quantised code is decided in that precision.
 * OpenMP (when available) only splits the loop over independent 256-element blocks.
 *
 * Parity status: every function is pinned by the CPU tests (closed forms, exhaustive
 * rounding sweeps, library cross-checks, hand-worked blocks, brute-force optimality of
 * each code). The relative-L2 error figures are reported only: the pages print none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BLOCK 256
#define ORACLE_MAX_RANKS 8

/* ---------------------------------------------------------------- bit helpers */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 is the upper half of an IEEE binary32 word, so widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Round a binary32 value to the nearest bfloat16, ties to even: keep the upper 16 bits
 * after adding half an ulp of the result (0x7FFF) plus the result's low bit (which turns
 * an exact half into a round-to-even). NaN stays a quiet NaN. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u = f32_bits(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* ---------------------------------------------------------------- FP8 E4M3 (OCP e4m3fn) */

/* Value of an e4m3fn code from the format definition: 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); 0x7F/0xFF are NaN and are
 * never produced here. [P1 "dual-scale": the group scale is an FP8 value] */
float oracle_e4m3_decode(uint8_t code) {
  int e = (code >> 3) & 15, m = code & 7;
  float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return (code & 0x80) ? -v : v;
}

/* Nearest e4m3fn code to r >= 0, ties to the even code, saturating at 448 (code 0x7E).
 * Plain nearest-neighbour search: locate r between two consecutive finite codes by
 * bisection over the increasing table of the 127 non-negative finite values, then keep the
 * closer one. Distances are exact in double (both operands are floats within 2^41 of each
 * other wherever a tie is possible). */
uint8_t oracle_e4m3_encode(float r) {
  if (!(r > 0.0f)) return 0;                 /* zero (and -0) */
  if (r >= 448.0f) return 0x7E;              /* saturate */
  int lo = 0, hi = 126;                      /* invariant: value(lo) <= r < value(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (oracle_e4m3_decode((uint8_t)mid) <= r) lo = mid; else hi = mid;
  }
  double dl = (double)r - (double)oracle_e4m3_decode((uint8_t)lo);
  double dh = (double)oracle_e4m3_decode((uint8_t)hi) - (double)r;
  if (dl < dh) return (uint8_t)lo;
  if (dh < dl) return (uint8_t)hi;
  return (uint8_t)((lo % 2 == 0) ? lo : hi);  /* tie: the even code */
}

/* ---------------------------------------------------------------- FP4 E2M1 */

static const float kE2M1Grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

/* Value of a 4-bit E2M1 code: bit 3 is the sign, bits 0..2 index the magnitude grid
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}. Code 0x8 is -0. [P4: E2M1 elements; P3 "4-bit
 * floating-point format"] */
float oracle_e2m1_decode(uint8_t code) {
  float v = kE2M1Grid[code & 7];
  return (code & 8) ? -v : v;
}

/* E2M1 code of q: the sign bit of q, and the grid magnitude nearest to |q| found by
 * exhaustive search over the 8 magnitudes, ties to the even code; |q| > 6 gives 6. */
uint8_t oracle_e2m1_encode(float q) {
  uint8_t sign = signbit(q) ? 8 : 0;
  double a = fabs((double)q);
  int best = 0;
  double bestd = a;                          /* distance to grid[0] = 0 */
  for (int k = 1; k < 8; ++k) {
    double d = fabs(a - (double)kE2M1Grid[k]);
    if (d < bestd || (d == bestd && (k % 2 == 0))) { best = k; bestd = d; }
  }
  return (uint8_t)(sign | best);
}

/* ---------------------------------------------------------------- E8M0 (MX scale) */

/* The microscaled variant [P4 problem statement: MXFP4 scales blocks of 32 E2M1 elements]
 * gives each group of 32 a power-of-two scale X stored as an 8-bit exponent (E8M0: code =
 * exponent + 127). The reading follows the open MX definition: X = 2^(floor(log2(amax)) -
 * 2), where 2 is the exponent of the largest E2M1 value (6 = 1.5 * 2^2), so amax / X lies
 * in [4, 8); the exponent is clamped below at -127 (code 0, which also serves amax = 0).
 * floor(log2(a)) comes from frexpf (a = m * 2^e with m in [0.5, 1)), exact for subnormals. */
uint8_t oracle_e8m0_scale(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e = 0;
  frexpf(amax, &e);
  int shared = (e - 1) - 2;
  if (shared < -127) shared = -127;
  return (uint8_t)(shared + 127);
}

/* Value of an E8M0 scale code: 2^(code - 127) (code 255 is NaN and never produced). */
float oracle_e8m0_decode(uint8_t code) { return ldexpf(1.0f, (int)code - 127); }

/* ---------------------------------------------------------------- FWHT */

/* Orthonormal Walsh-Hadamard transform of one 256-element block in Sylvester (natural)
 * order: butterflies with stride h = 1, 2, 4, ..., 128, each (a, b) -> (a + b, a - b) in
 * FP32, then a multiplication by 1/16. Strides below 16 mix the elements of one 16-element
 * group (level 1); strides of 16 and more mix the 16 groups (level 2), i.e.
 * H256 = H16 (x) H16. [P1 "hybrid two-level FWHT pipeline"; P3 "a fast transform"]
 * This is the forward transform of compress. */
void oracle_fwht256(float* v) {
  for (int h = 1; h < ORACLE_BLOCK; h <<= 1) {
    for (int j = 0; j < ORACLE_BLOCK; ++j) {
      if (j & h) continue;
      float a = v[j], b = v[j + h];
      v[j] = a + b;
      v[j + h] = a - b;
    }
  }
  for (int j = 0; j < ORACLE_BLOCK; ++j) v[j] = v[j] * 0.0625f;
}

/* Inverse transform used by every decode: the same butterflies in mirror order
 * (h = 128, 64, ..., 1: level 2 across groups first, then level 1 inside each group),
 * then a multiplication by 1/16. In exact arithmetic this equals oracle_fwht256 (the stages
 * commute and H * H = I); the order is fixed because FP32 rounding depends on it. */
void oracle_ifwht256(float* v) {
  for (int h = ORACLE_BLOCK / 2; h >= 1; h >>= 1) {
    for (int j = 0; j < ORACLE_BLOCK; ++j) {
      if (j & h) continue;
      float a = v[j], b = v[j + h];
      v[j] = a + b;
      v[j + h] = a - b;
    }
  }
  for (int j = 0; j < ORACLE_BLOCK; ++j) v[j] = v[j] * 0.0625f;
}

/* ---------------------------------------------------------------- payload layout */

static int64_t pad16(int64_t b) { return (b + 15) / 16 * 16; }

/* mx = 0: dual scales (E4M3 per group x FP32 per block), G = 16 or 32;
 * mx = 1: E8M0 power-of-two scale per group of 32, no block scale. */
static int valid(int64_t n, int G, int mx) {
  if (mx != 0 && mx != 1) return 0;
  if (mx ? G != 32 : (G != 16 && G != 32)) return 0;
  return n > 0 && n < ((int64_t)1 << 40);
}

/* Elements covered by the payload: n rounded up to whole blocks. A last partial block is
 * zero-padded (the build's reading; the pages say nothing about lengths that are not a
 * multiple of the block): its missing elements are +0 going in, and the decode writes
 * only the n real elements back. */
static int64_t padded(int64_t n) { return (n + ORACLE_BLOCK - 1) / ORACLE_BLOCK * ORACLE_BLOCK; }

/* Payload = [codes n/2 bytes][group scales n/G bytes, padded to 16][block scales n/256
 * float32; absent when mx]. [P3 "values are packed two per byte"; the layout itself is the
 * build's reading, the pages give none] Returns 0 on invalid arguments. */
int64_t oracle_payload_bytes(int64_t n, int G, int mx) {
  if (!valid(n, G, mx)) return 0;
  const int64_t m = padded(n);
  return m / 2 + pad16(m / G) + (mx ? 0 : 4 * (m / ORACLE_BLOCK));
}
int64_t oracle_gscale_offset(int64_t n, int G, int mx) { return valid(n, G, mx) ? padded(n) / 2 : 0; }
int64_t oracle_bscale_offset(int64_t n, int G, int mx) {
  return valid(n, G, mx) ? padded(n) / 2 + pad16(padded(n) / G) : 0;
}

/* ---------------------------------------------------------------- one block */

/* Dual-scale quantisation of one block of 256 transform-domain values y
 * [P1 "micro-grouped dual-scale FP4 quantization"; P3 "tiny clusters of values share
 * scaling factors"]:
 *   A = max|y|; all-zero block if A < 2688 * 2^-100;
 *   s_b = A / 2688; t_b = s_b * 6; per group r = amax / t_b, s_g = E4M3(r);
 *   S = value(s_g) * s_b; inv = 1/S (0 if S == 0); q = y * inv; code = E2M1(q).
 * Writes 256 codes (one per byte, unpacked), 256/G scale bytes, the block scale and,
 * when q_out is not NULL, every q (0 for an all-zero block). */
static void quantize_block(const float* y, int G, uint8_t* code, uint8_t* gs, float* bs,
                           float* q_out) {
  float A = 0.0f;
  for (int i = 0; i < ORACLE_BLOCK; ++i) {
    float a = fabsf(y[i]);
    if (a > A) A = a;
  }
  const float zero_limit = 2688.0f * 0x1p-100f;
  if (A < zero_limit) {
    *bs = 0.0f;
    for (int g = 0; g < ORACLE_BLOCK / G; ++g) gs[g] = 0;
    for (int i = 0; i < ORACLE_BLOCK; ++i) { code[i] = 0; if (q_out) q_out[i] = 0.0f; }
    return;
  }
  float s_b = A / 2688.0f;
  float t_b = s_b * 6.0f;
  *bs = s_b;
  for (int g = 0; g < ORACLE_BLOCK / G; ++g) {
    const float* yg = y + g * G;
    float amax = 0.0f;
    for (int i = 0; i < G; ++i) {
      float a = fabsf(yg[i]);
      if (a > amax) amax = a;
    }
    float r = amax / t_b;
    uint8_t s_g = oracle_e4m3_encode(r);
    gs[g] = s_g;
    float S = oracle_e4m3_decode(s_g) * s_b;
    float inv = (S > 0.0f) ? 1.0f / S : 0.0f;
    for (int i = 0; i < G; ++i) {
      float q = yg[i] * inv;
      code[g * G + i] = oracle_e2m1_encode(q);
      if (q_out) q_out[g * G + i] = q;
    }
  }
}

/* Decoded transform-domain values of one block: x~ = grid(code) * S, S = value(s_g) * s_b. */
static void dequantize_block(const uint8_t* packed, const uint8_t* gs, float s_b, int G,
                             float* out) {
  for (int i = 0; i < ORACLE_BLOCK; ++i) {
    uint8_t byte = packed[i / 2];
    uint8_t c = (i % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
    float S = oracle_e4m3_decode(gs[i / G]) * s_b;
    out[i] = oracle_e2m1_decode(c) * S;
  }
}

/* Microscaled quantisation of one block (8 groups of 32): per group X = E8M0 scale of
 * amax, q = y / X (a division by a power of two), code = E2M1(q). No block-level guard:
 * a group of zeros gets scale code 0 and codes 0x0 / 0x8 by the sign of each zero. */
static void quantize_block_mx(const float* y, uint8_t* code, uint8_t* gs, float* q_out) {
  for (int g = 0; g < ORACLE_BLOCK / 32; ++g) {
    const float* yg = y + g * 32;
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
      float a = fabsf(yg[i]);
      if (a > amax) amax = a;
    }
    uint8_t sc = oracle_e8m0_scale(amax);
    gs[g] = sc;
    float X = oracle_e8m0_decode(sc);
    for (int i = 0; i < 32; ++i) {
      float q = yg[i] / X;
      code[g * 32 + i] = oracle_e2m1_encode(q);
      if (q_out) q_out[g * 32 + i] = q;
    }
  }
}

/* Decoded transform-domain values of a microscaled block: x~ = grid(code) * X. */
static void dequantize_block_mx(const uint8_t* packed, const uint8_t* gs, float* out) {
  for (int i = 0; i < ORACLE_BLOCK; ++i) {
    uint8_t byte = packed[i / 2];
    uint8_t c = (i % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
    out[i] = oracle_e2m1_decode(c) * oracle_e8m0_decode(gs[i / 32]);
  }
}

/* Two codes per byte, the even element in the low nibble [P3 "packed two per byte"]. */
static void pack_block(const uint8_t* code, uint8_t* packed) {
  for (int k = 0; k < ORACLE_BLOCK / 2; ++k)
    packed[k] = (uint8_t)(code[2 * k] | (code[2 * k + 1] << 4));
}

/* ---------------------------------------------------------------- whole tensors */

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int t) {
#ifdef _OPENMP
  if (t > 0) omp_set_num_threads(t);
#else
  (void)t;
#endif
}

/* Compress of BF16 (x16) or FP32 (x32) input, exactly one of them non-NULL: per block,
 * widen (BF16) or take (FP32) the values, FWHT (if fwht), quantise, pack. Returns 0, or -1
 * on invalid arguments. q_out (optional) receives the pre-rounding q of every element. */
static int compress_any(const uint16_t* x16, const float* x32, int64_t n, uint8_t* payload, int G, int fwht,
                        int mx, float* q_out) {
  if (!valid(n, G, mx) || (fwht != 0 && fwht != 1) || (!x16 && !x32) || !payload) return -1;
  const int64_t m = padded(n), nb = m / ORACLE_BLOCK;
  uint8_t* codes = payload;
  uint8_t* gsc = payload + oracle_gscale_offset(n, G, mx);
  float* bsc = (float*)(payload + oracle_bscale_offset(n, G, mx));
  memset(gsc + m / G, 0, (size_t)(pad16(m / G) - m / G));
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nb; ++b) {
    float y[ORACLE_BLOCK];
    uint8_t code[ORACLE_BLOCK];
    float s_b;
    for (int i = 0; i < ORACLE_BLOCK; ++i) {
      const int64_t e = b * ORACLE_BLOCK + i;
      y[i] = e >= n ? 0.0f : x16 ? oracle_bf16_to_f32(x16[e]) : x32[e];
    }
    if (fwht) oracle_fwht256(y);
    float qb[ORACLE_BLOCK];
    if (mx) {
      quantize_block_mx(y, code, gsc + b * (ORACLE_BLOCK / 32), qb);
    } else {
      quantize_block(y, G, code, gsc + b * (ORACLE_BLOCK / G), &s_b, qb);
      memcpy(&bsc[b], &s_b, 4);
    }
    if (q_out)
      for (int i = 0; i < ORACLE_BLOCK && b * ORACLE_BLOCK + i < n; ++i) q_out[b * ORACLE_BLOCK + i] = qb[i];
    pack_block(code, codes + b * (ORACLE_BLOCK / 2));
  }
  return 0;
}

/* Compress: per block, widen BF16 to FP32, FWHT (if fwht), quantise, pack. */
int oracle_compress(const uint16_t* x, int64_t n, uint8_t* payload, int G, int fwht, int mx,
                    float* q_out) {
  if (!x) return -1;
  return compress_any(x, NULL, n, payload, G, fwht, mx, q_out);
}

/* Compress of FP32 input: the same steps with the input used as it is (no widening). */
int oracle_compress_f32(const float* x, int64_t n, uint8_t* payload, int G, int fwht, int mx,
                        float* q_out) {
  if (!x) return -1;
  return compress_any(NULL, x, n, payload, G, fwht, mx, q_out);
}

/* Decode block b of a payload to 256 FP32 values: x~ = grid(code) * S, then the inverse
 * FWHT (mirror stage order) when fwht is set. */
static void decode_all(const uint8_t* payload, int64_t n, int G, int fwht, int mx, int64_t b,
                       float* xh) {
  const uint8_t* codes = payload;
  const uint8_t* gsc = payload + oracle_gscale_offset(n, G, mx);
  if (mx) {
    dequantize_block_mx(codes + b * (ORACLE_BLOCK / 2), gsc + b * (ORACLE_BLOCK / 32), xh);
  } else {
    const uint8_t* bsc = payload + oracle_bscale_offset(n, G, mx);
    float s_b;
    memcpy(&s_b, bsc + 4 * b, 4);
    dequantize_block(codes + b * (ORACLE_BLOCK / 2), gsc + b * (ORACLE_BLOCK / G), s_b, G, xh);
  }
  if (fwht) oracle_ifwht256(xh);
}

/* Decompress-accumulate: dst = beta ? dst + x^ : x^ (dtype 0: bfloat16 dst, the sum formed
 * in FP32 and rounded once to nearest even; dtype 1: float32 dst). The receive side of the
 * compressed AllReduce [P3 "Read it as"]. Returns 0, or -1 on invalid arguments. */
int oracle_decompress_accumulate(const uint8_t* payload, int64_t n, void* dst, int dtype,
                                 int beta, int G, int fwht, int mx) {
  if (!valid(n, G, mx) || (fwht != 0 && fwht != 1) || (dtype != 0 && dtype != 1) ||
      (beta != 0 && beta != 1) || !payload || !dst)
    return -1;
  const int64_t nb = padded(n) / ORACLE_BLOCK;
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nb; ++b) {
    float xh[ORACLE_BLOCK];
    decode_all(payload, n, G, fwht, mx, b, xh);
    for (int i = 0; i < ORACLE_BLOCK && b * ORACLE_BLOCK + i < n; ++i) {
      int64_t e = b * ORACLE_BLOCK + i;
      if (dtype == 0) {
        uint16_t* d = (uint16_t*)dst;
        float v = beta ? oracle_bf16_to_f32(d[e]) + xh[i] : xh[i];
        d[e] = oracle_f32_to_bf16(v);
      } else {
        float* d = (float*)dst;
        d[e] = beta ? d[e] + xh[i] : xh[i];
      }
    }
  }
  return 0;
}

/* Roundtrip: y = bf16(decode(compress(x))), the definition of the fused fake-quantizer. */
int oracle_roundtrip(const uint16_t* x, int64_t n, uint16_t* y, int G, int fwht, int mx) {
  int64_t bytes = oracle_payload_bytes(n, G, mx);
  if (bytes == 0 || !x || !y) return -1;
  uint8_t* p = (uint8_t*)malloc((size_t)bytes);
  if (!p) return -2;
  int rc = oracle_compress(x, n, p, G, fwht, mx, NULL);
  if (rc == 0) rc = oracle_decompress_accumulate(p, n, y, 0, 0, G, fwht, mx);
  free(p);
  return rc;
}

/* FP32 roundtrip: y = decode(compress_f32(x)) in FP32 (no BF16 rounding of the output). */
int oracle_roundtrip_f32(const float* x, int64_t n, float* y, int G, int fwht, int mx) {
  int64_t bytes = oracle_payload_bytes(n, G, mx);
  if (bytes == 0 || !x || !y) return -1;
  uint8_t* p = (uint8_t*)malloc((size_t)bytes);
  if (!p) return -2;
  int rc = oracle_compress_f32(x, n, p, G, fwht, mx, NULL);
  if (rc == 0) rc = oracle_decompress_accumulate(p, n, y, 1, 0, G, fwht, mx);
  free(p);
  return rc;
}

/* Emulated R-way reduce: for each element z = x~_0 + x~_1 + ... in rank order (FP32,
 * decoded in the transform domain, no inverse FWHT), then the block is quantised and
 * packed again with no forward FWHT. [P3 "Read it as": the tensor-parallel AllReduce]
 * Returns 0, or -1 on invalid arguments. */
int oracle_reduce_requantize(const uint8_t* const* payloads, int R, int64_t n, uint8_t* out,
                             int G, int mx, float* q_out) {
  if (!valid(n, G, mx) || R < 1 || R > ORACLE_MAX_RANKS || !payloads || !out) return -1;
  for (int r = 0; r < R; ++r)
    if (!payloads[r]) return -1;
  const int64_t m = padded(n), nb = m / ORACLE_BLOCK;
  uint8_t* codes = out;
  uint8_t* gsc = out + oracle_gscale_offset(n, G, mx);
  float* bsc = (float*)(out + oracle_bscale_offset(n, G, mx));
  memset(gsc + m / G, 0, (size_t)(pad16(m / G) - m / G));
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nb; ++b) {
    float z[ORACLE_BLOCK], xr[ORACLE_BLOCK];
    uint8_t code[ORACLE_BLOCK];
    float s_b;
    decode_all(payloads[0], n, G, 0, mx, b, z);
    for (int r = 1; r < R; ++r) {
      decode_all(payloads[r], n, G, 0, mx, b, xr);
      for (int i = 0; i < ORACLE_BLOCK; ++i) z[i] = z[i] + xr[i];
    }
    float qb[ORACLE_BLOCK];
    if (mx) {
      quantize_block_mx(z, code, gsc + b * (ORACLE_BLOCK / 32), qb);
    } else {
      quantize_block(z, G, code, gsc + b * (ORACLE_BLOCK / G), &s_b, qb);
      memcpy(&bsc[b], &s_b, 4);
    }
    if (q_out)
      for (int i = 0; i < ORACLE_BLOCK && b * ORACLE_BLOCK + i < n; ++i) q_out[b * ORACLE_BLOCK + i] = qb[i];
    pack_block(code, codes + b * (ORACLE_BLOCK / 2));
  }
  return 0;
}

/* ---------------------------------------------------------------- array helpers for pins */

void oracle_e4m3_encode_array(const float* r, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(r[i]);
}

void oracle_e2m1_encode_array(const float* q, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(q[i]);
}

void oracle_e8m0_scale_array(const float* a, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e8m0_scale(a[i]);
}

void oracle_bf16_round_array(const float* f, uint16_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(f[i]);
}

/* Forward (inverse = 0) or inverse (inverse = 1) FWHT of nblk consecutive 256-element
 * blocks, in place. */
void oracle_fwht256_array(float* v, int64_t nblk, int inverse) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblk; ++b) {
    if (inverse) oracle_ifwht256(v + b * ORACLE_BLOCK);
    else oracle_fwht256(v + b * ORACLE_BLOCK);
  }
}

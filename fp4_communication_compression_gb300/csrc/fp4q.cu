// fp4q.cu - GB300 (sm_103a) kernels and C ABI of the FP4 communication codec.
//
// The method: "FP4Quant: Efficient 4-Bit Communication Compression for Model-Parallel LLM
// Training" (shd-paper.top summary, English abstract and technical framework): a hybrid
// two-level FWHT, micro-grouped dual-scale FP4 quantization and warp-cooperative packing of
// the tensors the tensor-parallel AllReduce exchanges ("4-bit compression speeds up LLM
// training by 56 percent", zot.news, lead paragraph and "Read it as"). The numeric contract
// (block 256, G = 16/32, E4M3 x FP32 scales, ties to even, payload layout, stage orders) is
// stated once in include/fp4q.h; every kernel here reproduces it bit for bit.
//
// Thread mapping (all kernels). A warp owns a tile of 8 consecutive 256-element blocks.
// Lane L works on block L >> 2 of the tile with 3 partner lanes; a block is a 16 x 16
// matrix M[g][p] (g = 16-element group, p = position in the group).
//   layout A: lane (L & 3) = a holds rows 4a .. 4a+3      (all p, g bits 0-1 in registers)
//   layout B: lane (L & 3) = b holds rows b, b+4, b+8, b+12 (all p, g bits 2-3 in registers)
// Values are kept as float2 pairs (p even, p odd) so that the butterflies run on the
// packed FP32x2 pipe (add/sub/mul.rn.f32x2). FWHT strides 1..32 act on layout A, strides
// 64 and 128 on layout B; one transpose through a padded, bank-conflict-free shared buffer
// (73 16-byte units per block) moves between them. Group and block maxima reduce over the
// 4 lanes of a block with two xor-shuffles.
//
// Exactness. Every floating-point step is a separately rounded FP32 operation: the file is
// built with -fmad=false, divisions and reciprocals are the IEEE-rounded __fdiv_rn and
// __frcp_rn, packed ops carry .rn, and no operation is reassociated. Two rewrites are
// bit-identical to the contract's literal order and are used to save work:
//   * compress never multiplies y by 1/16: max|y| = fl(max|z| / 16) because rounding is
//     monotone, and q = y * inv = z * (inv / 16) exactly whenever a code can depend on it
//     (inv / 16 is exact for |x| < 2^120; a y that underflows gives |q| < 2^-17, code +-0
//     with the sign of z either way);
//   * all E2M1 / E4M3 rounding is done by the sm_100-family cvt instructions, which round
//     to nearest even with saturation exactly as the contract states.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "fp4q.h"

namespace {

constexpr int kBlock = 256;
constexpr int kTileBlocks = 8;                  // 256-element blocks per warp tile
constexpr int kCtaWarps = 8;                    // warps per CTA
constexpr int kUnitsPerBlock = 73;              // 16-byte units per block in the transpose buffer
constexpr int kWarpSmemBytes = kTileBlocks * kUnitsPerBlock * 16;
constexpr int kCtaSmemBytes = kCtaWarps * kWarpSmemBytes;
constexpr float kZeroLimit = 2688.0f * 0x1p-100f;   // all-zero block guard on A_b
constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------------ packed FP32x2 ops

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 A, B, C;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t"
      "add.rn.f32x2 C, A, B;\n\tmov.b64 {%0, %1}, C;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 A, B, C;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t"
      "sub.rn.f32x2 C, A, B;\n\tmov.b64 {%0, %1}, C;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{.reg .b64 A, B, C;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t"
      "mul.rn.f32x2 C, A, B;\n\tmov.b64 {%0, %1}, C;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// (a, b) <- (a + b, a - b) on two pairs at once.
__device__ __forceinline__ void bfly2(float2& a, float2& b) {
  float2 s = add2(a, b), d = sub2(a, b);
  a = s;
  b = d;
}
// (x, y) <- (x + y, x - y) inside one pair (stride-1 butterfly).
__device__ __forceinline__ void bfly_in(float2& v) {
  float s = __fadd_rn(v.x, v.y), d = __fsub_rn(v.x, v.y);
  v = make_float2(s, d);
}

// ------------------------------------------------------------------ format conversions

// bfloat16 pair (low half = even element) -> float2, exact.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// float2 -> bfloat16 pair, round to nearest even (low half = x).
__device__ __forceinline__ uint32_t f2_to_bf16x2(float2 v) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(v.y), "f"(v.x));
  return r;
}
// Four value pairs -> one word of eight E2M1 codes; element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1_pack8(float2 q0, float2 q1, float2 q2, float2 q3) {
  uint32_t w;
  asm("{.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};}"
      : "=r"(w)
      : "f"(q0.x), "f"(q0.y), "f"(q1.x), "f"(q1.y), "f"(q2.x), "f"(q2.y), "f"(q3.x), "f"(q3.y));
  return w;
}
// One word of eight E2M1 codes -> the eight grid values (exact), element 2i+e in out[i].e.
__device__ __forceinline__ void e2m1_word_to_f2(uint32_t w, float2 out[4]) {
  uint32_t h[4];
  asm("{.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 t = *reinterpret_cast<__half2*>(&h[i]);
    out[i] = make_float2(__low2float(t), __high2float(t));
  }
}
// Two non-negative ratios -> two E4M3 codes (round to nearest even, saturate at 448);
// the code of lo is the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two E4M3 codes (low byte first) -> their values, exact.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t codes16) {
  uint32_t h2;
  uint16_t c = (uint16_t)codes16;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return make_float2(__low2float(h), __high2float(h));
}

// ------------------------------------------------------------------ FWHT pieces

// Rows of one lane: v[k][j] = pair j (positions 2j, 2j+1) of the lane's k-th row.
typedef float2 Rows[4][8];

// Level 1 (strides 1, 2, 4, 8 inside each row), forward order.
__device__ __forceinline__ void level1_fwd(Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int j = 0; j < 8; ++j) bfly_in(v[k][j]);
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!(j & h)) bfly2(v[k][j], v[k][j + h]);
  }
}
// Level 1 in mirror order (strides 8, 4, 2, 1).
__device__ __forceinline__ void level1_inv(Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!(j & h)) bfly2(v[k][j], v[k][j + h]);
#pragma unroll
    for (int j = 0; j < 8; ++j) bfly_in(v[k][j]);
  }
}
// Butterflies between the lane's rows k and k + hk (hk = 1 or 2), all positions.
__device__ __forceinline__ void rows_bfly(Rows v, int hk) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (!(k & hk))
#pragma unroll
      for (int j = 0; j < 8; ++j) bfly2(v[k][j], v[k + hk][j]);
}

// Transpose buffer addressing: block region of 73 units, row r at unit
// 4r + 2(r >> 2) + 2((r >> 1) & 1). Layout A rows 4a+k sit at 18a + 4k + 2(k >> 1);
// layout B rows b+4k at 4b + 2(b >> 1) + 18k. Eight consecutive lanes (two blocks, four
// rows each) then always touch eight distinct 16-byte bank groups.
__device__ __forceinline__ int unitA(int blk, int a) { return kUnitsPerBlock * blk + 18 * a; }
__device__ __forceinline__ int unitB(int blk, int b) { return kUnitsPerBlock * blk + 4 * b + 2 * (b >> 1); }
__device__ __forceinline__ int offA(int k) { return 4 * k + 2 * (k >> 1); }
__device__ __forceinline__ int offB(int k) { return 18 * k; }

// Write the lane's 4 rows from one layout, read 4 rows of the other. toB: A -> B.
template <bool toB>
__device__ __forceinline__ void transpose(Rows v, float4* buf, int blk, int l4) {
  const int wbase = toB ? unitA(blk, l4) : unitB(blk, l4);
  const int rbase = toB ? unitB(blk, l4) : unitA(blk, l4);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int o = toB ? offA(k) : offB(k);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      buf[wbase + o + c] = make_float4(v[k][2 * c].x, v[k][2 * c].y, v[k][2 * c + 1].x, v[k][2 * c + 1].y);
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int o = toB ? offB(k) : offA(k);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float4 t = buf[rbase + o + c];
      v[k][2 * c] = make_float2(t.x, t.y);
      v[k][2 * c + 1] = make_float2(t.z, t.w);
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ quantisation

// Result of quantising the lane's 4 rows of one block.
struct Quant {
  uint32_t code[4][2];   // 16 codes per row, 2 words per row
  uint32_t sg;           // the 4 group-scale codes of the lane's rows, row k in byte k
  float S[4];            // decode scale of each row's group
  float sb;              // block scale
};

// Dual-scale quantisation of the lane's rows (rows in layout A if !LB, layout B if LB).
// FOLD: the values are the unnormalised transform z = 16 y (see the file header).
template <int G, bool LB, bool FOLD>
__device__ __forceinline__ void quantize(const Rows v, Quant& o) {
  float am[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fmaxf(fabsf(v[k][j].x), fabsf(v[k][j].y)));
    am[k] = m;
  }
  float A = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));
  A = fmaxf(A, __shfl_xor_sync(kFull, A, 1));
  A = fmaxf(A, __shfl_xor_sync(kFull, A, 2));
  if (G == 32) {
    // a group is two consecutive rows: inside the lane in layout A, across lanes b, b^1 in B
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float other = LB ? __shfl_xor_sync(kFull, am[k], 1) : am[k ^ 1];
      am[k] = fmaxf(am[k], other);
    }
  }
  if (FOLD) {
    A = __fmul_rn(A, 0.0625f);
#pragma unroll
    for (int k = 0; k < 4; ++k) am[k] = __fmul_rn(am[k], 0.0625f);
  }
  const bool zero = !(A >= kZeroLimit);
  const float sb = zero ? 0.0f : __fdiv_rn(A, 2688.0f);
  const float tb = zero ? 1.0f : __fmul_rn(sb, 6.0f);
  float r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) r[k] = __fdiv_rn(am[k], tb);
  uint32_t c01 = e4m3x2(r[0], r[1]), c23 = e4m3x2(r[2], r[3]);
  if (zero) c01 = c23 = 0u;
  const float2 s01 = e4m3x2_to_f2(c01), s23 = e4m3x2_to_f2(c23);
  const float sgv[4] = {s01.x, s01.y, s23.x, s23.y};
  o.sg = c01 | (c23 << 16);
  o.sb = sb;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float S = __fmul_rn(sgv[k], sb);
    o.S[k] = S;
    float inv = S > 0.0f ? __frcp_rn(S) : 0.0f;
    if (FOLD) inv = __fmul_rn(inv, 0.0625f);
    const float2 iv = make_float2(inv, inv);
    uint32_t w0 = e2m1_pack8(mul2(v[k][0], iv), mul2(v[k][1], iv), mul2(v[k][2], iv), mul2(v[k][3], iv));
    uint32_t w1 = e2m1_pack8(mul2(v[k][4], iv), mul2(v[k][5], iv), mul2(v[k][6], iv), mul2(v[k][7], iv));
    if (zero) w0 = w1 = 0u;
    o.code[k][0] = w0;
    o.code[k][1] = w1;
  }
}

// Decode the lane's 4 rows from codes and per-row scales: x~ = grid(code) * S.
// The products use the IEEE __fmul_rn, which is never contracted: a packed mul.rn.f32x2
// whose result feeds a packed add was observed to be fused into an FMA by the toolchain
// (even with .rn and --fmad=false), which breaks bit parity in the sums that follow.
__device__ __forceinline__ void dequantize(const uint32_t code[4][2], const float S[4], Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      float2 g[4];
      e2m1_word_to_f2(code[k][w], g);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[k][4 * w + i] = make_float2(__fmul_rn(g[i].x, S[k]), __fmul_rn(g[i].y, S[k]));
    }
  }
}

// x^ = v / 16. A packed multiply is kept only where the product feeds a conversion or a
// store; before an accumulation the IEEE scalar multiply is used (see dequantize).
template <bool BEFORE_ADD>
__device__ __forceinline__ void scale16(Rows v) {
  const float2 s16 = make_float2(0.0625f, 0.0625f);
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      v[k][j] = BEFORE_ADD ? make_float2(__fmul_rn(v[k][j].x, 0.0625f), __fmul_rn(v[k][j].y, 0.0625f))
                           : mul2(v[k][j], s16);
}

// ------------------------------------------------------------------ payload addressing

struct Payload {
  uint8_t* codes;      // n/2 bytes
  uint8_t* gsc;        // n/G bytes (+ padding to 16)
  float* bsc;          // n/256 floats
  int64_t nb;          // number of blocks
};

__host__ __device__ inline int64_t pad16(int64_t b) { return (b + 15) / 16 * 16; }

__host__ __device__ inline Payload payload_of(void* base, int64_t n, int G) {
  uint8_t* p = static_cast<uint8_t*>(base);
  Payload s;
  s.codes = p;
  s.gsc = p + n / 2;
  s.bsc = reinterpret_cast<float*>(p + n / 2 + pad16(n / G));
  s.nb = n / 256;
  return s;
}

// Row of the lane's k-th row inside its block.
template <bool LB>
__device__ __forceinline__ int row_of(int l4, int k) { return LB ? l4 + 4 * k : 4 * l4 + k; }

// Store the lane's part of a quantised block (block index gb).
template <int G, bool LB>
__device__ __forceinline__ void store_block(const Payload& P, int64_t gb, int l4, const Quant& q) {
  if (LB) {
    // rows l4 + 4k: four separate 8-byte pieces
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint2*>(P.codes + gb * 128 + row_of<true>(l4, k) * 8) =
          make_uint2(q.code[k][0], q.code[k][1]);
  } else {
    // rows 4 l4 .. 4 l4 + 3 are 32 contiguous bytes
    uint4* dst = reinterpret_cast<uint4*>(P.codes + gb * 128 + l4 * 32);
    dst[0] = make_uint4(q.code[0][0], q.code[0][1], q.code[1][0], q.code[1][1]);
    dst[1] = make_uint4(q.code[2][0], q.code[2][1], q.code[3][0], q.code[3][1]);
  }
  if (G == 16) {
    if (LB) {
#pragma unroll
      for (int k = 0; k < 4; ++k) P.gsc[gb * 16 + l4 + 4 * k] = (uint8_t)(q.sg >> (8 * k));
    } else {
      *reinterpret_cast<uint32_t*>(P.gsc + gb * 16 + 4 * l4) = q.sg;
    }
  } else {
    if (LB) {
      // group m = (l4 + 4k) / 2 is shared by lanes l4 and l4 ^ 1; the even lane writes it
      if (!(l4 & 1)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) P.gsc[gb * 8 + ((l4 + 4 * k) >> 1)] = (uint8_t)(q.sg >> (8 * k));
      }
    } else {
      // rows 4 l4 + {0,1} form group 2 l4, rows 4 l4 + {2,3} group 2 l4 + 1
      const uint16_t two = (uint16_t)((q.sg & 0xffu) | ((q.sg >> 8) & 0xff00u));
      *reinterpret_cast<uint16_t*>(P.gsc + gb * 8 + 2 * l4) = two;
    }
  }
  if (l4 == 0) {
    P.bsc[gb] = q.sb;
    // G = 32 with an odd block count: the group-scale segment ends 8 bytes short of a
    // 16-byte boundary; the last block zeroes that padding
    if (G == 32 && (P.nb & 1) && gb == P.nb - 1)
      *reinterpret_cast<uint2*>(P.gsc + 8 * P.nb) = make_uint2(0u, 0u);
  }
}

// Load the lane's part of a payload block: codes of its 4 rows and each row's decode scale.
template <int G, bool LB>
__device__ __forceinline__ void load_block(const Payload& P, int64_t gb, int l4, uint32_t code[4][2],
                                           float S[4]) {
  if (LB) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint2 c = __ldg(reinterpret_cast<const uint2*>(P.codes + gb * 128 + (l4 + 4 * k) * 8));
      code[k][0] = c.x;
      code[k][1] = c.y;
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(P.codes + gb * 128 + l4 * 32);
    uint4 c0 = __ldg(src), c1 = __ldg(src + 1);
    code[0][0] = c0.x; code[0][1] = c0.y; code[1][0] = c0.z; code[1][1] = c0.w;
    code[2][0] = c1.x; code[2][1] = c1.y; code[3][0] = c1.z; code[3][1] = c1.w;
  }
  uint32_t sg;   // the 4 rows' group-scale codes, row k in byte k
  if (G == 16) {
    if (LB) {
      // row l4 + 4k uses byte l4 of word k
      uint4 all = __ldg(reinterpret_cast<const uint4*>(P.gsc + gb * 16));
      const uint32_t sel = 0x4440u | (uint32_t)l4;
      sg = __byte_perm(all.x, 0, sel) | (__byte_perm(all.y, 0, sel) << 8) |
           (__byte_perm(all.z, 0, sel) << 16) | (__byte_perm(all.w, 0, sel) << 24);
    } else {
      sg = __ldg(reinterpret_cast<const uint32_t*>(P.gsc + gb * 16 + 4 * l4));
    }
  } else {
    if (LB) {
      uint2 all = __ldg(reinterpret_cast<const uint2*>(P.gsc + gb * 8));
      // row l4 + 4k belongs to group (l4 >> 1) + 2k: byte (l4 >> 1) + 2(k & 1) of word k >> 1
      const uint32_t s0 = 0x4440u | (uint32_t)(l4 >> 1), s2 = s0 + 2;
      sg = __byte_perm(all.x, 0, s0) | (__byte_perm(all.x, 0, s2) << 8) |
           (__byte_perm(all.y, 0, s0) << 16) | (__byte_perm(all.y, 0, s2) << 24);
    } else {
      const uint32_t two = __ldg(reinterpret_cast<const uint16_t*>(P.gsc + gb * 8 + 2 * l4));
      sg = (two & 0xffu) * 0x0101u | ((two >> 8) & 0xffu) * 0x01010000u;
    }
  }
  const float sb = __ldg(P.bsc + gb);
  const float2 s01 = e4m3x2_to_f2(sg & 0xffffu), s23 = e4m3x2_to_f2(sg >> 16);
  S[0] = __fmul_rn(s01.x, sb);
  S[1] = __fmul_rn(s01.y, sb);
  S[2] = __fmul_rn(s23.x, sb);
  S[3] = __fmul_rn(s23.y, sb);
}

// Load the lane's 4 rows of bfloat16 input in layout A (64 contiguous elements).
__device__ __forceinline__ void load_rows_bf16_A(const uint16_t* x, int64_t gb, int a, Rows v) {
  const uint4* src = reinterpret_cast<const uint4*>(x + gb * kBlock + a * 64);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 t = __ldg(src + 2 * k + h);
      v[k][4 * h + 0] = bf16x2_to_f2(t.x);
      v[k][4 * h + 1] = bf16x2_to_f2(t.y);
      v[k][4 * h + 2] = bf16x2_to_f2(t.z);
      v[k][4 * h + 3] = bf16x2_to_f2(t.w);
    }
  }
}

__device__ __forceinline__ void zero_rows(Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j) v[k][j] = make_float2(0.0f, 0.0f);
}

// Accumulate decoded rows (layout A: 64 contiguous elements per lane) into dst.
template <int DT, int BETA>
__device__ __forceinline__ void accumulate_A(void* dst, int64_t gb, int a, const Rows v) {
  if (DT == FP4Q_BF16) {
    uint4* d = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + gb * kBlock + a * 64);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float2 x0 = v[k][4 * h], x1 = v[k][4 * h + 1], x2 = v[k][4 * h + 2], x3 = v[k][4 * h + 3];
        if (BETA) {
          uint4 o = d[2 * k + h];
          x0 = add2(bf16x2_to_f2(o.x), x0);
          x1 = add2(bf16x2_to_f2(o.y), x1);
          x2 = add2(bf16x2_to_f2(o.z), x2);
          x3 = add2(bf16x2_to_f2(o.w), x3);
        }
        d[2 * k + h] = make_uint4(f2_to_bf16x2(x0), f2_to_bf16x2(x1), f2_to_bf16x2(x2), f2_to_bf16x2(x3));
      }
    }
  } else {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(dst) + gb * kBlock + a * 64);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float2 x0 = v[k][2 * h], x1 = v[k][2 * h + 1];
        if (BETA) {
          float4 o = d[4 * k + h];
          x0 = add2(make_float2(o.x, o.y), x0);
          x1 = add2(make_float2(o.z, o.w), x1);
        }
        d[4 * k + h] = make_float4(x0.x, x0.y, x1.x, x1.y);
      }
    }
  }
}

// ------------------------------------------------------------------ kernels

struct TileLoop {
  int64_t tiles;     // number of 8-block tiles
  int64_t nb;        // number of 256-element blocks
};

__device__ __forceinline__ int64_t warp_global() {
  return (int64_t)blockIdx.x * kCtaWarps + (threadIdx.x >> 5);
}
__device__ __forceinline__ int64_t warp_count() { return (int64_t)gridDim.x * kCtaWarps; }

// K1: compress. x (bfloat16, n) -> payload.
template <int G, int FWHT>
__global__ void __launch_bounds__(kCtaWarps * 32)
compress_kernel(const uint16_t* __restrict__ x, Payload P, TileLoop T) {
  extern __shared__ __align__(16) uint8_t smem[];
  float4* buf = reinterpret_cast<float4*>(smem + (threadIdx.x >> 5) * kWarpSmemBytes);
  const int lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  for (int64_t t = warp_global(); t < T.tiles; t += warp_count()) {
    const int64_t gb = t * kTileBlocks + blk;
    const bool valid = gb < T.nb;
    Rows v;
    if (valid) load_rows_bf16_A(x, gb, l4, v); else zero_rows(v);
    Quant q;
    if (FWHT) {
      level1_fwd(v);
      rows_bfly(v, 1);             // h = 16
      rows_bfly(v, 2);             // h = 32
      transpose<true>(v, buf, blk, l4);
      rows_bfly(v, 1);             // h = 64
      rows_bfly(v, 2);             // h = 128
      quantize<G, true, true>(v, q);
      if (valid) store_block<G, true>(P, gb, l4, q);
    } else {
      quantize<G, false, false>(v, q);
      if (valid) store_block<G, false>(P, gb, l4, q);
    }
  }
}

// K2: decompress-accumulate. payload -> dst (dtype DT), dst = BETA ? dst + x^ : x^.
template <int G, int FWHT, int DT, int BETA>
__global__ void __launch_bounds__(kCtaWarps * 32)
decompress_kernel(Payload P, void* __restrict__ dst, TileLoop T) {
  extern __shared__ __align__(16) uint8_t smem[];
  float4* buf = reinterpret_cast<float4*>(smem + (threadIdx.x >> 5) * kWarpSmemBytes);
  const int lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  for (int64_t t = warp_global(); t < T.tiles; t += warp_count()) {
    const int64_t gb = t * kTileBlocks + blk;
    const bool valid = gb < T.nb;
    uint32_t code[4][2];
    float S[4];
    Rows v;
    if (FWHT) {
      if (valid) {
        load_block<G, true>(P, gb, l4, code, S);
        dequantize(code, S, v);
      } else {
        zero_rows(v);
      }
      rows_bfly(v, 2);             // h = 128
      rows_bfly(v, 1);             // h = 64
      transpose<false>(v, buf, blk, l4);
      rows_bfly(v, 2);             // h = 32
      rows_bfly(v, 1);             // h = 16
      level1_inv(v);
      scale16<BETA != 0>(v);
    } else {
      if (!valid) continue;
      load_block<G, false>(P, gb, l4, code, S);
      dequantize(code, S, v);
    }
    if (valid) accumulate_A<DT, BETA>(dst, gb, l4, v);
  }
}

// K3: fused roundtrip. x (bfloat16) -> y = bf16(decode(compress(x))), no payload.
template <int G, int FWHT>
__global__ void __launch_bounds__(kCtaWarps * 32)
roundtrip_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ y, TileLoop T) {
  extern __shared__ __align__(16) uint8_t smem[];
  float4* buf = reinterpret_cast<float4*>(smem + (threadIdx.x >> 5) * kWarpSmemBytes);
  const int lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  for (int64_t t = warp_global(); t < T.tiles; t += warp_count()) {
    const int64_t gb = t * kTileBlocks + blk;
    const bool valid = gb < T.nb;
    Rows v;
    if (valid) load_rows_bf16_A(x, gb, l4, v); else zero_rows(v);
    Quant q;
    if (FWHT) {
      level1_fwd(v);
      rows_bfly(v, 1);
      rows_bfly(v, 2);
      transpose<true>(v, buf, blk, l4);
      rows_bfly(v, 1);
      rows_bfly(v, 2);
      quantize<G, true, true>(v, q);
      dequantize(q.code, q.S, v);
      rows_bfly(v, 2);
      rows_bfly(v, 1);
      transpose<false>(v, buf, blk, l4);
      rows_bfly(v, 2);
      rows_bfly(v, 1);
      level1_inv(v);
      scale16<false>(v);
    } else {
      quantize<G, false, false>(v, q);
      dequantize(q.code, q.S, v);
    }
    if (valid) accumulate_A<FP4Q_BF16, 0>(y, gb, l4, v);
  }
}

// K4: emulated R-way reduce. R payloads -> transform-domain FP32 sum in rank order ->
// requantised payload (no transform).
struct RankPtrs {
  const uint8_t* p[FP4Q_MAX_RANKS];
};

template <int G>
__global__ void __launch_bounds__(kCtaWarps * 32)
reduce_kernel(RankPtrs in, int R, int64_t n, Payload out, TileLoop T) {
  const int lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  for (int64_t t = warp_global(); t < T.tiles; t += warp_count()) {
    const int64_t gb = t * kTileBlocks + blk;
    const bool valid = gb < T.nb;
    Rows z;
    if (valid) {
      uint32_t code[4][2];
      float S[4];
      load_block<G, false>(payload_of(const_cast<uint8_t*>(in.p[0]), n, G), gb, l4, code, S);
      dequantize(code, S, z);
#pragma unroll
      for (int r = 1; r < FP4Q_MAX_RANKS; ++r) {
        if (r >= R) break;
        Rows xr;
        load_block<G, false>(payload_of(const_cast<uint8_t*>(in.p[r]), n, G), gb, l4, code, S);
        dequantize(code, S, xr);
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int j = 0; j < 8; ++j) z[k][j] = add2(z[k][j], xr[k][j]);
      }
    } else {
      zero_rows(z);
    }
    Quant q;
    quantize<G, false, false>(z, q);
    if (valid) store_block<G, false>(out, gb, l4, q);
  }
}

// ------------------------------------------------------------------ host side

struct Launch {
  int grid;
  int smem;
};

int g_num_sms[64];

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (g_num_sms[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_num_sms[dev] = v;
  }
  return g_num_sms[dev];
}

// Persistent grid: as many CTAs as fit on all SMs at once, never more than the tiles need.
template <typename K>
fp4q_status plan(K kernel, int smem, int64_t tiles, Launch& L) {
  const int sms = num_sms();
  if (sms <= 0) return FP4Q_ERR_CUDA;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FP4Q_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCtaWarps * 32, smem) != cudaSuccess ||
      per_sm <= 0)
    return FP4Q_ERR_CUDA;
  const int64_t want = (tiles + kCtaWarps - 1) / kCtaWarps;
  const int64_t cap = (int64_t)per_sm * sms;
  L.grid = (int)(want < cap ? want : cap);
  L.smem = smem;
  return FP4Q_OK;
}

fp4q_status launched() {
  return cudaGetLastError() == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

fp4q_status check_params(const fp4q_params* p, int& G, int& fwht) {
  fp4q_params d = {FP4Q_GROUP_DEFAULT, FP4Q_BLOCK, 1};
  if (p) d = *p;
  if ((d.group != 16 && d.group != 32) || d.block != FP4Q_BLOCK || (d.fwht != 0 && d.fwht != 1))
    return FP4Q_ERR_PARAM;
  G = d.group;
  fwht = d.fwht;
  return FP4Q_OK;
}

bool size_ok(int64_t n) { return n > 0 && n % FP4Q_BLOCK == 0 && n < ((int64_t)1 << 40); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

TileLoop tiles_of(int64_t n) {
  TileLoop T;
  T.nb = n / FP4Q_BLOCK;
  T.tiles = (T.nb + kTileBlocks - 1) / kTileBlocks;
  return T;
}

template <int G, int F>
fp4q_status launch_compress(const void* x, int64_t n, void* payload, cudaStream_t s) {
  TileLoop T = tiles_of(n);
  auto k = compress_kernel<G, F>;
  Launch L;
  fp4q_status st = plan(k, F ? kCtaSmemBytes : 0, T.tiles, L);
  if (st != FP4Q_OK) return st;
  k<<<L.grid, kCtaWarps * 32, L.smem, s>>>(static_cast<const uint16_t*>(x), payload_of(payload, n, G), T);
  return launched();
}

template <int G, int F, int DT, int B>
fp4q_status launch_decompress(const void* payload, int64_t n, void* dst, cudaStream_t s) {
  TileLoop T = tiles_of(n);
  auto k = decompress_kernel<G, F, DT, B>;
  Launch L;
  fp4q_status st = plan(k, F ? kCtaSmemBytes : 0, T.tiles, L);
  if (st != FP4Q_OK) return st;
  k<<<L.grid, kCtaWarps * 32, L.smem, s>>>(payload_of(const_cast<void*>(payload), n, G), dst, T);
  return launched();
}

template <int G, int F>
fp4q_status launch_roundtrip(const void* x, int64_t n, void* y, cudaStream_t s) {
  TileLoop T = tiles_of(n);
  auto k = roundtrip_kernel<G, F>;
  Launch L;
  fp4q_status st = plan(k, F ? kCtaSmemBytes : 0, T.tiles, L);
  if (st != FP4Q_OK) return st;
  k<<<L.grid, kCtaWarps * 32, L.smem, s>>>(static_cast<const uint16_t*>(x), static_cast<uint16_t*>(y), T);
  return launched();
}

template <int G>
fp4q_status launch_reduce(const RankPtrs& in, int R, int64_t n, void* out, cudaStream_t s) {
  TileLoop T = tiles_of(n);
  auto k = reduce_kernel<G>;
  Launch L;
  fp4q_status st = plan(k, 0, T.tiles, L);
  if (st != FP4Q_OK) return st;
  k<<<L.grid, kCtaWarps * 32, 0, s>>>(in, R, n, payload_of(out, n, G), T);
  return launched();
}

size_t payload_bytes_of(int64_t n, int G) {
  return (size_t)(n / 2 + pad16(n / G) + 4 * (n / FP4Q_BLOCK));
}

}  // namespace

extern "C" {

size_t fp4q_payload_bytes(int64_t n, const fp4q_params* params) {
  int G, f;
  if (!size_ok(n) || check_params(params, G, f) != FP4Q_OK) return 0;
  return payload_bytes_of(n, G);
}

size_t fp4q_gscale_offset(int64_t n, const fp4q_params* params) {
  int G, f;
  if (!size_ok(n) || check_params(params, G, f) != FP4Q_OK) return 0;
  return (size_t)(n / 2);
}

size_t fp4q_bscale_offset(int64_t n, const fp4q_params* params) {
  int G, f;
  if (!size_ok(n) || check_params(params, G, f) != FP4Q_OK) return 0;
  return (size_t)(n / 2 + pad16(n / G));
}

fp4q_status fp4q_compress(const void* x_bf16, int64_t n, void* payload, const fp4q_params* params,
                          void* stream) {
  int G, F;
  fp4q_status st = check_params(params, G, F);
  if (st != FP4Q_OK) return st;
  if (!x_bf16 || !payload) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(x_bf16) || !aligned16(payload)) return FP4Q_ERR_ALIGN;
  if (overlap(x_bf16, (size_t)n * 2, payload, payload_bytes_of(n, G))) return FP4Q_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (G == 16) return F ? launch_compress<16, 1>(x_bf16, n, payload, s) : launch_compress<16, 0>(x_bf16, n, payload, s);
  return F ? launch_compress<32, 1>(x_bf16, n, payload, s) : launch_compress<32, 0>(x_bf16, n, payload, s);
}

fp4q_status fp4q_decompress_accumulate(const void* payload, int64_t n, void* dst, fp4q_dtype dtype,
                                       int32_t beta, const fp4q_params* params, void* stream) {
  int G, F;
  fp4q_status st = check_params(params, G, F);
  if (st != FP4Q_OK) return st;
  if ((dtype != FP4Q_BF16 && dtype != FP4Q_F32) || (beta != 0 && beta != 1)) return FP4Q_ERR_PARAM;
  if (!payload || !dst) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(payload) || !aligned16(dst)) return FP4Q_ERR_ALIGN;
  const size_t dbytes = (size_t)n * (dtype == FP4Q_BF16 ? 2 : 4);
  if (overlap(payload, payload_bytes_of(n, G), dst, dbytes)) return FP4Q_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int key = (G == 32) * 8 + F * 4 + (dtype == FP4Q_F32) * 2 + beta;
  switch (key) {
    case 0: return launch_decompress<16, 0, FP4Q_BF16, 0>(payload, n, dst, s);
    case 1: return launch_decompress<16, 0, FP4Q_BF16, 1>(payload, n, dst, s);
    case 2: return launch_decompress<16, 0, FP4Q_F32, 0>(payload, n, dst, s);
    case 3: return launch_decompress<16, 0, FP4Q_F32, 1>(payload, n, dst, s);
    case 4: return launch_decompress<16, 1, FP4Q_BF16, 0>(payload, n, dst, s);
    case 5: return launch_decompress<16, 1, FP4Q_BF16, 1>(payload, n, dst, s);
    case 6: return launch_decompress<16, 1, FP4Q_F32, 0>(payload, n, dst, s);
    case 7: return launch_decompress<16, 1, FP4Q_F32, 1>(payload, n, dst, s);
    case 8: return launch_decompress<32, 0, FP4Q_BF16, 0>(payload, n, dst, s);
    case 9: return launch_decompress<32, 0, FP4Q_BF16, 1>(payload, n, dst, s);
    case 10: return launch_decompress<32, 0, FP4Q_F32, 0>(payload, n, dst, s);
    case 11: return launch_decompress<32, 0, FP4Q_F32, 1>(payload, n, dst, s);
    case 12: return launch_decompress<32, 1, FP4Q_BF16, 0>(payload, n, dst, s);
    case 13: return launch_decompress<32, 1, FP4Q_BF16, 1>(payload, n, dst, s);
    case 14: return launch_decompress<32, 1, FP4Q_F32, 0>(payload, n, dst, s);
    default: return launch_decompress<32, 1, FP4Q_F32, 1>(payload, n, dst, s);
  }
}

fp4q_status fp4q_roundtrip(const void* x_bf16, int64_t n, void* y_bf16, const fp4q_params* params,
                           void* stream) {
  int G, F;
  fp4q_status st = check_params(params, G, F);
  if (st != FP4Q_OK) return st;
  if (!x_bf16 || !y_bf16) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(x_bf16) || !aligned16(y_bf16)) return FP4Q_ERR_ALIGN;
  if (overlap(x_bf16, (size_t)n * 2, y_bf16, (size_t)n * 2)) return FP4Q_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (G == 16) return F ? launch_roundtrip<16, 1>(x_bf16, n, y_bf16, s) : launch_roundtrip<16, 0>(x_bf16, n, y_bf16, s);
  return F ? launch_roundtrip<32, 1>(x_bf16, n, y_bf16, s) : launch_roundtrip<32, 0>(x_bf16, n, y_bf16, s);
}

fp4q_status fp4q_reduce_requantize(const void* const* payloads, int32_t R, int64_t n, void* out_payload,
                                   const fp4q_params* params, void* stream) {
  int G, F;
  fp4q_status st = check_params(params, G, F);
  if (st != FP4Q_OK) return st;
  if (R < 1 || R > FP4Q_MAX_RANKS) return FP4Q_ERR_PARAM;
  if (!payloads || !out_payload) return FP4Q_ERR_NULL;
  for (int r = 0; r < R; ++r)
    if (!payloads[r]) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(out_payload)) return FP4Q_ERR_ALIGN;
  for (int r = 0; r < R; ++r)
    if (!aligned16(payloads[r])) return FP4Q_ERR_ALIGN;
  const size_t pb = payload_bytes_of(n, G);
  for (int r = 0; r < R; ++r)
    if (overlap(payloads[r], pb, out_payload, pb)) return FP4Q_ERR_OVERLAP;
  RankPtrs in;
  for (int r = 0; r < FP4Q_MAX_RANKS; ++r) in.p[r] = r < R ? static_cast<const uint8_t*>(payloads[r]) : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return G == 16 ? launch_reduce<16>(in, R, n, out_payload, s) : launch_reduce<32>(in, R, n, out_payload, s);
}

const char* fp4q_status_string(fp4q_status status) {
  switch (status) {
    case FP4Q_OK: return "ok";
    case FP4Q_ERR_NULL: return "null pointer";
    case FP4Q_ERR_SIZE: return "n must be a positive multiple of 256 below 2^40";
    case FP4Q_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FP4Q_ERR_PARAM: return "invalid parameter (group, block, fwht, R, dtype or beta)";
    case FP4Q_ERR_OVERLAP: return "output overlaps an input";
    case FP4Q_ERR_CUDA: return "CUDA runtime error or failed launch";
  }
  return "unknown status";
}

int32_t fp4q_version(void) { return 100; }

}  // extern "C"

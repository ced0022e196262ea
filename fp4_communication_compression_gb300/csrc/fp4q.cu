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
// 64 and 128 on layout B; one transpose through a bank-conflict-free shared buffer moves
// between them. Compress and roundtrip move the two 8-column halves of a block one after
// the other through a padded 640-byte buffer (each lane addresses it as one base plus
// immediates, and the smaller buffer lets 5 CTAs share an SM); decompress and the tail
// kernels use a 1 KiB-per-block XOR-swizzled buffer (reduce has no transform). Group and block maxima reduce over
// the 4 lanes of a block with two xor-shuffles.
//
// Data movement and scheduling. Each warp streams its tiles through its own TMA pipeline
// (InPipe: mbarrier-tracked cp.async.bulk.tensor loads with bounded waits), and BF16 / FP32
// outputs leave by TMA stores from a swizzled staging buffer; where a tile needs one box per
// block (strided rows that do not hold whole tiles) eight lanes issue them. Tiles are
// assigned round robin to the warps of the grid; large tensors (compress and roundtrip of
// BF16 input, decompress-accumulate into BF16 with beta = 1, the reduce) instead run one CTA
// per SM whose warps claim the CTA's tiles from a shared-memory counter. Every kernel starts with
// griddepcontrol.wait and is launched with programmatic stream serialisation, so
// back-to-back codec kernels overlap launch and drain; for that overlap every kernel asks for
// the largest shared-memory carveout, and a cap on CTAs per SM is enforced by padding the
// dynamic shared memory (plan). The same kernels serve the E8M0 (microscaled) scales, FP32
// input, strided 2-D views (3-D tensor maps) and, through one-warp tail kernels, lengths that
// are not a multiple of 256.
//
// Exactness. Every floating-point step is a separately rounded FP32 operation: the file is
// built with -fmad=false, packed ops carry .rn, no operation is reassociated, and the scale
// chain's divisions and reciprocals are the correctly rounded, branch-free FMA refinements of
// fp4q_math.cuh (checked exhaustively against CUDA's IEEE __fdiv_rn / __frcp_rn over the
// operand ranges used here). Two rewrites are bit-identical to the contract's literal order
// and are used to save work:
//   * with dual scales compress never multiplies y by 1/16 (the E8M0 path does, since its
//     power-of-two scale would expose the difference): max|y| = fl(max|z| / 16) because rounding is
//     monotone, and q = y * inv = z * (inv / 16) exactly whenever a code can depend on it
//     (inv / 16 is exact for |x| < 2^120; a y that underflows gives |q| < 2^-17, code +-0
//     with the sign of z either way);
//   * all E2M1 / E4M3 rounding is done by the sm_100-family cvt instructions, which round
//     to nearest even with saturation exactly as the contract states.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <utility>

#include "fp4q.h"
#include "fp4q_math.cuh"

namespace {

constexpr int kTileBlocks = 8;                  // 256-element blocks per warp tile
// Warps per CTA and input stages per warp, per kernel (shared memory per warp decides how
// many warps fit on an SM: compress and roundtrip are issue/latency bound and want the
// most resident warps; one stage is enough because a tile's compute outlasts its load).
constexpr int kCompressWarps = 4, kCompressStages = 1, kCompressCtas = 5, kCompressCtasF32 = 4;
// Compress and roundtrip grids that would give a warp fewer than kSmallGridTiles tiles at
// their full CTAs per SM run kSmallGridCtas per SM instead (measured faster at 2^24 elements).
constexpr int kSmallGridTiles = 3, kSmallGridCtas = 4;
constexpr int kRoundtripWarps = 4, kRoundtripStages = 1, kRoundtripCtas = 5, kRoundtripCtasF32 = 4;
constexpr int kDecompressWarps = 4, kDecompressStages = 1, kDecompressCtas = 4;
constexpr int kDecompressGridCtas = 4;     // resident CTAs per SM the grid is sized for
// (5 for beta = 0, which has no destination stage, lost: 0.445 -> 0.397 of the copy peak at
// 2^24 elements, 0.63 -> 0.52 back to back)
constexpr int kReduceWarps = 4;
// Large reduces (at least kReduceDynTilesPerSm tiles per SM) run one CTA of
// ReduceCfg<R>::kDynWarps warps per SM with dynamic tile claims (InPipe DYN): warps of one SM were
// measured finishing up to 9 us apart under the round-robin assignment.
constexpr int64_t kReduceDynTilesPerSm = 384;
// R <= 2 (two stages, 20-warp CTAs) already gains from 8 tiles per warp (R = 2: 35.0 -> 33.0 us
// at 2^26, 59.9 -> 57.7 us at 2^27, equal at 2^25); R = 8 lost there (45.2 -> 53.6 us at 2^25)
constexpr int64_t kReduceDynTilesPerWarpR2 = 8;
// Compress and roundtrip of BF16 input with at least kCompressDynTilesPerWarp tiles per warp
// run the same way: one CTA of kCompressDynWarps warps (the 5 x 4 warps as one CTA) per SM,
// tiles claimed dynamically. The five CTAs of an SM were measured finishing up to 12 us apart
// at 2^26 elements (the warps of one CTA within 1 us), the SM's last stretch running on few
// warps; claimed dynamically they end within 2 us (compress 38.9 -> 37.4 us at 2^26, 69.6 ->
// 67.7 at 2^27; roundtrip 61.4 -> 59.4, 113.5 -> 110.1). From 4 tiles per warp (2^25
// elements) it still gains a little: launched back to back, compress 0.650 -> 0.655 of the
// copy peak, roundtrip 0.636 -> 0.643, decompress-accumulate (beta = 1) 0.86 -> 0.90. For the
// reduce below 384 tiles per SM it lost (R = 8 at 2^25: 47.2 -> 54.9 us).
// 24 warps (80 registers, about 70 bytes of spill) lost: compress 0.83 -> 0.79 of the copy peak
// at 2^29, 0.75 -> 0.72 at 2^27; roundtrip unchanged.
constexpr int kCompressDynWarps = 20;
// Decompress-accumulate into BF16 likewise (its 4 CTAs x 4 warps as one CTA). beta = 1:
// 48.2 -> 47.0 us at 2^26, 96.2 -> 95.7 us at 2^27, equal at 2^28 - 2^29. beta = 0 (no
// destination pipeline; the warps claim from the counter directly): 0.72 -> 0.73 of the copy
// peak at 2^26, 0.78 -> 0.81 at 2^27, 0.86 -> 0.89 at 2^29, within the timer's step at 2^25.
constexpr int kDecompressDynWarps = 16;
// beta = 0 has no destination stage, so its claiming CTA holds 20 warps (96 registers, no
// spill): 0.81 -> 0.83 of the copy peak at 2^27, 0.89 -> 0.915 at 2^29, equal below.
template <int BETA> constexpr int kDecDynWarps = BETA ? kDecompressDynWarps : 20;
constexpr int64_t kCompressDynTilesPerWarp = 4;
constexpr int kDynHeaderBytes = 2048;      // barriers of up to 31 warps, the claim counter last
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
// a * b + c on two pairs at once (one rounding each).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{.reg .b64 A, B, C, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\tmov.b64 C, {%6, %7};\n\t"
      "fma.rn.f32x2 D, A, B, C;\n\tmov.b64 {%0, %1}, D;}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
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

// Three-input maximum (sm_100 family), used for the absolute-maximum trees.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
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

// Level 1 strides 2, 4, 8 inside each row, forward order (stride 1 is done while the
// bfloat16 pairs are widened, see bf16x2_bfly).
__device__ __forceinline__ void level1_fwd_from2(Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
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

// Shared-memory vector accesses by 32-bit shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Transpose buffer: block blk's 16 x 16 FP32 values fill 64 16-byte units (1 KiB, no
// padding). Unit u = 4r + c (row r, 4-value chunk c) is stored at (u & ~7) | ((u & 7) ^ H)
// with H = ((r >> 2) ^ (r & 3)) & 3 | (blk & 1) << 2. Then the 8 lanes of every access phase
// (two blocks, four lanes each) hit 8 distinct 16-byte bank groups both when lanes own rows
// 4a..4a+3 (layout A) and when they own rows b, b+4, b+8, b+12 (layout B), and the unit of
// every access is a per-lane base (8 for layout A, 4 for layout B) plus an immediate.
struct XposeAddr {
  uint32_t a[8];   // layout A: unit base for (S ^ key), S = ((4 (j & 1) + c) ^ j) & 7
  uint32_t b[4];   // layout B: unit base for ((c ^ k) & 3) ^ key
};

__device__ __forceinline__ XposeAddr xpose_addr(uint32_t xbuf, int blk, int l4) {
  XposeAddr x;
  const uint32_t blkb = xbuf + (uint32_t)blk * 1024u, beta4 = (uint32_t)(blk & 1) << 2;
  const uint32_t keyA = (uint32_t)l4 | beta4;
  const uint32_t keyB = ((4u * (uint32_t)(l4 & 1)) ^ (uint32_t)l4 ^ beta4) & 7u;
  const uint32_t baseA = blkb + 256u * (uint32_t)l4, baseB = blkb + 128u * (uint32_t)(l4 >> 1);
#pragma unroll
  for (uint32_t s = 0; s < 8; ++s) x.a[s] = baseA + 16u * (s ^ keyA);
#pragma unroll
  for (uint32_t s = 0; s < 4; ++s) x.b[s] = baseB + 16u * (s ^ keyB);
  return x;
}
// row 4 l4 + j, chunk c (layout A)
__device__ __forceinline__ uint32_t xaddr_A(const XposeAddr& x, int j, int c) {
  return x.a[((4 * (j & 1) + c) ^ j) & 7] + 128u * (uint32_t)(j >> 1);
}
// row l4 + 4k, chunk c (layout B)
__device__ __forceinline__ uint32_t xaddr_B(const XposeAddr& x, int k, int c) {
  return x.b[(c ^ k) & 3] + 256u * (uint32_t)k;
}

// Write the lane's 4 rows from one layout, read 4 rows of the other. toB: A -> B.
template <bool toB>
__device__ __forceinline__ void transpose(Rows v, const XposeAddr& x) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      sts128(toB ? xaddr_A(x, k, c) : xaddr_B(x, k, c),
             make_uint4(__float_as_uint(v[k][2 * c].x), __float_as_uint(v[k][2 * c].y),
                        __float_as_uint(v[k][2 * c + 1].x), __float_as_uint(v[k][2 * c + 1].y)));
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 t = lds128(toB ? xaddr_B(x, k, c) : xaddr_A(x, k, c));
      v[k][2 * c] = make_float2(__uint_as_float(t.x), __uint_as_float(t.y));
      v[k][2 * c + 1] = make_float2(__uint_as_float(t.z), __uint_as_float(t.w));
    }
  __syncwarp();
}

// Half-width transpose buffer: the two 8-column halves of every block go through it one
// after the other, 640 bytes per block. Unit (row r = 4a + j, chunk cc of the half) is
// stored at 10 a + 2 j + beta + cc (beta = block parity). The 8 lanes of an access phase
// (two blocks, four lanes each) then hit 8 distinct 16-byte bank groups in layout A (lane a
// writes its row j at 2a + beta + const mod 8) and in layout B (lane b reads its row k at
// 2b + beta + const mod 8), and every unit is one per-lane base plus an immediate.
constexpr int kXHalfBlockBytes = 640;

struct XposeHalf {
  uint32_t a, b;   // layout A base (unit 10 l4 + beta), layout B base (unit 2 l4 + beta)
};

__device__ __forceinline__ XposeHalf xpose_half_addr(uint32_t xbuf, int blk, int l4) {
  const uint32_t blkb = xbuf + (uint32_t)blk * kXHalfBlockBytes, beta = (uint32_t)(blk & 1);
  return {blkb + 16u * (10u * (uint32_t)l4 + beta), blkb + 16u * (2u * (uint32_t)l4 + beta)};
}

// transpose<toB> through the half-width buffer, one half of the columns at a time.
template <bool toB>
__device__ __forceinline__ void transpose_half(Rows v, const XposeHalf& x) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * h + cc;
        sts128(toB ? x.a + 16u * (2 * k + cc) : x.b + 16u * (10 * k + cc),
               make_uint4(__float_as_uint(v[k][2 * c].x), __float_as_uint(v[k][2 * c].y),
                          __float_as_uint(v[k][2 * c + 1].x), __float_as_uint(v[k][2 * c + 1].y)));
      }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * h + cc;
        const uint4 t = lds128(toB ? x.b + 16u * (10 * k + cc) : x.a + 16u * (2 * k + cc));
        v[k][2 * c] = make_float2(__uint_as_float(t.x), __uint_as_float(t.y));
        v[k][2 * c + 1] = make_float2(__uint_as_float(t.z), __uint_as_float(t.w));
      }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ quantisation

// Result of quantising the lane's 4 rows of one block.
struct Quant {
  uint32_t code[4][2];   // 16 codes per row, 2 words per row
  uint32_t sg;           // the 4 group-scale codes of the lane's rows, row k in byte k
  float S[4];            // decode scale of each row's group
  float sb;              // block scale
};

// Dual scales of the lane's rows (rows in layout A if !LB, layout B if LB): the group-scale
// codes, the decode scale S and the quantisation multiplier inv of each row, the block scale.
// FOLD: the values are the unnormalised transform z = 16 y (see the file header).
struct DualScales {
  float S[4], inv[4], sb;
  uint32_t sg;
  bool zero;
};

template <int G, bool LB, bool FOLD>
__device__ __forceinline__ void dual_scales(const Rows v, DualScales& o) {
  float am[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      a[2 * j] = fabsf(v[k][j].x);
      a[2 * j + 1] = fabsf(v[k][j].y);
    }
    const float m0 = max3(a[0], a[1], a[2]), m1 = max3(a[3], a[4], a[5]), m2 = max3(a[6], a[7], a[8]);
    const float m3 = max3(a[9], a[10], a[11]), m4 = max3(a[12], a[13], a[14]);
    am[k] = max3(max3(m0, m1, m2), fmaxf(m3, m4), a[15]);
  }
  float A = max3(fmaxf(am[0], am[1]), am[2], am[3]);
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
  // s_b = RN(A / 2688), r = RN(amax / t_b) and inv = RN(1 / S) with the branch-free
  // correctly rounded division and reciprocal of fp4q_math.cuh (one reciprocal of t_b per
  // lane serves its four group ratios)
  const bool zero = !(A >= kZeroLimit);
  const float sb = zero ? 0.0f : fp4q_math::div_rn_2688(A);
  const float tb = zero ? 1.0f : __fmul_rn(sb, 6.0f);
  const fp4q_math::Divider by_tb(tb);
  float r[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) r[k] = by_tb.div(am[k]);
  uint32_t c01 = e4m3x2(r[0], r[1]), c23 = e4m3x2(r[2], r[3]);
  if (zero) c01 = c23 = 0u;
  const float2 s01 = e4m3x2_to_f2(c01), s23 = e4m3x2_to_f2(c23);
  const float sgv[4] = {s01.x, s01.y, s23.x, s23.y};
  o.sg = c01 | (c23 << 16);
  o.sb = sb;
  o.zero = zero;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float S = __fmul_rn(sgv[k], sb);
    o.S[k] = S;
    float inv = S > 0.0f ? fp4q_math::rcp_rn(S) : 0.0f;
    if (FOLD) inv = __fmul_rn(inv, 0.0625f);
    o.inv[k] = inv;
  }
}

// Dual-scale quantisation of the lane's rows: codes, scales.
template <int G, bool LB, bool FOLD>
__device__ __forceinline__ void quantize(const Rows v, Quant& o) {
  DualScales sc;
  dual_scales<G, LB, FOLD>(v, sc);
  o.sg = sc.sg;
  o.sb = sc.sb;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    o.S[k] = sc.S[k];
    const float2 iv = make_float2(sc.inv[k], sc.inv[k]);
    uint32_t w0 = e2m1_pack8(mul2(v[k][0], iv), mul2(v[k][1], iv), mul2(v[k][2], iv), mul2(v[k][3], iv));
    uint32_t w1 = e2m1_pack8(mul2(v[k][4], iv), mul2(v[k][5], iv), mul2(v[k][6], iv), mul2(v[k][7], iv));
    if (sc.zero) w0 = w1 = 0u;
    o.code[k][0] = w0;
    o.code[k][1] = w1;
  }
}

// One value pair -> its E2M1 codes -> their grid values (exact): the code byte never leaves
// the conversion, for the fused roundtrip, which writes no payload.
__device__ __forceinline__ float2 e2m1_round_pair(float2 q) {
  uint32_t h;
  asm("{.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %2, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;}"
      : "=r"(h) : "f"(q.x), "f"(q.y));
  const __half2 t = *reinterpret_cast<const __half2*>(&h);
  return make_float2(__low2float(t), __high2float(t));
}

// quantize followed by dequantize, for the fused roundtrip: v (the transform values) becomes
// x~ * dscale (dscale = 1/16 folds the inverse transform's normalisation into the decode
// scale, as scale_by_16th does). Bit-identical to the two steps: the same conversions in the
// same order, without packing the codes into words and unpacking them again; an all-zero block
// decodes to +0, as its zeroed codes do.
template <int G, bool LB, bool FOLD>
__device__ __forceinline__ void quantize_decode(Rows v, float dscale, float nz) {
  DualScales sc;
  dual_scales<G, LB, FOLD>(v, sc);
  const float2 z2 = make_float2(nz, nz);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 iv = make_float2(sc.inv[k], sc.inv[k]);
    const float Sd = __fmul_rn(sc.S[k], dscale);
    const float2 s = make_float2(Sd, Sd);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[k][j] = fma2(e2m1_round_pair(mul2(v[k][j], iv)), s, z2);
  }
  if (sc.zero) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) v[k][j] = make_float2(0.0f, 0.0f);
  }
}

// Microscaled quantisation (scales = e8m0, groups of 32 = two rows; rows in layout A if
// !LB, layout B if LB): per group X = 2^(floor(log2 amax) - 2), stored as the E8M0 code
// max(E - 2, 0) where E is the biased exponent field of amax (subnormal and zero maxima all
// clamp to code 0, X = 2^-127); q = y * 2^(127 - code), an exact power-of-two scaling that
// rounds like y / X; code = E2M1(q). The values are the normalised transform y.
template <bool LB>
__device__ __forceinline__ void quantize_mx(const Rows v, Quant& o) {
  float am[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      a[2 * j] = fabsf(v[k][j].x);
      a[2 * j + 1] = fabsf(v[k][j].y);
    }
    const float m0 = max3(a[0], a[1], a[2]), m1 = max3(a[3], a[4], a[5]), m2 = max3(a[6], a[7], a[8]);
    const float m3 = max3(a[9], a[10], a[11]), m4 = max3(a[12], a[13], a[14]);
    am[k] = max3(max3(m0, m1, m2), fmaxf(m3, m4), a[15]);
  }
  // a group is two consecutive rows: inside the lane in layout A, across lanes b, b^1 in B
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float other = LB ? __shfl_xor_sync(kFull, am[k], 1) : am[k ^ 1];
    am[k] = fmaxf(am[k], other);
  }
  uint32_t sg = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int E = (int)(__float_as_uint(am[k]) >> 23);
    const uint32_t c = (uint32_t)(E > 2 ? E - 2 : 0);
    sg |= c << (8 * k);
    o.S[k] = __uint_as_float(c ? c << 23 : 0x00400000u);
    const float m = __uint_as_float((254u - c) << 23);
    const float2 iv = make_float2(m, m);
    o.code[k][0] = e2m1_pack8(mul2(v[k][0], iv), mul2(v[k][1], iv), mul2(v[k][2], iv), mul2(v[k][3], iv));
    o.code[k][1] = e2m1_pack8(mul2(v[k][4], iv), mul2(v[k][5], iv), mul2(v[k][6], iv), mul2(v[k][7], iv));
  }
  o.sg = sg;
  o.sb = 0.0f;
}

// Value of an E8M0 scale code: 2^(code - 127) (code 0 is the subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t c) { return __uint_as_float(c ? c << 23 : 0x00400000u); }

// Multiply every value of the lane's rows by 1/16 (exact scaling of the unnormalised
// transform back to y, rounded as the contract's final step rounds it).
__device__ __forceinline__ void scale_rows_16th(Rows v) {
  const float2 s = make_float2(0.0625f, 0.0625f);
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j) v[k][j] = mul2(v[k][j], s);
}

// Decode the lane's 4 rows from codes and per-row scales: x~ = grid(code) * S.
// A packed mul.rn.f32x2 whose product feeds a packed add was observed to be fused into an
// FMA by the toolchain (even with .rn and --fmad=false), which breaks bit parity in the sums
// that follow. The products are therefore formed as fma.rn.f32x2(g, S, nz) with nz = -0.0
// passed in from the host: a * b + (-0) is exactly RN(a * b) (signed zeros included), and an
// FMA cannot absorb the addition that follows.
__device__ __forceinline__ void dequantize(const uint32_t code[4][2], const float S[4], Rows v, float nz) {
  const float2 z2 = make_float2(nz, nz);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 s = make_float2(S[k], S[k]);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      float2 g[4];
      e2m1_word_to_f2(code[k][w], g);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[k][4 * w + i] = fma2(g[i], s, z2);
    }
  }
}

// v += x~ for the lane's 4 rows (x~ = grid(code) * S as in dequantize, each product rounded on
// its own before the add): the reduce's running sum, decoded a word at a time so that no
// second 64-value array is live.
__device__ __forceinline__ void dequantize_add(const uint32_t code[4][2], const float S[4], Rows v, float nz) {
  const float2 z2 = make_float2(nz, nz);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 s = make_float2(S[k], S[k]);
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      float2 g[4];
      e2m1_word_to_f2(code[k][w], g);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[k][4 * w + i] = add2(v[k][4 * w + i], fma2(g[i], s, z2));
    }
  }
}

// The decode's final multiplication by 1/16 is folded into the decode scales: x~/16 =
// RN(grid * (S/16)) exactly (S/16 is exact, and the product stays normal: S >= 2^-109
// because a non-zero block has s_b >= 2^-100 and s_g >= 2^-9), and every butterfly of the
// inverse transform then works on values divided by 16. All of them are multiples of 2^-137
// (decoded values are normal with ulp >= 2^-133), so each sum is either exact (below 2^-114)
// or rounded in a binade where scaling by 2^4 commutes with the rounding: the result is
// bit-identical to transforming x~ and multiplying by 1/16 last. Payloads from compress and
// reduce always satisfy s_b = 0 or s_b >= 2^-100.
__device__ __forceinline__ void scale_by_16th(float S[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) S[k] = __fmul_rn(S[k], 0.0625f);
}

// ------------------------------------------------------------------ payload addressing

struct Payload {
  uint8_t* codes;      // n/2 bytes
  uint8_t* gsc;        // n/G bytes (+ padding to 16)
  float* bsc;          // n/256 floats (NULL for the microscaled variant)
  int64_t nb;          // number of blocks
};

__host__ __device__ inline int64_t pad16(int64_t b) { return (b + 15) / 16 * 16; }

__host__ __device__ inline Payload payload_of(void* base, int64_t n, int G, bool mx = false) {
  uint8_t* p = static_cast<uint8_t*>(base);
  Payload s;
  s.codes = p;
  s.gsc = p + n / 2;
  s.bsc = mx ? nullptr : reinterpret_cast<float*>(p + n / 2 + pad16(n / G));
  s.nb = n / 256;
  return s;
}

// Row of the lane's k-th row inside its block.
template <bool LB>
__device__ __forceinline__ int row_of(int l4, int k) { return LB ? l4 + 4 * k : 4 * l4 + k; }

// Store the lane's part of a quantised block (block index gb).
template <int G, bool LB, bool MX = false>
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
    if (!MX) P.bsc[gb] = q.sb;
    // G = 32 with an odd block count: the group-scale segment ends 8 bytes short of a
    // 16-byte boundary; the last block zeroes that padding
    if (G == 32 && (P.nb & 1) && gb == P.nb - 1)
      *reinterpret_cast<uint2*>(P.gsc + 8 * P.nb) = make_uint2(0u, 0u);
  }
}

// ------------------------------------------------------------------ prefetchable payload reads

// Raw payload words of the lane's part of one block, loaded one tile ahead of their use.
struct PayRaw {
  uint32_t code[4][2];
  uint32_t g[4];   // group-scale bytes: layout B = the block's 16 (G=16) or 8 (G=32) bytes;
                   // layout A = the lane's own 4 (G=16) or 2 (G=32) bytes in g[0]
  float sb;
};

__device__ __forceinline__ void pay_zero(PayRaw& r) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    r.code[k][0] = r.code[k][1] = 0u;
    r.g[k] = 0u;
  }
  r.sb = 0.0f;
}

template <int G, bool LB, bool MX = false>
__device__ __forceinline__ void pay_load(const Payload& P, int64_t gb, int l4, PayRaw& r) {
  if (LB) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint2 c = __ldg(reinterpret_cast<const uint2*>(P.codes + gb * 128 + (l4 + 4 * k) * 8));
      r.code[k][0] = c.x;
      r.code[k][1] = c.y;
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(P.codes + gb * 128 + l4 * 32);
    uint4 c0 = __ldg(src), c1 = __ldg(src + 1);
    r.code[0][0] = c0.x; r.code[0][1] = c0.y; r.code[1][0] = c0.z; r.code[1][1] = c0.w;
    r.code[2][0] = c1.x; r.code[2][1] = c1.y; r.code[3][0] = c1.z; r.code[3][1] = c1.w;
  }
  if (G == 16) {
    if (LB) {
      uint4 all = __ldg(reinterpret_cast<const uint4*>(P.gsc + gb * 16));
      r.g[0] = all.x; r.g[1] = all.y; r.g[2] = all.z; r.g[3] = all.w;
    } else {
      r.g[0] = __ldg(reinterpret_cast<const uint32_t*>(P.gsc + gb * 16 + 4 * l4));
    }
  } else {
    if (LB) {
      uint2 all = __ldg(reinterpret_cast<const uint2*>(P.gsc + gb * 8));
      r.g[0] = all.x; r.g[1] = all.y;
    } else {
      r.g[0] = __ldg(reinterpret_cast<const uint16_t*>(P.gsc + gb * 8 + 2 * l4));
    }
  }
  r.sb = MX ? 0.0f : __ldg(P.bsc + gb);
}

// Decode scale S = value(s_g) * s_b of each of the lane's 4 rows.
template <int G, bool LB, bool MX = false>
__device__ __forceinline__ void pay_scales(const PayRaw& r, int l4, float S[4]) {
  uint32_t sg;   // row k's group-scale code in byte k
  if (G == 16) {
    if (LB) {
      // row l4 + 4k uses byte l4 of word k
      const uint32_t sel = 0x4440u | (uint32_t)l4;
      sg = __byte_perm(r.g[0], 0, sel) | (__byte_perm(r.g[1], 0, sel) << 8) |
           (__byte_perm(r.g[2], 0, sel) << 16) | (__byte_perm(r.g[3], 0, sel) << 24);
    } else {
      sg = r.g[0];
    }
  } else {
    if (LB) {
      // row l4 + 4k belongs to group (l4 >> 1) + 2k: byte (l4 >> 1) + 2(k & 1) of word k >> 1
      const uint32_t s0 = 0x4440u | (uint32_t)(l4 >> 1), s2 = s0 + 2;
      sg = __byte_perm(r.g[0], 0, s0) | (__byte_perm(r.g[0], 0, s2) << 8) |
           (__byte_perm(r.g[1], 0, s0) << 16) | (__byte_perm(r.g[1], 0, s2) << 24);
    } else {
      // rows 4 l4 + {0,1} form group 2 l4, rows 4 l4 + {2,3} group 2 l4 + 1
      sg = (r.g[0] & 0xffu) * 0x0101u | ((r.g[0] >> 8) & 0xffu) * 0x01010000u;
    }
  }
  if (MX) {
#pragma unroll
    for (int k = 0; k < 4; ++k) S[k] = e8m0_value((sg >> (8 * k)) & 0xffu);
    return;
  }
  const float2 s01 = e4m3x2_to_f2(sg & 0xffffu), s23 = e4m3x2_to_f2(sg >> 16);
  S[0] = __fmul_rn(s01.x, r.sb);
  S[1] = __fmul_rn(s01.y, r.sb);
  S[2] = __fmul_rn(s23.x, r.sb);
  S[3] = __fmul_rn(s23.y, r.sb);
}

// ------------------------------------------------------------------ TMA pipelines

// Programmatic dependent launch: a kernel launched with programmatic stream serialisation
// may start while the previous kernel on the stream is finishing. griddepcontrol.wait blocks
// until that kernel has completed and its memory operations are visible, so every kernel
// calls it before its first global-memory access (read or write); launch_dependents lets the
// next kernel's CTAs be scheduled as soon as SM resources free up.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Fetch a tensor map's descriptor before the first copy that uses it. A kernel parameter is
// not written by an earlier kernel, so this may run before grid_dependency_wait: under
// programmatic serialisation the fetch then overlaps the previous kernel's tail.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Shared-memory primitives (sm_90+ PTX: mbarrier, cp.async.bulk.tensor, proxy fences).
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// One poll of a barrier phase. Without a suspend-time hint the hardware holds the thread for at
// most a short, implementation-defined window while the phase is incomplete; with a hint
// (an earlier version passed 1000 ns) a wait that was entered a little early could sleep
// well past the phase's completion.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Nanoseconds of the GPU's global timer (used only to bound waits).
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t c0, int32_t c1, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// Device fault word: set when a bounded wait gives up (the kernel then drains its own copies
// in flight, with a bound, and returns). Read by fp4q_fault_flags.
__device__ unsigned int g_fp4q_fault;
constexpr unsigned kFaultLoadWait = 1u;    // a TMA load did not complete within the bound
constexpr unsigned kFaultDrainWait = 2u;   // a copy still in flight after a fault did not complete
constexpr unsigned kFaultSelftest = 4u;    // the self-test wait ran out (expected)

// A wait is declared failed after kWaitLimitNs of the global timer (about a second) or after
// its poll budget, whichever comes first.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kSpinLimit = 1u << 30;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t polls) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < polls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u && global_ns() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

constexpr int kTileLinesBF16 = 32;         // 128-byte lines per 8-block bf16 tile (4 KiB)
constexpr int kTileLinesF32 = 64;          // 128-byte lines per 8-block f32 tile (8 KiB)
constexpr int kXBufBytes = 8192;           // full-width transpose buffer / output staging per warp
constexpr int kCompressXBytes = kTileBlocks * kXHalfBlockBytes;   // compress: half-width transpose
// roundtrip: half-width transpose; the buffer also stages the output tile (8 KiB for FP32)
template <bool XF>
struct RoundtripXBytes {
  static constexpr int value = XF ? kXBufBytes : kCompressXBytes;
};
constexpr int kHeaderBytes = 1024;         // per-CTA header: every warp's stage barriers

// CTA shared memory: [alignment slack][header: 64 bytes of barriers per warp][warp regions],
// each warp region = [input stages][xbuf of XB bytes], 1024-byte aligned (the 128-byte TMA
// swizzle repeats every 1024 bytes).
template <int WARPS, int STAGES, int IN_BYTES, int XB = kXBufBytes, int HDR = kHeaderBytes>
struct WarpSmemLayout {
  static constexpr int kRegion = STAGES * IN_BYTES + XB;
  static_assert(kRegion % 1024 == 0, "warp regions must stay 1024-byte aligned");
  static_assert(64 * WARPS <= HDR - 8, "the header holds 64 bytes of barriers per warp");
  static constexpr int kCtaBytes = 1024 + HDR + WARPS * kRegion;
};
// Shared address of a DYN CTA's claim counter: the last word of its header.
__device__ __forceinline__ uint32_t dyn_counter_addr(uint8_t* raw) {
  return ((smem_addr(raw) + 1023u) & ~1023u) + (uint32_t)kDynHeaderBytes - 8u;
}

struct WarpSmem {
  uint32_t stage0, xbuf, bar0;
};

template <int STAGES, int IN_BYTES, int XB = kXBufBytes, int HDR = kHeaderBytes>
__device__ __forceinline__ WarpSmem warp_smem(uint8_t* raw, int warp) {
  constexpr int region = STAGES * IN_BYTES + XB;
  const uint32_t base = (smem_addr(raw) + 1023u) & ~1023u;
  WarpSmem w;
  w.stage0 = base + HDR + (uint32_t)(warp * region);
  w.xbuf = w.stage0 + STAGES * IN_BYTES;
  w.bar0 = base + 64u * (uint32_t)warp;
  return w;
}

// Per-warp input pipeline over STAGES stage buffers of BYTES bytes: STAGES tiles stay in
// flight (issue(buf, bar, t) arms the barrier and starts the copies of tile t; lane 0 calls
// it, or every lane when ALL_LANES, for copies spread over lanes); every lane waits on the
// tile's barrier, reads the stage, and the stage is refilled with the warp's next tile.
// Tiles come round robin (warp w of W takes w, w + W, ...), or with DYN from the CTA's
// claim counter in shared memory: CTA c's tiles are c, c + G, c + 2G, ... (G = gridDim.x)
// and its warps take them in the order they ask, so warps that run ahead do more tiles.
// With `defer` the start loads only the first stage and the first refill the others, so
// that every warp's first tile reaches the head of the memory queue (the 3- and 4-rank
// reduce: 0.554 -> 0.581 of the copy peak at 2^25 back to back, 0.603 -> 0.617 at 2^26; the
// 2-rank reduce gains with it once it also reads its scales directly; no gain for the
// other kernels).
template <int STAGES, int BYTES, bool ALL_LANES = false, bool DYN = false>
struct InPipe {
  uint32_t stage0, bar0;
  int64_t t0, W, tiles;
  int i, issued, deferred;      // iterations whose copies were issued, stages the start left out
  uint32_t ctr, asked;          // DYN: the CTA's counter (shared address), lane 0's claim
  int64_t tid[DYN ? STAGES : 1];  // DYN: the tile each stage holds

  __device__ __forceinline__ int64_t claim_tile(uint32_t claim) const {
    return (int64_t)blockIdx.x + (int64_t)__shfl_sync(kFull, claim, 0) * gridDim.x;
  }
  __device__ __forceinline__ uint32_t claim_ask(int lane) const {
    uint32_t c = 0;
    if (lane == 0) asm volatile("atom.shared.add.u32 %0, [%1], 1;" : "=r"(c) : "r"(ctr) : "memory");
    return c;
  }

  __device__ __forceinline__ uint32_t buf(int s) const { return stage0 + (uint32_t)(s * BYTES); }
  __device__ __forceinline__ uint32_t bar(int s) const { return bar0 + 8u * (uint32_t)s; }

  template <class Issue>
  __device__ __forceinline__ void start(uint32_t stage0_, uint32_t bar0_, int64_t t0_, int64_t W_,
                                        int64_t tiles_, int lane, Issue&& issue, bool defer = false) {
    stage0 = stage0_;
    bar0 = bar0_;
    t0 = t0_;
    W = W_;
    tiles = tiles_;
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) mbar_init(bar(s), 1);
      fence_barrier_init();
    }
    __syncwarp();
    issued = 0;
    deferred = defer ? STAGES - 1 : 0;
    for (int s = 0; s < STAGES - deferred; ++s) {
      const int64_t t = t0 + (int64_t)s * W;
      if (t < tiles) {
        if (ALL_LANES || lane == 0) issue(buf(s), bar(s), t);
        ++issued;
      }
    }
    i = 0;
  }
  // DYN start: the CTA's counter at shared address ctr_ (zeroed, with a CTA barrier, by
  // dyn_counter_init before any warp gets here).
  template <class Issue>
  __device__ __forceinline__ void start_dyn(uint32_t stage0_, uint32_t bar0_, uint32_t ctr_, int64_t tiles_, int lane,
                                            Issue&& issue, bool defer = false) {
    static_assert(DYN, "start_dyn needs DYN");
    stage0 = stage0_;
    bar0 = bar0_;
    ctr = ctr_;
    tiles = tiles_;
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) mbar_init(bar(s), 1);
      fence_barrier_init();
    }
    __syncwarp();
    issued = 0;
    deferred = defer ? STAGES - 1 : 0;
    for (int s = 0; s < STAGES; ++s) {
      tid[s] = claim_tile(claim_ask(lane));
      if (s < STAGES - deferred && tid[s] < tiles) {
        if (ALL_LANES || lane == 0) issue(buf(s), bar(s), tid[s]);
        ++issued;
      }
    }
    i = 0;
  }
  // The current tile and the one after it.
  __device__ __forceinline__ int64_t tile() const { return DYN ? tid[i % STAGES] : t0 + (int64_t)i * W; }
  __device__ __forceinline__ int64_t next_tile() const {
    static_assert(!DYN || STAGES > 1, "with one stage the next tile is claimed at the refill");
    return DYN ? tid[(i + 1) % STAGES] : t0 + (int64_t)(i + 1) * W;
  }
  // DYN: claim the tile the next refill loads, at the top of an iteration, so the counter's
  // latency hides behind the wait and the reading of the stage.
  __device__ __forceinline__ void ask(int lane) {
    if (DYN) asked = claim_ask(lane);
  }
  // DYN: the tile that claim is for (every lane; the next refill loads it).
  __device__ __forceinline__ int64_t asked_tile() const { return claim_tile(asked); }
  __device__ __forceinline__ uint32_t cur() const { return buf(i % STAGES); }
  // Wait for the current tile. On failure record the fault, wait (bounded) for every copy
  // still in flight into this warp's stages, and return false: the caller must stop.
  __device__ __forceinline__ bool wait() {
    bool ok = mbar_wait(bar(i % STAGES), (uint32_t)((i / STAGES) & 1), kSpinLimit);
    ok = __all_sync(kFull, ok);
    if (!ok) {
      if ((threadIdx.x & 31) == 0) atomicOr(&g_fp4q_fault, kFaultLoadWait);
      for (int k = i; k < issued; ++k)
        if (!mbar_wait(bar(k % STAGES), (uint32_t)((k / STAGES) & 1), kSpinLimit) && (threadIdx.x & 31) == 0)
          atomicOr(&g_fp4q_fault, kFaultDrainWait);
    }
    return ok;
  }
  // The current stage has been read: refill it with the tile STAGES iterations ahead. The
  // lanes' shared-memory reads (generic proxy) must be ordered before the TMA write (async
  // proxy) into the same stage: every lane fences across proxies, then the warp syncs, then
  // lane 0 issues the copy. Without the fence a refill overtook an outstanding read.
  template <class Issue>
  __device__ __forceinline__ void refill(int lane, Issue&& issue) {
    fence_proxy_async();
    __syncwarp();
    if (deferred) {
      for (int s = STAGES - deferred; s < STAGES; ++s) {
        const int64_t t = DYN ? tid[s] : t0 + (int64_t)s * W;
        if (t < tiles) {
          if (ALL_LANES || lane == 0) issue(buf(s), bar(s), t);
          ++issued;
        }
      }
      deferred = 0;
    }
    const int64_t tn = DYN ? claim_tile(asked) : t0 + (int64_t)(i + STAGES) * W;
    if (DYN) tid[i % STAGES] = tn;
    if (tn < tiles) {
      if (ALL_LANES || lane == 0) issue(buf(i % STAGES), bar(i % STAGES), tn);
      ++issued;
    }
    ++i;
  }
};

// Tile I/O in the 128-byte-swizzled shared layout the TMA writes and reads: 16-byte chunk c
// of line l sits at chunk position c ^ (l & 7). Layout A: lane (blk, a) owns line 4 blk + a
// of a bf16 tile (its 4 rows), or lines 8 blk + 2a + {0, 1} of an f32 tile.
__device__ __forceinline__ void tile_read_bf16(uint32_t buf, int blk, int a, Rows v) {
  const int line = 4 * blk + a;
  const uint32_t base = buf + (uint32_t)line * 128u, sw = (uint32_t)(line & 7);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 t = lds128(base + ((((uint32_t)c) ^ sw) << 4));
    const int k = c >> 1, j = 4 * (c & 1);
    v[k][j + 0] = bf16x2_to_f2(t.x);
    v[k][j + 1] = bf16x2_to_f2(t.y);
    v[k][j + 2] = bf16x2_to_f2(t.z);
    v[k][j + 3] = bf16x2_to_f2(t.w);
  }
}
// bfloat16 pair (x0 low, x1 high) -> (x0 + x1, x0 - x1): the stride-1 butterfly fused with
// the widening, by the mixed-precision add/sub (bf16 operand widened exactly, one rounding).
__device__ __forceinline__ float2 bf16x2_bfly(uint32_t w) {
  float s, d;
  const float hi = __uint_as_float(w & 0xffff0000u);
  asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, l, %3;}"
      : "=f"(s), "=f"(d) : "r"(w), "f"(hi));
  return make_float2(s, d);
}
// As tile_read_bf16, with the stride-1 butterfly applied to every pair.
__device__ __forceinline__ void tile_read_bf16_bfly(uint32_t buf, int blk, int a, Rows v) {
  const int line = 4 * blk + a;
  const uint32_t base = buf + (uint32_t)line * 128u, sw = (uint32_t)(line & 7);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 t = lds128(base + ((((uint32_t)c) ^ sw) << 4));
    const int k = c >> 1, j = 4 * (c & 1);
    v[k][j + 0] = bf16x2_bfly(t.x);
    v[k][j + 1] = bf16x2_bfly(t.y);
    v[k][j + 2] = bf16x2_bfly(t.z);
    v[k][j + 3] = bf16x2_bfly(t.w);
  }
}
// The input tile of compress / roundtrip: BF16 (stride-1 butterfly fused into the widening
// when BFLY) or FP32 (the same butterfly applied to each pair in FP32).
template <bool XF, bool BFLY>
__device__ __forceinline__ void tile_read_in(uint32_t buf, int blk, int a, Rows v);

__device__ __forceinline__ void tile_write_bf16(uint32_t buf, int blk, int a, const Rows v) {
  const int line = 4 * blk + a;
  const uint32_t base = buf + (uint32_t)line * 128u, sw = (uint32_t)(line & 7);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int k = c >> 1, j = 4 * (c & 1);
    sts128(base + ((((uint32_t)c) ^ sw) << 4),
           make_uint4(f2_to_bf16x2(v[k][j]), f2_to_bf16x2(v[k][j + 1]), f2_to_bf16x2(v[k][j + 2]),
                      f2_to_bf16x2(v[k][j + 3])));
  }
}
__device__ __forceinline__ void tile_read_f32(uint32_t buf, int blk, int a, Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int line = 8 * blk + 2 * a + (k >> 1);
    const uint32_t base = buf + (uint32_t)line * 128u, sw = (uint32_t)(line & 7);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint32_t c = (uint32_t)(4 * (k & 1) + cc);
      const uint4 t = lds128(base + ((c ^ sw) << 4));
      v[k][2 * cc] = make_float2(__uint_as_float(t.x), __uint_as_float(t.y));
      v[k][2 * cc + 1] = make_float2(__uint_as_float(t.z), __uint_as_float(t.w));
    }
  }
}
__device__ __forceinline__ void tile_write_f32(uint32_t buf, int blk, int a, const Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int line = 8 * blk + 2 * a + (k >> 1);
    const uint32_t base = buf + (uint32_t)line * 128u, sw = (uint32_t)(line & 7);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint32_t c = (uint32_t)(4 * (k & 1) + cc);
      sts128(base + ((c ^ sw) << 4),
             make_uint4(__float_as_uint(v[k][2 * cc].x), __float_as_uint(v[k][2 * cc].y),
                        __float_as_uint(v[k][2 * cc + 1].x), __float_as_uint(v[k][2 * cc + 1].y)));
    }
  }
}

__device__ __forceinline__ void pair_bfly(Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j) v[k][j] = make_float2(__fadd_rn(v[k][j].x, v[k][j].y), __fsub_rn(v[k][j].x, v[k][j].y));
}

template <bool XF, bool BFLY>
__device__ __forceinline__ void tile_read_in(uint32_t buf, int blk, int a, Rows v) {
  if (XF) {
    tile_read_f32(buf, blk, a, v);
    if (BFLY) pair_bfly(v);
  } else if (BFLY) {
    tile_read_bf16_bfly(buf, blk, a, v);
  } else {
    tile_read_bf16(buf, blk, a, v);
  }
}

// ------------------------------------------------------------------ kernels

struct TileLoop {
  int64_t tiles;     // number of 8-block tiles
  int64_t nb;        // number of 256-element blocks
  int64_t bpr;       // 0: the data tensor is contiguous; else blocks per row of a strided 2-D tensor
  int64_t tpr;       // strided rows holding whole tiles (bpr % 8 == 0): tiles per row, else 0
  float negzero;     // -0.0f, set by the host so the compiler cannot see its value
};

// TMA traffic of one tile of a data tensor (x, y or dst) with LPB 128-byte lines per block
// (4 for BF16, 8 for FP32); every lane of the warp calls these. Tile and block indices fit in
// 32 bits (n < 2^37: fewer than 2^29 blocks), so the row divisions are 32-bit. Contiguous data is a 2-D map
// of lines and a tile is one box, issued by lane 0. A strided 2-D tensor is a 3-D map
// {line, line in row, row}: a tile is one box when rows hold whole tiles (tpr), else one box
// per existing block (blocks never straddle rows: cols is a multiple of 256), lane b issuing
// block b's box after lane 0 has armed the barrier for all of them. Each block lands at the
// same shared-memory offset either way, so the swizzled tile layout is unchanged.
// One box per existing block of tile t (nb blocks in all, bpr per row, lpb lines per block).
// Kept out of line: it runs only for strided tensors whose rows do not hold whole tiles, and
// inlined its registers weighed on every kernel's common path.
__device__ __noinline__ void blocks_load(const CUtensorMap* map, uint32_t nb, uint32_t bpr, uint32_t t, uint32_t buf,
                                         uint32_t bar, int lane, uint32_t lpb) {
  const uint32_t gb0 = t * kTileBlocks, bpb = 128u * lpb;
  const int nv = (int)(nb - gb0 < (uint32_t)kTileBlocks ? nb - gb0 : (uint32_t)kTileBlocks);
  if (lane == 0) mbar_expect_tx(bar, (uint32_t)nv * bpb);
  __syncwarp();
  if (lane < nv) {
    const uint32_t gb = gb0 + (uint32_t)lane, row = gb / bpr;
    tma_load_3d(buf + (uint32_t)lane * bpb, map, 0, (int32_t)((gb - row * bpr) * lpb), (int32_t)row, bar);
  }
}
__device__ __noinline__ void blocks_store(const CUtensorMap* map, uint32_t nb, uint32_t bpr, uint32_t t, uint32_t src,
                                          int lane, uint32_t lpb) {
  const uint32_t gb0 = t * kTileBlocks, bpb = 128u * lpb;
  const int nv = (int)(nb - gb0 < (uint32_t)kTileBlocks ? nb - gb0 : (uint32_t)kTileBlocks);
  if (lane < nv) {
    const uint32_t gb = gb0 + (uint32_t)lane, row = gb / bpr;
    tma_store_3d(map, 0, (int32_t)((gb - row * bpr) * lpb), (int32_t)row, src + (uint32_t)lane * bpb);
    bulk_commit();
  }
}

template <int LPB>
__device__ __forceinline__ void tile_load(const CUtensorMap* map, const TileLoop& T, int64_t t, uint32_t buf,
                                          uint32_t bar, int lane) {
  constexpr uint32_t BPB = 128u * LPB;
  if (T.bpr == 0 || T.tpr) {
    if (lane != 0) return;
    mbar_expect_tx(bar, kTileBlocks * BPB);
    if (T.bpr == 0) {
      tma_load_2d(buf, map, 0, (int32_t)(t * kTileBlocks * LPB), bar);
    } else {
      const uint32_t row = (uint32_t)t / (uint32_t)T.tpr;
      tma_load_3d(buf, map, 0, (int32_t)(((uint32_t)t - row * (uint32_t)T.tpr) * kTileBlocks * LPB), (int32_t)row, bar);
    }
    return;
  }
  blocks_load(map, (uint32_t)T.nb, (uint32_t)T.bpr, (uint32_t)t, buf, bar, lane, LPB);
}
// Store tile t from the staging buffer; each issuing lane commits its own bulk group.
template <int LPB>
__device__ __forceinline__ void tile_store(const CUtensorMap* map, const TileLoop& T, int64_t t, uint32_t src,
                                           int lane) {
  if (T.bpr == 0 || T.tpr) {
    if (lane != 0) return;
    if (T.bpr == 0) {
      tma_store_2d(map, 0, (int32_t)(t * kTileBlocks * LPB), src);
    } else {
      const uint32_t row = (uint32_t)t / (uint32_t)T.tpr;
      tma_store_3d(map, 0, (int32_t)(((uint32_t)t - row * (uint32_t)T.tpr) * kTileBlocks * LPB), (int32_t)row, src);
    }
    bulk_commit();
    return;
  }
  blocks_store(map, (uint32_t)T.nb, (uint32_t)T.bpr, (uint32_t)t, src, lane, LPB);
}

// Zero a CTA's tile counter before any warp claims from it.
__device__ __forceinline__ void dyn_counter_init(uint32_t ctr) {
  if (threadIdx.x == 0) asm volatile("st.shared.u32 [%0], 0;" ::"r"(ctr) : "memory");
  __syncthreads();
}
// One tile claimed from a CTA's counter by a warp with no load pipeline (InPipe DYN claims
// the same way): CTA c's tiles are c, c + G, c + 2G, ... (G = gridDim.x); every lane gets it.
__device__ __forceinline__ int64_t claim_plain(uint32_t ctr, int lane) {
  uint32_t c = 0;
  if (lane == 0) asm volatile("atom.shared.add.u32 %0, [%1], 1;" : "=r"(c) : "r"(ctr) : "memory");
  return (int64_t)blockIdx.x + (int64_t)__shfl_sync(kFull, c, 0) * gridDim.x;
}

template <int WARPS>
__device__ __forceinline__ int64_t warp_global() {
  return (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5);
}
template <int WARPS>
__device__ __forceinline__ int64_t warp_count() { return (int64_t)gridDim.x * WARPS; }

// Wait until the warp's TMA stores have finished reading the staging buffer (every lane waits
// for the bulk groups it committed itself).
__device__ __forceinline__ void staging_free() {
  bulk_wait_read_all();
  __syncwarp();
}
// Publish the staging buffer (written with st.shared) to the TMA store of tile t.
template <int LPB>
__device__ __forceinline__ void staging_store(const CUtensorMap* map, const TileLoop& T, int64_t t, uint32_t xbuf,
                                              int lane) {
  fence_proxy_async();
  __syncwarp();
  tile_store<LPB>(map, T, t, xbuf, lane);
}

#include "fp4q_tc.cuh"

// K1: compress. x (bfloat16, n) -> payload. Input tiles arrive by TMA.
// XF: FP32 input (8 KiB tiles of 64 lines) instead of BF16 (4 KiB, 32 lines).
// DYN: one CTA of kCompressDynWarps warps per SM claiming its tiles dynamically (InPipe DYN).
template <int G, int FWHT, bool MX, bool XF, bool DYN = false>
__global__ void __launch_bounds__(DYN ? kCompressDynWarps * 32 : kCompressWarps * 32,
                                  DYN ? 1 : (XF ? kCompressCtasF32 : kCompressCtas))
compress_kernel(const __grid_constant__ CUtensorMap xmap, Payload P, TileLoop T) {
  constexpr int IN = XF ? 8192 : 4096;
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) prefetch_tensormap(&xmap);
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  const WarpSmem ws = warp_smem<kCompressStages, IN, kCompressXBytes, DYN ? kDynHeaderBytes : kHeaderBytes>(smem_raw, warp);
  const XposeHalf xa = xpose_half_addr(ws.xbuf, blk, l4);
  auto issue = [&](uint32_t buf, uint32_t bar, int64_t t) { tile_load<XF ? 8 : 4>(&xmap, T, t, buf, bar, lane); };
  InPipe<kCompressStages, IN, true, DYN> pipe{};
  if constexpr (DYN) {
    const uint32_t ctr = dyn_counter_addr(smem_raw);
    dyn_counter_init(ctr);
    pipe.start_dyn(ws.stage0, ws.bar0, ctr, T.tiles, lane, issue);
  } else {
    pipe.start(ws.stage0, ws.bar0, warp_global<kCompressWarps>(), warp_count<kCompressWarps>(), T.tiles, lane, issue);
  }
  for (int64_t t = DYN ? pipe.tile() : pipe.t0; t < T.tiles; t = DYN ? pipe.tile() : t + pipe.W) {
    pipe.ask(lane);
    const int64_t gb = t * kTileBlocks + blk;
    const bool valid = gb < T.nb;
    if (!pipe.wait()) return;
    Rows v;
    tile_read_in<XF, FWHT != 0>(pipe.cur(), blk, l4, v);
    pipe.refill(lane, issue);
    Quant q;
    if (FWHT) {
      level1_fwd_from2(v);
      rows_bfly(v, 1);             // h = 16
      rows_bfly(v, 2);             // h = 32
      transpose_half<true>(v, xa);
      rows_bfly(v, 1);             // h = 64
      rows_bfly(v, 2);             // h = 128
      if (MX) {
        scale_rows_16th(v);
        quantize_mx<true>(v, q);
      } else {
        quantize<G, true, true>(v, q);
      }
      if (valid) store_block<G, true, MX>(P, gb, l4, q);
    } else {
      if (MX) quantize_mx<false>(v, q); else quantize<G, false, false>(v, q);
      if (valid) store_block<G, false, MX>(P, gb, l4, q);
    }
  }
}

// K2: decompress-accumulate. payload -> dst (dtype DT), dst = BETA ? dst + x^ : x^.
// The payload of the next tile is prefetched into registers; dst tiles are read (BETA) and
// written through the swizzled shared staging buffer by TMA.
// DYN (BF16 dst): one CTA of kDecDynWarps<BETA> warps per SM claiming its tiles dynamically;
// the payload prefetch follows the claims (the tile claimed at the top of an iteration is the
// one the refill loads next with BETA = 1, the one the next iteration decodes with BETA = 0).
template <int G, int FWHT, int DT, int BETA, bool MX, bool DYN = false>
__global__ void __launch_bounds__(DYN ? kDecDynWarps<BETA> * 32 : kDecompressWarps * 32, DYN ? 1 : kDecompressCtas)
decompress_kernel(const __grid_constant__ CUtensorMap dmap, Payload P, TileLoop T) {
  static_assert(!DYN || DT == FP4Q_BF16, "dynamic claims: BF16 destinations");
  constexpr int TB = DT == FP4Q_BF16 ? 4096 : 8192;
  constexpr int LPB = DT == FP4Q_BF16 ? 4 : 8;   // 128-byte lines per block of dst
  constexpr bool LB = FWHT != 0;
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) prefetch_tensormap(&dmap);
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  const WarpSmem ws = warp_smem<kDecompressStages, BETA ? TB : 0, kXBufBytes, DYN ? kDynHeaderBytes : kHeaderBytes>(smem_raw, warp);
  const XposeAddr xa = xpose_addr(ws.xbuf, blk, l4);
  auto issue = [&](uint32_t buf, uint32_t bar, int64_t t) { tile_load<LPB>(&dmap, T, t, buf, bar, lane); };
  InPipe<kDecompressStages, TB, true, DYN && BETA> pipe{};
  int64_t t0, W;
  uint32_t ctr = 0;
  if constexpr (DYN) {
    ctr = dyn_counter_addr(smem_raw);
    dyn_counter_init(ctr);
    if constexpr (BETA) {
      pipe.start_dyn(ws.stage0, ws.bar0, ctr, T.tiles, lane, issue);
      t0 = pipe.tile();
    } else {
      t0 = claim_plain(ctr, lane);    // no destination pipeline: the counter directly
    }
    W = 0;
  } else {
    t0 = warp_global<kDecompressWarps>();
    W = warp_count<kDecompressWarps>();
    if (BETA) pipe.start(ws.stage0, ws.bar0, t0, W, T.tiles, lane, issue);
  }
  PayRaw cur, nxt;
  if (t0 < T.tiles && t0 * kTileBlocks + blk < T.nb) pay_load<G, LB, MX>(P, t0 * kTileBlocks + blk, l4, cur);
  else pay_zero(cur);
  int64_t tn = 0;
  for (int64_t t = t0; t < T.tiles; t = DYN ? (BETA ? pipe.tile() : tn) : t + W) {
    if constexpr (DYN && BETA) {
      pipe.ask(lane);
      tn = pipe.asked_tile();
    } else if constexpr (DYN) {
      tn = claim_plain(ctr, lane);
    } else {
      tn = t + W;
    }
    const int64_t gbn = tn * kTileBlocks + blk;
    if (tn < T.tiles && gbn < T.nb) pay_load<G, LB, MX>(P, gbn, l4, nxt); else pay_zero(nxt);
    float S[4];
    pay_scales<G, LB, MX>(cur, l4, S);
    if (FWHT) scale_by_16th(S);
    Rows v;
    dequantize(cur.code, S, v, T.negzero);
    staging_free();
    if (FWHT) {
      rows_bfly(v, 2);             // h = 128
      rows_bfly(v, 1);             // h = 64
      transpose<false>(v, xa);
      rows_bfly(v, 2);             // h = 32
      rows_bfly(v, 1);             // h = 16
      level1_inv(v);
    }
    if (BETA) {
      if (!pipe.wait()) break;
      Rows d;
      if (DT == FP4Q_BF16) tile_read_bf16(pipe.cur(), blk, l4, d); else tile_read_f32(pipe.cur(), blk, l4, d);
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) v[k][j] = add2(d[k][j], v[k][j]);
      pipe.refill(lane, issue);
    }
    if (DT == FP4Q_BF16) tile_write_bf16(ws.xbuf, blk, l4, v); else tile_write_f32(ws.xbuf, blk, l4, v);
    staging_store<LPB>(&dmap, T, t, ws.xbuf, lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cur.code[k][0] = nxt.code[k][0];
      cur.code[k][1] = nxt.code[k][1];
      cur.g[k] = nxt.g[k];
    }
    cur.sb = nxt.sb;
  }
  bulk_wait_all();
}

// K3: fused roundtrip. x (bfloat16) -> y = bf16(decode(compress(x))), no payload.
// XF: FP32 input and output instead of BF16.
// DYN: one CTA of kCompressDynWarps warps per SM claiming its tiles dynamically (as compress).
template <int G, int FWHT, bool MX, bool XF, bool DYN = false>
__global__ void __launch_bounds__(DYN ? kCompressDynWarps * 32 : kRoundtripWarps * 32,
                                  DYN ? 1 : (XF ? kRoundtripCtasF32 : kRoundtripCtas))
roundtrip_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap ymap, TileLoop T) {
  constexpr int IN = XF ? 8192 : 4096;
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) prefetch_tensormap(&xmap);
  if (threadIdx.x == 32) prefetch_tensormap(&ymap);
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  const WarpSmem ws =
      warp_smem<kRoundtripStages, IN, RoundtripXBytes<XF>::value, DYN ? kDynHeaderBytes : kHeaderBytes>(smem_raw, warp);
  const XposeHalf xa = xpose_half_addr(ws.xbuf, blk, l4);
  auto issue = [&](uint32_t buf, uint32_t bar, int64_t t) { tile_load<XF ? 8 : 4>(&xmap, T, t, buf, bar, lane); };
  InPipe<kRoundtripStages, IN, true, DYN> pipe{};
  if constexpr (DYN) {
    const uint32_t ctr = dyn_counter_addr(smem_raw);
    dyn_counter_init(ctr);
    pipe.start_dyn(ws.stage0, ws.bar0, ctr, T.tiles, lane, issue);
  } else {
    pipe.start(ws.stage0, ws.bar0, warp_global<kRoundtripWarps>(), warp_count<kRoundtripWarps>(), T.tiles, lane,
               issue);
  }
  for (int64_t t = DYN ? pipe.tile() : pipe.t0; t < T.tiles; t = DYN ? pipe.tile() : t + pipe.W) {
    pipe.ask(lane);
    if (!pipe.wait()) break;
    Rows v;
    tile_read_in<XF, FWHT != 0>(pipe.cur(), blk, l4, v);
    pipe.refill(lane, issue);
    Quant q;
    if (FWHT) {
      level1_fwd_from2(v);
      rows_bfly(v, 1);
      rows_bfly(v, 2);
      staging_free();
      transpose_half<true>(v, xa);
      rows_bfly(v, 1);
      rows_bfly(v, 2);
      if (MX) {
        scale_rows_16th(v);
        quantize_mx<true>(v, q);
        scale_by_16th(q.S);
        dequantize(q.code, q.S, v, T.negzero);
      } else {
        quantize_decode<G, true, true>(v, 0.0625f, T.negzero);
      }
      rows_bfly(v, 2);
      rows_bfly(v, 1);
      transpose_half<false>(v, xa);
      rows_bfly(v, 2);
      rows_bfly(v, 1);
      level1_inv(v);
    } else {
      if (MX) {
        quantize_mx<false>(v, q);
        dequantize(q.code, q.S, v, T.negzero);
      } else {
        quantize_decode<G, false, false>(v, 1.0f, T.negzero);
      }
      staging_free();
    }
    if (XF) tile_write_f32(ws.xbuf, blk, l4, v); else tile_write_bf16(ws.xbuf, blk, l4, v);
    staging_store<XF ? 8 : 4>(&ymap, T, t, ws.xbuf, lane);
  }
  bulk_wait_all();
}

// K4: emulated R-way reduce. R payloads -> transform-domain FP32 sum in rank order ->
// requantised payload (no transform). Each rank's tile of codes (1 KiB), group scales (128 or
// 64 bytes) and block scales (32 bytes) is contiguous in its payload and arrives by plain
// bulk copies. Their sizes are exact for the last, partial tile (never reading past a
// payload); the bulk copy moves whole 16-byte units, so up to three block scales of that
// last tile are read with plain loads instead.
constexpr int kRankStageBytes = 1024 + 128 + 32;   // codes | group scales | block scales

struct RankPtrs {
  const uint8_t* codes[FP4Q_MAX_RANKS];
  const uint8_t* gsc[FP4Q_MAX_RANKS];
  const float* bsc[FP4Q_MAX_RANKS];
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

constexpr bool kReduceDirectScales = true;

template <int R>
struct ReduceCfg {
  // R = 2 - 4 (dual scales): the scales are read straight from global memory one tile ahead,
  // so the bulk copies carry only the codes (at 2^28 elements R = 4 gains 5%). R = 2 gains
  // since the pipeline start was deferred (0.48 -> 0.52 of the copy peak back to back at 2^25,
  // 0.57 -> 0.61 at 2^26, 0.61 -> 0.66 at 2^27); before, the extra load latency cost more
  // than the two copies per rank saved. The E8M0 scales are only 2 bytes per lane, and above
  // R = 4 the single stage leaves no next tile to prefetch for.
  static constexpr bool kDirectScales = kReduceDirectScales && R >= 2 && R <= 4;
  // stages per warp: 2 up to R = 4 (3 for R = 2 lost: 0.52 -> 0.39 of the copy peak back to
  // back at 2^25, 0.61 -> 0.56 at 2^26), 1 above
  static constexpr int kStagesR = R <= 4 ? 2 : 1;
  // launch bound (CTAs per SM): 5 where the kernel fits 96 registers without spilling its
  // running sum (R = 2: 21.6 -> 20.5 us, R = 8: 49.2 -> 47.1 us at 2^25 elements; R = 2 with
  // the direct scales spills 8 bytes at G = 16 and is faster all the same: at 4 CTAs, spill-
  // free, 0.61 -> 0.60 of the copy peak back to back at 2^26, 0.66 -> 0.65 at 2^27); the R = 3, 4
  // variants prefetch every rank's scales into registers and keep 4 (at 5 they spill: R = 4
  // went from 29.4 to 36.8 us); R = 2 at 6 (80 registers, spilling) lost at every size (0.48 ->
  // 0.41 of the copy peak back to back at 2^25)
  static constexpr int kMinCtas = (R == 3 || R == 4) ? 4 : 5;
  // dynamic-claim CTAs (InPipe DYN) hold as many warps as that fixed grid has per SM
  static constexpr int kDynWarps = 4 * kMinCtas;
  static constexpr int cta_bytes(int warps) { return warps * kRegion + 128 + 16; }   // + DYN counter
  static constexpr int kStageBytes = R * kRankStageBytes;
  static constexpr int kRegion = kStagesR * kStageBytes + 128;       // + barriers

};

template <int G, int R, bool MX, bool DYN>
__global__ void __launch_bounds__(DYN ? ReduceCfg<R>::kDynWarps * 32 : kReduceWarps * 32, DYN ? 1 : ReduceCfg<R>::kMinCtas)
reduce_kernel(RankPtrs in, Payload out, TileLoop T) {
  typedef ReduceCfg<R> C;
  constexpr bool DS = C::kDirectScales && !MX;
  extern __shared__ uint8_t smem_raw[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, blk = lane >> 2, l4 = lane & 3;
  const uint32_t base = ((smem_addr(smem_raw) + 127u) & ~127u) + (uint32_t)(warp * C::kRegion);
  constexpr uint32_t gs_per_block = G == 16 ? 16 : 8;
  // lane r < R copies rank r's segments; its three source pointers live in registers
  const uint8_t* my_codes = in.codes[0];
  const uint8_t* my_gsc = in.gsc[0];
  const float* my_bsc = in.bsc[0];
#pragma unroll
  for (int r = 1; r < R; ++r)
    if (lane == r) {
      my_codes = in.codes[r];
      my_gsc = in.gsc[r];
      my_bsc = in.bsc[r];
    }
  auto issue = [&](uint32_t buf, uint32_t bar, int64_t t) {
    const int64_t left = T.nb - t * kTileBlocks;
    const uint32_t nblk = (uint32_t)(left < kTileBlocks ? left : kTileBlocks);
    const uint32_t cbytes = nblk * 128u, gbytes = (nblk * gs_per_block + 15u) & ~15u;
    const uint32_t sbytes = MX ? 0u : (nblk * 4u) & ~15u;
    // arm the barrier for all R ranks before any of their copies is issued
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)R * (DS ? cbytes : cbytes + gbytes + sbytes));
    __syncwarp();
    if (lane < R) {
      const uint32_t b = buf + (uint32_t)(lane * kRankStageBytes);
      bulk_load(b, my_codes + t * 1024, cbytes, bar);
      if (!DS) {
        bulk_load(b + 1024, my_gsc + t * (kTileBlocks * gs_per_block), gbytes, bar);
        if (sbytes) bulk_load(b + 1152, my_bsc + t * kTileBlocks, sbytes, bar);
      }
    }
  };
  // direct scales: this lane's group-scale bytes and block scale of every rank, for the
  // current tile (cg, cs) and the warp's next tile (ng, ns)
  uint32_t cg[R], ng[R];
  float cs[R], ns[R];
  auto load_scales = [&](int64_t tt, uint32_t* g, float* sb) {
    const int64_t b = tt * kTileBlocks + blk;
    const bool ok = tt < T.tiles && b < T.nb;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      g[r] = !ok ? 0u : G == 16 ? __ldg(reinterpret_cast<const uint32_t*>(in.gsc[r] + b * 16 + 4 * l4))
                                : (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(in.gsc[r] + b * 8 + 2 * l4));
      sb[r] = (!ok || MX) ? 0.0f : __ldg(in.bsc[r] + b);
    }
  };
  InPipe<C::kStagesR, C::kStageBytes, true, DYN> pipe{};
  // the direct-scale variants (R = 2 - 4) defer all but their first stage (see InPipe)
  if constexpr (DYN) {
    const uint32_t ctr = ((smem_addr(smem_raw) + 127u) & ~127u) + (uint32_t)(C::kDynWarps * C::kRegion);
    dyn_counter_init(ctr);
    pipe.start_dyn(base, base + (uint32_t)(C::kStagesR * C::kStageBytes), ctr, T.tiles, lane, issue, DS);
  } else {
    pipe.start(base, base + (uint32_t)(C::kStagesR * C::kStageBytes), warp_global<kReduceWarps>(),
               warp_count<kReduceWarps>(), T.tiles, lane, issue, DS);
  }
  if (DS) load_scales(DYN ? pipe.tile() : pipe.t0, cg, cs);
  for (int64_t t = DYN ? pipe.tile() : pipe.t0; t < T.tiles; t = DYN ? pipe.tile() : t + pipe.W) {
    pipe.ask(lane);
    if constexpr (DS) load_scales(DYN ? pipe.next_tile() : t + pipe.W, ng, ns);
    const int64_t gb = t * kTileBlocks + blk;
    const bool valid = gb < T.nb;
    // a block scale outside the bulk-copied whole 16-byte units of the last tile
    const int64_t left = T.nb - t * kTileBlocks;
    const bool direct_sb = !MX && valid && left < kTileBlocks && blk >= (int)(left & ~3);
    if (!pipe.wait()) return;
    Rows z;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t b = pipe.cur() + (uint32_t)(r * kRankStageBytes);
      PayRaw raw;
      const uint4 c0 = lds128(b + (uint32_t)(blk * 128 + l4 * 32));
      const uint4 c1 = lds128(b + (uint32_t)(blk * 128 + l4 * 32 + 16));
      raw.code[0][0] = c0.x; raw.code[0][1] = c0.y; raw.code[1][0] = c0.z; raw.code[1][1] = c0.w;
      raw.code[2][0] = c1.x; raw.code[2][1] = c1.y; raw.code[3][0] = c1.z; raw.code[3][1] = c1.w;
      if (DS) {
        raw.g[0] = cg[r];
        raw.sb = cs[r];
      } else {
        raw.g[0] = G == 16 ? lds32(b + 1024u + (uint32_t)(blk * 16 + 4 * l4))
                           : lds16(b + 1024u + (uint32_t)(blk * 8 + 2 * l4));
        raw.sb = MX ? 0.0f : direct_sb ? __ldg(in.bsc[r] + gb) : __uint_as_float(lds32(b + 1152u + (uint32_t)(4 * blk)));
      }
      float S[4];
      pay_scales<G, false, MX>(raw, l4, S);
      if (r == 0) dequantize(raw.code, S, z, T.negzero); else dequantize_add(raw.code, S, z, T.negzero);
    }
    pipe.refill(lane, issue);
    Quant q;
    if (MX) quantize_mx<false>(z, q); else quantize<G, false, false>(z, q);
    if (valid) store_block<G, false, MX>(out, gb, l4, q);
    if (DS) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        cg[r] = ng[r];
        cs[r] = ns[r];
      }
    }
  }
}

// Last partial block of a tensor whose length is not a multiple of 256 (it is zero-padded
// to 256 elements): one warp loads it with bounds checks and runs the same per-block steps
// as the tiled kernels. All 8 four-lane groups of the warp work on that block, so the
// transpose and the shuffles see a full warp; only the first group stores.
constexpr int kTailThreads = 32;

// Row 4 l4 + k, pair j = elements 16 (4 l4 + k) + 2j and + 1 of the block (layout A); with
// bfly, each pair goes through the stride-1 butterfly in FP32, as the fused BF16 load does.
template <bool XF>
__device__ __forceinline__ float tail_elem(const void* x, int e) {
  return XF ? static_cast<const float*>(x)[e] : __uint_as_float((uint32_t)static_cast<const uint16_t*>(x)[e] << 16);
}
template <bool XF>
__device__ __forceinline__ void tail_load(const void* x, int len, int l4, Rows v, bool bfly) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 16 * (4 * l4 + k) + 2 * j;
      const float a = e < len ? tail_elem<XF>(x, e) : 0.0f;
      const float b = e + 1 < len ? tail_elem<XF>(x, e + 1) : 0.0f;
      v[k][j] = bfly ? make_float2(__fadd_rn(a, b), __fsub_rn(a, b)) : make_float2(a, b);
    }
}

// dst[e] = BETA ? dst[e] + v : v for the block's elements below len (layout A rows).
template <int DT, int BETA>
__device__ __forceinline__ void tail_store(void* dst, int len, int l4, const Rows v) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = 16 * (4 * l4 + k) + 2 * j + h;
        if (e >= len) continue;
        const float x = h ? v[k][j].y : v[k][j].x;
        if (DT == FP4Q_BF16) {
          uint16_t* d = static_cast<uint16_t*>(dst);
          const float o = BETA ? __fadd_rn(__uint_as_float((uint32_t)d[e] << 16), x) : x;
          d[e] = (uint16_t)(f2_to_bf16x2(make_float2(o, 0.0f)) & 0xffffu);
        } else {
          float* d = static_cast<float*>(dst);
          d[e] = BETA ? __fadd_rn(d[e], x) : x;
        }
      }
}

// Forward steps of compress / roundtrip on a loaded block; leaves the codes and scales in q
// and the values in layout B (FWHT) or A.
template <int G, int FWHT, bool MX>
__device__ __forceinline__ void tail_quantize(Rows v, const XposeAddr& xa, Quant& q) {
  if (FWHT) {
    level1_fwd_from2(v);
    rows_bfly(v, 1);
    rows_bfly(v, 2);
    transpose<true>(v, xa);
    rows_bfly(v, 1);
    rows_bfly(v, 2);
    if (MX) {
      scale_rows_16th(v);
      quantize_mx<true>(v, q);
    } else {
      quantize<G, true, true>(v, q);
    }
  } else {
    if (MX) quantize_mx<false>(v, q); else quantize<G, false, false>(v, q);
  }
}

// Inverse transform of decoded values (layout B in, layout A out).
__device__ __forceinline__ void tail_inverse(Rows v, const XposeAddr& xa) {
  rows_bfly(v, 2);
  rows_bfly(v, 1);
  transpose<false>(v, xa);
  rows_bfly(v, 2);
  rows_bfly(v, 1);
  level1_inv(v);
}

template <int G, int FWHT, bool MX, bool XF>
__global__ void __launch_bounds__(kTailThreads)
tail_compress_kernel(const void* x, int len, Payload P, int64_t gb) {
  __shared__ __align__(1024) uint8_t xbuf[kXBufBytes];
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x, blk = lane >> 2, l4 = lane & 3;
  const XposeAddr xa = xpose_addr(smem_addr(xbuf), blk, l4);
  Rows v;
  tail_load<XF>(x, len, l4, v, FWHT != 0);
  Quant q;
  tail_quantize<G, FWHT, MX>(v, xa, q);
  if (blk == 0) store_block<G, FWHT != 0, MX>(P, gb, l4, q);
}

template <int G, int FWHT, int DT, int BETA, bool MX>
__global__ void __launch_bounds__(kTailThreads)
tail_decompress_kernel(Payload P, int64_t gb, void* dst, int len, float negzero) {
  __shared__ __align__(1024) uint8_t xbuf[kXBufBytes];
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x, blk = lane >> 2, l4 = lane & 3;
  const XposeAddr xa = xpose_addr(smem_addr(xbuf), blk, l4);
  PayRaw r;
  pay_load<G, FWHT != 0, MX>(P, gb, l4, r);
  float S[4];
  pay_scales<G, FWHT != 0, MX>(r, l4, S);
  if (FWHT) scale_by_16th(S);
  Rows v;
  dequantize(r.code, S, v, negzero);
  if (FWHT) tail_inverse(v, xa);
  if (blk == 0) tail_store<DT, BETA>(dst, len, l4, v);
}

template <int G, int FWHT, bool MX, bool XF>
__global__ void __launch_bounds__(kTailThreads)
tail_roundtrip_kernel(const void* x, void* y, int len, float negzero) {
  __shared__ __align__(1024) uint8_t xbuf[kXBufBytes];
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x, blk = lane >> 2, l4 = lane & 3;
  const XposeAddr xa = xpose_addr(smem_addr(xbuf), blk, l4);
  Rows v;
  tail_load<XF>(x, len, l4, v, FWHT != 0);
  Quant q;
  tail_quantize<G, FWHT, MX>(v, xa, q);
  if (FWHT) scale_by_16th(q.S);
  dequantize(q.code, q.S, v, negzero);
  if (FWHT) tail_inverse(v, xa);
  if (blk == 0) tail_store<XF ? FP4Q_F32 : FP4Q_BF16, 0>(y, len, l4, v);
}

// Self-test of the bounded wait: one warp waits on a barrier phase that nothing completes;
// the wait gives up after `polls` polls and records kFaultSelftest.
__global__ void selftest_wait_kernel(uint32_t polls) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(b, 0u, polls);
  if (!__all_sync(kFull, ok) && threadIdx.x == 0) atomicOr(&g_fp4q_fault, kFaultSelftest);
}

// ------------------------------------------------------------------ host side

// Per-device attribute caches: written once per device with the same value by whichever
// thread gets there first (atomics, so concurrent first calls are well defined).
std::atomic<int> g_num_sms[64];

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int v = g_num_sms[dev].load();
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_num_sms[dev].store(v);
  }
  return v;
}

// Resident CTAs per SM of a kernel instance on the current device, with its dynamic
// shared-memory limit raised as needed. Both runtime queries are made once per (kernel,
// device) and cached: they cost microseconds of host time, which would otherwise be paid on
// every call.
struct PlanEntry {
  const void* fn;
  int dev, threads, smem, per_sm;
};
std::mutex g_plan_mu;
PlanEntry g_plan[512];
int g_plan_count = 0;

int resident_ctas(const void* fn, int threads, int smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (int i = 0; i < g_plan_count; ++i) {
      const PlanEntry& e = g_plan[i];
      if (e.fn == fn && e.dev == dev && e.threads == threads && e.smem == smem) return e.per_sm;
    }
  }
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  // every codec kernel asks for the largest shared-memory carveout: kernels whose carveouts
  // differ cannot share an SM, which would stop a programmatically launched kernel's CTAs
  // from starting beside the previous kernel's last CTAs (a chain of two compresses, a reduce
  // and a decompress-accumulate of 2^24 elements: 48.8 us with it, 50.6-50.9 us without)
  if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess) return -1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess || per_sm <= 0)
    return -1;
  std::lock_guard<std::mutex> lock(g_plan_mu);
  if (g_plan_count < (int)(sizeof(g_plan) / sizeof(g_plan[0]))) g_plan[g_plan_count++] = {fn, dev, threads, smem, per_sm};
  return per_sm;
}

struct Launch {
  int grid;
  int smem;
};

// CTAs per SM cap for a grid of `warps`-warp CTAs over `tiles` tiles, `ctas` per SM at most
// (0: as many as fit).
int small_grid_cap(int64_t tiles, int warps, int ctas) {
  const int sms = num_sms();
  return sms > 0 && tiles < (int64_t)kSmallGridTiles * warps * ctas * sms ? kSmallGridCtas : 0;
}

// Shared memory of one SM and the part of it reserved per CTA, on the current device
// (queried once per device).
bool smem_per_sm(int& total, int& reserved) {
  static std::atomic<int> g_total[64], g_reserved[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int t = g_total[dev].load();
  int r = g_reserved[dev].load();
  if (t == 0) {
    if (cudaDeviceGetAttribute(&t, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&r, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess || t <= 0)
      return false;
    g_reserved[dev].store(r);   // before total: a reader that sees total also sees reserved
    g_total[dev].store(t);
  }
  total = t;
  reserved = r;
  return true;
}

// Persistent grid: as many CTAs as fit on all SMs at once (at most max_per_sm per SM when it
// is given), never more than the tiles need. A cap below what fits is also enforced by
// resources: the dynamic shared memory is padded just enough that a (max_per_sm + 1)-th CTA
// of the kernel no longer fits on an SM. A grid merely sized for fewer CTAs per SM than fit
// is packed unevenly when the kernel starts while the previous kernel drains (programmatic
// launch): SMs that free up first take the extra CTAs. Measured on a chain of two compresses,
// a reduce and a decompress-accumulate of 2^24 elements with compress capped at 4 CTAs of 5:
// 48.8 us per chain with the padded cap, 54.0 us with the grid size alone.
template <typename K>
fp4q_status plan(K kernel, int warps, int smem, int64_t tiles, Launch& L, int max_per_sm = 0) {
  const int sms = num_sms();
  if (sms <= 0) return FP4Q_ERR_CUDA;
  int per_sm = resident_ctas(reinterpret_cast<const void*>(kernel), warps * 32, smem);
  if (per_sm <= 0) return FP4Q_ERR_CUDA;
  if (max_per_sm > 0 && per_sm > max_per_sm) {
    int total = 0, reserved = 0;
    if (smem_per_sm(total, reserved)) {
      const int padded = total / (max_per_sm + 1) - reserved + 1;
      if (padded > smem &&
          resident_ctas(reinterpret_cast<const void*>(kernel), warps * 32, padded) == max_per_sm)
        smem = padded;
    }
    per_sm = max_per_sm;
  }
  const int64_t want = (tiles + warps - 1) / warps;
  const int64_t cap = (int64_t)per_sm * sms;
  L.grid = (int)(want < cap ? want : cap);
  L.smem = smem;
  return FP4Q_OK;
}

// Launch with programmatic stream serialisation (see grid_dependency_wait).
template <class... KArgs, class... Args>
fp4q_status launch_pdl(void (*kernel)(KArgs...), const Launch& L, int threads, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)L.grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)L.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA;
}

fp4q_status launched() { return cudaGetLastError() == cudaSuccess ? FP4Q_OK : FP4Q_ERR_CUDA; }

// cuTensorMapEncodeTiled from the driver, looked up once.
typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encode_fn() {
  static EncodeTiled fn = []() -> EncodeTiled {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// 2-D view of a contiguous buffer as 128-byte lines, one 8-block tile per box, 128-byte
// swizzle (bfloat16: 64 elements per line, 32 lines per tile; float32: 32 and 64).
bool line_map(CUtensorMap* m, const void* ptr, int64_t n, bool f32, int box_lines = 0) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t per_line = f32 ? 32 : 64;
  const cuuint64_t dims[2] = {per_line, (cuuint64_t)(n / (int64_t)per_line)};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {(cuuint32_t)per_line,
                             (cuuint32_t)(box_lines ? box_lines : (f32 ? kTileLinesF32 : kTileLinesBF16))};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Strided 2-D tensor [rows, cols] with row stride ld elements, as a 3-D map of 128-byte
// lines {line, line in row, row}; one box is one 256-element block.
bool rows_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool f32) {
  // one box per tile when whole tiles fit in a row (cols a multiple of 2048), else per block
  const bool tiles = cols % (kTileBlocks * FP4Q_BLOCK) == 0;
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t per_line = f32 ? 32 : 64, esz = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {per_line, (cuuint64_t)cols / per_line, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {128, (cuuint64_t)ld * esz};
  const cuuint32_t box[3] = {(cuuint32_t)per_line, (f32 ? 8u : 4u) * (tiles ? (cuuint32_t)kTileBlocks : 1u), 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

fp4q_status check_params(const fp4q_params* p, int& G, int& fwht, bool& mx) {
  fp4q_params d = {FP4Q_GROUP_DEFAULT, FP4Q_BLOCK, 1, FP4Q_SCALES_DUAL};
  if (p) d = *p;
  if ((d.group != 16 && d.group != 32) || d.block != FP4Q_BLOCK || d.fwht < 0 || d.fwht > 2 ||
      (d.scales != FP4Q_SCALES_DUAL && d.scales != FP4Q_SCALES_E8M0) ||
      (d.scales == FP4Q_SCALES_E8M0 && d.group != 32))
    return FP4Q_ERR_PARAM;
  G = d.group;
  fwht = d.fwht;
  mx = d.scales == FP4Q_SCALES_E8M0;
  return FP4Q_OK;
}

// The kernels address tiles with 32-bit TMA line coordinates: n < 2^37 keeps them in range.
bool size_ok(int64_t n) { return n > 0 && n < ((int64_t)1 << 37); }

// Elements the payload covers: n rounded up to whole blocks (the last one zero-padded).
int64_t padded_n(int64_t n) { return (n + FP4Q_BLOCK - 1) / FP4Q_BLOCK * FP4Q_BLOCK; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

TileLoop tiles_of(int64_t n) {
  TileLoop T;
  T.nb = n / FP4Q_BLOCK;
  T.tiles = (T.nb + kTileBlocks - 1) / kTileBlocks;
  T.bpr = 0;
  T.tpr = 0;
  T.negzero = -0.0f;
  return T;
}

// Tail launch: one warp for the last partial block.
template <class K, class... Args>
fp4q_status launch_tail(K kernel, cudaStream_t s, Args&&... args) {
  Launch L;
  L.grid = 1;
  L.smem = 0;
  return launch_pdl(kernel, L, kTailThreads, s, std::forward<Args>(args)...);
}

// Full blocks through the tiled kernel, then the zero-padded last block (if any) through
// the one-warp tail kernel; the payload layout is that of the padded length.
template <int G, int F, bool MX, bool XF>
fp4q_status launch_compress(const void* x, int64_t n, const Payload& P, cudaStream_t s) {
  const int64_t nfull = n / FP4Q_BLOCK * FP4Q_BLOCK;
  if (nfull > 0) {
    TileLoop T = tiles_of(nfull);
    CUtensorMap xm;
    if (!line_map(&xm, x, nfull, XF)) return FP4Q_ERR_CUDA;
    const int sms = num_sms();
    fp4q_status st = FP4Q_OK;
    bool dyn = false;
    if constexpr (!XF) {
      dyn = sms > 0 && T.tiles >= kCompressDynTilesPerWarp * kCompressDynWarps * sms;
      if (dyn) {
        auto k = compress_kernel<G, F, MX, false, true>;
        Launch L;
        st = plan(k, kCompressDynWarps,
                  WarpSmemLayout<kCompressDynWarps, kCompressStages, 4096, kCompressXBytes, kDynHeaderBytes>::kCtaBytes,
                  T.tiles, L, 1);
        if (st == FP4Q_OK) st = launch_pdl(k, L, kCompressDynWarps * 32, s, xm, P, T);
      }
    }
    if (!dyn) {
      auto k = compress_kernel<G, F, MX, XF>;
      Launch L;
      st = plan(k, kCompressWarps,
                WarpSmemLayout<kCompressWarps, kCompressStages, XF ? 8192 : 4096, kCompressXBytes>::kCtaBytes, T.tiles, L,
                small_grid_cap(T.tiles, kCompressWarps, kCompressCtas));
      if (st == FP4Q_OK) st = launch_pdl(k, L, kCompressWarps * 32, s, xm, P, T);
    }
    if (st != FP4Q_OK) return st;
  }
  if (n == nfull) return FP4Q_OK;
  const void* xt = static_cast<const uint8_t*>(x) + nfull * (XF ? 4 : 2);
  return launch_tail(tail_compress_kernel<G, F, MX, XF>, s, xt, (int)(n - nfull), P, (int64_t)(nfull / FP4Q_BLOCK));
}

// Tensor-core compress (fwht = 2): full blocks through compress_tc_kernel, persistent, one CTA
// per SM (its TMEM allocation is the SM's 512 columns); a last partial block through the
// one-warp tail kernel with the butterfly transform.
template <int G, bool MX>
fp4q_status launch_compress_tc(const void* x, int64_t n, const Payload& P, cudaStream_t s) {
  const int64_t nfull = n / FP4Q_BLOCK * FP4Q_BLOCK;
  if (nfull > 0) {
    const int64_t nb = nfull / FP4Q_BLOCK, batches = (nb + kTcBatchBlocks - 1) / kTcBatchBlocks;
    CUtensorMap xm;   // 128-byte lines (quarter-blocks), boxes of 256 lines (64 blocks), two per batch
    if (!line_map(&xm, x, nfull, false, 2 * kTcBatchBlocks)) return FP4Q_ERR_CUDA;
    auto k = compress_tc_kernel<G, MX>;
    Launch L;
    // plan() sizes the grid as (units / warps) CTAs: one unit per warp and batch gives one CTA
    // per batch, capped at one per SM
    constexpr int warps = kTcThreads / 32;
    fp4q_status st = plan(k, warps, kTcSmemBytes, warps * batches, L, 1);
    if (st == FP4Q_OK) st = launch_pdl(k, L, kTcThreads, s, xm, P, nb, batches);
    if (st != FP4Q_OK) return st;
  }
  if (n == nfull) return FP4Q_OK;
  const void* xt = static_cast<const uint8_t*>(x) + nfull * 2;
  return launch_tail(tail_compress_kernel<G, 1, MX, false>, s, xt, (int)(n - nfull), P, (int64_t)(nfull / FP4Q_BLOCK));
}

template <int G, int F, int DT, int B, bool MX>
fp4q_status launch_decompress(const Payload& P, int64_t n, void* dst, cudaStream_t s) {
  const int64_t nfull = n / FP4Q_BLOCK * FP4Q_BLOCK;
  if (nfull > 0) {
    TileLoop T = tiles_of(nfull);
    CUtensorMap dm;
    if (!line_map(&dm, dst, nfull, DT == FP4Q_F32)) return FP4Q_ERR_CUDA;
    constexpr int TB = DT == FP4Q_BF16 ? 4096 : 8192;
    const int sms = num_sms();
    fp4q_status st = FP4Q_OK;
    bool dyn = false;
    if constexpr (DT == FP4Q_BF16) {
      dyn = sms > 0 && T.tiles >= kCompressDynTilesPerWarp * kDecDynWarps<B> * sms;
      if (dyn) {
        auto k = decompress_kernel<G, F, DT, B, MX, true>;
        Launch L;
        st = plan(k, kDecDynWarps<B>,
                  WarpSmemLayout<kDecDynWarps<B>, kDecompressStages, B ? TB : 0, kXBufBytes, kDynHeaderBytes>::kCtaBytes,
                  T.tiles, L, 1);
        if (st == FP4Q_OK) st = launch_pdl(k, L, kDecDynWarps<B> * 32, s, dm, P, T);
      }
    }
    if (!dyn) {
      auto k = decompress_kernel<G, F, DT, B, MX>;
      Launch L;
      st = plan(k, kDecompressWarps, WarpSmemLayout<kDecompressWarps, kDecompressStages, B ? TB : 0>::kCtaBytes, T.tiles,
                L, kDecompressGridCtas);
      if (st == FP4Q_OK) st = launch_pdl(k, L, kDecompressWarps * 32, s, dm, P, T);
    }
    if (st != FP4Q_OK) return st;
  }
  if (n == nfull) return FP4Q_OK;
  void* dtail = static_cast<uint8_t*>(dst) + nfull * (DT == FP4Q_BF16 ? 2 : 4);
  return launch_tail(tail_decompress_kernel<G, F, DT, B, MX>, s, P, (int64_t)(nfull / FP4Q_BLOCK), dtail,
                     (int)(n - nfull), -0.0f);
}

template <int G, int F, bool MX, bool XF>
fp4q_status launch_roundtrip(const void* x, int64_t n, void* y, cudaStream_t s) {
  const int64_t nfull = n / FP4Q_BLOCK * FP4Q_BLOCK;
  if (nfull > 0) {
    TileLoop T = tiles_of(nfull);
    CUtensorMap xm, ym;
    if (!line_map(&xm, x, nfull, XF) || !line_map(&ym, y, nfull, XF)) return FP4Q_ERR_CUDA;
    const int sms = num_sms();
    fp4q_status st = FP4Q_OK;
    bool dyn = false;
    if constexpr (!XF) {
      dyn = sms > 0 && T.tiles >= kCompressDynTilesPerWarp * kCompressDynWarps * sms;
      if (dyn) {
        auto k = roundtrip_kernel<G, F, MX, false, true>;
        Launch L;
        st = plan(k, kCompressDynWarps,
                  WarpSmemLayout<kCompressDynWarps, kRoundtripStages, 4096, RoundtripXBytes<false>::value,
                                 kDynHeaderBytes>::kCtaBytes,
                  T.tiles, L, 1);
        if (st == FP4Q_OK) st = launch_pdl(k, L, kCompressDynWarps * 32, s, xm, ym, T);
      }
    }
    if (!dyn) {
      auto k = roundtrip_kernel<G, F, MX, XF>;
      Launch L;
      st = plan(k, kRoundtripWarps,
                WarpSmemLayout<kRoundtripWarps, kRoundtripStages, XF ? 8192 : 4096, RoundtripXBytes<XF>::value>::kCtaBytes,
                T.tiles, L, XF ? 0 : small_grid_cap(T.tiles, kRoundtripWarps, kRoundtripCtas));
      if (st == FP4Q_OK) st = launch_pdl(k, L, kRoundtripWarps * 32, s, xm, ym, T);
    }
    if (st != FP4Q_OK) return st;
  }
  if (n == nfull) return FP4Q_OK;
  const size_t es = XF ? 4 : 2;
  return launch_tail(tail_roundtrip_kernel<G, F, MX, XF>, s,
                     static_cast<const void*>(static_cast<const uint8_t*>(x) + nfull * es),
                     static_cast<void*>(static_cast<uint8_t*>(y) + nfull * es), (int)(n - nfull), -0.0f);
}

// Strided 2-D launches (rows x cols, cols a multiple of 256, row strides in elements).
// The kernels are the contiguous ones; only the tensor maps and TileLoop.bpr differ.
TileLoop tiles_2d(int64_t rows, int64_t cols) {
  TileLoop T = tiles_of(rows * cols);
  T.bpr = cols / FP4Q_BLOCK;
  T.tpr = T.bpr % kTileBlocks == 0 ? T.bpr / kTileBlocks : 0;
  return T;
}

template <int G, int F, bool MX>
fp4q_status launch_compress_2d(const void* x, int64_t rows, int64_t cols, int64_t ld, void* payload, cudaStream_t s) {
  const TileLoop T = tiles_2d(rows, cols);
  CUtensorMap xm;
  if (!rows_map(&xm, x, rows, cols, ld, false)) return FP4Q_ERR_CUDA;
  auto k = compress_kernel<G, F, MX, false>;
  Launch L;
  fp4q_status st = plan(k, kCompressWarps, WarpSmemLayout<kCompressWarps, kCompressStages, 4096, kCompressXBytes>::kCtaBytes,
                        T.tiles, L, small_grid_cap(T.tiles, kCompressWarps, kCompressCtas));
  if (st != FP4Q_OK) return st;
  return launch_pdl(k, L, kCompressWarps * 32, s, xm, payload_of(payload, rows * cols, G, MX), T);
}

template <int G, int F, int DT, int B, bool MX>
fp4q_status launch_decompress_2d(const void* payload, int64_t rows, int64_t cols, void* dst, int64_t ld,
                                 cudaStream_t s) {
  const TileLoop T = tiles_2d(rows, cols);
  CUtensorMap dm;
  if (!rows_map(&dm, dst, rows, cols, ld, DT == FP4Q_F32)) return FP4Q_ERR_CUDA;
  auto k = decompress_kernel<G, F, DT, B, MX>;
  constexpr int TB = DT == FP4Q_BF16 ? 4096 : 8192;
  Launch L;
  fp4q_status st = plan(k, kDecompressWarps,
                        WarpSmemLayout<kDecompressWarps, kDecompressStages, B ? TB : 0>::kCtaBytes, T.tiles, L,
                        kDecompressGridCtas);
  if (st != FP4Q_OK) return st;
  return launch_pdl(k, L, kDecompressWarps * 32, s, dm,
                    payload_of(const_cast<void*>(payload), rows * cols, G, MX), T);
}

template <int G, int F, bool MX>
fp4q_status launch_roundtrip_2d(const void* x, int64_t rows, int64_t cols, int64_t ldx, void* y, int64_t ldy,
                                cudaStream_t s) {
  const TileLoop T = tiles_2d(rows, cols);
  CUtensorMap xm, ym;
  if (!rows_map(&xm, x, rows, cols, ldx, false) || !rows_map(&ym, y, rows, cols, ldy, false)) return FP4Q_ERR_CUDA;
  auto k = roundtrip_kernel<G, F, MX, false>;
  Launch L;
  fp4q_status st = plan(k, kRoundtripWarps, WarpSmemLayout<kRoundtripWarps, kRoundtripStages, 4096, RoundtripXBytes<false>::value>::kCtaBytes,
                        T.tiles, L, small_grid_cap(T.tiles, kRoundtripWarps, kRoundtripCtas));
  if (st != FP4Q_OK) return st;
  return launch_pdl(k, L, kRoundtripWarps * 32, s, xm, ym, T);
}

template <int G, int R, bool MX>
fp4q_status launch_reduce_r(const RankPtrs& in, int64_t n, const Payload& P, cudaStream_t s) {
  n = padded_n(n);   // the reduce works on whole (zero-padded) blocks of the payloads
  TileLoop T = tiles_of(n);
  const int sms = num_sms();
  const int64_t dyn_min = R <= 2 ? kReduceDynTilesPerWarpR2 * ReduceCfg<R>::kDynWarps : kReduceDynTilesPerSm;
  const bool dyn = sms > 0 && T.tiles >= dyn_min * sms;
  auto k = dyn ? reduce_kernel<G, R, MX, true> : reduce_kernel<G, R, MX, false>;
  const int warps = dyn ? ReduceCfg<R>::kDynWarps : kReduceWarps;
  Launch L;
  fp4q_status st = plan(k, warps, ReduceCfg<R>::cta_bytes(warps), T.tiles, L);
  if (st != FP4Q_OK) return st;
  return launch_pdl(k, L, warps * 32, s, in, P, T);
}

template <int G, bool MX>
fp4q_status launch_reduce(const Payload* ins, int R, int64_t n, const Payload& out, cudaStream_t s) {
  RankPtrs in;
  memset(&in, 0, sizeof(in));
  for (int r = 0; r < R; ++r) {
    in.codes[r] = ins[r].codes;
    in.gsc[r] = ins[r].gsc;
    in.bsc[r] = ins[r].bsc;
  }
  switch (R) {
    case 1: return launch_reduce_r<G, 1, MX>(in, n, out, s);
    case 2: return launch_reduce_r<G, 2, MX>(in, n, out, s);
    case 3: return launch_reduce_r<G, 3, MX>(in, n, out, s);
    case 4: return launch_reduce_r<G, 4, MX>(in, n, out, s);
    case 5: return launch_reduce_r<G, 5, MX>(in, n, out, s);
    case 6: return launch_reduce_r<G, 6, MX>(in, n, out, s);
    case 7: return launch_reduce_r<G, 7, MX>(in, n, out, s);
    default: return launch_reduce_r<G, 8, MX>(in, n, out, s);
  }
}

size_t payload_bytes_of(int64_t n, int G, bool mx) {
  const int64_t m = padded_n(n);
  return (size_t)(m / 2 + pad16(m / G) + (mx ? 0 : 4 * (m / FP4Q_BLOCK)));
}

template <int G, bool MX>
fp4q_status dispatch_decompress(int key, const Payload& payload, int64_t n, void* dst, cudaStream_t s) {
  switch (key) {
    case 0: return launch_decompress<G, 0, FP4Q_BF16, 0, MX>(payload, n, dst, s);
    case 1: return launch_decompress<G, 0, FP4Q_BF16, 1, MX>(payload, n, dst, s);
    case 2: return launch_decompress<G, 0, FP4Q_F32, 0, MX>(payload, n, dst, s);
    case 3: return launch_decompress<G, 0, FP4Q_F32, 1, MX>(payload, n, dst, s);
    case 4: return launch_decompress<G, 1, FP4Q_BF16, 0, MX>(payload, n, dst, s);
    case 5: return launch_decompress<G, 1, FP4Q_BF16, 1, MX>(payload, n, dst, s);
    case 6: return launch_decompress<G, 1, FP4Q_F32, 0, MX>(payload, n, dst, s);
    default: return launch_decompress<G, 1, FP4Q_F32, 1, MX>(payload, n, dst, s);
  }
}

template <bool XF>
fp4q_status dispatch_compress(int G, int F, bool MX, const void* x, int64_t n, const Payload& P, cudaStream_t s) {
  if (F == 2) {   // tensor-core transform: BF16 input
    if (XF) return FP4Q_ERR_PARAM;
    if (MX) return launch_compress_tc<32, true>(x, n, P, s);
    return G == 16 ? launch_compress_tc<16, false>(x, n, P, s) : launch_compress_tc<32, false>(x, n, P, s);
  }
  if (MX) return F ? launch_compress<32, 1, true, XF>(x, n, P, s) : launch_compress<32, 0, true, XF>(x, n, P, s);
  if (G == 16) return F ? launch_compress<16, 1, false, XF>(x, n, P, s) : launch_compress<16, 0, false, XF>(x, n, P, s);
  return F ? launch_compress<32, 1, false, XF>(x, n, P, s) : launch_compress<32, 0, false, XF>(x, n, P, s);
}

template <bool MX>
fp4q_status dispatch_reduce(int G, const Payload* ins, int R, int64_t n, const Payload& out, cudaStream_t s) {
  if (MX) return launch_reduce<32, true>(ins, R, n, out, s);
  return G == 16 ? launch_reduce<16, false>(ins, R, n, out, s) : launch_reduce<32, false>(ins, R, n, out, s);
}

fp4q_status dispatch_decompress_all(int G, int F, bool MX, const Payload& P, int64_t n, void* dst, fp4q_dtype dtype,
                                    int beta, cudaStream_t s) {
  const int key = F * 4 + (dtype == FP4Q_F32) * 2 + beta;
  if (MX) return dispatch_decompress<32, true>(key, P, n, dst, s);
  return G == 16 ? dispatch_decompress<16, false>(key, P, n, dst, s) : dispatch_decompress<32, false>(key, P, n, dst, s);
}

// Argument checks and dispatch of compress / roundtrip for BF16 (XF = false) or FP32 input.
template <bool XF>
fp4q_status compress_entry(const void* x, int64_t n, void* payload, const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (!x || !payload) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(x) || !aligned16(payload)) return FP4Q_ERR_ALIGN;
  if (overlap(x, (size_t)n * (XF ? 4 : 2), payload, payload_bytes_of(n, G, MX))) return FP4Q_ERR_OVERLAP;
  return dispatch_compress<XF>(G, F, MX, x, n, payload_of(payload, padded_n(n), G, MX), static_cast<cudaStream_t>(stream));
}

template <bool XF>
fp4q_status roundtrip_entry(const void* x, int64_t n, void* y, const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (F == 2) return FP4Q_ERR_PARAM;   // the tensor-core transform is an encoder option only
  if (!x || !y) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(x) || !aligned16(y)) return FP4Q_ERR_ALIGN;
  const size_t bytes = (size_t)n * (XF ? 4 : 2);
  if (overlap(x, bytes, y, bytes)) return FP4Q_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (MX) return F ? launch_roundtrip<32, 1, true, XF>(x, n, y, s) : launch_roundtrip<32, 0, true, XF>(x, n, y, s);
  if (G == 16) return F ? launch_roundtrip<16, 1, false, XF>(x, n, y, s) : launch_roundtrip<16, 0, false, XF>(x, n, y, s);
  return F ? launch_roundtrip<32, 1, false, XF>(x, n, y, s) : launch_roundtrip<32, 0, false, XF>(x, n, y, s);
}

// A payload given as three separately placed segments (fp4q_segments): each 16-byte aligned,
// sized as in the contiguous payload of n elements (codes m/2, group scales pad16(m/G), block
// scales 4 m/256 bytes, m = n rounded up to whole blocks); the block scales are absent (NULL)
// for E8M0 scales.
struct SegSizes {
  size_t codes, gsc, bsc;
};
SegSizes seg_sizes(int64_t n, int G, bool mx) {
  const int64_t m = padded_n(n);
  return {(size_t)(m / 2), (size_t)pad16(m / G), mx ? (size_t)0 : (size_t)(4 * (m / FP4Q_BLOCK))};
}
fp4q_status segments_of(const fp4q_segments* sg, int64_t n, int G, bool mx, Payload& P) {
  if (!sg || !sg->codes || !sg->gscales || (!mx && !sg->bscales)) return FP4Q_ERR_NULL;
  if (!aligned16(sg->codes) || !aligned16(sg->gscales) || (!mx && !aligned16(sg->bscales))) return FP4Q_ERR_ALIGN;
  P.codes = static_cast<uint8_t*>(sg->codes);
  P.gsc = static_cast<uint8_t*>(sg->gscales);
  P.bsc = mx ? nullptr : static_cast<float*>(sg->bscales);
  P.nb = padded_n(n) / FP4Q_BLOCK;
  return FP4Q_OK;
}
// Does any segment of P overlap [a, a + na)?
bool seg_overlap(const Payload& P, const SegSizes& z, const void* a, size_t na) {
  return overlap(P.codes, z.codes, a, na) || overlap(P.gsc, z.gsc, a, na) || (P.bsc && overlap(P.bsc, z.bsc, a, na));
}
// Do two segment sets overlap anywhere (or, with self, do a set's own segments overlap)?
bool segs_overlap(const Payload& A, const Payload& B, const SegSizes& z) {
  return seg_overlap(B, z, A.codes, z.codes) || seg_overlap(B, z, A.gsc, z.gsc) ||
         (A.bsc && seg_overlap(B, z, A.bsc, z.bsc));
}
bool segs_self_overlap(const Payload& P, const SegSizes& z) {
  return overlap(P.codes, z.codes, P.gsc, z.gsc) ||
         (P.bsc && (overlap(P.codes, z.codes, P.bsc, z.bsc) || overlap(P.gsc, z.gsc, P.bsc, z.bsc)));
}

// A strided 2-D view: rows >= 1, cols a positive multiple of 256, rows * cols < 2^37,
// cols <= ld < 2^37 with 16-byte aligned rows (ld * element size a multiple of 16).
fp4q_status check_2d(int64_t rows, int64_t cols, int64_t ld, int esz) {
  const int64_t lim = (int64_t)1 << 37;
  if (rows < 1 || cols < FP4Q_BLOCK || cols % FP4Q_BLOCK != 0 || cols >= lim || rows >= lim / cols)
    return FP4Q_ERR_SIZE;
  if (ld < cols || ld >= lim) return FP4Q_ERR_PARAM;
  if ((ld * esz) % 16 != 0) return FP4Q_ERR_ALIGN;
  return FP4Q_OK;
}
// Bytes spanned by a strided view.
size_t span_2d(int64_t rows, int64_t cols, int64_t ld, int esz) { return (size_t)((rows - 1) * ld + cols) * esz; }

}  // namespace

extern "C" {

size_t fp4q_payload_bytes(int64_t n, const fp4q_params* params) {
  int G, f;
  bool mx;
  if (!size_ok(n) || check_params(params, G, f, mx) != FP4Q_OK) return 0;
  return payload_bytes_of(n, G, mx);
}

size_t fp4q_gscale_offset(int64_t n, const fp4q_params* params) {
  int G, f;
  bool mx;
  if (!size_ok(n) || check_params(params, G, f, mx) != FP4Q_OK) return 0;
  return (size_t)(padded_n(n) / 2);
}

size_t fp4q_bscale_offset(int64_t n, const fp4q_params* params) {
  int G, f;
  bool mx;
  if (!size_ok(n) || check_params(params, G, f, mx) != FP4Q_OK) return 0;
  return (size_t)(padded_n(n) / 2 + pad16(padded_n(n) / G));
}

fp4q_status fp4q_compress(const void* x_bf16, int64_t n, void* payload, const fp4q_params* params,
                          void* stream) {
  return compress_entry<false>(x_bf16, n, payload, params, stream);
}

fp4q_status fp4q_compress_f32(const void* x_f32, int64_t n, void* payload, const fp4q_params* params,
                              void* stream) {
  return compress_entry<true>(x_f32, n, payload, params, stream);
}

fp4q_status fp4q_decompress_accumulate(const void* payload, int64_t n, void* dst, fp4q_dtype dtype,
                                       int32_t beta, const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (F == 2) F = 1;   // a tensor-core-encoded payload is decoded like any fwht = 1 payload
  if ((dtype != FP4Q_BF16 && dtype != FP4Q_F32) || (beta != 0 && beta != 1)) return FP4Q_ERR_PARAM;
  if (!payload || !dst) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(payload) || !aligned16(dst)) return FP4Q_ERR_ALIGN;
  const size_t dbytes = (size_t)n * (dtype == FP4Q_BF16 ? 2 : 4);
  if (overlap(payload, payload_bytes_of(n, G, MX), dst, dbytes)) return FP4Q_ERR_OVERLAP;
  return dispatch_decompress_all(G, F, MX, payload_of(const_cast<void*>(payload), padded_n(n), G, MX), n, dst, dtype,
                                 beta, static_cast<cudaStream_t>(stream));
}

fp4q_status fp4q_roundtrip(const void* x_bf16, int64_t n, void* y_bf16, const fp4q_params* params,
                           void* stream) {
  return roundtrip_entry<false>(x_bf16, n, y_bf16, params, stream);
}

fp4q_status fp4q_roundtrip_f32(const void* x_f32, int64_t n, void* y_f32, const fp4q_params* params,
                               void* stream) {
  return roundtrip_entry<true>(x_f32, n, y_f32, params, stream);
}

fp4q_status fp4q_compress_2d(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld, void* payload,
                             const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (F == 2) return FP4Q_ERR_PARAM;   // the tensor-core transform takes contiguous input only
  if (!x_bf16 || !payload) return FP4Q_ERR_NULL;
  if ((st = check_2d(rows, cols, ld, 2)) != FP4Q_OK) return st;
  if (!aligned16(x_bf16) || !aligned16(payload)) return FP4Q_ERR_ALIGN;
  const int64_t n = rows * cols;
  if (overlap(x_bf16, span_2d(rows, cols, ld, 2), payload, payload_bytes_of(n, G, MX))) return FP4Q_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ld == cols) return fp4q_compress(x_bf16, n, payload, params, stream);
  if (MX) return F ? launch_compress_2d<32, 1, true>(x_bf16, rows, cols, ld, payload, s)
                   : launch_compress_2d<32, 0, true>(x_bf16, rows, cols, ld, payload, s);
  if (G == 16) return F ? launch_compress_2d<16, 1, false>(x_bf16, rows, cols, ld, payload, s)
                        : launch_compress_2d<16, 0, false>(x_bf16, rows, cols, ld, payload, s);
  return F ? launch_compress_2d<32, 1, false>(x_bf16, rows, cols, ld, payload, s)
           : launch_compress_2d<32, 0, false>(x_bf16, rows, cols, ld, payload, s);
}

fp4q_status fp4q_decompress_accumulate_2d(const void* payload, int64_t rows, int64_t cols, void* dst, int64_t ld,
                                          fp4q_dtype dtype, int32_t beta, const fp4q_params* params,
                                          void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (F == 2) F = 1;   // a tensor-core-encoded payload is decoded like any fwht = 1 payload
  if ((dtype != FP4Q_BF16 && dtype != FP4Q_F32) || (beta != 0 && beta != 1)) return FP4Q_ERR_PARAM;
  if (!payload || !dst) return FP4Q_ERR_NULL;
  const int esz = dtype == FP4Q_BF16 ? 2 : 4;
  if ((st = check_2d(rows, cols, ld, esz)) != FP4Q_OK) return st;
  if (!aligned16(payload) || !aligned16(dst)) return FP4Q_ERR_ALIGN;
  const int64_t n = rows * cols;
  if (overlap(payload, payload_bytes_of(n, G, MX), dst, span_2d(rows, cols, ld, esz))) return FP4Q_ERR_OVERLAP;
  if (ld == cols) return fp4q_decompress_accumulate(payload, n, dst, dtype, beta, params, stream);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int key = F * 4 + (dtype == FP4Q_F32) * 2 + beta;
#define FP4Q_D2(GG, MM)                                                                        \
  switch (key) {                                                                               \
    case 0: return launch_decompress_2d<GG, 0, FP4Q_BF16, 0, MM>(payload, rows, cols, dst, ld, s); \
    case 1: return launch_decompress_2d<GG, 0, FP4Q_BF16, 1, MM>(payload, rows, cols, dst, ld, s); \
    case 2: return launch_decompress_2d<GG, 0, FP4Q_F32, 0, MM>(payload, rows, cols, dst, ld, s);  \
    case 3: return launch_decompress_2d<GG, 0, FP4Q_F32, 1, MM>(payload, rows, cols, dst, ld, s);  \
    case 4: return launch_decompress_2d<GG, 1, FP4Q_BF16, 0, MM>(payload, rows, cols, dst, ld, s); \
    case 5: return launch_decompress_2d<GG, 1, FP4Q_BF16, 1, MM>(payload, rows, cols, dst, ld, s); \
    case 6: return launch_decompress_2d<GG, 1, FP4Q_F32, 0, MM>(payload, rows, cols, dst, ld, s);  \
    default: return launch_decompress_2d<GG, 1, FP4Q_F32, 1, MM>(payload, rows, cols, dst, ld, s); \
  }
  if (MX) FP4Q_D2(32, true)
  if (G == 16) FP4Q_D2(16, false)
  FP4Q_D2(32, false)
#undef FP4Q_D2
}

fp4q_status fp4q_roundtrip_2d(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx, void* y_bf16,
                              int64_t ldy, const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (F == 2) return FP4Q_ERR_PARAM;   // the tensor-core transform takes contiguous input only
  if (!x_bf16 || !y_bf16) return FP4Q_ERR_NULL;
  if ((st = check_2d(rows, cols, ldx, 2)) != FP4Q_OK || (st = check_2d(rows, cols, ldy, 2)) != FP4Q_OK) return st;
  if (!aligned16(x_bf16) || !aligned16(y_bf16)) return FP4Q_ERR_ALIGN;
  if (overlap(x_bf16, span_2d(rows, cols, ldx, 2), y_bf16, span_2d(rows, cols, ldy, 2))) return FP4Q_ERR_OVERLAP;
  if (ldx == cols && ldy == cols) return fp4q_roundtrip(x_bf16, rows * cols, y_bf16, params, stream);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (MX) return F ? launch_roundtrip_2d<32, 1, true>(x_bf16, rows, cols, ldx, y_bf16, ldy, s)
                   : launch_roundtrip_2d<32, 0, true>(x_bf16, rows, cols, ldx, y_bf16, ldy, s);
  if (G == 16) return F ? launch_roundtrip_2d<16, 1, false>(x_bf16, rows, cols, ldx, y_bf16, ldy, s)
                        : launch_roundtrip_2d<16, 0, false>(x_bf16, rows, cols, ldx, y_bf16, ldy, s);
  return F ? launch_roundtrip_2d<32, 1, false>(x_bf16, rows, cols, ldx, y_bf16, ldy, s)
           : launch_roundtrip_2d<32, 0, false>(x_bf16, rows, cols, ldx, y_bf16, ldy, s);
}

fp4q_status fp4q_reduce_requantize(const void* const* payloads, int32_t R, int64_t n, void* out_payload,
                                   const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (R < 1 || R > FP4Q_MAX_RANKS) return FP4Q_ERR_PARAM;
  if (!payloads || !out_payload) return FP4Q_ERR_NULL;
  for (int r = 0; r < R; ++r)
    if (!payloads[r]) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  if (!aligned16(out_payload)) return FP4Q_ERR_ALIGN;
  for (int r = 0; r < R; ++r)
    if (!aligned16(payloads[r])) return FP4Q_ERR_ALIGN;
  const size_t pb = payload_bytes_of(n, G, MX);
  for (int r = 0; r < R; ++r)
    if (overlap(payloads[r], pb, out_payload, pb)) return FP4Q_ERR_OVERLAP;
  Payload ins[FP4Q_MAX_RANKS];
  for (int r = 0; r < R; ++r) ins[r] = payload_of(const_cast<void*>(payloads[r]), padded_n(n), G, MX);
  const Payload out = payload_of(out_payload, padded_n(n), G, MX);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return MX ? dispatch_reduce<true>(G, ins, R, n, out, s) : dispatch_reduce<false>(G, ins, R, n, out, s);
}

fp4q_status fp4q_segment_bytes(int64_t n, const fp4q_params* params, size_t* codes, size_t* gscales,
                               size_t* bscales) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (!codes || !gscales || !bscales) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  const SegSizes z = seg_sizes(n, G, MX);
  *codes = z.codes;
  *gscales = z.gsc;
  *bscales = z.bsc;
  return FP4Q_OK;
}

fp4q_status fp4q_compress_segments(const void* x, fp4q_dtype x_dtype, int64_t n, const fp4q_segments* out,
                                   const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (x_dtype != FP4Q_BF16 && x_dtype != FP4Q_F32) return FP4Q_ERR_PARAM;
  if (!x || !out) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  Payload P;
  if ((st = segments_of(out, n, G, MX, P)) != FP4Q_OK) return st;
  if (!aligned16(x)) return FP4Q_ERR_ALIGN;
  const SegSizes z = seg_sizes(n, G, MX);
  const bool xf = x_dtype == FP4Q_F32;
  if (segs_self_overlap(P, z) || seg_overlap(P, z, x, (size_t)n * (xf ? 4 : 2))) return FP4Q_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return xf ? dispatch_compress<true>(G, F, MX, x, n, P, s) : dispatch_compress<false>(G, F, MX, x, n, P, s);
}

fp4q_status fp4q_decompress_accumulate_segments(const fp4q_segments* in, int64_t n, void* dst, fp4q_dtype dtype,
                                                int32_t beta, const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (F == 2) F = 1;   // a tensor-core-encoded payload is decoded like any fwht = 1 payload
  if ((dtype != FP4Q_BF16 && dtype != FP4Q_F32) || (beta != 0 && beta != 1)) return FP4Q_ERR_PARAM;
  if (!in || !dst) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  Payload P;
  if ((st = segments_of(in, n, G, MX, P)) != FP4Q_OK) return st;
  if (!aligned16(dst)) return FP4Q_ERR_ALIGN;
  if (seg_overlap(P, seg_sizes(n, G, MX), dst, (size_t)n * (dtype == FP4Q_BF16 ? 2 : 4))) return FP4Q_ERR_OVERLAP;
  return dispatch_decompress_all(G, F, MX, P, n, dst, dtype, beta, static_cast<cudaStream_t>(stream));
}

fp4q_status fp4q_reduce_requantize_segments(const fp4q_segments* in, int32_t R, int64_t n, const fp4q_segments* out,
                                            const fp4q_params* params, void* stream) {
  int G, F;
  bool MX;
  fp4q_status st = check_params(params, G, F, MX);
  if (st != FP4Q_OK) return st;
  if (R < 1 || R > FP4Q_MAX_RANKS) return FP4Q_ERR_PARAM;
  if (!in || !out) return FP4Q_ERR_NULL;
  if (!size_ok(n)) return FP4Q_ERR_SIZE;
  Payload ins[FP4Q_MAX_RANKS], P;
  for (int r = 0; r < R; ++r)
    if ((st = segments_of(&in[r], n, G, MX, ins[r])) != FP4Q_OK) return st;
  if ((st = segments_of(out, n, G, MX, P)) != FP4Q_OK) return st;
  const SegSizes z = seg_sizes(n, G, MX);
  if (segs_self_overlap(P, z)) return FP4Q_ERR_OVERLAP;
  for (int r = 0; r < R; ++r)
    if (segs_overlap(ins[r], P, z)) return FP4Q_ERR_OVERLAP;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return MX ? dispatch_reduce<true>(G, ins, R, n, P, s) : dispatch_reduce<false>(G, ins, R, n, P, s);
}

fp4q_status fp4q_fault_flags(uint32_t* flags, int32_t clear) {
  if (!flags) return FP4Q_ERR_NULL;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fp4q_fault, sizeof(v)) != cudaSuccess) return FP4Q_ERR_CUDA;
  *flags = v;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fp4q_fault, &zero, sizeof(zero)) != cudaSuccess) return FP4Q_ERR_CUDA;
  }
  return FP4Q_OK;
}

fp4q_status fp4q_selftest_wait_timeout(uint32_t polls, void* stream) {
  if (polls == 0 || polls > (1u << 20)) return FP4Q_ERR_PARAM;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(polls);
  return launched();
}

const char* fp4q_status_string(fp4q_status status) {
  switch (status) {
    case FP4Q_OK: return "ok";
    case FP4Q_ERR_NULL: return "null pointer";
    case FP4Q_ERR_SIZE: return "n must be positive and below 2^37";
    case FP4Q_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FP4Q_ERR_PARAM: return "invalid parameter (group, block, fwht, scales, R, dtype, beta or polls)";
    case FP4Q_ERR_OVERLAP: return "output overlaps an input";
    case FP4Q_ERR_CUDA: return "CUDA runtime error or failed launch";
  }
  return "unknown status";
}

int32_t fp4q_version(void) { return 300; }

}  // extern "C"

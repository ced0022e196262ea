/*
 * fp4q.h - C ABI of the FP4 communication codec (compress, decompress-accumulate,
 * fused roundtrip, emulated R-way reduce) for NVIDIA GB300 (sm_103a).
 *
 * Source of the method:
 *   [P1] "FP4Quant: Efficient 4-Bit Communication Compression for Model-Parallel LLM
 *        Training" (shd-paper.top summary of arXiv 2611.04323), English abstract and the
 *        method section's "technical framework" paragraph: micro-grouped dual-scale FP4
 *        quantization, warp-cooperative FP4 packing, hybrid two-level FWHT.
 *   [P3] "4-bit compression speeds up LLM training by 56 percent with minimal accuracy
 *        loss" (zot.news), lead paragraph and "Read it as": small clusters of values share
 *        scaling factors, values are packed two per byte, a fast transform keeps errors
 *        low; the compressed tensors are the ones the tensor-parallel AllReduce exchanges.
 *   [P4] "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"
 *        (gist.science), technical summary, problem statement: FP4 elements are E2M1, and
 *        the microscaled MXFP4 format scales blocks of 32 of them.
 *
 * The pages fix the shape of the method but none of its numbers. This header is the one
 * place where the numbers are fixed; every kernel and the CPU oracle implement exactly
 * this contract:
 *
 *   Block.   The tensor is cut into blocks of FP4Q_BLOCK = 256 consecutive elements.
 *            Any n >= 1: a last partial block is zero-padded to 256 elements (+0), the
 *            payload covers ceil(n/256) blocks, and every decode writes back only the n
 *            elements (the pages say nothing about other lengths; this is the build's
 *            reading).
 *   FWHT.    (fwht = 1) per block, y = (1/16) * H256 * x with H256 the Sylvester-ordered
 *            Walsh-Hadamard matrix, H256 = H16 (x) H16. It is evaluated as the butterfly
 *            sequence h = 1, 2, 4, ..., 128: for every j with (j & h) == 0,
 *            (y[j], y[j+h]) <- (y[j] + y[j+h], y[j] - y[j+h]) in FP32 round-to-nearest,
 *            then y <- y * 0.0625f. Stages h < 16 act inside a 16-element group (level 1),
 *            stages h >= 16 act across the 16 groups of a block (level 2). [P1 "hybrid
 *            two-level FWHT pipeline"; P3 "a fast transform keeps errors low"]
 *   Scales.  Two levels [P1 "dual-scale"; P3 "tiny clusters of values share scaling
 *            factors"]:
 *              A_b = max |y| over the block.
 *              If A_b < 2688 * 2^-100 the block is all-zero: s_b = 0, every group scale
 *              byte 0x00, every code 0x0.
 *              Otherwise s_b = A_b / 2688.0f   (2688 = 6 * 448, FP32 IEEE division).
 *              t_b = s_b * 6.0f; per group of G elements r_g = amax_g / t_b (IEEE div);
 *              s_g = E4M3(r_g): round to nearest, ties to the even code, saturating at
 *              448 (OCP e4m3fn, codes 0x00..0x7E, never 0x7F).
 *   Scales, microscaled variant (scales = FP4Q_SCALES_E8M0, group 32 only) [P4 problem
 *            statement: MXFP4 scales blocks of 32 E2M1 elements]: no block scale; per group
 *            X = 2^(floor(log2 amax_g) - 2), stored as the E8M0 byte e + 127 with the
 *            exponent e clamped below at -127 (amax_g = 0 and subnormal maxima give byte 0),
 *            so amax_g / X lies in [4, 8); q = y / X (exact), code as below; decode
 *            x~ = grid(code) * X. No all-zero guard: a zero keeps its sign (0x0 / 0x8).
 *   Codes.   S_g = float(s_g) * s_b; inv_g = S_g > 0 ? 1.0f / S_g : 0.0f (IEEE);
 *            q = y * inv_g; code = sign(q) << 3 | E2M1(|q|), E2M1 = round to nearest,
 *            ties to the even code, onto {0, 0.5, 1, 1.5, 2, 3, 4, 6} (codes 0..7),
 *            saturating at 6. The sign is kept: a negative q that rounds to 0 gives 0x8.
 *            [P4 "E2M1"; P1 "FP4"]
 *   Packing. byte k of the code segment = code[2k] | code[2k+1] << 4 (even element in
 *            the low nibble). [P3 "packed two per byte"]
 *   Payload. One contiguous byte buffer, structure of arrays:
 *              [codes: n/2 bytes][group scales: n/G bytes, zero-padded to a multiple of
 *              16][block scales: n/256 x float32, little endian; absent for E8M0 scales]
 *            Every segment starts 16-byte aligned when the buffer does. A contiguous range
 *            of blocks can be cut out of each segment.
 *   Decode.  x~ = grid(code) * S_g (signed, FP32); if fwht, the inverse transform: the
 *            same butterflies in mirror order h = 128, 64, ..., 1 (level 2, then level 1),
 *            followed by * 0.0625f (H is symmetric and H*H = I, so the stages of the forward
 *            transform undone in reverse order give the inverse).
 *   Reduce.  z = x~_0 + x~_1 + ... + x~_{R-1} (FP32, in rank order, no FMA), decoded in
 *            the transform domain (no inverse FWHT), then Scales/Codes/Packing on z with
 *            no forward FWHT. [P3 "Read it as": the AllReduce of tensor parallelism]
 *   Tensor-core encoder (fwht = 2; relaxed, opt-in) [P1 "hybrid two-level FWHT pipeline",
 *            "GPU-aware execution optimization"]: the same y = H256 x / 16, with the two
 *            butterfly stages that mix the four quarter-blocks of a block (strides 64 and 128)
 *            computed first, as a +-1 BF16 matrix product on the tensor cores (exact products,
 *            FP32 accumulation in the hardware's order), then the other six stages as FP32
 *            butterflies. y agrees with the FWHT step above to FP32 rounding only (about 1e-6
 *            of the block maximum), so a scale
 *            or a code whose contract value lies on a rounding boundary can differ; the
 *            payload format is unchanged and decodes as an fwht = 1 payload. Contiguous
 *            BF16 input only, either scale format (fp4q_compress, fp4q_compress_segments); the
 *            decoders and the reduce accept fwht = 2 as fwht = 1; the other producers reject
 *            it (FP4Q_ERR_PARAM).
 *
 * Every floating-point step is a separately rounded FP32 operation (no FMA contraction),
 * so the GPU result is bit-identical to a plain scalar evaluation of the steps above.
 *
 * Preconditions on data (not checked): inputs finite and |x| < 2^120.
 *
 * Threading and ownership: the caller owns every buffer, and the library allocates no device
 * memory. The library holds process-wide state of two kinds: a cache, per kernel variant
 * and device, of the launch plan (shared-memory attributes set once, the occupancy query),
 * guarded by a mutex; and one 4-byte fault word per device (a __device__ variable, read and
 * cleared by fp4q_fault_flags). Nothing else persists between calls. All entry points are
 * asynchronous on the given stream and never synchronise. Argument errors are returned
 * before anything is launched. A failed launch returns FP4Q_ERR_CUDA (the CUDA error is left
 * to the caller's next runtime call to report). FP4Q_OK means the kernels were launched, not
 * that they completed: a kernel whose bounded wait on a copy gives up returns early with its
 * outputs incomplete and records this in the fault word, which the caller must read (after
 * synchronising) to know that every call since the word was cleared ran to completion.
 * Kernels are launched with programmatic stream serialisation:
 * a codec kernel may be scheduled while the previous kernel on the stream is finishing,
 * but it waits for that kernel to complete (and for its memory to be visible) before its
 * first global-memory access, so stream order is preserved exactly. The first call of each
 * kernel variant on a device sets that kernel's dynamic shared-memory limit and preferred
 * shared-memory carveout (the largest) and queries its occupancy; the results are cached per
 * kernel and device, and the library's own kernels are the only ones it configures.
 * Calls may be captured in a CUDA graph once each kernel variant has run on the device (so
 * that the first-call configuration above happens outside the capture): a launch carries
 * everything it needs as kernel parameters (tensor maps of the given buffers included) and
 * keeps no host state, so a replay on new contents of the same buffers computes what the
 * same calls would. Several host threads may call the library at once, each on its own
 * stream.
 */
#ifndef FP4Q_H
#define FP4Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP4Q_BLOCK 256              /* elements per block (FWHT length, block scale)   */
#define FP4Q_GROUP_DEFAULT 16       /* elements per micro-group (E4M3 scale)           */
#define FP4Q_MAX_RANKS 8            /* largest R accepted by fp4q_reduce_requantize    */
#define FP4Q_E4M3_MAX 448.0f        /* largest finite e4m3fn value                      */
#define FP4Q_E2M1_MAX 6.0f          /* largest E2M1 value                               */
#define FP4Q_BLOCK_DENOM 2688.0f    /* FP4Q_E4M3_MAX * FP4Q_E2M1_MAX                    */
#define FP4Q_SCALES_DUAL 0          /* E4M3 group scale x FP32 block scale (default)     */
#define FP4Q_SCALES_E8M0 1          /* power-of-two E8M0 scale per group of 32          */

typedef enum fp4q_status {
  FP4Q_OK = 0,
  FP4Q_ERR_NULL = 1,     /* a required pointer is NULL                                  */
  FP4Q_ERR_SIZE = 2,     /* n <= 0 or n >= 2^37                                         */
  FP4Q_ERR_ALIGN = 3,    /* a data pointer is not 16-byte aligned                       */
  FP4Q_ERR_PARAM = 4,    /* bad params: group not 16/32, block not 256, fwht not 0/1/2,
                            scales not 0/1 or E8M0 with group != 32, R outside [1, 8],
                            unknown dtype, beta not 0/1                                 */
  FP4Q_ERR_OVERLAP = 5,  /* an output buffer overlaps an input buffer                   */
  FP4Q_ERR_CUDA = 6      /* a CUDA runtime call or a kernel launch failed               */
} fp4q_status;

typedef struct fp4q_params {
  int32_t group;  /* G: 16 (default) or 32 elements per group scale                    */
  int32_t block;  /* must be 256                                                        */
  int32_t fwht;   /* 1: apply the FWHT (default); 0: quantize the raw values; 2: the FWHT
                     with the tensor-core encoder (relaxed; see above)                     */
  int32_t scales; /* FP4Q_SCALES_DUAL (default) or FP4Q_SCALES_E8M0 (needs group 32)    */
} fp4q_params;

typedef enum fp4q_dtype {
  FP4Q_BF16 = 0,  /* destination is bfloat16, rounded to nearest even                   */
  FP4Q_F32 = 1    /* destination is float32                                             */
} fp4q_dtype;

/* Bytes of the payload for n elements, with m = n rounded up to a multiple of 256:
 * m/2 + pad16(m/G) + 4*(m/256) (dual scales) or m/2 + pad16(m/32) (E8M0 scales).
 * Returns 0 when n or params are invalid.
 * params == NULL means the defaults {16, 256, 1, FP4Q_SCALES_DUAL}. */
size_t fp4q_payload_bytes(int64_t n, const fp4q_params* params);

/* Byte offsets of the group-scale and block-scale segments inside the payload
 * (the code segment starts at offset 0). Return 0 on invalid arguments. */
size_t fp4q_gscale_offset(int64_t n, const fp4q_params* params);
size_t fp4q_bscale_offset(int64_t n, const fp4q_params* params);

/* Compress: x_bf16 (device, n bfloat16, 16-byte aligned) -> payload (device,
 * fp4q_payload_bytes(n) bytes, 16-byte aligned). Steps FWHT, Scales, Codes, Packing
 * above [P1 abstract: micro-grouped dual-scale FP4 quantization, warp-cooperative
 * packing, two-level FWHT]. payload must not overlap x (FP4Q_ERR_OVERLAP).
 * stream: a cudaStream_t (NULL = legacy default stream). */
fp4q_status fp4q_compress(const void* x_bf16, int64_t n, void* payload,
                          const fp4q_params* params, void* stream);

/* Compress of FP32 input: x_f32 (device, n float32, 16-byte aligned) -> payload, the same
 * steps with the input values used as they are instead of widened from BF16 (general
 * shapes: FP32 tensors such as FP32 gradients). A BF16-exact input gives the payload
 * fp4q_compress gives. payload must not overlap x (FP4Q_ERR_OVERLAP). */
fp4q_status fp4q_compress_f32(const void* x_f32, int64_t n, void* payload,
                              const fp4q_params* params, void* stream);

/* Decompress-accumulate: payload (device) -> dst (device, n elements of dtype, 16-byte
 * aligned). dst = beta ? dst + x^ : x^, where x^ is the Decode step above; for a bfloat16
 * dst the sum is formed in FP32 and rounded to nearest even once. This is the receive side
 * of the compressed AllReduce [P3 "Read it as"]. dst may not overlap payload. The payload
 * is expected as fp4q_compress / fp4q_reduce_requantize write it (every block scale 0 or
 * >= 2^-100); for other block scales the result can differ from the contract's decode in
 * the last bit of values in the subnormal range. */
fp4q_status fp4q_decompress_accumulate(const void* payload, int64_t n, void* dst,
                                       fp4q_dtype dtype, int32_t beta,
                                       const fp4q_params* params, void* stream);

/* Fused roundtrip (fake quantization): y_bf16 = bf16(decode(compress(x_bf16))) without
 * writing a payload. Bit-identical to fp4q_compress followed by
 * fp4q_decompress_accumulate(..., FP4Q_BF16, beta = 0). y must not overlap x. */
fp4q_status fp4q_roundtrip(const void* x_bf16, int64_t n, void* y_bf16,
                           const fp4q_params* params, void* stream);

/* Fused roundtrip of FP32 data: y_f32 = decode(compress_f32(x_f32)) in FP32 (no BF16
 * rounding), bit-identical to fp4q_compress_f32 followed by
 * fp4q_decompress_accumulate(..., FP4Q_F32, beta = 0). y must not overlap x. */
fp4q_status fp4q_roundtrip_f32(const void* x_f32, int64_t n, void* y_f32,
                               const fp4q_params* params, void* stream);

/* Strided 2-D variants (general shapes): a row-major [rows, cols] view with a row stride of
 * ld elements (ld >= cols, ld * element size a multiple of 16 bytes, cols a multiple of
 * 256, rows * cols < 2^37). The payload is that of the dense row-major [rows, cols] tensor
 * (n = rows * cols) and is interchangeable with the 1-D entry points'; only the data
 * tensors are strided. Each block is one TMA box of a 3-D map {line, line in row, row}.
 * Errors as for the 1-D calls; a bad shape gives FP4Q_ERR_SIZE, ld < cols FP4Q_ERR_PARAM,
 * a misaligned row stride FP4Q_ERR_ALIGN. ld == cols runs the 1-D call. */
fp4q_status fp4q_compress_2d(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                             void* payload, const fp4q_params* params, void* stream);
fp4q_status fp4q_decompress_accumulate_2d(const void* payload, int64_t rows, int64_t cols,
                                          void* dst, int64_t ld, fp4q_dtype dtype, int32_t beta,
                                          const fp4q_params* params, void* stream);
fp4q_status fp4q_roundtrip_2d(const void* x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                              void* y_bf16, int64_t ldy, const fp4q_params* params,
                              void* stream);

/* Emulated R-way reduce: payloads is a HOST array of R device pointers, each a payload of
 * n elements made with the same params; out_payload (device) receives the requantized sum
 * (Reduce step above). This is the fused decompress-sum-requantize step of a
 * reduce-scatter/all-gather AllReduce with all R rank buffers resident on one GPU
 * [P3 "Read it as"]. params->fwht only records the domain of the payloads; the reduce never
 * transforms. out_payload may not overlap any input payload. 1 <= R <= FP4Q_MAX_RANKS. */
fp4q_status fp4q_reduce_requantize(const void* const* payloads, int32_t R, int64_t n,
                                   void* out_payload, const fp4q_params* params,
                                   void* stream);

/* A payload placed as three separate device buffers instead of one contiguous one (the
 * Payload step above, segment by segment): codes (m/2 bytes), group scales (m/G bytes
 * zero-padded to a multiple of 16) and block scales (4 m/256 bytes; NULL for E8M0 scales),
 * m = n rounded up to a multiple of 256. Each pointer must be 16-byte aligned. The segments
 * of a tensor's payload can then be cut at block boundaries and scattered / gathered by a
 * collective (reduce-scatter, all-gather) without any repacking: the compressed AllReduce
 * of tensor parallelism [P3 "Read it as"] exchanges exactly such slices. */
typedef struct fp4q_segments {
  void* codes;
  void* gscales;
  void* bscales;
} fp4q_segments;

/* Sizes in bytes of the three segments of a payload of n elements (as above); bscales is 0
 * for E8M0 scales. Errors: FP4Q_ERR_PARAM, FP4Q_ERR_NULL, FP4Q_ERR_SIZE. */
fp4q_status fp4q_segment_bytes(int64_t n, const fp4q_params* params, size_t* codes, size_t* gscales,
                               size_t* bscales);

/* fp4q_compress / fp4q_compress_f32 (x_dtype FP4Q_BF16 or FP4Q_F32) writing the payload into
 * separately placed segments. Bit-identical to the contiguous call. No segment may overlap x
 * or another segment (FP4Q_ERR_OVERLAP). */
fp4q_status fp4q_compress_segments(const void* x, fp4q_dtype x_dtype, int64_t n, const fp4q_segments* out,
                                   const fp4q_params* params, void* stream);

/* fp4q_decompress_accumulate reading a payload from separately placed segments. */
fp4q_status fp4q_decompress_accumulate_segments(const fp4q_segments* in, int64_t n, void* dst, fp4q_dtype dtype,
                                                int32_t beta, const fp4q_params* params, void* stream);

/* fp4q_reduce_requantize over R payloads given as segments (in: a HOST array of R segment
 * sets), writing the requantized sum into the segments of out. This is the shard owner's
 * step of a compressed reduce-scatter: in[r] are the slices of rank r's payload that cover
 * the owner's shard, in rank order [P3 "Read it as": the AllReduce of tensor parallelism].
 * 1 <= R <= FP4Q_MAX_RANKS; out may not overlap any input or itself. */
fp4q_status fp4q_reduce_requantize_segments(const fp4q_segments* in, int32_t R, int64_t n, const fp4q_segments* out,
                                            const fp4q_params* params, void* stream);

/* Device fault word of the current device. The kernels wait on TMA copies with bounded
 * waits (about a second); a wait that gives up sets a bit here, waits (bounded) for the
 * warp's copies still in flight and returns early, leaving that call's outputs incomplete:
 *   bit 0: a TMA load did not complete within the bound;
 *   bit 1: a copy still in flight after such a fault did not complete either;
 *   bit 2: fp4q_selftest_wait_timeout ran out (expected).
 * The word is sticky across calls. This call synchronises with the device (it reads device
 * memory); clear != 0 resets the word to 0 afterwards. No counterpart in the pages: it
 * reports the health of this implementation's asynchronous copies. */
fp4q_status fp4q_fault_flags(uint32_t* flags, int32_t clear);

/* Self-test of the bounded wait: launches one warp that waits on a barrier phase nothing
 * completes, giving up after `polls` polls (1 <= polls <= 2^20) and setting bit 2 of the
 * fault word. Asynchronous on `stream`. No counterpart in the pages. */
fp4q_status fp4q_selftest_wait_timeout(uint32_t polls, void* stream);

/* Static string naming a status code (never NULL). */
const char* fp4q_status_string(fp4q_status status);

/* Library version as 10000*major + 100*minor + patch. */
int32_t fp4q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP4Q_H */

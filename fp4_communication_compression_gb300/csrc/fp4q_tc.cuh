// fp4q_tc.cuh - compress with the transform on the tensor cores (fp4q_params.fwht = 2).
// Included by fp4q.cu inside its anonymous namespace, after the shared helpers.
//
// The method: "FP4Quant" (shd-paper.top), technical framework: a hybrid two-level FWHT in a
// GPU-aware pipeline. A block of 256 elements is x[g][p] (g = group of 16, p = position in
// the group) and H256 = H16 (x) H16; with H16 = H4 (x) H4 the group index splits further into
// g = 4 gh + gl. This encoder evaluates the part of the transform that mixes the four
// quarter-blocks (gh, two butterfly stages) as a +-1 matrix product on the 5th-generation
// tensor cores and the remaining six stages in registers:
//   D = Hq * Xq    (tcgen05.mma kind::f16, BF16 operands, FP32 accumulation in TMEM)
// where Xq is the BF16 input of 4 x 32 consecutive blocks exactly as the TMA loads it (128-byte
// lines of 64 elements, each a quarter-block (block, gh); 128-byte swizzle): the four 32-block
// sub-batches side by side form a K x N = 128 x 256 MN-major operand whose K index (block within
// the sub-batch, gh) they share. Hq is the block-diagonal 128 x 128 matrix of 32 H4 blocks, applied as
// eight K = 16 slices (slice j holds four H4 blocks in rows 16j .. 16j+15; every slice is a
// window of one 240-row buffer that has them in rows 112 .. 127 and zeros elsewhere). TMEM
// lane (block, gh') then holds the 64 values (gl, p) of that quarter-block after the mixing;
// its thread loads them with tcgen05.ld, applies H4 across gl and H16 along p with FP32
// butterflies and holds the four groups 4 gh' + gl' of the block: the row layout of the
// tiled kernels (four lanes per block, four groups per lane), so the same quantisation (dual
// or E8M0 scales) and store run on it.
//
// The products are exact (BF16 times +-1) but the tensor core accumulates each 4-term sum in
// its own order and the stages run in another order than the contract's butterfly sequence,
// so y matches the contract only to FP32 rounding: scales and codes can differ where the
// contract's value sits on a rounding boundary. The payload format is the contract's, and
// every decoder reads it as an fwht = 1 payload.
//
// Pipeline (warp-specialised, one persistent CTA per SM). A batch is 128 consecutive blocks
// (four sub-batches of 32, side by side in the MMA's N dimension: N = 256, so each MMA
// instruction covers 4 x 32 blocks; at N = 64 the producer spent ~80 cycles issuing each
// MMA and paced the whole pipeline). A producer warp keeps kTcStages - kTcRefillLag batches
// in flight by TMA and issues the eight MMAs of each batch into one of two 256-column TMEM
// accumulators as soon as its input has landed and the accumulator is free; each of the
// kTcGroups consumer warpgroups takes one sub-batch (64 columns) of every batch, copies it
// to registers (one tcgen05.ld of 64 columns), frees it, then applies the in-register stages
// and quantises while the tensor cores fill the other accumulator. MMA completion is signalled
// with tcgen05.commit to mbarriers (accumulator full, input stage free). Every wait is
// bounded; a wait that gives up sets the fault word and a CTA-wide stop flag, the producer
// waits (bounded) for the copies and products it issued, and the CTA frees its TMEM.

constexpr int kTcGroups = 4;                         // consumer warpgroups = sub-batches per batch
constexpr int kTcSubBlocks = 32;                     // blocks per sub-batch (128 quarter-block rows = MMA M, K)
constexpr int kTcBatchBlocks = kTcGroups * kTcSubBlocks;
constexpr int kTcSubBytes = kTcSubBlocks * 512;      // BF16 input of one sub-batch (16 KiB)
constexpr int kTcBatchBytes = kTcGroups * kTcSubBytes;
constexpr int kTcAcc = 2;                            // TMEM accumulators
constexpr int kTcAccCols = 64 * kTcGroups;           // MMA N: 256 FP32 columns per accumulator
constexpr uint32_t kTcTmemCols = kTcAcc * kTcAccCols;  // 512: the whole TMEM of the SM
constexpr int kTcStages = 3;                         // input batches buffered per CTA
constexpr int kTcRefillLag = 1;                      // a stage is refilled this many batches after its MMAs
constexpr int kTcZBytes = 8192;                      // A operand buffer (240 rows used)
constexpr int kTcThreads = 32 * (4 * kTcGroups + 1);   // consumers + one producer warp
constexpr int kTcSmemBytes = 1024 + kTcZBytes + kTcStages * kTcBatchBytes;

// Shared-memory matrix descriptor of tcgen05.mma: start address, leading and stride byte
// offsets (16-byte units), the sm_100 descriptor version (bit 46) and the swizzle mode.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | (uint64_t)((lbo >> 4) & 0x3FFFu) << 16 |
         (uint64_t)((sbo >> 4) & 0x3FFFu) << 32 | (uint64_t)1 << 46 | (uint64_t)swizzle << 61;
}
constexpr uint32_t kUmmaSwizzle32B = 6;
// Instruction descriptor (kind::f16): D FP32, A and B BF16, A K-major, B MN-major,
// N = kTcAccCols, M = 128.
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                              ((uint32_t)(kTcAccCols >> 3) << 17) | ((128u >> 4) << 24);
// Operand layouts (checked on the hardware against a CPU product): A K-major without swizzle,
// core matrices of 8 rows x 16 bytes, K-group stride 128 bytes (LBO), row-group stride 256
// (SBO); B MN-major with the 128-byte swizzle the TMA writes, rows of 64 elements, 8-row group
// stride 1024 bytes (SBO), 64-column group stride one sub-batch (LBO).
constexpr uint32_t kTcALbo = 128, kTcASbo = 256, kTcBLbo = kTcSubBytes, kTcBSbo = 1024;
constexpr uint32_t kUmmaSwizzle128B = 2;

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               ::"r"(d_tmem), "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate)
               : "memory");
}
// Arrive on an mbarrier once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive 32-bit TMEM columns of the warp's 32 lanes (one row per thread), without
// waiting: the registers are valid after tmem_ld_wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t r[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// One poll loop of the pipeline: bounded, and it also gives up when another thread of the CTA
// has already given up (stop flag in shared memory).
// BACKOFF: sleep between polls (consumer warps, which wait for most of a batch: spinning, they
// would take issue slots from the producer warp that shares their sub-partition).
template <bool BACKOFF>
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, const volatile uint32_t* stop) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  uint32_t sleep_ns = 32;
  for (uint32_t k = 1; k < kSpinLimit; ++k) {
    if (BACKOFF) {
      __nanosleep(sleep_ns);
      if (sleep_ns < 256) sleep_ns <<= 1;
    }
    if (mbar_try_wait(bar, parity)) return true;
    if ((k & 63u) == 0u && (*stop || global_ns() - t0 > kWaitLimitNs)) return false;
  }
  return false;
}

template <int G, bool MX>
__global__ void __launch_bounds__(kTcThreads, 1)
compress_tc_kernel(const __grid_constant__ CUtensorMap xmap, Payload P, int64_t nb, int64_t batches) {
  extern __shared__ uint8_t smem_raw[];
  // mbarriers: input stage full (TMA), input stage free (MMA done), accumulator full (MMA done),
  // accumulator free (its 4 consumer warps have read it)
  __shared__ __align__(8) uint64_t bars[2 * kTcStages + 2 * kTcAcc];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile uint32_t stop;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t zbuf = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t stage0 = zbuf + kTcZBytes;
  const uint32_t full0 = smem_addr(&bars[0]), sfree0 = full0 + 8u * kTcStages;
  const uint32_t afull0 = sfree0 + 8u * kTcStages, afree0 = afull0 + 8u * kTcAcc;

  // A operand: row r, column k at (r / 8) * 256 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2;
  // rows 112 .. 127 hold four H4 blocks on the diagonal (entry (i, k) = (-1)^popcount(i & k)
  // when i / 4 == k / 4, exact in BF16), the rest 0.
  for (int u = tid; u < kTcZBytes / 16; u += kTcThreads) {
    const int r = 8 * (u >> 4) + (u & 7), k0 = 8 * ((u >> 3) & 1);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (r >= 112 && r < 128) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = r - 112, k = k0 + e;
        if ((i >> 2) != (k >> 2)) continue;
        const uint32_t h = (__popc((uint32_t)(i & k & 3)) & 1) ? 0xBF80u : 0x3F80u;
        w[e >> 1] |= h << (16 * (e & 1));
      }
    }
    sts128(zbuf + 16u * (uint32_t)u, make_uint4(w[0], w[1], w[2], w[3]));
  }
  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(sfree0 + 8u * s, 1);
    }
    for (int a = 0; a < kTcAcc; ++a) {
      mbar_init(afull0 + 8u * a, 1);
      mbar_init(afree0 + 8u * a, 4 * kTcGroups);
    }
    stop = 0u;
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                 "r"(kTcTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_proxy_async();                       // the A operand, written by threads, read by the MMA
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  grid_dependency_wait();
  grid_launch_dependents();

  const int64_t first = blockIdx.x, step = gridDim.x;
  const int64_t mine = first < batches ? (batches - 1 - first) / step + 1 : 0;
  if (warp == 4 * kTcGroups) {
    // ---------------------------------------------------------------- producer warp
    int64_t loaded = 0, issued = 0;
    bool ok = true;
    auto load = [&](int64_t i) {               // lane 0: TMA of batch i into stage i % kTcStages
      const uint32_t st = stage0 + (uint32_t)((i % kTcStages) * kTcBatchBytes), bar = full0 + 8u * (uint32_t)(i % kTcStages);
      if (lane == 0) {
        // two boxes of 256 lines = 128 blocks (lines past the tensor's end read as zeros)
        const int32_t line0 = (int32_t)((first + i * step) * (4 * kTcBatchBlocks));
        mbar_expect_tx(bar, (uint32_t)kTcBatchBytes);
        tma_load_2d(st, &xmap, 0, line0, bar);
        tma_load_2d(st + kTcBatchBytes / 2, &xmap, 0, line0 + 2 * kTcBatchBlocks, bar);
      }
    };
    // descriptors: the A slices are fixed; a B slice differs from the first stage's first slice
    // only in the start-address field (address >> 4, which stays below 2^14 inside shared memory)
    uint64_t adesc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) adesc[j] = umma_desc(zbuf + (uint32_t)(14 - 2 * j) * 256u, kTcALbo, kTcASbo, 0);
    const uint64_t bdesc0 = umma_desc(stage0, kTcBLbo, kTcBSbo, kUmmaSwizzle128B);
    for (; loaded < kTcStages && loaded < mine; ++loaded) load(loaded);
    for (int64_t i = 0; i < mine && ok; ++i) {
      const int s = (int)(i % kTcStages), a = (int)(i % kTcAcc);
      ok = __all_sync(kFull, tc_wait<false>(full0 + 8u * s, (uint32_t)((i / kTcStages) & 1), &stop));
      if (ok && i >= kTcAcc) ok = __all_sync(kFull, tc_wait<false>(afree0 + 8u * a, (uint32_t)(((i / kTcAcc) - 1) & 1), &stop));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d = tmem + (uint32_t)(a * kTcAccCols);
        const uint64_t bd = bdesc0 + (uint64_t)((uint32_t)(s * kTcBatchBytes) >> 4);   // + 128 per K-slice (16 rows)
#pragma unroll
        for (int j = 0; j < 8; ++j) umma_bf16(d, adesc[j], bd + (uint64_t)(128u * (uint32_t)j), j > 0);
        umma_commit(afull0 + 8u * a);
        umma_commit(sfree0 + 8u * s);
      }
      __syncwarp();
      issued = i + 1;
      // refill the stage of batch i - kTcRefillLag (its products finished long ago) with batch
      // i - kTcRefillLag + kTcStages: the copies stay kTcStages - kTcRefillLag batches ahead
      const int64_t k = i - kTcRefillLag;
      if (k >= 0 && loaded < mine) {
        ok = __all_sync(kFull, tc_wait<false>(sfree0 + 8u * (uint32_t)(k % kTcStages), (uint32_t)((k / kTcStages) & 1), &stop));
        if (!ok) break;
        load(loaded++);
      }
    }
    if (!ok) {
      if (lane == 0) {
        stop = 1u;
        atomicOr(&g_fp4q_fault, kFaultLoadWait);
      }
      // wait (bounded) for the copies and products still in flight before the TMEM is freed
      for (int64_t k = issued; k < loaded; ++k)
        if (!mbar_wait(full0 + 8u * (uint32_t)(k % kTcStages), (uint32_t)((k / kTcStages) & 1), kSpinLimit) && lane == 0)
          atomicOr(&g_fp4q_fault, kFaultDrainWait);
      for (int64_t k = issued > kTcStages ? issued - kTcStages : 0; k < issued; ++k)   // no later use of those stages
        if (!mbar_wait(sfree0 + 8u * (uint32_t)(k % kTcStages), (uint32_t)((k / kTcStages) & 1), kSpinLimit) && lane == 0)
          atomicOr(&g_fp4q_fault, kFaultDrainWait);
    }
  } else {
    // ---------------------------------------------------------------- consumer warpgroups
    const int grp = warp >> 2, wq = warp & 3;   // warpgroup (= sub-batch), its quarter of the TMEM lanes
    const int l4 = lane & 3;                    // gh' of the lane's quarter-block (four lanes per block)
    for (int64_t i = 0; i < mine; ++i) {
      const int a = (int)(i % kTcAcc);
      if (!__all_sync(kFull, tc_wait<true>(afull0 + 8u * a, (uint32_t)((i / kTcAcc) & 1), &stop))) {
        if (lane == 0) {
          stop = 1u;
          atomicOr(&g_fp4q_fault, kFaultLoadWait);
        }
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(a * kTcAccCols + 64 * grp);
      uint32_t r[4][16];
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_ld16(acc + 16u * (uint32_t)k, r[k]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(afree0 + 8u * a) : "memory");
      Rows v;                                   // v[gl][j]: positions 2j, 2j + 1 of group gl
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) v[k][j] = make_float2(__uint_as_float(r[k][2 * j]), __uint_as_float(r[k][2 * j + 1]));
      rows_bfly(v, 1);                          // H4 across gl
      rows_bfly(v, 2);
#pragma unroll
      for (int k = 0; k < 4; ++k)               // H16 along p (strides 1, 2, 4, 8)
#pragma unroll
        for (int j = 0; j < 8; ++j) bfly_in(v[k][j]);
      level1_fwd_from2(v);
      Quant q;
      if (MX) {
        scale_rows_16th(v);                     // the power-of-two scale sees y itself
        quantize_mx<false>(v, q);
      } else {
        quantize<G, false, true>(v, q);
      }
      const int64_t gb = (first + i * step) * kTcBatchBlocks + kTcSubBlocks * grp + 8 * wq + (lane >> 2);
      if (gb < nb) store_block<G, false, MX>(P, gb, l4, q);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols) : "memory");
}

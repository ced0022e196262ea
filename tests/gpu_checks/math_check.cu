// Exhaustive check of the codec's branch-free reciprocal and division (fp4q_math.cuh)
// against CUDA's IEEE __frcp_rn / __fdiv_rn. Prints one "name bad=<count> tested=<count>"
// line per check; every count of mismatches must be 0.
#include <cstdio>
#include <cstdint>
#include "fp4q_math.cuh"

__device__ unsigned long long g_bad[4], g_tested[4], g_nfail;
__device__ float g_fail[8][2];

// every significand of every exponent in [e0, e1]: reciprocal
__global__ void rcp_all(int e0, int e1) {
  const uint64_t total = (uint64_t)(e1 - e0 + 1) << 23;
  unsigned long long bad = 0, tested = 0;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total; i += (uint64_t)gridDim.x * blockDim.x) {
    const int e = e0 + (int)(i >> 23);
    const float b = __uint_as_float(((uint32_t)(127 + e) << 23) | (uint32_t)(i & 0x7fffff));
    bad += __float_as_uint(fp4q_math::rcp_rn(b)) != __float_as_uint(__frcp_rn(b));
    ++tested;
  }
  atomicAdd(&g_bad[0], bad);
  atomicAdd(&g_tested[0], tested);
}

// every significand of every exponent in [e0, e1]: division by 2688
__global__ void div2688_all(int e0, int e1) {
  const uint64_t total = (uint64_t)(e1 - e0 + 1) << 23;
  unsigned long long bad = 0, tested = 0;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total; i += (uint64_t)gridDim.x * blockDim.x) {
    const int e = e0 + (int)(i >> 23);
    const float a = __uint_as_float(((uint32_t)(127 + e) << 23) | (uint32_t)(i & 0x7fffff));
    bad += __float_as_uint(fp4q_math::div_rn_2688(a)) != __float_as_uint(__fdiv_rn(a, 2688.0f));
    ++tested;
  }
  atomicAdd(&g_bad[1], bad);
  atomicAdd(&g_tested[1], tested);
}

__device__ __forceinline__ uint32_t mix(uint64_t x) {     // splitmix64 finaliser
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return (uint32_t)(x ^ (x >> 31));
}

// random divisors b = 2^[-98, 116) * [1, 2) and quotients 2^[-20, 9) * [1, 2), plus
// quotients steered onto and next to the midpoints of the float grid (a = RN(m * b) for a
// midpoint m of two consecutive floats), the hardest cases for a residual correction
__global__ void div_pairs(uint64_t count) {
  unsigned long long bad = 0, tested = 0;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t h0 = mix(3 * i), h1 = mix(3 * i + 1), h2 = mix(3 * i + 2);
    const int eb = -98 + (int)(h0 % 214u);
    const float b = __uint_as_float(((uint32_t)(127 + eb) << 23) | (h1 & 0x7fffff));
    const int eq = -20 + (int)((h0 >> 8) % 29u);
    float q = __uint_as_float(((uint32_t)(127 + eq) << 23) | (h2 & 0x7fffff));
    float a;
    if (h0 & 0x80000000u) {
      // midpoint between q and its successor, perturbed by -1, 0, +1 ulp of a
      const float qn = __uint_as_float(__float_as_uint(q) + 1);
      const double m = 0.5 * ((double)q + (double)qn);
      a = (float)(m * (double)b);
      const int k = (int)((h1 >> 23) % 3u) - 1;
      a = __uint_as_float(__float_as_uint(a) + k);
    } else {
      a = __fmul_rn(q, b);
    }
    const fp4q_math::Divider d(b);
    const bool wrong = __float_as_uint(d.div(a)) != __float_as_uint(__fdiv_rn(a, b));
    bad += wrong;
    ++tested;
    if (wrong) {
      const unsigned long long slot = atomicAdd(&g_nfail, 1ull);
      if (slot < 8) {
        g_fail[slot][0] = a;
        g_fail[slot][1] = b;
      }
    }
  }
  atomicAdd(&g_bad[2], bad);
  atomicAdd(&g_tested[2], tested);
}

// every significand of the codec's block sizes: the scale chain t_b = 6 * RN(A / 2688) and
// the group ratio r = RN(amax / t_b) for amax = A * 2^-k (k = 0..24) and amax just below A
__global__ void chain_all(int e0, int e1) {
  const uint64_t total = (uint64_t)(e1 - e0 + 1) << 23;
  unsigned long long bad = 0, tested = 0;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total; i += (uint64_t)gridDim.x * blockDim.x) {
    const int e = e0 + (int)(i >> 23);
    const float A = __uint_as_float(((uint32_t)(127 + e) << 23) | (uint32_t)(i & 0x7fffff));
    const float tb = __fmul_rn(__fdiv_rn(A, 2688.0f), 6.0f);
    const fp4q_math::Divider d(tb);
    const uint32_t h = (uint32_t)(i * 2654435761u);
    const float amax[3] = {A, __uint_as_float(__float_as_uint(A) - 1 - (h & 0xff)),
                           __fmul_rn(A, __uint_as_float((uint32_t)(127 - (int)(h >> 27)) << 23))};
    for (int k = 0; k < 3; ++k) {
      bad += __float_as_uint(d.div(amax[k])) != __float_as_uint(__fdiv_rn(amax[k], tb));
      ++tested;
    }
  }
  atomicAdd(&g_bad[3], bad);
  atomicAdd(&g_tested[3], tested);
}

int main() {
  rcp_all<<<4096, 256>>>(-110, 122);
  div2688_all<<<4096, 256>>>(-89, 123);
  div_pairs<<<4096, 256>>>(1ull << 30);
  chain_all<<<4096, 256>>>(-88, 123);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    printf("cuda error\n");
    return 1;
  }
  unsigned long long bad[4], tested[4];
  cudaMemcpyFromSymbol(bad, g_bad, sizeof(bad));
  cudaMemcpyFromSymbol(tested, g_tested, sizeof(tested));
  const char* names[4] = {"rcp_rn", "div_rn_2688", "divider", "scale_chain"};
  for (int i = 0; i < 4; ++i) printf("%s bad=%llu tested=%llu\n", names[i], bad[i], tested[i]);
  float fail[8][2];
  unsigned long long nfail = 0;
  cudaMemcpyFromSymbol(fail, g_fail, sizeof(fail));
  cudaMemcpyFromSymbol(&nfail, g_nfail, sizeof(nfail));
  for (unsigned long long k = 0; k < nfail && k < 8; ++k) printf("divider failure a=%a b=%a\n", fail[k][0], fail[k][1]);
  return 0;
}

// Per-block softmax arithmetic shared by the forward kernels: the
// probabilities of one row's block of raw scores against a reference, and
// the row maximum. Scores are fp32 bit patterns as tcgen05.ld returns them;
// log2(e) and the logit scale are folded into `sl`.
#pragma once

#include <math.h>
#include <stdint.h>

#include "sm103.cuh"

namespace moda {
namespace sm103 {

// p = 2^(s*sl - m) for the N raw scores x (fp32 bits) as bf16 pairs into pk;
// returns the fp32 sum. One packed FMA per pair, then the exponential unit;
// the sum through eight packed accumulators.
template <int N>
__device__ __forceinline__ float exp_block(const uint32_t* x, uint32_t* pk, float sl, float m) {
  static_assert(N >= 16 && N % 16 == 0, "whole accumulator rounds");
  const float nbase = (m == -INFINITY) ? 0.f : -m;
  const uint64_t sl2 = f2(sl, sl), nb2 = f2(nbase, nbase);
  uint64_t acc[8];
#pragma unroll
  for (int c = 0; c < N / 2; ++c) {
    float u, w;
    f2_split(ffma2(f2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])), sl2, nb2), u, w);
    const float e0 = ex2_approx(u), e1 = ex2_approx(w);
    pk[c] = pack_bf16x2(e0, e1);
    acc[c & 7] = c < 8 ? f2(e0, e1) : fadd2(acc[c & 7], f2(e0, e1));
  }
  acc[0] = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
  acc[4] = fadd2(fadd2(acc[4], acc[5]), fadd2(acc[6], acc[7]));
  acc[0] = fadd2(acc[0], acc[4]);
  float u, w;
  f2_split(acc[0], u, w);
  return u + w;
}

// Row maximum of raw scores by three-input max trees.
__device__ __forceinline__ float raw_max128(const uint32_t* x) {
  float a1[43];
#pragma unroll
  for (int i = 0; i < 42; ++i)
    a1[i] = max3f(__uint_as_float(x[3 * i]), __uint_as_float(x[3 * i + 1]), __uint_as_float(x[3 * i + 2]));
  a1[42] = fmaxf(__uint_as_float(x[126]), __uint_as_float(x[127]));
  float a2[15];
#pragma unroll
  for (int i = 0; i < 14; ++i) a2[i] = max3f(a1[3 * i], a1[3 * i + 1], a1[3 * i + 2]);
  a2[14] = a1[42];
  float a3[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) a3[i] = max3f(a2[3 * i], a2[3 * i + 1], a2[3 * i + 2]);
  return fmaxf(max3f(a3[0], a3[1], a3[2]), fmaxf(a3[3], a3[4]));
}
__device__ __forceinline__ float raw_max32(const uint32_t* x) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i)
    a[i] = max3f(__uint_as_float(x[3 * i]), __uint_as_float(x[3 * i + 1]), __uint_as_float(x[3 * i + 2]));
  a[10] = fmaxf(__uint_as_float(x[30]), __uint_as_float(x[31]));
  return fmaxf(max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), max3f(a[6], a[7], a[8])),
               fmaxf(a[9], a[10]));
}

}  // namespace sm103
}  // namespace moda

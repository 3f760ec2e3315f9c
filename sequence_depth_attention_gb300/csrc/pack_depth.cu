// Depth-stream relayout: [L, T, Hk, d] -> [Hk, T, L, d], bf16, bit-exact.
//
// Mixture-of-Depths Attention, Sec. 3.2: the "flash-compatible" layout puts
// the L depth slots of each position next to each other, and the
// "chunk-aware" reading makes the slots of a run of positions one contiguous
// region. Per KV head, [T, L, d] is both.
//
// The copy is HBM-bound: every byte is read once and written once. Each
// (l, t, hk) row of d bf16 is contiguous in both layouts (128 or 256 bytes),
// so the kernel moves 16-byte vectors; a warp covers whole rows on both
// sides, so every DRAM sector it touches is fully used. The destination is
// walked in order (coalesced stores); consecutive destination rows come from
// source rows T*Hk*d elements apart.
#include "moda_internal.h"

namespace moda {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // independent 16-byte loads in flight per lane

// One warp copies the L*d bf16 of one (hk, t) pair at a time: the L source
// rows src[0..L)[t][hk][:] (each contiguous, T*Hk*d elements apart) become one
// contiguous run dst[hk][t][0..L)[:]. Index math stays 32-bit and per-vector
// work is a shift and a mask.
__global__ void __launch_bounds__(kThreads)
pack_depth_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                  int L, int T, int Hk, int lg_vpr) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = kThreads / 32;
  const int64_t npairs = (int64_t)Hk * T;
  const int vpr = 1 << lg_vpr;                  // 16-byte vectors per row
  const int per_pair = L << lg_vpr;             // vectors per (hk, t)
  const int64_t lstride = (int64_t)T * Hk * vpr;  // source vectors between slots
  for (int64_t pair = (int64_t)blockIdx.x * warps_per_block + (threadIdx.x >> 5);
       pair < npairs; pair += (int64_t)gridDim.x * warps_per_block) {
    const int hk = (int)(pair / T);
    const int t = (int)(pair - (int64_t)hk * T);
    const uint4* s = src + ((int64_t)t * Hk + hk) * vpr;
    uint4* dp = dst + pair * per_pair;
    for (int i0 = 0; i0 < per_pair; i0 += 32 * kUnroll) {
      uint4 val[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < per_pair) val[u] = __ldg(s + (int64_t)(i >> lg_vpr) * lstride + (i & (vpr - 1)));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < per_pair) dp[i] = val[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_pack_depth(const void* src, void* dst, int L, int T, int Hk,
                              int d, cudaStream_t stream) {
  const int lg_vpr = (d == 128) ? 4 : 3;  // d/8 vectors of 8 bf16
  const int64_t npairs = (int64_t)Hk * T;
  if (npairs == 0 || L == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  const int warps_per_block = kThreads / 32;
  int64_t blocks = (npairs + warps_per_block - 1) / warps_per_block;
  const int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread blocks per SM
  if (blocks > cap) blocks = cap;
  pack_depth_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(
      (const uint4*)src, (uint4*)dst, L, T, Hk, lg_vpr);
  return cudaGetLastError();
}

}  // namespace moda

// Depth-stream write: one layer's K (or V) rows go straight into slot `slot`
// of the packed depth stream, dst[hk][t][slot][:] = src[t][hk][:].
//
// Mixture-of-Depths Attention, Sec. 2.2 ("write" step): each attention layer
// appends its K, V to the depth stream and each FFN layer the KV projection
// of its input. Writing into the packed, per-position-contiguous layout as
// the layers run removes the separate relayout of the whole stream.
//
// HBM-bound copy of 16-byte vectors: consecutive lanes walk the d/8 vectors
// of one (t, hk) row, so reads are contiguous and each destination row of
// d*2 bytes is written whole; each thread keeps four loads in flight.
#include "moda_internal.h"

namespace moda {
namespace {

constexpr int kThreads = 256;

// slot_dev (may be null): the slot is read from device memory, as chosen by a
// kernel earlier on the stream; one outside [0, L) writes nothing and latches
// MODA_ERR_INVALID_ARG in the device error word.
__global__ void __launch_bounds__(kThreads)
depth_write_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int T, int Hk, int L,
                   int slot, const int* __restrict__ slot_dev, unsigned int* err, int lg_vpr,
                   int64_t total_vec) {
  if (slot_dev) {
    slot = *slot_dev;
    if (slot < 0 || slot >= L) {
      if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(err, 0u, (unsigned int)MODA_ERR_INVALID_ARG);
      return;
    }
  }
  const int vpr = 1 << lg_vpr;
  auto put = [&](int64_t n, const uint4& v) {
    const int c = (int)(n & (vpr - 1));
    const int64_t row = n >> lg_vpr;  // t*Hk + hk
    const int t = (int)(row / Hk);
    const int hk = (int)(row - (int64_t)t * Hk);
    dst[(((int64_t)hk * T + t) * L + slot) * vpr + c] = v;
  };
  // four loads in flight per thread before their stores, so that an SM keeps
  // enough bytes in flight to cover the memory latency
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t n = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  for (; n + 3 * stride < total_vec; n += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __ldg(src + n + j * stride);
#pragma unroll
    for (int j = 0; j < 4; ++j) put(n + j * stride, v[j]);
  }
  for (; n < total_vec; n += stride) put(n, __ldg(src + n));
}

}  // namespace

cudaError_t launch_depth_write(const void* src, void* dst, int T, int Hk, int d, int L, int slot,
                               const int* slot_dev, unsigned int* err, int num_sms,
                               cudaStream_t stream) {
  const int lg_vpr = d == 128 ? 4 : 3;
  const int64_t total = (int64_t)T * Hk << lg_vpr;
  int64_t blocks = (total + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)(num_sms > 0 ? num_sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  depth_write_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(
      (const uint4*)src, (uint4*)dst, T, Hk, L, slot, slot_dev, err, lg_vpr, total);
  return cudaGetLastError();
}

}  // namespace moda

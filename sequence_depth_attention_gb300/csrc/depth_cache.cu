// Bounded depth KV cache (summary, Sec. 6.2 "bounded depth KV slot cache"):
// a fixed budget of S slots in the packed depth stream, and a policy that
// decides which depth entries stay once more than S have been written.
//
//   depth_mass_kernel   utility of every slot: the probability mass the joint
//                       softmax (Sec. 2.2) gave it in one layer's read,
//                       mass[hk][l] = sum_t sum_{h in group hk}
//                                     exp(scale q[t,h].kd[hk,t,l] - lse[t,h]);
//                       per-CTA partial sums, then a fixed-order reduction,
//                       so the result does not depend on scheduling
//   cache_admit_kernel  the slot the next entry goes into: an empty slot if
//                       any, else, of the entries outside the `recent` most
//                       recent ones, the one with the least utility (ties:
//                       the older, then the lower slot)
//   depth_write_kernel  (depth_write.cu) writes the entry into that slot,
//                       reading the slot index from device memory
// All three run on the stream, so a layer loop needs no host round trip.
#include <cuda_bf16.h>

#include "moda_internal.h"

namespace moda {
namespace {

constexpr int kWarps = 8;
constexpr int kChunk = 64;  // positions per CTA of the mass kernel
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
depth_mass_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kd,
                  const float* __restrict__ lse, int T, int Hq, int L, float scale_log2,
                  float* __restrict__ partial) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // [kWarps][G][D] query rows of the position a warp works on, then
  // [kWarps][L] per-warp slot sums
  __nv_bfloat16* qs_all = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  float* acc_all = reinterpret_cast<float*>(smem_raw + (size_t)kWarps * G * D * 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, hk = blockIdx.y, nchunks = gridDim.x;
  __nv_bfloat16* qs = qs_all + (size_t)warp * G * D;
  float* acc = acc_all + (size_t)warp * L;
  for (int l = lane; l < L; l += 32) acc[l] = 0.f;
  for (int tt = warp; tt < kChunk; tt += kWarps) {
    const int t = chunk * kChunk + tt;
    if (t >= T) break;
    const int64_t row0 = (int64_t)t * Hq + hk * G;
    __syncwarp();
    for (int idx = lane; idx < G * D / 8; idx += 32)
      reinterpret_cast<uint4*>(qs)[idx] = __ldg(reinterpret_cast<const uint4*>(q + row0 * D) + idx);
    float lg[G];
#pragma unroll
    for (int g = 0; g < G; ++g) lg[g] = __ldg(lse + row0 + g) * kLog2e;
    __syncwarp();
    const int64_t slot0 = ((int64_t)hk * T + t) * L;
    for (int l = lane; l < L; l += 32) {
      // lane owns slot l: its G logits from one read of the slot's key row
      const uint4* kr = reinterpret_cast<const uint4*>(kd + (slot0 + l) * D);
      float s[G];
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = 0.f;
#pragma unroll 4
      for (int ch = 0; ch < D / 8; ++ch) {
        const uint4 kc = __ldg(kr + ch);
        const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kc);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint4 qc = reinterpret_cast<const uint4*>(qs + g * D)[ch];
          const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qc);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(q2[i]), b = __bfloat1622float2(k2[i]);
            s[g] = fmaf(a.x, b.x, fmaf(a.y, b.y, s[g]));
          }
        }
      }
      float m = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) m += exp2f(s[g] * scale_log2 - lg[g]);
      acc[l] += m;
    }
  }
  __syncthreads();
  // this CTA's partial sums, warps added in a fixed order
  float* out = partial + ((int64_t)hk * nchunks + chunk) * L;
  for (int l = threadIdx.x; l < L; l += kWarps * 32) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += acc_all[(size_t)w * L + l];
    out[l] = s;
  }
}

__global__ void depth_mass_reduce_kernel(const float* __restrict__ partial, int Hk, int nchunks,
                                         int L, float* __restrict__ mass) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Hk * L) return;
  const int hk = i / L, l = i - hk * L;
  const float* p = partial + (int64_t)hk * nchunks * L + l;
  float s = 0.f;
  for (int c = 0; c < nchunks; ++c) s += p[(int64_t)c * L];
  mass[i] = s;
}

template <int D, int G>
cudaError_t launch_mass_dg(const DepthMassArgs& a, cudaStream_t st) {
  const int nchunks = (a.T + kChunk - 1) / kChunk;
  const size_t smem = (size_t)kWarps * G * D * 2 + (size_t)kWarps * a.L * 4;
  cudaError_t e = cudaFuncSetAttribute(depth_mass_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  depth_mass_kernel<D, G><<<dim3(nchunks, a.Hk), kWarps * 32, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kd, a.lse, a.T, a.Hq, a.L,
      a.scale * kLog2e, a.work);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = a.Hk * a.L;
  depth_mass_reduce_kernel<<<(n + 255) / 256, 256, 0, st>>>(a.work, a.Hk, nchunks, a.L, a.mass);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_mass_d(const DepthMassArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 1: return launch_mass_dg<D, 1>(a, st);
    case 2: return launch_mass_dg<D, 2>(a, st);
    case 4: return launch_mass_dg<D, 4>(a, st);
    case 8: return launch_mass_dg<D, 8>(a, st);
    default: return launch_mass_dg<D, 16>(a, st);
  }
}

// Eviction order: (utility, age, slot) ascending; the first one leaves. NaN
// utilities order as the largest.
struct Key {
  float u;
  int age, slot;
};
__device__ __forceinline__ bool before(const Key& a, const Key& b) {
  const bool an = a.u != a.u, bn = b.u != b.u;
  if (an != bn) return bn;
  if (!an && a.u != b.u) return a.u < b.u;
  if (a.age != b.age) return a.age < b.age;
  return a.slot < b.slot;
}

// One CTA of S (rounded up to 32) threads; thread s looks at slot s.
__global__ void cache_admit_kernel(int* __restrict__ ages, const float* __restrict__ mass, int Hk,
                                   int S, int recent, int new_age, int* __restrict__ slot_out) {
  __shared__ int s_age[1024];
  __shared__ int s_empty;
  __shared__ Key s_best[32];
  const int s = threadIdx.x, warp = s >> 5, lane = s & 31;
  if (s == 0) s_empty = S;
  if (s < S) s_age[s] = ages[s];
  __syncthreads();
  if (s < S && s_age[s] < 0) atomicMin(&s_empty, s);
  __syncthreads();
  if (s_empty < S) {
    if (s == 0) {
      ages[s_empty] = new_age;
      *slot_out = s_empty;
    }
    return;
  }
  // the keep - 1 newest cached entries stay with the new one (rank by age,
  // newest first; equal ages by slot)
  const int keep = max(0, min(recent, S) - 1);
  Key k{__int_as_float(0x7fc00000), 0x7fffffff, 0x7fffffff};  // "no candidate": orders last
  bool cand = false;
  if (s < S) {
    int rank = 0;
    const int a = s_age[s];
    for (int o = 0; o < S; ++o) {
      const int b = s_age[o];
      rank += (b > a) || (b == a && o < s);
    }
    if (rank >= keep) {
      float u = 0.f;
      for (int h = 0; h < Hk; ++h) u += mass[(int64_t)h * S + s];  // heads in order
      k = Key{u, a, s};
      cand = true;
    }
  }
  if (!cand) k.slot = 0x7fffffff;
  for (int off = 16; off >= 1; off >>= 1) {
    Key o;
    o.u = __shfl_xor_sync(0xffffffffu, k.u, off);
    o.age = __shfl_xor_sync(0xffffffffu, k.age, off);
    o.slot = __shfl_xor_sync(0xffffffffu, k.slot, off);
    const bool o_valid = o.slot != 0x7fffffff, k_valid = k.slot != 0x7fffffff;
    if (o_valid && (!k_valid || before(o, k))) k = o;
  }
  if (lane == 0) s_best[warp] = k;
  __syncthreads();
  if (s == 0) {
    Key b = s_best[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
      const Key o = s_best[w];
      if (o.slot != 0x7fffffff && (b.slot == 0x7fffffff || before(o, b))) b = o;
    }
    ages[b.slot] = new_age;
    *slot_out = b.slot;
  }
}

}  // namespace

size_t depth_mass_workspace_floats(int T, int Hk, int L) {
  return (size_t)((T + kChunk - 1) / kChunk) * Hk * L;
}

cudaError_t launch_depth_mass(const DepthMassArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_mass_d<128>(a, stream) : launch_mass_d<64>(a, stream);
}

cudaError_t launch_cache_admit(int* ages, const float* mass, int Hk, int S, int recent,
                               int new_age, int* slot_out, cudaStream_t stream) {
  const int threads = (S + 31) / 32 * 32;
  cache_admit_kernel<<<1, threads, 0, stream>>>(ages, mass, Hk, S, recent, new_age, slot_out);
  return cudaGetLastError();
}

}  // namespace moda

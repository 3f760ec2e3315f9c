// The depth part of the MoDA forward on CUDA cores, as a second pass that is
// merged exactly into the result of the sequence part (the forward with
// L = 0). This is the measured alternative to the depth blocks that the
// tcgen05 forward runs under the block-diagonal mask (Mixture-of-Depths
// Attention, Sec. 3.3); moda_fwd_depth_cc exposes it.
//
// One warp per (KV head hk, position t): the G query rows of the group see
// the same L slots kd[hk][t][0..L) (one contiguous run of the packed stream).
//   phase 1  lane l scores slot l0 + l for every head of the group (a full
//            dot product over d from 16-byte loads of its row), then the 32
//            scores of the chunk update the running max and sum of each head
//            (five shuffles per head and chunk);
//   phase 2  lanes split the d columns and accumulate sum_l p_l vd[l] with
//            p broadcast from shared memory (coalesced rows of vd).
// Merge: with the sequence part's lse_s and normalised o_s (as moda_fwd left
// them) and the depth part's max m, sum l and unnormalised o_d,
//   lse = log(e^lse_s + l e^m),  o = (e^lse_s o_s + e^m o_d) / e^lse.
#include <cuda_bf16.h>

#include "moda_internal.h"

namespace moda {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int G>
struct alignas(16) DepthCcSmem {
  __nv_bfloat16 qs[G][D];
  float P[G][32];
};

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
fwd_depth_cc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kd,
                    const __nv_bfloat16* __restrict__ vd, int T, int Hq, int Hk, int L,
                    float scale_log2, __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  constexpr int E = D / 32;  // columns per lane in phase 2
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  DepthCcSmem<D, G>& sm = reinterpret_cast<DepthCcSmem<D, G>*>(smem_raw)[warp];
  const int64_t pair = (int64_t)blockIdx.x * kWarps + warp;
  if (pair >= (int64_t)Hk * T) return;
  const int hk = (int)(pair / T), t = (int)(pair - (int64_t)hk * T);
  const int64_t row0 = (int64_t)t * Hq + hk * G;  // row of head g is row0 + g
  for (int idx = lane; idx < G * D / 8; idx += 32) {
    const int g = idx / (D / 8), ch = idx % (D / 8);
    reinterpret_cast<uint4*>(&sm.qs[g][0])[ch] = reinterpret_cast<const uint4*>(q + (row0 + g) * D)[ch];
  }
  __syncwarp();

  float m[G], l[G], od[G][E];  // per head: running max (log2 units), sum, unnormalised o
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) od[g][e] = 0.f;
  }
  const int64_t slot0 = ((int64_t)hk * T + t) * L;  // packed row of slot 0
  for (int l0 = 0; l0 < L; l0 += 32) {
    // ---- phase 1: lane owns slot l0 + lane
    const int li = l0 + lane;
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = 0.f;
    if (li < L) {
      const uint4* kr = reinterpret_cast<const uint4*>(kd + (slot0 + li) * D);
#pragma unroll 4
      for (int ch = 0; ch < D / 8; ++ch) {
        const uint4 kc = __ldg(kr + ch);
        const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kc);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const uint4 qc = reinterpret_cast<const uint4*>(&sm.qs[g][0])[ch];
          const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qc);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(q2[i]), b = __bfloat1622float2(k2[i]);
            s[g] = fmaf(a.x, b.x, fmaf(a.y, b.y, s[g]));
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sg = li < L ? s[g] * scale_log2 : -INFINITY;
      float mx = sg;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[g], mx);  // finite: the chunk holds at least one slot
      const float alpha = exp2f(m[g] - mn);
      const float p = exp2f(sg - mn);
      float ps = p;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[g] = l[g] * alpha + ps;
      m[g] = mn;
#pragma unroll
      for (int e = 0; e < E; ++e) od[g][e] *= alpha;
      sm.P[g][lane] = p;
    }
    __syncwarp();
    // ---- phase 2: lane owns columns lane*E .. lane*E+E-1
    const int nl = min(32, L - l0);
    for (int jj = 0; jj < nl; ++jj) {
      const __nv_bfloat16* vr = vd + (slot0 + l0 + jj) * D + lane * E;
      float vv[E];
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vr + e));
        vv[e] = f.x;
        vv[e + 1] = f.y;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pg = sm.P[g][jj];
#pragma unroll
        for (int e = 0; e < E; ++e) od[g][e] = fmaf(pg, vv[e], od[g][e]);
      }
    }
    __syncwarp();
  }
  // ---- merge with the sequence part (log2 units)
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int64_t row = row0 + g;
    const float ls = lse[row] * kLog2e;
    const float md = m[g] + log2f(l[g]);  // the depth part's log-sum
    const float M = fmaxf(ls, md);
    const float as = exp2f(ls - M), ad = exp2f(m[g] - M);
    const float tot = as + l[g] * ad;
    const float inv = 1.f / tot;
    __nv_bfloat16* orow = o + row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 os = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(orow + e));
      const float r0 = (as * os.x + ad * od[g][e]) * inv;
      const float r1 = (as * os.y + ad * od[g][e + 1]) * inv;
      *reinterpret_cast<__nv_bfloat162*>(orow + e) = __floats2bfloat162_rn(r0, r1);
    }
    if (lane == 0) lse[row] = (M + log2f(tot)) * kLn2;
  }
}

template <int D, int G>
cudaError_t launch_dg(const FwdArgs& a, cudaStream_t st) {
  const size_t smem = kWarps * sizeof(DepthCcSmem<D, G>);
  cudaError_t e = cudaFuncSetAttribute(fwd_depth_cc_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t pairs = (int64_t)a.Hk * a.T;
  fwd_depth_cc_kernel<D, G><<<(unsigned)((pairs + kWarps - 1) / kWarps), kWarps * 32, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kd, (const __nv_bfloat16*)a.vd, a.T, a.Hq,
      a.Hk, a.L, a.scale * kLog2e, (__nv_bfloat16*)a.o, a.lse);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 1: return launch_dg<D, 1>(a, st);
    case 2: return launch_dg<D, 2>(a, st);
    case 4: return launch_dg<D, 4>(a, st);
    case 8: return launch_dg<D, 8>(a, st);
    default: return launch_dg<D, 16>(a, st);
  }
}

}  // namespace

cudaError_t launch_fwd_depth_cc(const FwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

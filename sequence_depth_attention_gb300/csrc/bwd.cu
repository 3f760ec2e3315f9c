// MoDA backward (gradients of the joint-softmax forward of Mixture-of-Depths
// Attention, Sec. 2.2): the CUDA-core kernels and the dispatch.
//
// For a row (t, h) with joint probabilities p over its candidates c (keys
// j <= t of its KV head, then the L depth slots of position t):
//   D = <dO, o>,  dp_c = <dO, v_c>,  ds_c = p_c (dp_c - D),
//   dq += scale ds_c key_c,  dkey_c += scale ds_c q,  dval_c += p_c dO.
// p is recomputed from the forward's lse: p_c = exp(scale q.key_c - lse).
//
// Four launches, every output row with one owner (no atomics):
//   1. delta     D[t,h] = <dO[t,h], o[t,h]>                   (caller workspace)
//   2. depth     one warp per (hk, t): the G rows x L slots of that position
//                on CUDA cores -> dkd, dvd (in the layout of kd, vd: packed
//                or layer-major) and dq's depth share, written as dq's
//                initial value
//   3. dq        tcgen05 (bwd_dq_tc.cu), added to dq
//   4. dk/dv     tcgen05 (bwd_dkdv_tc.cu)
// All gradients are fp32.
#include <cuda_bf16.h>

#include "moda_internal.h"

namespace moda {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- 1. delta
template <int D>
__global__ void __launch_bounds__(256)
bwd_delta_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
                 float* __restrict__ delta, int64_t rows) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int E = D / 32;  // elements per lane
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(o + row * D + lane * E);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(dO + row * D + lane * E);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    const float2 x = __bfloat1622float2(a[i]), y = __bfloat1622float2(b[i]);
    s += x.x * y.x + x.y * y.y;
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[row] = s;
}

// ---------------------------------------------------------------- 2. depth
// Per-warp shared state; 16-byte aligned so that every warp's q/dO rows take
// 16-byte accesses.
template <int D, int G, bool STAGE>
struct alignas(16) DepthWarpSmem {
  // staged rows only: the chunk's 32 kd and vd rows, 16-byte piece c of row r
  // at c ^ (r % (D/8))
  uint4 kr[STAGE ? 32 : 1][D / 8];
  uint4 vr[STAGE ? 32 : 1][D / 8];
  __nv_bfloat16 qs[G][D];
  __nv_bfloat16 ds_[G][D];  // dO rows
  float P[G][32];
  float S[G][32];           // ds values
  float lse2[G];
  float Dd[G];
};

// One warp per (hk, t), 32 slots at a time. Phase 1: lane l computes, for its
// slot and every head g of the group, p and ds (full-length dot products).
// Phase 2: lanes split the d columns and walk the 32 slots of the chunk,
// producing dvd and dkd rows (coalesced) and accumulating dq's depth share.
// LM: depth layout, packed [Hk,T,L,d] (a position's slots are adjacent rows)
// or layer-major [L,T,Hk,d] (the slots lie T*Hk rows apart). STAGE: the
// chunk's kd and vd rows are first staged in shared memory with coalesced
// 16-byte loads, each lane then reading its row in a swizzled order that puts
// the 32 lanes' rows in distinct banks; without it each lane reads its own
// row straight from global memory. Staging pays for layer-major rows and for
// d = 64 rows (128 bytes); packed d = 128 rows keep the direct reads, where
// the 16 KB of staging per warp costs more resident warps than it saves.
template <int D, int G, bool LM, bool STAGE>
__global__ void __launch_bounds__(128)
bwd_depth_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kd,
                 const __nv_bfloat16* __restrict__ vd, const __nv_bfloat16* __restrict__ dO,
                 const float* __restrict__ lse, const float* __restrict__ delta, int T, int Hq,
                 int Hk, int L, float scale_log2, float scale, float* __restrict__ dq,
                 float* __restrict__ dkd, float* __restrict__ dvd) {
  constexpr int E = D / 32;  // columns per lane in phase 2
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  DepthWarpSmem<D, G, STAGE>& sm = reinterpret_cast<DepthWarpSmem<D, G, STAGE>*>(smem_raw)[warp];
  const int64_t pair = (int64_t)blockIdx.x * 4 + warp;
  if (pair >= (int64_t)Hk * T) return;
  const int hk = (int)(pair / T), t = (int)(pair - (int64_t)hk * T);
  const int64_t row0 = (int64_t)t * Hq + hk * G;  // row of head g is row0 + g

  // stage q and dO rows of the group (16-byte chunks)
  for (int idx = lane; idx < G * D / 8; idx += 32) {
    const int g = idx / (D / 8), ch = idx % (D / 8);
    reinterpret_cast<uint4*>(&sm.qs[g][0])[ch] =
        reinterpret_cast<const uint4*>(q + (row0 + g) * D)[ch];
    reinterpret_cast<uint4*>(&sm.ds_[g][0])[ch] =
        reinterpret_cast<const uint4*>(dO + (row0 + g) * D)[ch];
  }
  if (lane < G) {
    sm.lse2[lane] = lse[row0 + lane] * kLog2e;
    sm.Dd[lane] = delta[row0 + lane];
  }
  __syncwarp();

  float dqa[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < E; ++e) dqa[g][e] = 0.f;

  // row (of D values) of slot l: slot0 + l * lstride, in kd/vd and in dkd/dvd
  // alike; packed [Hk, T, L, d] or layer-major [L, T, Hk, d]
  const int64_t slot0 = LM ? (int64_t)t * Hk + hk : ((int64_t)hk * T + t) * L;
  const int64_t lstride = LM ? (int64_t)T * Hk : 1;
  constexpr int CH = D / 8;  // 16-byte pieces per row
  for (int l0 = 0; l0 < L; l0 += 32) {
    const int nl = min(32, L - l0);
    if constexpr (STAGE) {
      // ---- stage the chunk's rows
#pragma unroll 4
      for (int idx = lane; idx < 32 * CH; idx += 32) {
        const int r = idx / CH, c = idx % CH;
        uint4 kc = make_uint4(0u, 0u, 0u, 0u), vc = kc;
        if (r < nl) {
          const int64_t row = slot0 + (int64_t)(l0 + r) * lstride;
          kc = __ldg(reinterpret_cast<const uint4*>(kd + row * D) + c);
          vc = __ldg(reinterpret_cast<const uint4*>(vd + row * D) + c);
        }
        sm.kr[r][c ^ (r & (CH - 1))] = kc;
        sm.vr[r][c ^ (r & (CH - 1))] = vc;
      }
      __syncwarp();
    }
    // ---- phase 1: lane owns slot l0 + lane
    {
      const int l = l0 + lane;
      float s[G], dp[G];
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = dp[g] = 0.f;
      if (l < L) {
        const uint4* kg = reinterpret_cast<const uint4*>(kd + (slot0 + l * lstride) * D);
        const uint4* vg = reinterpret_cast<const uint4*>(vd + (slot0 + l * lstride) * D);
        for (int ch = 0; ch < CH; ++ch) {
          uint4 kc, vc;
          if constexpr (STAGE) {
            kc = sm.kr[lane][ch ^ (lane & (CH - 1))];
            vc = sm.vr[lane][ch ^ (lane & (CH - 1))];
          } else {
            kc = __ldg(kg + ch);
            vc = __ldg(vg + ch);
          }
          const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kc);
          const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vc);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const uint4 qc = reinterpret_cast<const uint4*>(&sm.qs[g][0])[ch];
            const uint4 oc = reinterpret_cast<const uint4*>(&sm.ds_[g][0])[ch];
            const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&qc);
            const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&oc);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 a = __bfloat1622float2(q2[i]), b = __bfloat1622float2(k2[i]);
              const float2 c = __bfloat1622float2(o2[i]), dd = __bfloat1622float2(v2[i]);
              s[g] = fmaf(a.x, b.x, fmaf(a.y, b.y, s[g]));
              dp[g] = fmaf(c.x, dd.x, fmaf(c.y, dd.y, dp[g]));
            }
          }
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = l < L ? exp2f(s[g] * scale_log2 - sm.lse2[g]) : 0.f;
        sm.P[g][lane] = p;
        sm.S[g][lane] = p * (dp[g] - sm.Dd[g]);
      }
    }
    __syncwarp();
    // ---- phase 2: lane owns columns lane*E .. lane*E+E-1
    for (int jj = 0; jj < nl; ++jj) {
      const int64_t prow = slot0 + (l0 + jj) * lstride;
      float kdv[E];
      {
        // layer-major: columns lane*E.. lie in piece (lane*E)/8 of staged row
        // jj, at its swizzled place
        const int col = lane * E;
        const __nv_bfloat16* kr =
            STAGE ? reinterpret_cast<const __nv_bfloat16*>(&sm.kr[jj][(col >> 3) ^ (jj & (CH - 1))]) +
                     (col & 7)
               : kd + prow * D + col;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kr + e));
          kdv[e] = f.x;
          kdv[e + 1] = f.y;
        }
      }
      float dvv[E], dkv[E];
#pragma unroll
      for (int e = 0; e < E; ++e) dvv[e] = dkv[e] = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pg = sm.P[g][jj], dsg = sm.S[g][jj];
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 qq = __bfloat1622float2(
              *reinterpret_cast<const __nv_bfloat162*>(&sm.qs[g][lane * E + e]));
          const float2 oo = __bfloat1622float2(
              *reinterpret_cast<const __nv_bfloat162*>(&sm.ds_[g][lane * E + e]));
          dvv[e] = fmaf(pg, oo.x, dvv[e]);
          dvv[e + 1] = fmaf(pg, oo.y, dvv[e + 1]);
          dkv[e] = fmaf(dsg, qq.x, dkv[e]);
          dkv[e + 1] = fmaf(dsg, qq.y, dkv[e + 1]);
          dqa[g][e] = fmaf(dsg, kdv[e], dqa[g][e]);
          dqa[g][e + 1] = fmaf(dsg, kdv[e + 1], dqa[g][e + 1]);
        }
      }
      float* dvo = dvd + prow * D + lane * E;
      float* dko = dkd + prow * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        *reinterpret_cast<float2*>(dvo + e) = make_float2(dvv[e], dvv[e + 1]);
        *reinterpret_cast<float2*>(dko + e) = make_float2(dkv[e] * scale, dkv[e + 1] * scale);
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float* out = dq + (row0 + g) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
      *reinterpret_cast<float2*>(out + e) = make_float2(dqa[g][e] * scale, dqa[g][e + 1] * scale);
  }
}

template <int D, int G, bool LM, bool STAGE>
cudaError_t launch_depth_layout(const BwdArgs& a, cudaStream_t st) {
  const size_t smem = 4 * sizeof(DepthWarpSmem<D, G, STAGE>);
  cudaError_t e = cudaFuncSetAttribute(bwd_depth_kernel<D, G, LM, STAGE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t pairs = (int64_t)a.Hk * a.T;
  bwd_depth_kernel<D, G, LM, STAGE><<<(unsigned)((pairs + 3) / 4), 128, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kd, (const __nv_bfloat16*)a.vd,
      (const __nv_bfloat16*)a.dO, a.lse, a.delta, a.T, a.Hq, a.Hk, a.L, a.scale * kLog2e, a.scale,
      a.dq, a.dkd, a.dvd);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_depth(const BwdArgs& a, cudaStream_t st) {
  if (a.layer_major) return launch_depth_layout<D, G, true, true>(a, st);
  return D == 64 ? launch_depth_layout<D, G, false, true>(a, st)
                 : launch_depth_layout<D, G, false, false>(a, st);
}

template <int D>
cudaError_t launch_d(const BwdArgs& a, cudaStream_t st) {
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int64_t rows = (int64_t)a.T * a.Hq;
  bwd_delta_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(
      (const __nv_bfloat16*)a.o, (const __nv_bfloat16*)a.dO, a.delta, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.L > 0) {
    switch (a.G) {
      case 1: e = launch_depth<D, 1>(a, st); break;
      case 2: e = launch_depth<D, 2>(a, st); break;
      case 4: e = launch_depth<D, 4>(a, st); break;
      case 8: e = launch_depth<D, 8>(a, st); break;
      default: e = launch_depth<D, 16>(a, st); break;
    }
    if (e != cudaSuccess) return e;
  }
  e = launch_bwd_dq_tc(a, st);
  if (e != cudaSuccess) return e;
  return launch_bwd_dkdv_tc(a, st);
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

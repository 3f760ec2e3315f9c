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
//                on warp-level MMAs -> dkd, dvd (in the layout of kd, vd:
//                packed or layer-major) and dq's depth share, written as dq's
//                initial value
//   3. dq        tcgen05 (bwd_dq_tc.cu), added to dq
//   4. dk/dv     tcgen05 (bwd_dkdv_tc.cu)
// All gradients are fp32.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "warp_mma.cuh"

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
// One warp per (KV head hk, position t): the G query rows of the pair against
// the L depth slots of t, 32 slots per chunk, on warp-level tensor-core MMAs
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation; the G rows are rows
// 0..G-1 of the 16-row A tiles, the rest zero):
//   S = Q Kd^T, dP = dO Vd^T                          (16 x 32 per chunk)
//   P = exp2(S scale log2e - lse log2e), dS = P (dP - D)   (in registers)
//   dvd = P^T dO, dkd = scale dS^T Q                  (32 x d per chunk, stored)
//   dq = scale dS Kd                                  (16 x d, over all chunks)
// P and dS are rounded to bf16 as MMA operands, as in the sequence kernels.
// LM: depth layout, packed [Hk,T,L,d] (a position's slots are adjacent rows)
// or layer-major [L,T,Hk,d] (the slots lie T*Hk rows apart); each chunk's kd
// and vd rows are copied to shared memory by 16-byte cp.async, piece c of row
// r at c ^ (r % (D/8)) so that the ldmatrix row reads hit distinct banks.
template <int D, int G>
struct alignas(16) DepthWarpSmem {
  static constexpr int R = G < 8 ? 8 : G;  // q/dO rows held (rows >= G are zero)
  static constexpr int QS = D + 8;         // padded q/dO row: ldmatrix rows in distinct banks
  uint4 kr[32][D / 8];
  uint4 vr[32][D / 8];
  __nv_bfloat16 qs[R][QS];
  __nv_bfloat16 os[R][QS];  // dO rows
};

template <int D, int G, bool LM>
__global__ void __launch_bounds__(128)
bwd_depth_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kd,
                 const __nv_bfloat16* __restrict__ vd, const __nv_bfloat16* __restrict__ dO,
                 const float* __restrict__ lse, const float* __restrict__ delta, int T, int Hq,
                 int Hk, int L, float scale_log2, float scale, float* __restrict__ dq,
                 float* __restrict__ dkd, float* __restrict__ dvd) {
  using W = DepthWarpSmem<D, G>;
  using namespace wmma16;
  constexpr int CH = D / 8;    // 16-byte pieces per row
  constexpr int NT = D / 8;    // 8-column tiles of a d-wide row
  constexpr bool kHi = G > 8;  // rows 8..15 of the A tiles hold query heads
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  W& sm = reinterpret_cast<W*>(smem_raw)[warp];
  const int64_t pair = (int64_t)blockIdx.x * 4 + warp;
  if (pair >= (int64_t)Hk * T) return;
  const int hk = (int)(pair / T), t = (int)(pair - (int64_t)hk * T);
  const int64_t row0 = (int64_t)t * Hq + hk * G;  // row of head g is row0 + g

  // q and dO rows of the group; rows G..R-1 zero
  for (int idx = lane; idx < W::R * CH; idx += 32) {
    const int g = idx / CH, ch = idx % CH;
    uint4 qv = make_uint4(0u, 0u, 0u, 0u), ov = qv;
    if (g < G) {
      qv = __ldg(reinterpret_cast<const uint4*>(q + (row0 + g) * D) + ch);
      ov = __ldg(reinterpret_cast<const uint4*>(dO + (row0 + g) * D) + ch);
    }
    *reinterpret_cast<uint4*>(&sm.qs[g][ch * 8]) = qv;
    *reinterpret_cast<uint4*>(&sm.os[g][ch * 8]) = ov;
  }
  // this thread's rows of the accumulator fragments: g_lo and g_lo + 8
  const int g_lo = lane >> 2;
  const float lse_lo = g_lo < G ? __ldg(lse + row0 + g_lo) * kLog2e : 0.f;
  const float d_lo = g_lo < G ? __ldg(delta + row0 + g_lo) : 0.f;
  const float lse_hi = kHi ? __ldg(lse + row0 + g_lo + 8) * kLog2e : 0.f;
  const float d_hi = kHi ? __ldg(delta + row0 + g_lo + 8) : 0.f;

  float dqa[NT][4];
#pragma unroll
  for (int c = 0; c < NT; ++c) dqa[c][0] = dqa[c][1] = dqa[c][2] = dqa[c][3] = 0.f;

  // row (of D values) of slot l: slot0 + l * lstride, in kd/vd and in dkd/dvd
  // alike; packed [Hk, T, L, d] or layer-major [L, T, Hk, d]
  const int64_t slot0 = LM ? (int64_t)t * Hk + hk : ((int64_t)hk * T + t) * L;
  const int64_t lstride = LM ? (int64_t)T * Hk : 1;
  const uint32_t kr0 = sm103::smem_u32(&sm.kr[0][0]), vr0 = sm103::smem_u32(&sm.vr[0][0]);
  const uint32_t qs0 = sm103::smem_u32(&sm.qs[0][0]), os0 = sm103::smem_u32(&sm.os[0][0]);
  // byte offset of 16-byte piece c of staged row r
  auto piece = [](int r, int c) -> uint32_t { return (uint32_t)((r * CH + (c ^ (r & (CH - 1)))) * 16); };
  const int lr = lane & 7, lm = lane >> 3;  // ldmatrix: the row this lane addresses, its matrix

  for (int l0 = 0; l0 < L; l0 += 32) {
    const int nl = min(32, L - l0);
    __syncwarp();  // the previous chunk's reads of the staged rows are done
#pragma unroll 4
    for (int idx = lane; idx < 32 * CH; idx += 32) {
      const int r = idx / CH, c = idx % CH;
      const bool ok = r < nl;
      const int64_t row = slot0 + (int64_t)(l0 + (ok ? r : 0)) * lstride;
      cp_async16(kr0 + piece(r, c), kd + row * D + c * 8, ok ? 16u : 0u);
      cp_async16(vr0 + piece(r, c), vd + row * D + c * 8, ok ? 16u : 0u);
    }
    cp_async_wait_all();
    __syncwarp();

    // ---- S = Q Kd^T, dP = dO Vd^T: n-tile nt holds slots 8nt..8nt+7
    float sc[4][4], dpc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[nt][i] = dpc[nt][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t aq[4], ao[4];
      if constexpr (kHi) {
        // matrices: rows 0-7 | rows 8-15, columns 16ks.. | 16ks+8..
        const uint32_t off = (uint32_t)(((lm & 1) * 8 + lr) * W::QS + ks * 16 + (lm >> 1) * 8) * 2;
        ldsm_x4(qs0 + off, aq[0], aq[1], aq[2], aq[3]);
        ldsm_x4(os0 + off, ao[0], ao[1], ao[2], ao[3]);
      } else {
        const uint32_t off = (uint32_t)(lr * W::QS + ks * 16 + (lm & 1) * 8) * 2;
        ldsm_x2(qs0 + off, aq[0], aq[2]);
        ldsm_x2(os0 + off, ao[0], ao[2]);
        aq[1] = aq[3] = ao[1] = ao[3] = 0u;
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        // matrices: kd pieces 2ks, 2ks+1, vd pieces 2ks, 2ks+1 of slots 8nt..8nt+7
        const int r = nt * 8 + lr;
        const uint32_t base = (lm < 2 ? kr0 : vr0) + piece(r, 2 * ks + (lm & 1));
        uint32_t bk0, bk1, bv0, bv1;
        ldsm_x4(base, bk0, bk1, bv0, bv1);
        mma_bf16(sc[nt], aq, bk0, bk1);
        mma_bf16(dpc[nt], ao, bv0, bv1);
      }
    }
    // ---- P and dS as bf16 pairs: [nt][0] row g_lo, [nt][1] row g_lo + 8,
    // slots 8nt + 2(lane%4) and +1; zero for rows >= G and slots >= nl
    uint32_t pa[4][2], da[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int sl = nt * 8 + 2 * (lane & 3);
      const bool v0 = sl < nl, v1 = sl + 1 < nl;
      {
        const bool row_ok = g_lo < G;
        const float p0 = row_ok && v0 ? exp2f(sc[nt][0] * scale_log2 - lse_lo) : 0.f;
        const float p1 = row_ok && v1 ? exp2f(sc[nt][1] * scale_log2 - lse_lo) : 0.f;
        pa[nt][0] = pack_bf16(p0, p1);
        da[nt][0] = pack_bf16(p0 * (dpc[nt][0] - d_lo), p1 * (dpc[nt][1] - d_lo));
      }
      if constexpr (kHi) {
        const float p0 = v0 ? exp2f(sc[nt][2] * scale_log2 - lse_hi) : 0.f;
        const float p1 = v1 ? exp2f(sc[nt][3] * scale_log2 - lse_hi) : 0.f;
        pa[nt][1] = pack_bf16(p0, p1);
        da[nt][1] = pack_bf16(p0 * (dpc[nt][2] - d_hi), p1 * (dpc[nt][3] - d_hi));
      } else {
        pa[nt][1] = da[nt][1] = 0u;
      }
    }
    // ---- dq += dS Kd: k-step kk covers slots 16kk..16kk+15; B = Kd read
    // transposed (k = slot, n = column)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t a[4] = {da[2 * kk][0], da[2 * kk][1], da[2 * kk + 1][0], da[2 * kk + 1][1]};
#pragma unroll
      for (int ct = 0; ct < NT; ct += 2) {
        // matrices: slots 16kk..+7 | 16kk+8..+15, columns 8ct.. | 8ct+8..
        const int r = 16 * kk + (lm & 1) * 8 + lr;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(kr0 + piece(r, ct + (lm >> 1)), b0, b1, b2, b3);
        mma_bf16(dqa[ct], a, b0, b1);
        mma_bf16(dqa[ct + 1], a, b2, b3);
      }
    }
    // ---- dvd = P^T dO, dkd = scale dS^T Q: m-tile mt covers slots
    // 16mt..16mt+15 (A = the transposed P / dS blocks), B = dO / Q read
    // transposed (k = row g, n = column)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const uint32_t ap[4] = {movmatrix_t(pa[2 * mt][0]), movmatrix_t(pa[2 * mt + 1][0]),
                              kHi ? movmatrix_t(pa[2 * mt][1]) : 0u,
                              kHi ? movmatrix_t(pa[2 * mt + 1][1]) : 0u};
      const uint32_t ad[4] = {movmatrix_t(da[2 * mt][0]), movmatrix_t(da[2 * mt + 1][0]),
                              kHi ? movmatrix_t(da[2 * mt][1]) : 0u,
                              kHi ? movmatrix_t(da[2 * mt + 1][1]) : 0u};
      const int s_lo = 16 * mt + g_lo, s_hi = s_lo + 8;  // chunk-local slots of this thread's rows
      float* dv_lo = dvd + (slot0 + (int64_t)(l0 + s_lo) * lstride) * D + 2 * (lane & 3);
      float* dk_lo = dkd + (slot0 + (int64_t)(l0 + s_lo) * lstride) * D + 2 * (lane & 3);
      float* dv_hi = dvd + (slot0 + (int64_t)(l0 + s_hi) * lstride) * D + 2 * (lane & 3);
      float* dk_hi = dkd + (slot0 + (int64_t)(l0 + s_hi) * lstride) * D + 2 * (lane & 3);
#pragma unroll
      for (int ct = 0; ct < NT; ++ct) {
        uint32_t bo0, bo1, bq0, bq1;
        if constexpr (kHi) {
          // matrices: dO rows 0-7, 8-15, Q rows 0-7, 8-15 at columns 8ct..
          const uint32_t off = (uint32_t)(((lm & 1) * 8 + lr) * W::QS + ct * 8) * 2;
          ldsm_x4_t((lm < 2 ? os0 : qs0) + off, bo0, bo1, bq0, bq1);
        } else {
          const uint32_t off = (uint32_t)(lr * W::QS + ct * 8) * 2;
          ldsm_x2_t((lm & 1 ? qs0 : os0) + off, bo0, bq0);
          bo1 = bq1 = 0u;
        }
        float cv[4] = {0.f, 0.f, 0.f, 0.f}, ck[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16(cv, ap, bo0, bo1);
        mma_bf16(ck, ad, bq0, bq1);
        if (s_lo < nl) {
          *reinterpret_cast<float2*>(dv_lo + ct * 8) = make_float2(cv[0], cv[1]);
          *reinterpret_cast<float2*>(dk_lo + ct * 8) = make_float2(ck[0] * scale, ck[1] * scale);
        }
        if (s_hi < nl) {
          *reinterpret_cast<float2*>(dv_hi + ct * 8) = make_float2(cv[2], cv[3]);
          *reinterpret_cast<float2*>(dk_hi + ct * 8) = make_float2(ck[2] * scale, ck[3] * scale);
        }
      }
    }
  }
  // dq's depth share (its initial value; the sequence share is added later)
#pragma unroll
  for (int ct = 0; ct < NT; ++ct) {
    const int col = ct * 8 + 2 * (lane & 3);
    if (g_lo < G)
      *reinterpret_cast<float2*>(dq + (row0 + g_lo) * D + col) =
          make_float2(dqa[ct][0] * scale, dqa[ct][1] * scale);
    if (kHi)
      *reinterpret_cast<float2*>(dq + (row0 + g_lo + 8) * D + col) =
          make_float2(dqa[ct][2] * scale, dqa[ct][3] * scale);
  }
}

template <int D, int G, bool LM>
cudaError_t launch_depth_layout(const BwdArgs& a, cudaStream_t st) {
  const size_t smem = 4 * sizeof(DepthWarpSmem<D, G>);
  cudaError_t e = cudaFuncSetAttribute(bwd_depth_kernel<D, G, LM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t pairs = (int64_t)a.Hk * a.T;
  bwd_depth_kernel<D, G, LM><<<(unsigned)((pairs + 3) / 4), 128, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kd, (const __nv_bfloat16*)a.vd,
      (const __nv_bfloat16*)a.dO, a.lse, a.delta, a.T, a.Hq, a.Hk, a.L, a.scale * kLog2e, a.scale,
      a.dq, a.dkd, a.dvd);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_depth(const BwdArgs& a, cudaStream_t st) {
  return a.layer_major ? launch_depth_layout<D, G, true>(a, st) : launch_depth_layout<D, G, false>(a, st);
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

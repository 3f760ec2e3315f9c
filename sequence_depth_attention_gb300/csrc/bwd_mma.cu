// MoDA backward (gradients of the joint-softmax forward of Mixture-of-Depths
// Attention, Sec. 2.2) on warp-level MMA and CUDA cores.
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
//                on CUDA cores -> dkd, dvd (packed layout) and dq's depth
//                share, written as dq's initial value
//   3. dq        64 G-stacked query rows per CTA over the causal key blocks
//                (S = Q K^T, dP = dO V^T, dS, dQ += dS K), added to dq
//   4. dk/dv     64 keys of one KV head per CTA over the query blocks that
//                see them (S^T, dP^T, dV += P^T dO, dK += dS^T Q)
// Tensor-core steps use mma.sync m16n8k16 (bf16 in, fp32 accumulate); P and
// dS are rounded to bf16 as MMA operands. All gradients are fp32.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "warp_mma.cuh"

namespace moda {
namespace {

using namespace wmma16;

constexpr int BM = 64;  // query rows (dq) / keys (dk, dv) per CTA
constexpr int BN = 64;  // keys (dq) / query rows (dk, dv) per inner block
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

// Stage 64 rows into a swizzled [64][D] tile; row i from row_ptr(i), rows with
// row_ptr(i) == nullptr zero-filled.
template <int D, typename RowPtr>
__device__ __forceinline__ void stage_rows(__nv_bfloat16* tile, RowPtr row_ptr,
                                           const __nv_bfloat16* any_valid) {
  constexpr int kChunks = D / 8;
  for (int idx = threadIdx.x; idx < 64 * kChunks; idx += kThreads) {
    const int row = idx / kChunks, ch = idx % kChunks;
    const __nv_bfloat16* src = row_ptr(row);
    const bool ok = src != nullptr;
    cp_async16(smem_u32(tile + swz<D>(row, ch * 8)), ok ? src + ch * 8 : any_valid, ok);
  }
}

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
template <int D, int G>
struct alignas(16) DepthWarpSmem {
  __nv_bfloat16 qs[G][D];
  __nv_bfloat16 ds_[G][D];  // dO rows
  float P[G][32];
  float S[G][32];           // ds values
  float lse2[G];
  float Dd[G];
};

// One warp per (hk, t). Phase 1: lane l computes, for its slot and every head
// g of the group, p and ds (full-length dot products). Phase 2: lanes split
// the d columns and walk the 32 slots of the chunk, producing dvd and dkd
// rows (coalesced) and accumulating dq's depth share.
template <int D, int G>
__global__ void __launch_bounds__(128)
bwd_depth_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kd,
                 const __nv_bfloat16* __restrict__ vd, const __nv_bfloat16* __restrict__ dO,
                 const float* __restrict__ lse, const float* __restrict__ delta, int T, int Hq,
                 int Hk, int L, float scale_log2, float scale, float* __restrict__ dq,
                 float* __restrict__ dkd, float* __restrict__ dvd) {
  constexpr int E = D / 32;  // columns per lane in phase 2
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  DepthWarpSmem<D, G>& sm = reinterpret_cast<DepthWarpSmem<D, G>*>(smem_raw)[warp];
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

  const int64_t slot0 = ((int64_t)hk * T + t) * L;  // packed row of slot 0
  for (int l0 = 0; l0 < L; l0 += 32) {
    // ---- phase 1: lane owns slot l0 + lane
    {
      const int l = l0 + lane;
      float s[G], dp[G];
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = dp[g] = 0.f;
      if (l < L) {
        const uint4* kr = reinterpret_cast<const uint4*>(kd + (slot0 + l) * D);
        const uint4* vr = reinterpret_cast<const uint4*>(vd + (slot0 + l) * D);
        for (int ch = 0; ch < D / 8; ++ch) {
          const uint4 kc = __ldg(kr + ch), vc = __ldg(vr + ch);
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
    const int nl = min(32, L - l0);
    for (int jj = 0; jj < nl; ++jj) {
      const int64_t prow = slot0 + l0 + jj;
      float kdv[E];
      {
        const __nv_bfloat16* kr = kd + prow * D + lane * E;
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

// ---------------------------------------------------------------- 3. dq
template <int D>
__global__ void __launch_bounds__(kThreads)
bwd_dq_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
              const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ dO,
              const float* __restrict__ lse, const float* __restrict__ delta, int T, int Hq, int Hk,
              int lgG, int ntiles, float scale_log2, float scale, float* __restrict__ dq,
              int accumulate) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sO = sQ + BM * D;      // dO tile
  __nv_bfloat16* sK = sO + BM * D;      // 2 stages
  __nv_bfloat16* sV = sK + 2 * BN * D;  // 2 stages
  const int G = 1 << lgG;
  const int P = BM >> lgG;
  const int tile = ntiles - 1 - (int)(blockIdx.x / Hk);  // longest first
  const int hk = (int)(blockIdx.x % Hk);
  const int p0 = tile * P;
  const int t_last = min(p0 + P, T) - 1;
  const int nblocks = t_last / BN + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t kv_stride = (int64_t)Hk * D;

  auto qrow = [&](const __nv_bfloat16* base, int r) -> const __nv_bfloat16* {
    const int t = p0 + (r >> lgG);
    return t < T ? base + ((int64_t)t * Hq + hk * G + (r & (G - 1))) * D : nullptr;
  };
  stage_rows<D>(sQ, [&](int r) { return qrow(q, r); }, q);
  stage_rows<D>(sO, [&](int r) { return qrow(dO, r); }, dO);
  auto load_block = [&](int b, int stage) {
    const int j0 = b * BN;
    stage_rows<D>(sK + stage * BN * D,
                  [&](int r) { return j0 + r < T ? k + (int64_t)(j0 + r) * kv_stride + hk * D : nullptr; }, k);
    stage_rows<D>(sV + stage * BN * D,
                  [&](int r) { return j0 + r < T ? v + (int64_t)(j0 + r) * kv_stride + hk * D : nullptr; }, v);
  };
  load_block(0, 0);
  cp_async_commit();

  const int rA = warp * 16 + (lane >> 2), rB = rA + 8;
  const int tA = p0 + (rA >> lgG), tB = p0 + (rB >> lgG);
  const int64_t iA = (int64_t)tA * Hq + hk * G + (rA & (G - 1));
  const int64_t iB = (int64_t)tB * Hq + hk * G + (rB & (G - 1));
  // invalid rows: lse = +inf makes every p zero
  const float lse2A = tA < T ? lse[iA] * kLog2e : INFINITY;
  const float lse2B = tB < T ? lse[iB] * kLog2e : INFINITY;
  const float DA = tA < T ? delta[iA] : 0.f, DB = tB < T ? delta[iB] : 0.f;
  const int lp_lo = (warp * 16) >> lgG;
  const bool warp_live = p0 + lp_lo < T;
  const int t_lo = p0 + lp_lo, t_hi = min(p0 + ((warp * 16 + 15) >> lgG), T - 1);

  uint32_t qf[D / 16][4];
  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  for (int b = 0; b < nblocks; ++b) {
    const int stage = b & 1;
    if (b + 1 < nblocks) {
      load_block(b + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (b == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int row = warp * 16 + (lane & 15), col = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(smem_u32(sQ + swz<D>(row, col)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    if (warp_live && b * BN <= t_hi) {
      const __nv_bfloat16* tK = sK + stage * BN * D;
      const __nv_bfloat16* tV = sV + stage * BN * D;
      float s[BN / 8][4], dp[BN / 8][4];
#pragma unroll
      for (int i = 0; i < BN / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[i][e] = dp[i][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t of[4];  // dO fragment of this k-step, reloaded to save registers
        ldsm_x4(smem_u32(sO + swz<D>(warp * 16 + (lane & 15), kk * 16 + (lane >> 4) * 8)), of[0],
                of[1], of[2], of[3]);
#pragma unroll
        for (int n2 = 0; n2 < BN / 16; ++n2) {
          const int key = n2 * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int col = kk * 16 + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(tK + swz<D>(key, col)), b0, b1, b2, b3);
          mma_bf16(s[2 * n2], qf[kk], b0, b1);
          mma_bf16(s[2 * n2 + 1], qf[kk], b2, b3);
          ldsm_x4(smem_u32(tV + swz<D>(key, col)), b0, b1, b2, b3);
          mma_bf16(dp[2 * n2], of, b0, b1);
          mma_bf16(dp[2 * n2 + 1], of, b2, b3);
        }
      }
      const int j0 = b * BN;
      const bool need_mask = j0 + BN - 1 > t_lo;
      uint32_t dsf[BN / 16][4];
#pragma unroll
      for (int nt = 0; nt < BN / 8; ++nt) {
        float d4[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + nt * 8 + (lane & 3) * 2 + e;
          const float pA = (!need_mask || j <= tA) ? exp2f(s[nt][e] * scale_log2 - lse2A) : 0.f;
          const float pB = (!need_mask || j <= tB) ? exp2f(s[nt][2 + e] * scale_log2 - lse2B) : 0.f;
          d4[e] = pA * (dp[nt][e] - DA);
          d4[2 + e] = pB * (dp[nt][2 + e] - DB);
        }
        dsf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(d4[0], d4[1]);
        dsf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(d4[2], d4[3]);
      }
      // dQ += dS K : B = K[key][dim] read transposed
#pragma unroll
      for (int jk = 0; jk < BN / 16; ++jk) {
#pragma unroll
        for (int dn2 = 0; dn2 < D / 16; ++dn2) {
          const int key = jk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int col = dn2 * 16 + (lane >> 4) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(tK + swz<D>(key, col)), b0, b1, b2, b3);
          mma_bf16(acc[2 * dn2], dsf[jk], b0, b1);
          mma_bf16(acc[2 * dn2 + 1], dsf[jk], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  const int64_t idx[2] = {iA, iB};
  const bool ok[2] = {tA < T, tB < T};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!ok[i]) continue;
    float* out = dq + idx[i] * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      const int col = dn * 8 + (lane & 3) * 2;
      float2 val = make_float2(acc[dn][2 * i] * scale, acc[dn][2 * i + 1] * scale);
      if (accumulate) {
        const float2 old = *reinterpret_cast<const float2*>(out + col);
        val.x += old.x;
        val.y += old.y;
      }
      *reinterpret_cast<float2*>(out + col) = val;
    }
  }
}

// ---------------------------------------------------------------- 4. dk, dv
template <int D>
__global__ void __launch_bounds__(kThreads)
bwd_dkdv_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ dO,
                const float* __restrict__ lse, const float* __restrict__ delta, int T, int Hq,
                int Hk, int lgG, float scale_log2, float scale, float* __restrict__ dk,
                float* __restrict__ dv) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sV = sK + BM * D;
  __nv_bfloat16* sQ = sV + BM * D;      // 2 stages
  __nv_bfloat16* sO = sQ + 2 * BN * D;  // 2 stages
  float* sL = reinterpret_cast<float*>(sO + 2 * BN * D);  // [2][64] lse * log2 e
  float* sD = sL + 2 * BN;                                // [2][64] delta
  const int G = 1 << lgG;
  const int P = BN >> lgG;  // positions per query block
  const int ktile = (int)(blockIdx.x / Hk);  // low keys (most query blocks) first
  const int hk = (int)(blockIdx.x % Hk);
  const int j0 = ktile * BM;
  const int qb0 = j0 / P;            // first query block holding a position >= j0
  const int nqb = (T - 1) / P - qb0 + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t kv_stride = (int64_t)Hk * D;

  stage_rows<D>(sK, [&](int r) { return j0 + r < T ? k + (int64_t)(j0 + r) * kv_stride + hk * D : nullptr; }, k);
  stage_rows<D>(sV, [&](int r) { return j0 + r < T ? v + (int64_t)(j0 + r) * kv_stride + hk * D : nullptr; }, v);
  auto load_block = [&](int i, int stage) {
    const int pq = (qb0 + i) * P;
    auto rowp = [&](const __nv_bfloat16* base, int r) -> const __nv_bfloat16* {
      const int t = pq + (r >> lgG);
      return t < T ? base + ((int64_t)t * Hq + hk * G + (r & (G - 1))) * D : nullptr;
    };
    stage_rows<D>(sQ + stage * BN * D, [&](int r) { return rowp(q, r); }, q);
    stage_rows<D>(sO + stage * BN * D, [&](int r) { return rowp(dO, r); }, dO);
    for (int r = threadIdx.x; r < BN; r += kThreads) {
      const int t = pq + (r >> lgG);
      const int64_t ri = (int64_t)t * Hq + hk * G + (r & (G - 1));
      sL[stage * BN + r] = t < T ? lse[ri] * kLog2e : INFINITY;
      sD[stage * BN + r] = t < T ? delta[ri] : 0.f;
    }
  };
  load_block(0, 0);
  cp_async_commit();

  const int kA = j0 + warp * 16 + (lane >> 2), kB = kA + 8;  // keys owned in C fragments
  float accK[D / 8][4], accV[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) accK[i][e] = accV[i][e] = 0.f;
  const bool warp_live = j0 + warp * 16 < T;

  for (int i = 0; i < nqb; ++i) {
    const int stage = i & 1;
    if (i + 1 < nqb) {
      load_block(i + 1, stage ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (warp_live) {
      const __nv_bfloat16* tQ = sQ + stage * BN * D;
      const __nv_bfloat16* tO = sO + stage * BN * D;
      const float* tL = sL + stage * BN;
      const float* tD = sD + stage * BN;
      const int pq = (qb0 + i) * P;
      float st[BN / 8][4], dpt[BN / 8][4];
#pragma unroll
      for (int n = 0; n < BN / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[n][e] = dpt[n][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t kf[4], vf[4];
        const int row = warp * 16 + (lane & 15), col = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(smem_u32(sK + swz<D>(row, col)), kf[0], kf[1], kf[2], kf[3]);
        ldsm_x4(smem_u32(sV + swz<D>(row, col)), vf[0], vf[1], vf[2], vf[3]);
#pragma unroll
        for (int n2 = 0; n2 < BN / 16; ++n2) {
          const int r = n2 * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int c = kk * 16 + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(tQ + swz<D>(r, c)), b0, b1, b2, b3);
          mma_bf16(st[2 * n2], kf, b0, b1);
          mma_bf16(st[2 * n2 + 1], kf, b2, b3);
          ldsm_x4(smem_u32(tO + swz<D>(r, c)), b0, b1, b2, b3);
          mma_bf16(dpt[2 * n2], vf, b0, b1);
          mma_bf16(dpt[2 * n2 + 1], vf, b2, b3);
        }
      }
      const bool need_mask = pq < j0 + BM;
      uint32_t pf[BN / 16][4], dsf[BN / 16][4];
#pragma unroll
      for (int nt = 0; nt < BN / 8; ++nt) {
        float p4[4], d4[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = nt * 8 + (lane & 3) * 2 + e;  // query row in the block
          const int t = pq + (r >> lgG);
          const float l2 = tL[r], dd = tD[r];
          const float pA = (!need_mask || kA <= t) ? exp2f(st[nt][e] * scale_log2 - l2) : 0.f;
          const float pB = (!need_mask || kB <= t) ? exp2f(st[nt][2 + e] * scale_log2 - l2) : 0.f;
          p4[e] = pA;
          p4[2 + e] = pB;
          d4[e] = pA * (dpt[nt][e] - dd);
          d4[2 + e] = pB * (dpt[nt][2 + e] - dd);
        }
        pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p4[0], p4[1]);
        pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p4[2], p4[3]);
        dsf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(d4[0], d4[1]);
        dsf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(d4[2], d4[3]);
      }
      // dV += P^T dO and dK += dS^T Q : B operands read transposed
#pragma unroll
      for (int jr = 0; jr < BN / 16; ++jr) {
#pragma unroll
        for (int dn2 = 0; dn2 < D / 16; ++dn2) {
          const int r = jr * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int c = dn2 * 16 + (lane >> 4) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(tO + swz<D>(r, c)), b0, b1, b2, b3);
          mma_bf16(accV[2 * dn2], pf[jr], b0, b1);
          mma_bf16(accV[2 * dn2 + 1], pf[jr], b2, b3);
          ldsm_x4_t(smem_u32(tQ + swz<D>(r, c)), b0, b1, b2, b3);
          mma_bf16(accK[2 * dn2], dsf[jr], b0, b1);
          mma_bf16(accK[2 * dn2 + 1], dsf[jr], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  const int keys[2] = {kA, kB};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (keys[i] >= T) continue;
    float* ok_ = dk + ((int64_t)keys[i] * Hk + hk) * D;
    float* ov = dv + ((int64_t)keys[i] * Hk + hk) * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      const int col = dn * 8 + (lane & 3) * 2;
      *reinterpret_cast<float2*>(ok_ + col) =
          make_float2(accK[dn][2 * i] * scale, accK[dn][2 * i + 1] * scale);
      *reinterpret_cast<float2*>(ov + col) = make_float2(accV[dn][2 * i], accV[dn][2 * i + 1]);
    }
  }
}

template <int D, int G>
cudaError_t launch_depth(const BwdArgs& a, cudaStream_t st) {
  const size_t smem = 4 * sizeof(DepthWarpSmem<D, G>);
  cudaError_t e = cudaFuncSetAttribute(bwd_depth_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t pairs = (int64_t)a.Hk * a.T;
  bwd_depth_kernel<D, G><<<(unsigned)((pairs + 3) / 4), 128, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kd, (const __nv_bfloat16*)a.vd,
      (const __nv_bfloat16*)a.dO, a.lse, a.delta, a.T, a.Hq, a.Hk, a.L, a.scale * kLog2e, a.scale,
      a.dq, a.dkd, a.dvd);
  return cudaGetLastError();
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

template <int D>
cudaError_t launch_dq_mma(const BwdArgs& a, cudaStream_t st) {
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int P = BM >> lgG;
  const int ntiles = (a.T + P - 1) / P;
  const size_t smem = (size_t)(2 * BM + 4 * BN) * D * sizeof(__nv_bfloat16);
  cudaError_t e =
      cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  bwd_dq_kernel<D><<<(unsigned)((int64_t)ntiles * a.Hk), kThreads, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
      (const __nv_bfloat16*)a.dO, a.lse, a.delta, a.T, a.Hq, a.Hk, lgG, ntiles,
      a.scale * kLog2e, a.scale, a.dq, a.L > 0 ? 1 : 0);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dkdv_mma(const BwdArgs& a, cudaStream_t st) {
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int nk = (a.T + BM - 1) / BM;
  const size_t smem = (size_t)(2 * BM + 4 * BN) * D * sizeof(__nv_bfloat16) + 4 * BN * sizeof(float);
  cudaError_t e =
      cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  bwd_dkdv_kernel<D><<<(unsigned)((int64_t)nk * a.Hk), kThreads, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
      (const __nv_bfloat16*)a.dO, a.lse, a.delta, a.T, a.Hq, a.Hk, lgG, a.scale * kLog2e,
      a.scale, a.dk, a.dv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_mma(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_dkdv_mma<128>(a, stream) : launch_dkdv_mma<64>(a, stream);
}

cudaError_t launch_bwd_dq_mma(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_dq_mma<128>(a, stream) : launch_dq_mma<64>(a, stream);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

// MoDA forward on warp-level MMA (mma.sync m16n8k16, bf16 in, fp32 acc).
//
// Mixture-of-Depths Attention, Sec. 3.3 (fused kernel) restated:
//   * group-aware query tile: BM = 64 rows hold 64/G positions x the G query
//     heads of one KV head (row r -> position p0 + r/G, head hk*G + r%G), so
//     each K/V tile staged in shared memory serves all G heads (Sec. 3.2
//     "group-aware depth KV computation");
//   * depth blocks first: the packed depth keys of the tile's positions are
//     one contiguous run of (64/G)*L rows of kd[hk] (chunk-aware layout);
//     row r keeps depth column j iff floor(j/L) == r/G (block-diagonal mask,
//     Sec. 3.3 mask equation). Processing order does not matter to an exact
//     online softmax, and depth first seeds the running max early;
//   * then the sequence blocks with the grouped causal mask key <= t(r);
//   * one running (m, l, O) state per row across both, normalised once.
// Exponentials are exp2 with log2(e) folded into the scale.
//
// This is the portable warp-MMA path; the tensor-memory path for sm_103a
// replaces it where it applies.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "warp_mma.cuh"

namespace moda {
namespace {

using namespace wmma16;

constexpr int BM = 64;   // query rows per CTA
constexpr int BN = 64;   // keys per block
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Stage 64 rows of D bf16 into a swizzled tile. Row i comes from
// base + i*row_stride (elements); rows >= nvalid are zero-filled.
template <int D>
__device__ __forceinline__ void load_rows(__nv_bfloat16* tile, const __nv_bfloat16* base,
                                          int64_t row_stride, int nvalid) {
  constexpr int kChunks = D / 8;
  for (int idx = threadIdx.x; idx < BN * kChunks; idx += kThreads) {
    const int row = idx / kChunks, ch = idx % kChunks;
    const bool ok = row < nvalid;
    const __nv_bfloat16* src = ok ? base + row * row_stride + ch * 8 : base;
    cp_async16(smem_u32(tile + swz<D>(row, ch * 8)), src, ok);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
moda_fwd_mma_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ kd,
                    const __nv_bfloat16* __restrict__ vd, int T, int Hq, int Hk, int L,
                    int lgG, int ntiles, float scale_log2, __nv_bfloat16* __restrict__ o,
                    float* __restrict__ lse) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sK = sQ + BM * D;       // 2 stages
  __nv_bfloat16* sV = sK + 2 * BN * D;   // 2 stages

  const int G = 1 << lgG;
  const int P = BM >> lgG;  // positions per tile
  const int bid = blockIdx.x;
  const int tile = ntiles - 1 - bid / Hk;  // longest (latest positions) first
  const int hk = bid % Hk;
  const int p0 = tile * P;
  const int npos = min(P, T - p0);
  const int t_last = p0 + npos - 1;
  const int nd = npos * L;  // packed depth rows of this tile
  const int n_depth_blocks = (nd + BN - 1) / BN;
  const int n_seq_blocks = t_last / BN + 1;
  const int nblocks = n_depth_blocks + n_seq_blocks;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t kv_row_stride = (int64_t)Hk * D;
  const __nv_bfloat16* kd_base = kd ? kd + ((int64_t)hk * T + p0) * L * D : nullptr;
  const __nv_bfloat16* vd_base = vd ? vd + ((int64_t)hk * T + p0) * L * D : nullptr;

  // ---- stage the Q tile: row r -> (p0 + r/G, hk*G + r%G) ----
  {
    constexpr int kChunks = D / 8;
    for (int idx = threadIdx.x; idx < BM * kChunks; idx += kThreads) {
      const int row = idx / kChunks, ch = idx % kChunks;
      const int t = p0 + (row >> lgG);
      const int h = hk * G + (row & (G - 1));
      const bool ok = t < T;
      const __nv_bfloat16* src = ok ? q + ((int64_t)t * Hq + h) * D + ch * 8 : q;
      cp_async16(smem_u32(sQ + swz<D>(row, ch * 8)), src, ok);
    }
  }
  auto load_block = [&](int b, int stage) {
    if (b < n_depth_blocks) {
      const int r0 = b * BN;
      load_rows<D>(sK + stage * BN * D, kd_base + (int64_t)r0 * D, D, nd - r0);
      load_rows<D>(sV + stage * BN * D, vd_base + (int64_t)r0 * D, D, nd - r0);
    } else {
      const int j0 = (b - n_depth_blocks) * BN;
      load_rows<D>(sK + stage * BN * D, k + (int64_t)j0 * kv_row_stride + hk * D, kv_row_stride, T - j0);
      load_rows<D>(sV + stage * BN * D, v + (int64_t)j0 * kv_row_stride + hk * D, kv_row_stride, T - j0);
    }
  };
  load_block(0, 0);
  cp_async_commit();

  // rows owned by this thread: r0 = 16*warp + lane/4 and r0 + 8
  const int rA = warp * 16 + (lane >> 2), rB = rA + 8;
  const int lpA = rA >> lgG, lpB = rB >> lgG;       // local positions
  const int tA = min(p0 + lpA, T - 1), tB = min(p0 + lpB, T - 1);  // clamped for masking
  const int lp_lo = (warp * 16) >> lgG, lp_hi = (warp * 16 + 15) >> lgG;
  const bool warp_live = p0 + lp_lo < T;
  const int t_lo = p0 + lp_lo, t_hi = min(p0 + lp_hi, T - 1);

  uint32_t qf[D / 16][4];
  float acc_o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc_o[i][0] = acc_o[i][1] = acc_o[i][2] = acc_o[i][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

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
        const int row = warp * 16 + (lane & 15);
        const int col = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(smem_u32(sQ + swz<D>(row, col)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const bool is_depth = b < n_depth_blocks;
    bool relevant;
    if (is_depth) {
      const int j0 = b * BN;
      relevant = warp_live && j0 < (lp_hi + 1) * L && j0 + BN > lp_lo * L;
    } else {
      relevant = warp_live && (b - n_depth_blocks) * BN <= t_hi;
    }
    if (relevant) {
      const __nv_bfloat16* tK = sK + stage * BN * D;
      const __nv_bfloat16* tV = sV + stage * BN * D;
      float s[BN / 8][4];
#pragma unroll
      for (int i = 0; i < BN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int n2 = 0; n2 < BN / 16; ++n2) {
          const int key = n2 * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int col = kk * 16 + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(tK + swz<D>(key, col)), b0, b1, b2, b3);
          mma_bf16(s[2 * n2], qf[kk], b0, b1);
          mma_bf16(s[2 * n2 + 1], qf[kk], b2, b3);
        }
      }
      // scale, mask, running max
      float mx[2] = {-INFINITY, -INFINITY};
      if (is_depth) {
        const int j0 = b * BN;
        const int loA = lpA * L, hiA = min((lpA + 1) * L, nd);
        const int loB = lpB * L, hiB = min((lpB + 1) * L, nd);
#pragma unroll
        for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = j0 + nt * 8 + (lane & 3) * 2 + e;
            s[nt][e] = (j >= loA && j < hiA) ? s[nt][e] * scale_log2 : -INFINITY;
            s[nt][2 + e] = (j >= loB && j < hiB) ? s[nt][2 + e] * scale_log2 : -INFINITY;
          }
        }
      } else {
        const int j0 = (b - n_depth_blocks) * BN;
        const bool need_mask = j0 + BN - 1 > t_lo;
#pragma unroll
        for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = j0 + nt * 8 + (lane & 3) * 2 + e;
            s[nt][e] = (!need_mask || j <= tA) ? s[nt][e] * scale_log2 : -INFINITY;
            s[nt][2 + e] = (!need_mask || j <= tB) ? s[nt][2 + e] * scale_log2 : -INFINITY;
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < BN / 8; ++nt) {
        mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      }
      float alpha[2], base[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float mn = fmaxf(m[i], mx[i]);
        base[i] = (mn == -INFINITY) ? 0.f : mn;
        alpha[i] = exp2f(m[i] - base[i]);  // m = -inf -> 0
        m[i] = mn;
      }
      float rs[2] = {0.f, 0.f};
      uint32_t pf[BN / 16][4];
#pragma unroll
      for (int nt = 0; nt < BN / 8; ++nt) {
        const float p0v = exp2f(s[nt][0] - base[0]);
        const float p1v = exp2f(s[nt][1] - base[0]);
        const float p2v = exp2f(s[nt][2] - base[1]);
        const float p3v = exp2f(s[nt][3] - base[1]);
        rs[0] += p0v + p1v;
        rs[1] += p2v + p3v;
        pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0v, p1v);
        pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2v, p3v);
      }
      l[0] = l[0] * alpha[0] + rs[0];
      l[1] = l[1] * alpha[1] + rs[1];
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        acc_o[dn][0] *= alpha[0];
        acc_o[dn][1] *= alpha[0];
        acc_o[dn][2] *= alpha[1];
        acc_o[dn][3] *= alpha[1];
      }
#pragma unroll
      for (int j = 0; j < BN / 16; ++j) {
        // A fragment: rows (lane/4, +8) x keys 16j.., from pf
        const uint32_t a[4] = {pf[j][0], pf[j][1], pf[j][2], pf[j][3]};
#pragma unroll
        for (int dn2 = 0; dn2 < D / 16; ++dn2) {
          const int key = j * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int col = dn2 * 16 + (lane >> 4) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(tV + swz<D>(key, col)), b0, b1, b2, b3);
          mma_bf16(acc_o[2 * dn2], a, b0, b1);
          mma_bf16(acc_o[2 * dn2 + 1], a, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // ---- epilogue: o = O / l, lse = m*ln2 + ln(l) ----
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
  }
  const int rows[2] = {rA, rB};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = p0 + (rows[i] >> lgG);
    if (t >= T) continue;
    const int h = hk * G + (rows[i] & (G - 1));
    const float inv = 1.f / l[i];
    __nv_bfloat16* orow = o + ((int64_t)t * Hq + h) * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      const int col = dn * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(orow + col) =
          pack_bf16(acc_o[dn][2 * i] * inv, acc_o[dn][2 * i + 1] * inv);
    }
    if (lse && (lane & 3) == 0) lse[(int64_t)t * Hq + h] = m[i] * kLn2 + logf(l[i]);
  }
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t stream) {
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int P = BM >> lgG;
  const int ntiles = (a.T + P - 1) / P;
  const size_t smem = (size_t)(BM + 4 * BN) * D * sizeof(__nv_bfloat16);
  cudaError_t e = cudaFuncSetAttribute(moda_fwd_mma_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = (int64_t)ntiles * a.Hk;
  moda_fwd_mma_kernel<D><<<(unsigned)grid, kThreads, smem, stream>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v,
      (const __nv_bfloat16*)a.kd, (const __nv_bfloat16*)a.vd, a.T, a.Hq, a.Hk, a.L, lgG, ntiles,
      a.scale * kLog2e, (__nv_bfloat16*)a.o, a.lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_mma(const FwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

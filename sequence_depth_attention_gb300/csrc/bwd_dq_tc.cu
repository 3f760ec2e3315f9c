// dQ of the MoDA backward on the 5th-generation tensor core (sm_103a).
//
// For a tile of 128 G-stacked query rows (row r <-> position p0 + r/G, head
// hk*G + r%G, one 3-D TMA box as in the forward) and each causal key block
// j of 128 keys:
//   S_j  = Q K_j^T,   dP_j = dO V_j^T                  (tcgen05, into TMEM)
//   dS_j = exp2(S_j scale log2e - lse log2e) * (dP_j - D)  (CUDA cores; lse from
//          the forward, so no running max and no cross-column reduction)
//   dQ  += dS_j K_j                                      (tcgen05, dS read from
//          TMEM as the A operand, K_j from shared memory as an MN-major B)
// The depth slots' share of dq is written beforehand by the depth kernel;
// this kernel adds the sequence share.
//
// Roles (12 warps): warp 0 TMA for Q, dO and K; warp 2 TMA for V; warp 1
// issues MMAs; warps 4-7 and 8-11 each own 64 columns of S and dP for all 128
// rows (thread = row = TMEM lane). TMEM: S [0,128), dP [128,256), dQ
// [256,256+d), dS double buffer [384,448) [448,512) as bf16 pairs.
// Issue order: S_0, dP_0, then per block j: S_{j+1}, dP_{j+1} once the
// softmax has read S_j and dP_j, then dQ += dS_j K_j once dS_j is written.
// All waits are bounded; on expiry the CTA drains and latches MODA_ERR_TIMEOUT.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "tensor_map.h"

namespace moda {
namespace {

using namespace sm103;

constexpr int BM = 128, BN = 128;
constexpr int kThreads = 384;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DqCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = 128 * 64 * 2;
  static constexpr int kNSK = 3, kNSV = 2;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffO = kOffQ + kTileBytes;  // dO tile
  static constexpr int kOffK = kOffO + kTileBytes;
  static constexpr int kOffV = kOffK + kNSK * kTileBytes;
  static constexpr int kOffBar = kOffV + kNSV * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr uint32_t kColS = 0, kColP = 128, kColQ = 256, kColDS = 384;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct alignas(8) DqBars {
  uint64_t q_full;
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full, s_free;
  uint64_t ds_full[2], dq_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqBars) <= 256, "barrier block");

struct DqParams {
  int T, Hq, Hk, lgG, ntiles, accumulate;
  float scale_log2, scale;
  const float* lse;
  const float* delta;
  float* dq;
  unsigned int* err;
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

// dS = exp2(S scale log2e - lse log2e) (dP - D) for 64 columns of one row,
// packed to bf16 pairs; columns >= span are zero when kMask.
template <bool kMask>
__device__ __forceinline__ void ds_pack(const uint32_t* x, const uint32_t* y, uint64_t sl2,
                                        uint64_t nl2, uint64_t nD2, int span, uint32_t* pk) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float a0, a1, d0, d1;
    f2_split(ffma2(f2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])), sl2, nl2), a0, a1);
    const uint64_t dd = fadd2(f2(__uint_as_float(y[2 * c]), __uint_as_float(y[2 * c + 1])), nD2);
    f2_split(fmul2(f2(ex2_approx(a0), ex2_approx(a1)), dd), d0, d1);
    if (kMask) {
      d0 = 2 * c < span ? d0 : 0.f;
      d1 = 2 * c + 1 < span ? d1 : 0.f;
    }
    pk[c] = pack_bf16x2(d0, d1);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const DqParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  DqBars* bars = reinterpret_cast<DqBars*>(smem + C::kOffBar);
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sO = smem_u32(smem + C::kOffO);
  const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = 1 << p.lgG;
  const int P = BM >> p.lgG;
  const int tile = p.ntiles - 1 - (int)(blockIdx.x / p.Hk);  // longest first
  const int hk = (int)(blockIdx.x % p.Hk);
  const int p0 = tile * P;
  const int t_last = min(p0 + P, p.T) - 1;
  const int nb = t_last / BN + 1;

  if (tid == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->k_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->v_empty[s]), 1);
      mbar_init(smem_u32(&bars->ds_full[s]), 256);
      mbar_init(smem_u32(&bars->dq_done[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->s_free), 256);
    mbar_init(smem_u32(&bars->mma_done), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------ TMA producers
    const bool leader = elect_one();
    const bool is_k = warp == 0;
    const int NS = is_k ? C::kNSK : C::kNSV;
    const uint32_t sbase = is_k ? sK : sV;
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    uint64_t* full = is_k ? bars->k_full : bars->v_full;
    uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
    if (is_k && leader) {
      const uint32_t qb = smem_u32(&bars->q_full);
      mbar_arrive_expect_tx(qb, 2 * C::kTileBytes);
      for (int c = 0; c < C::kBoxes; ++c) {
        tma_load_3d(sQ + c * C::kBoxBytes, &tmQ, qb, c * 64, hk * G, p0);
        tma_load_3d(sO + c * C::kBoxBytes, &tmO, qb, c * 64, hk * G, p0);
      }
    }
    int issued = 0;
    for (int j = 0; j < nb; ++j) {
      const int s = j % NS;
      const bool ok = mbar_wait_bounded(smem_u32(&empty[s]), ((j / NS) & 1) ^ 1, abort, kTimeoutNs);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (leader) {
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, C::kTileBytes);
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_3d(sbase + s * C::kTileBytes + c * C::kBoxBytes, map, fb, c * 64, hk, j * BN);
      }
      __syncwarp();
      issued = j + 1;
    }
    if (leader) {
      int never = 0;
      for (int j = max(0, issued - NS); j < issued; ++j)
        mbar_wait_bounded(smem_u32(&full[j % NS]), (j / NS) & 1, &never, kTimeoutNs);
      if (is_k) mbar_wait_bounded(smem_u32(&bars->q_full), 0, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    // One thread runs the whole schedule, waits included: the tensor core
    // queues few MMAs, so every instruction on this thread between two MMAs
    // can leave it idle, and the elementwise warps share its issue slots.
    if (elect_one()) {
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false);  // S, dP: K-major A and B
      constexpr uint32_t idQ = idesc_bf16_f32(BM, D, true);    // dQ: B = K read MN-major
      // every descriptor here has the same high word (SBO 1024, 128-byte
      // swizzle); tile offsets are 32-bit adds to the start address field
      const uint64_t dq_ = sdesc_sw128(sQ, 16, 1024);
      const uint32_t hi = (uint32_t)(dq_ >> 32), q_lo = (uint32_t)dq_;
      const uint32_t o_lo = (uint32_t)sdesc_sw128(sO, 16, 1024);
      const uint32_t k_lo = (uint32_t)sdesc_sw128(sK, 16, 1024), v_lo = (uint32_t)sdesc_sw128(sV, 16, 1024);
      const uint32_t kmn_lo = (uint32_t)sdesc_sw128(sK, C::kBoxBytes, 1024);
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return mbar_wait_bounded(smem_u32(bar), parity, abort, kTimeoutNs);
      };
      auto issue_s = [&](int j) {  // S_j
        const int ks = j % C::kNSK;
        const uint32_t kb = k_lo + ((uint32_t)(ks * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tbase + C::kColS, desc_join(q_lo + off, hi), desc_join(kb + off, hi), idS, kk > 0);
        }
      };
      auto issue_dp = [&](int j) {  // dP_j; frees V_j when done, completes block j
        const int vs = j % C::kNSV;
        const uint32_t vb = v_lo + ((uint32_t)(vs * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tbase + C::kColP, desc_join(o_lo + off, hi), desc_join(vb + off, hi), idS, kk > 0);
        }
        tc_commit(smem_u32(&bars->v_empty[vs]));
        tc_commit(smem_u32(&bars->s_full));
      };
      auto issue_dq = [&](int j) {  // dQ += dS_j K_j; frees K_j when done
        const int ks = j % C::kNSK, b = j & 1;
        const uint32_t kb = kmn_lo + ((uint32_t)(ks * C::kTileBytes) >> 4);
        const uint32_t acol = tbase + C::kColDS + b * 64;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tbase + C::kColQ, acol + kk * 8, desc_join(kb + ((uint32_t)(kk * 2048) >> 4), hi), idQ,
                 kk > 0 ? 1u : acc0);
        tc_commit(smem_u32(&bars->k_empty[ks]));
        tc_commit(smem_u32(&bars->dq_done[b]));
      };
      bool ok = wait(&bars->q_full, 0) && wait(&bars->k_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        ok = wait(&bars->v_full[0], 0);
        if (ok) issue_dp(0);
      }
      for (int j = 0; ok && j < nb; ++j) {
        if (j + 1 < nb) {
          // S_{j+1}, dP_{j+1} as soon as the softmax holds S_j, dP_j in registers;
          // S needs only K_{j+1}, so it runs while V_{j+1} may still be landing
          uint64_t* kf = &bars->k_full[(j + 1) % C::kNSK];
          const uint32_t kpar = ((j + 1) / C::kNSK) & 1;
          if (!mbar_test_both(smem_u32(&bars->s_free), j & 1, smem_u32(kf), kpar)) {
            if (!wait(&bars->s_free, j & 1)) break;
            if (!wait(kf, kpar)) break;
          }
          tc_fence_after();
          issue_s(j + 1);
          if (!wait(&bars->v_full[(j + 1) % C::kNSV], ((j + 1) / C::kNSV) & 1)) break;
          tc_fence_after();
          issue_dp(j + 1);
        }
        if (!wait(&bars->ds_full[j & 1], (j >> 1) & 1)) break;
        tc_fence_after();
        issue_dq(j);
      }
      int never = 0;
      tc_commit(smem_u32(&bars->mma_done));
      mbar_wait_bounded(smem_u32(&bars->mma_done), 0, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------ dS (two column halves)
    const int half = (warp - 4) >> 2, q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)q4 * 32;
    const int t_row = p0 + (row >> p.lgG);
    const int h_row = hk * G + (row & (G - 1));
    const bool valid = t_row < p.T;
    const int64_t ri = (int64_t)t_row * p.Hq + h_row;
    // invalid rows: lse = +inf makes every p zero
    const float lse2 = valid ? p.lse[ri] * kLog2e : INFINITY;
    const float Dr = valid ? p.delta[ri] : 0.f;
    const int t_mask = min(t_row, p.T - 1);
    const uint64_t sl2 = f2(p.scale_log2, p.scale_log2), nl2 = f2(-lse2, -lse2), nD2 = f2(-Dr, -Dr);
    bool ok = true;
    for (int j = 0; j < nb && ok; ++j) {
      if (!warp_wait(smem_u32(&bars->s_full), j & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x[64], y[64];
      tmem_ld32(tmem_addr(tbase, lane_base, C::kColS + half * 64), x);
      tmem_ld32(tmem_addr(tbase, lane_base, C::kColS + half * 64 + 32), x + 32);
      tmem_ld32(tmem_addr(tbase, lane_base, C::kColP + half * 64), y);
      tmem_ld32(tmem_addr(tbase, lane_base, C::kColP + half * 64 + 32), y + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->s_free));
      // causal mask (key <= t_row), needed only on the blocks that reach past p0
      const int k0 = j * BN + half * 64;
      uint32_t pk[32];
      if (j * BN + BN - 1 > p0) {
        const int span = max(0, min(64, t_mask - k0 + 1));
        ds_pack<true>(x, y, sl2, nl2, nD2, span, pk);
      } else {
        ds_pack<false>(x, y, sl2, nl2, nD2, 64, pk);
      }
      // dS_j reuses the buffer of dS_{j-2}: the tensor core must have consumed it
      if (j >= 2) {
        if (!warp_wait(smem_u32(&bars->dq_done[j & 1]), ((j - 2) >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tmem_addr(tbase, lane_base, C::kColDS + (j & 1) * 64 + half * 32), pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->ds_full[j & 1]));
    }
    if (ok) {
      ok = warp_wait(smem_u32(&bars->dq_done[(nb - 1) & 1]), ((nb - 1) >> 1) & 1, abort);
      if (ok && nb >= 2)
        ok = warp_wait(smem_u32(&bars->dq_done[(nb - 2) & 1]), ((nb - 2) >> 1) & 1, abort);
    }
    if (ok) {
      tc_fence_after();
      constexpr int HD = D / 2;
      float* out = p.dq + ri * D + half * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tbase, lane_base, C::kColQ + half * HD + c * 32), r);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float4 v = make_float4(__uint_as_float(r[i]) * p.scale, __uint_as_float(r[i + 1]) * p.scale,
                                   __uint_as_float(r[i + 2]) * p.scale, __uint_as_float(r[i + 3]) * p.scale);
            float4* dst = reinterpret_cast<float4*>(out + c * 32 + i);
            if (p.accumulate) {
              const float4 old = *dst;
              v.x += old.x; v.y += old.y; v.z += old.z; v.w += old.w;
            }
            *dst = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (tid == 0 && bars->abort) atomicCAS(p.err, 0u, (unsigned int)MODA_ERR_TIMEOUT);
}

template <int D>
cudaError_t launch_d(const BwdArgs& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int P = BM >> lgG;
  const int ntiles = (a.T + P - 1) / P;
  CUtensorMap tq, to, tk, tv;
  const uint64_t row = (uint64_t)D * 2;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)a.T};
    const uint64_t str[2] = {row, row * a.Hq};
    const uint32_t box[3] = {64, (uint32_t)a.G, (uint32_t)P};
    if (encode_bf16_sw128(&tq, a.q, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&to, a.dO, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hk, (uint64_t)a.T};
    const uint64_t str[2] = {row, row * a.Hk};
    const uint32_t box[3] = {64, 1, BN};
    if (encode_bf16_sw128(&tk, a.k, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tv, a.v, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  DqParams prm;
  prm.T = a.T; prm.Hq = a.Hq; prm.Hk = a.Hk; prm.lgG = lgG; prm.ntiles = ntiles;
  prm.accumulate = a.L > 0 ? 1 : 0;
  prm.scale_log2 = a.scale * kLog2e;
  prm.scale = a.scale;
  prm.lse = a.lse;
  prm.delta = a.delta;
  prm.dq = a.dq;
  prm.err = a.err;
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  bwd_dq_tc_kernel<D><<<(unsigned)((int64_t)ntiles * a.Hk), kThreads, C::kSmemBytes, stream>>>(
      tq, to, tk, tv, prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_tc(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

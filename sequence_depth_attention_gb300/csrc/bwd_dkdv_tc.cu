// dK and dV of the MoDA backward on the 5th-generation tensor core (sm_103a).
//
// One CTA owns a block of 128 keys of one KV head (K and V stay in shared
// memory) and walks over the query rows that can see it in sub-tiles of 64
// G-stacked rows (64/G positions x G heads, one 3-D TMA box as in the
// forward). For each sub-tile c:
//   S^T_c  = K Q_c^T,  dP^T_c = V dO_c^T             (tcgen05, 128 x 64 into TMEM)
//   P^T_c  = exp2(S^T_c scale log2e - lse log2e)      (per column: the query's lse)
//   dS^T_c = P^T_c * (dP^T_c - D)                     (CUDA cores, lane = key)
//   dV += P^T_c dO_c,  dK += dS^T_c Q_c               (tcgen05, A from TMEM,
//                                                      Q_c / dO_c read MN-major)
// Only the sequence keys are handled here; the depth slots' gradients come
// from the depth kernel. dk is written times the softmax scale.
//
// Roles (12 warps): warp 0 TMA (K, V once, then the Q/dO ring); warp 1 issues
// MMAs; warps 4-7 and 8-11 are the two elementwise warpgroups. Either each
// group takes 32 of the 64 columns of every sub-tile, or (ping-pong: always at
// d = 64, where the elementwise work per MMA flop doubles, and for long
// sequences at d = 128) the groups take alternate sub-tiles, all 64 columns
// each, so that two sub-tiles are worked on at once.
// TMEM columns: B buffers b of S^T [128b,128b+64) and dP^T [128b+64,128b+128)
// (B = 2 at d = 128, 3 at d = 64), sub-tile c in buffer c%B; the elementwise
// warps write P^T|dS^T over the S^T columns they read (per column half: 16
// columns of P^T then 16 of dS^T, bf16 pairs); dV [128B,128B+d) and dK
// [128B+d,128B+2d), 512 columns in all.
// Issue order: dP_c S_c for c < B, then per c: dV_c dK_c once P^T_c and dS^T_c
// are stored, dP_{c+B} (its columns were free once the elementwise warps read
// dP_c), and S_{c+B} once dV_c and dK_c have read buffer c%B. The tensor core
// works on one sub-tile while the elementwise warps work on the next ones.
// All waits are bounded; on expiry the CTA drains and latches MODA_ERR_TIMEOUT.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "tensor_map.h"

namespace moda {
namespace {

using namespace sm103;

constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 64;   // G-stacked query rows per sub-tile
constexpr int kThreads = 384;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct KvCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kKBox = BK * 128;  // bytes of one 64-column box of K or V
  static constexpr int kQBox = BQ * 128;  // bytes of one 64-column box of a Q or dO sub-tile
  static constexpr int kKTile = kBoxes * kKBox;
  static constexpr int kQTile = kBoxes * kQBox;
  static constexpr int kNS = D == 128 ? 4 : 6;  // Q/dO ring stages
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKTile;
  static constexpr int kOffQ = kOffV + kKTile;           // stage s: Q at kOffQ + s*2*kQTile
  static constexpr int kOffRow = kOffQ + kNS * 2 * kQTile;  // per-warp lse2 / D staging
  static constexpr int kB = D == 64 ? 3 : 2;  // S^T|dP^T buffers: 128*kB + 2*D = 512
  static constexpr int kOffBar = kOffRow + 8 * 2 * 64 * 4;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr uint32_t kColS = 0, kColP = 64, kColBuf = 128, kColV = 128 * kB,
                            kColK = 128 * kB + D;
  static_assert(kColK + D == 512, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct alignas(8) KvBars {
  uint64_t kv_full;
  uint64_t q_full[6], q_empty[6];
  uint64_t s_full[3];               // S^T, dP^T of buffer b computed
  uint64_t pd_full[3], pd_done[3];  // P^T|dS^T of buffer b stored / consumed
  uint64_t mma_done;                // every product of the CTA has completed
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(KvBars) <= 256, "barrier block");

struct KvParams {
  int T, Hq, Hk, lgG;
  float scale_log2, scale;
  const float* lse;
  const float* delta;
  float* dk;
  float* dv;
  unsigned int* err;
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

// For 32 columns of one key row: P^T = exp2(S^T scale log2e - lse log2e) and
// dS^T = P^T (dP^T - D), packed to bf16 pairs (P^T in pk[0,16), dS^T in
// pk[16,32)). nrow holds -lse log2e in [0,32) and -D in [32,64) per column.
// Columns below `first` are zero when kMask.
template <bool kMask>
__device__ __forceinline__ void pds_pack(const uint32_t* x, const uint32_t* y, const float* nrow,
                                         uint64_t sl2, int first, uint32_t* pk) {
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float4 l4 = *reinterpret_cast<const float4*>(nrow + c);
    const float4 d4 = *reinterpret_cast<const float4*>(nrow + 32 + c);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = c + 2 * h;
      const uint64_t nl = h ? f2(l4.z, l4.w) : f2(l4.x, l4.y);
      const uint64_t nd = h ? f2(d4.z, d4.w) : f2(d4.x, d4.y);
      float a0, a1, s0, s1;
      f2_split(ffma2(f2(__uint_as_float(x[e]), __uint_as_float(x[e + 1])), sl2, nl), a0, a1);
      float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
      const uint64_t dd = fadd2(f2(__uint_as_float(y[e]), __uint_as_float(y[e + 1])), nd);
      f2_split(fmul2(f2(p0, p1), dd), s0, s1);
      if (kMask) {
        p0 = e >= first ? p0 : 0.f;
        p1 = e + 1 >= first ? p1 : 0.f;
        s0 = e >= first ? s0 : 0.f;
        s1 = e + 1 >= first ? s1 : 0.f;
      }
      pk[e / 2] = pack_bf16x2(p0, p1);
      pk[16 + e / 2] = pack_bf16x2(s0, s1);
    }
  }
}

// PP: the elementwise warpgroups take alternate sub-tiles (ping-pong)
template <int D, bool PP>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const KvParams p) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  KvBars* bars = reinterpret_cast<KvBars*>(smem + C::kOffBar);
  const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = 1 << p.lgG;
  const int PQ = BQ >> p.lgG;  // positions per sub-tile
  const int kb = (int)(blockIdx.x / p.Hk);  // longest first: early keys see the most queries
  const int hk = (int)(blockIdx.x % p.Hk);
  const int q0 = kb * BK;                   // first query position that sees this block
  const int n = (p.T - q0 + PQ - 1) / PQ;   // sub-tiles
  constexpr bool pp = PP;

  if (tid == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->kv_full), 1);
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 1);
      mbar_init(smem_u32(&bars->q_empty[s]), 1);
    }
    for (int b = 0; b < C::kB; ++b) {
      mbar_init(smem_u32(&bars->s_full[b]), 1);
      mbar_init(smem_u32(&bars->pd_full[b]), pp ? 128 : 256);
      mbar_init(smem_u32(&bars->pd_done[b]), 1);
    }
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

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    const bool leader = elect_one();
    if (leader) {
      const uint32_t kvb = smem_u32(&bars->kv_full);
      mbar_arrive_expect_tx(kvb, 2 * C::kKTile);
      for (int c = 0; c < C::kBoxes; ++c) {
        tma_load_3d(sK + c * C::kKBox, &tmK, kvb, c * 64, hk, q0);
        tma_load_3d(sV + c * C::kKBox, &tmV, kvb, c * 64, hk, q0);
      }
    }
    int issued = 0;
    for (int i = 0; i < n; ++i) {
      const int s = i % C::kNS;
      if (!warp_wait(smem_u32(&bars->q_empty[s]), ((i / C::kNS) & 1) ^ 1, abort)) break;
      if (leader) {
        const uint32_t fb = smem_u32(&bars->q_full[s]);
        const uint32_t dst = sQ + s * 2 * C::kQTile;
        mbar_arrive_expect_tx(fb, 2 * C::kQTile);
        for (int c = 0; c < C::kBoxes; ++c) {
          tma_load_3d(dst + c * C::kQBox, &tmQ, fb, c * 64, hk * G, q0 + i * PQ);
          tma_load_3d(dst + C::kQTile + c * C::kQBox, &tmO, fb, c * 64, hk * G, q0 + i * PQ);
        }
      }
      __syncwarp();
      issued = i + 1;
    }
    if (leader) {
      int never = 0;
      for (int i = max(0, issued - C::kNS); i < issued; ++i)
        mbar_wait_bounded(smem_u32(&bars->q_full[i % C::kNS]), (i / C::kNS) & 1, &never, kTimeoutNs);
      mbar_wait_bounded(smem_u32(&bars->kv_full), 0, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    // One thread runs the whole schedule, waits included: the tensor core
    // queues few MMAs, so every instruction on this thread between two MMAs
    // can leave it idle, and the elementwise warps share its issue slots.
    if (elect_one()) {
      constexpr uint32_t idS = idesc_bf16_f32(BK, BQ, false);  // S^T, dP^T: K-major A and B
      constexpr uint32_t idG = idesc_bf16_f32(BK, D, true);    // dV, dK: B read MN-major
      // every descriptor here has the same high word (SBO 1024, 128-byte
      // swizzle); tile offsets are 32-bit adds to the start address field
      const uint64_t dq_ = sdesc_sw128(sQ, 16, 1024);
      const uint32_t hi = (uint32_t)(dq_ >> 32), q_lo = (uint32_t)dq_;
      const uint32_t k_lo = (uint32_t)sdesc_sw128(sK, 16, 1024), v_lo = (uint32_t)sdesc_sw128(sV, 16, 1024);
      const uint32_t qmn_lo = (uint32_t)sdesc_sw128(sQ, C::kQBox, 1024);
      auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return mbar_wait_bounded(smem_u32(bar), parity, abort, kTimeoutNs);
      };
      auto stage_of = [&](int i) { return (uint32_t)((i % C::kNS) * 2 * C::kQTile) >> 4; };
      auto issue_dp = [&](int i) {  // dP^T_i = V dO_i^T into buffer i%B
        const uint32_t qs = q_lo + stage_of(i) + (C::kQTile >> 4);
        const uint32_t acc = tbase + (i % C::kB) * C::kColBuf + C::kColP;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = ((kk >> 2) * C::kKBox + (kk & 3) * 32) >> 4;
          const uint32_t qa = ((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4;
          mma_ss(acc, desc_join(v_lo + ka, hi), desc_join(qs + qa, hi), idS, kk > 0);
        }
      };
      auto issue_s = [&](int i) {  // S^T_i = K Q_i^T into buffer i%B; buffer i%B is then complete
        const uint32_t qs = q_lo + stage_of(i);
        const uint32_t acc = tbase + (i % C::kB) * C::kColBuf + C::kColS;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ka = ((kk >> 2) * C::kKBox + (kk & 3) * 32) >> 4;
          const uint32_t qa = ((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4;
          mma_ss(acc, desc_join(k_lo + ka, hi), desc_join(qs + qa, hi), idS, kk > 0);
        }
        tc_commit(smem_u32(&bars->s_full[i % C::kB]));
      };
      auto issue_grad = [&](int i) {  // dV += P^T_i dO_i, dK += dS^T_i Q_i; frees stage and buffer
        const int s = i % C::kNS, b = i % C::kB;
        const uint32_t qs = qmn_lo + stage_of(i);
        const uint32_t abuf = tbase + b * C::kColBuf + C::kColS;
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint32_t acol = abuf + (kk >> 1) * 32 + (kk & 1) * 8;
          const uint32_t boff = (uint32_t)(kk * 2048) >> 4;
          mma_ts(tbase + C::kColV, acol, desc_join(qs + (C::kQTile >> 4) + boff, hi), idG, kk > 0 ? 1u : acc0);
          mma_ts(tbase + C::kColK, acol + 16, desc_join(qs + boff, hi), idG, kk > 0 ? 1u : acc0);
        }
        tc_commit(smem_u32(&bars->q_empty[s]));
        tc_commit(smem_u32(&bars->pd_done[b]));
      };
      bool ok = wait(&bars->kv_full, 0);
      for (int i = 0; ok && i < n && i < C::kB; ++i) {
        ok = wait(&bars->q_full[i], 0);
        if (ok) {
          tc_fence_after();
          issue_dp(i);
          issue_s(i);
        }
      }
      for (int i = 0; ok && i < n; ++i) {
        if (!wait(&bars->pd_full[i % C::kB], (i / C::kB) & 1)) break;
        tc_fence_after();
        issue_grad(i);
        const int j = i + C::kB;
        if (j < n) {
          if (!wait(&bars->q_full[j % C::kNS], (j / C::kNS) & 1)) break;
          tc_fence_after();
          issue_dp(j);
          // S^T_j overwrites the P^T|dS^T columns that dV_i and dK_i read
          if (!wait(&bars->pd_done[i % C::kB], (i / C::kB) & 1)) break;
          tc_fence_after();
          issue_s(j);
        }
      }
      int never = 0;
      tc_commit(smem_u32(&bars->mma_done));
      mbar_wait_bounded(smem_u32(&bars->mma_done), 0, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------ P^T and dS^T
    const int half = (warp - 4) >> 2, q4 = warp & 3;
    const int row = q4 * 32 + lane;  // key within the block
    const uint32_t lane_base = (uint32_t)q4 * 32;
    const int key = q0 + row;
    // group `half` takes column half `half` of every sub-tile, or with
    // ping-pong sub-tiles half, half + 2, ..., both column halves
    constexpr int halves = pp ? 2 : 1;  // column halves per thread and sub-tile
    const int i0 = pp ? half : 0, di = pp ? 2 : 1;
    const int h0 = pp ? 0 : half;  // first column half of this thread
    // per column half: -lse log2e of its 32 columns, then -D
    float* rowbuf = reinterpret_cast<float*>(smem + C::kOffRow) + (warp - 4) * 128;
    const uint64_t sl2 = f2(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int i = i0; i < n && ok; i += di) {
      const int t0 = q0 + i * PQ;
      __syncwarp();  // the previous sub-tile's reads of rowbuf are done
#pragma unroll
      for (int hh = 0; hh < halves; ++hh) {
        const int col = (h0 + hh) * 32 + lane;  // the column this lane fetches lse and D for
        const int t = t0 + (col >> p.lgG);
        const int64_t ri = (int64_t)t * p.Hq + hk * G + (col & (G - 1));
        const bool valid = t < p.T;
        rowbuf[hh * 64 + lane] = valid ? -__ldg(p.lse + ri) * kLog2e : -INFINITY;
        rowbuf[hh * 64 + 32 + lane] = valid ? -__ldg(p.delta + ri) : 0.f;
      }
      __syncwarp();
      const uint32_t buf = (i % C::kB) * C::kColBuf;
      if (!warp_wait(smem_u32(&bars->s_full[i % C::kB]), (i / C::kB) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int hh = 0; hh < halves; ++hh) {
        const int h = h0 + hh;
        uint32_t x[32], y[32];
        tmem_ld32(tmem_addr(tbase, lane_base, buf + C::kColS + h * 32), x);
        tmem_ld32(tmem_addr(tbase, lane_base, buf + C::kColP + h * 32), y);
        tmem_ld_wait();
        // causal: column c (position t0 + c/G) sees this key iff key <= position;
        // sub-tiles at or after the block's last key need no mask
        uint32_t pk[32];
        if (t0 < q0 + BK - 1) {
          const int first = (key - t0) * G - h * 32;  // first visible local column
          pds_pack<true>(x, y, rowbuf + hh * 64, sl2, first, pk);
        } else {
          pds_pack<false>(x, y, rowbuf + hh * 64, sl2, 0, pk);
        }
        // in place over the S^T columns this thread has just read
        tmem_st32(tmem_addr(tbase, lane_base, buf + C::kColS + h * 32), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->pd_full[i % C::kB]));
    }
    // every product has completed once the issuer's final commit arrives
    // (with ping-pong the other group may still be on its last sub-tile, so
    // waiting on a pd_done phase here could look two uses ahead of the barrier)
    if (ok) ok = warp_wait(smem_u32(&bars->mma_done), 0, abort);
    if (ok) {
      tc_fence_after();
      // half 0 writes dV, half 1 writes dK (times the softmax scale)
      const uint32_t c0 = half ? C::kColK : C::kColV;
      const float mul = half ? p.scale : 1.f;
      float* out = (half ? p.dk : p.dv) + ((int64_t)key * p.Hk + hk) * D;
      const bool valid = key < p.T;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tbase, lane_base, c0 + c * 32), r);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(out + c * 32 + e) =
                make_float4(__uint_as_float(r[e]) * mul, __uint_as_float(r[e + 1]) * mul,
                            __uint_as_float(r[e + 2]) * mul, __uint_as_float(r[e + 3]) * mul);
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
  using C = KvCfg<D>;
  const int lgG = __builtin_ctz((unsigned)a.G);
  const int PQ = BQ >> lgG;
  const int nk = (a.T + BK - 1) / BK;
  CUtensorMap tq, to, tk, tv;
  const uint64_t row = (uint64_t)D * 2;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)a.T};
    const uint64_t str[2] = {row, row * a.Hq};
    const uint32_t box[3] = {64, (uint32_t)a.G, (uint32_t)PQ};
    if (encode_bf16_sw128(&tq, a.q, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&to, a.dO, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hk, (uint64_t)a.T};
    const uint64_t str[2] = {row, row * a.Hk};
    const uint32_t box[3] = {64, 1, BK};
    if (encode_bf16_sw128(&tk, a.k, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tv, a.v, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  KvParams prm;
  prm.T = a.T; prm.Hq = a.Hq; prm.Hk = a.Hk; prm.lgG = lgG;
  prm.scale_log2 = a.scale * kLog2e;
  prm.scale = a.scale;
  prm.lse = a.lse;
  prm.delta = a.delta;
  prm.dk = a.dk;
  prm.dv = a.dv;
  prm.err = a.err;
  // Ping-pong always at d = 64; at d = 128 it pays once blocks see thousands
  // of sub-tiles (measured: 2-4 % faster at T = 32768 and 65536, 2-4 % slower
  // at T <= 16384).
  auto kern = bwd_dkdv_tc_kernel<D, true>;
  if constexpr (D == 128) {
    if (a.T < 32768) kern = bwd_dkdv_tc_kernel<D, false>;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)((int64_t)nk * a.Hk), kThreads, C::kSmemBytes, stream>>>(tq, to, tk, tv, prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_tc(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

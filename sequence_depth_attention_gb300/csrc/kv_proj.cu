// Depth K/V of an FFN layer, written straight into its slot of the packed
// depth streams (tcgen05 GEMM with a slot-scatter epilogue, sm_103a).
//
//   K[t, hk*d + j] = sum_c x[t, c] wk[hk*d + j, c],  V likewise with wv,
//   kd[hk, t, slot, j] = bf16(K[t, hk*d + j]),  vd[hk, t, slot, j] = bf16(V[...])
//
// An FFN layer's depth pair is a light KV projection of the FFN's input
// (reading notes Sec. 二.3; summary Sec. 2.2, the "write" step). Writing it in
// the GEMM's epilogue means the pair never exists outside the packed stream.
//
// One tile = 128 positions x one KV head: the B tile stacks that head's d rows
// of wk over its d rows of wv, so one MMA of N = 2d yields K and V side by side
// in TMEM. Persistent CTAs (one per SM) walk tiles id = blockIdx.x + i*gridDim.x
// with the KV heads of one row block adjacent, so the Hk CTAs that share an x
// row block run together and x is read from HBM about once.
// Roles (8 warps): warp 0 TMA (x box 64 x 128, wk and wv boxes 64 x d) into an
// NS-stage ring; warp 1 issues the MMAs; warps 4-7 drain the accumulator
// (thread = row = TMEM lane), round to bf16 and store 16-byte vectors. The
// accumulator is double-buffered in TMEM so the epilogue of tile i overlaps
// the MMAs of tile i+1. All waits are bounded; on expiry the CTA drains and
// latches MODA_ERR_TIMEOUT.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "tensor_map.h"

namespace moda {
namespace {

using namespace sm103;

constexpr int BM = 128;
constexpr int kThreads = 256;
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D>
struct ProjCfg {
  static constexpr int kN = 2 * D;           // K and V columns of one head
  static constexpr int kABytes = BM * 128;   // 128 rows x 64 bf16
  static constexpr int kBBytes = kN * 128;   // 2d rows x 64 bf16
  static constexpr int kStage = kABytes + kBBytes;
  static constexpr int kNS = D == 128 ? 4 : 6;
  static constexpr int kOffBar = kNS * kStage;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr uint32_t kTmemCols = 2 * kN < 32 ? 32 : 2 * kN;  // two accumulators
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct alignas(8) ProjBars {
  uint64_t full[6], empty[6];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(ProjBars) <= 256, "barrier block");

struct ProjParams {
  int T, Dm, Hk, L, slot, ntiles;
  __nv_bfloat16* kd;
  __nv_bfloat16* vd;
  unsigned int* err;
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort, kTimeoutNs);
  return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
kv_proj_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWk,
               const __grid_constant__ CUtensorMap tmWv, const ProjParams p) {
  using C = ProjCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  ProjBars* bars = reinterpret_cast<ProjBars*>(smem + C::kOffBar);
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nk = p.Dm / 64;

  if (tid == 0) {
    bars->abort = 0;
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(smem_u32(&bars->full[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars->acc_full[b]), 1);
      mbar_init(smem_u32(&bars->acc_empty[b]), 128);
    }
    mbar_init(smem_u32(&bars->mma_done), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmWk);
    tma_prefetch_desc(&tmWv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    const bool leader = elect_one();
    int it = 0;
    bool ok = true;
    for (int id = blockIdx.x; ok && id < p.ntiles; id += gridDim.x) {
      const int mt = id / p.Hk, hk = id % p.Hk;
      for (int kc = 0; kc < nk; ++kc, ++it) {
        const int s = it % C::kNS;
        if (!warp_wait(smem_u32(&bars->empty[s]), ((it / C::kNS) & 1) ^ 1, abort)) {
          ok = false;
          break;
        }
        if (leader) {
          const uint32_t fb = smem_u32(&bars->full[s]);
          const uint32_t a = sbase + s * C::kStage, b = a + C::kABytes;
          mbar_arrive_expect_tx(fb, C::kStage);
          tma_load_2d(a, &tmX, fb, kc * 64, mt * BM);
          tma_load_2d(b, &tmWk, fb, kc * 64, hk * D);
          tma_load_2d(b + D * 128, &tmWv, fb, kc * 64, hk * D);
        }
        __syncwarp();
      }
    }
    if (leader) {  // wait for the copies still in flight before the CTA exits
      int never = 0;
      for (int j = max(0, it - C::kNS); j < it; ++j)
        mbar_wait_bounded(smem_u32(&bars->full[j % C::kNS]), (j / C::kNS) & 1, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_bf16_f32(BM, C::kN, false);
    const uint64_t d0 = sdesc_sw128(sbase, 16, 1024);
    int it = 0, i = 0;
    bool ok = true;
    for (int id = blockIdx.x; ok && id < p.ntiles; id += gridDim.x, ++i) {
      const int b = i & 1;
      if (!warp_wait(smem_u32(&bars->acc_empty[b]), ((i >> 1) & 1) ^ 1, abort)) break;
      tc_fence_after();
      const uint32_t acc = tbase + b * C::kN;
      for (int kc = 0; kc < nk; ++kc, ++it) {
        const int s = it % C::kNS;
        if (!warp_wait(smem_u32(&bars->full[s]), (it / C::kNS) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) {
          const uint64_t da = d0 + (uint64_t)((s * C::kStage) >> 4);
          const uint64_t db = da + (uint64_t)(C::kABytes >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(acc, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc, (kc | kk) != 0);
          tc_commit(smem_u32(&bars->empty[s]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) tc_commit(smem_u32(&bars->acc_full[b]));
      __syncwarp();
    }
    if (leader) {
      int never = 0;
      tc_commit(smem_u32(&bars->mma_done));
      mbar_wait_bounded(smem_u32(&bars->mma_done), 0, &never, kTimeoutNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------ epilogue
    const uint32_t lane_base = (uint32_t)(warp & 3) * 32;
    const int row = (warp & 3) * 32 + lane;
    int i = 0;
    for (int id = blockIdx.x; id < p.ntiles; id += gridDim.x, ++i) {
      const int b = i & 1;
      if (!warp_wait(smem_u32(&bars->acc_full[b]), (i >> 1) & 1, abort)) break;
      tc_fence_after();
      const int mt = id / p.Hk, hk = id % p.Hk;
      const int t = mt * BM + row;
      const bool valid = t < p.T;
      const int64_t off = (((int64_t)hk * p.T + (valid ? t : 0)) * p.L + p.slot) * D;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4* dst = reinterpret_cast<uint4*>((half ? p.vd : p.kd) + off);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tbase, lane_base, b * C::kN + half * D + c * 32), r);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->acc_empty[b]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
  if (tid == 0 && bars->abort) atomicCAS(p.err, 0u, (unsigned int)MODA_ERR_TIMEOUT);
}

template <int D>
cudaError_t launch_d(const KvProjArgs& a, cudaStream_t stream) {
  using C = ProjCfg<D>;
  CUtensorMap tx, twk, twv;
  {
    const uint64_t dims[2] = {(uint64_t)a.Dm, (uint64_t)a.T};
    const uint64_t str[1] = {(uint64_t)a.Dm * 2};
    const uint32_t box[2] = {64, BM};
    if (encode_bf16_sw128(&tx, a.x, 2, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)a.Dm, (uint64_t)a.Hk * D};
    const uint64_t str[1] = {(uint64_t)a.Dm * 2};
    const uint32_t box[2] = {64, (uint32_t)D};
    if (encode_bf16_sw128(&twk, a.wk, 2, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&twv, a.wv, 2, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  ProjParams prm;
  prm.T = a.T; prm.Dm = a.Dm; prm.Hk = a.Hk; prm.L = a.L; prm.slot = a.slot;
  prm.ntiles = ((a.T + BM - 1) / BM) * a.Hk;
  prm.kd = static_cast<__nv_bfloat16*>(a.kd);
  prm.vd = static_cast<__nv_bfloat16*>(a.vd);
  prm.err = a.err;
  cudaError_t e = cudaFuncSetAttribute(kv_proj_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = prm.ntiles < a.num_sms ? prm.ntiles : a.num_sms;
  kv_proj_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(tx, twk, twv, prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_proj(const KvProjArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

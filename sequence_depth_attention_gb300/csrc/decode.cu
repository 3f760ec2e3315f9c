// MoDA decode: one new token at position t = Tctx-1 attends, under one
// softmax, to the whole sequence KV cache (positions 0..t, its own K/V
// included) and to the L depth slots of position t (Mixture-of-Depths
// Attention, Sec. 2.2; the decode-time depth cache of Table 1 is these L
// slots of the current token).
//
// HBM-bound: every cached K/V row is read once and used by the G query heads
// of its KV head (about G flop per byte), so the work runs on CUDA cores.
//   pass 1  grid (nsplit + 1, Hk): CTA (s, hk) walks a contiguous chunk of the
//           cache (the last CTA the depth slots) for the G heads of hk with
//           an online softmax; TMA streams 64-key K and V boxes through a
//           3-stage shared-memory ring while 8 warps (lanes split d) consume.
//           Each writes a partial (m, l, unnormalised o) to the workspace.
//   pass 2  grid Hq: merge the nsplit + 1 partials of each head, o = O / l.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "tensor_map.h"

namespace moda {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// A lane's E = D/32 consecutive bf16 of a row, loaded in one access.
template <int E> struct LaneRow;
template <> struct LaneRow<4> {
  using T = uint2;
  __device__ static void unpack(const T& r, float* f) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
};
template <> struct LaneRow<2> {
  using T = uint32_t;
  __device__ static void unpack(const T& r, float* f) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r));
    f[0] = a.x; f[1] = a.y;
  }
};

// Keys of the CTA stream through a ring of kStages shared-memory stages of
// kKB keys (K and V), filled by TMA (one elected thread) and tracked by
// mbarriers, so kStages*kKB*d*4 bytes are in flight per CTA while its 8
// warps work on the oldest stage: warp w takes keys w*kU .. w*kU+kU-1 of a
// stage, lanes split d. A block-wide vote releases a stage, so a bounded
// wait that gives up ends every thread of the CTA together.
constexpr int kW = 8;       // warps
constexpr int kKB = 64;     // keys per stage
constexpr int kU = kKB / kW;
constexpr int kStages = 3;
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D, int G>
struct DecodeSmem {
  union {
    __nv_bfloat16 kv[kStages][2][kKB][D];  // [stage][K or V][key][d] while streaming
    struct {                                // the warps' states for the final merge
      float o[kW][G][D];
      float ml[kW][G][2];
    } merge;
  } u;
  uint64_t full[kStages];
  int abort;
};

template <int D, int G>
__global__ void __launch_bounds__(kW * 32)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmKd, const __grid_constant__ CUtensorMap tmVd,
                    const __nv_bfloat16* __restrict__ q, int Tctx, int Hq, int L,
                    int keys_per_split, int nsplit, float scale_log2, float* __restrict__ part,
                    unsigned int* __restrict__ err) {
  constexpr int E = D / 32;  // columns per lane
  using Row = LaneRow<E>;
  using RowT = typename Row::T;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // TMA destinations need 128-byte alignment: align the base explicitly
  DecodeSmem<D, G>& sm = *reinterpret_cast<DecodeSmem<D, G>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const int split = blockIdx.x, hk = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool depth = split == nsplit;
  const int j0 = depth ? 0 : split * keys_per_split;
  const int j1 = depth ? L : min(Tctx, j0 + keys_per_split);
  const int nblk = (j1 - j0 + kKB - 1) / kKB;
  constexpr uint32_t kStageBytes = 2u * kKB * D * 2u;

  if (tid == 0) {
    sm.abort = 0;
    for (int s = 0; s < kStages; ++s) sm103::mbar_init(sm103::smem_u32(&sm.full[s]), 1);
    sm103::fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int b) {  // block b -> stage b % kStages
    const int s = b % kStages;
    const uint32_t bar = sm103::smem_u32(&sm.full[s]);
    sm103::mbar_arrive_expect_tx(bar, kStageBytes);
    const uint32_t dk = sm103::smem_u32(&sm.u.kv[s][0][0][0]);
    const uint32_t dv = sm103::smem_u32(&sm.u.kv[s][1][0][0]);
    const int jb = j0 + b * kKB;
    if (depth) {
      sm103::tma_load_3d(dk, &tmKd, bar, 0, jb, hk);
      sm103::tma_load_3d(dv, &tmVd, bar, 0, jb, hk);
    } else {
      sm103::tma_load_3d(dk, &tmK, bar, 0, hk, jb);
      sm103::tma_load_3d(dv, &tmV, bar, 0, hk, jb);
    }
  };
  if (tid == 0)
    for (int b = 0; b < min(kStages, nblk); ++b) issue(b);

  float qv[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float f[E];
    Row::unpack(*reinterpret_cast<const RowT*>(q + (int64_t)(hk * G + g) * D + lane * E), f);
#pragma unroll
    for (int e = 0; e < E; ++e) qv[g][e] = f[e] * scale_log2;  // fold the scale into q
  }
  float m[G], l[G], o[G][E];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[g][e] = 0.f;
  }
  int issued = min(kStages, nblk);
  for (int b = 0; b < nblk; ++b) {
    const int s = b % kStages;
    bool ok = sm103::mbar_wait_bounded(sm103::smem_u32(&sm.full[s]), (b / kStages) & 1,
                                       &sm.abort, kTimeoutNs);
    if (!__syncthreads_and(ok)) break;
    const int jb = j0 + b * kKB + warp * kU;  // this warp's first key
    float s_[G][kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float kf[E];
      Row::unpack(*reinterpret_cast<const RowT*>(&sm.u.kv[s][0][warp * kU + u][lane * E]), kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc = fmaf(qv[g][e], kf[e], acc);
        s_[g][u] = acc;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int u = 0; u < kU; ++u) s_[g][u] += __shfl_xor_sync(0xffffffffu, s_[g][u], off);
    if (jb < j1) {  // the warp holds at least one valid key
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (jb + u >= j1)
#pragma unroll
          for (int g = 0; g < G; ++g) s_[g][u] = -INFINITY;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mx = s_[g][0];
#pragma unroll
        for (int u = 1; u < kU; ++u) mx = fmaxf(mx, s_[g][u]);
        const float mn = fmaxf(m[g], mx);
        const float alpha = exp2f(m[g] - mn);
        l[g] *= alpha;
#pragma unroll
        for (int e = 0; e < E; ++e) o[g][e] *= alpha;
        m[g] = mn;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        float vf[E];
        Row::unpack(*reinterpret_cast<const RowT*>(&sm.u.kv[s][1][warp * kU + u][lane * E]), vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = exp2f(s_[g][u] - m[g]);
          l[g] += p;
#pragma unroll
          for (int e = 0; e < E; ++e) o[g][e] = fmaf(p, vf[e], o[g][e]);
        }
      }
    }
    __syncthreads();  // stage s is free
    if (tid == 0 && issued < nblk) {
      issue(issued);
      ++issued;
    }
  }
  // in-flight copies land before the CTA exits (only after an abort)
  if (tid == 0) {
    int never = 0;
    for (int b = max(0, issued - kStages); b < issued; ++b)
      sm103::mbar_wait_bounded(sm103::smem_u32(&sm.full[b % kStages]), (b / kStages) & 1, &never,
                               kTimeoutNs);
    if (sm.abort) atomicCAS(err, 0u, (unsigned int)MODA_ERR_TIMEOUT);
  }
  // merge the warps of the CTA (the ring is idle now: every copy has landed)
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int e = 0; e < E; ++e) sm.u.merge.o[warp][g][lane * E + e] = o[g][e];
    if (lane == 0) {
      sm.u.merge.ml[warp][g][0] = m[g];
      sm.u.merge.ml[warp][g][1] = l[g];
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kW * 32) {
    const int g = idx / D, c = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW; ++w) M = fmaxf(M, sm.u.merge.ml[w][g][0]);
    float oo = 0.f, ll = 0.f;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const float a = M == -INFINITY ? 0.f : exp2f(sm.u.merge.ml[w][g][0] - M);
      oo = fmaf(a, sm.u.merge.o[w][g][c], oo);
      ll = fmaf(a, sm.u.merge.ml[w][g][1], ll);
    }
    float* pr = part + ((int64_t)split * Hq + hk * G + g) * (D + 2);
    pr[c] = oo;
    if (c == 0) {
      pr[D] = M;
      pr[D + 1] = ll;
    }
  }
}

// One CTA per query head: 8 warps take the partials round-robin (each lane
// its D/32 columns). Every warp loads all of its partials before merging any,
// so the loads overlap instead of costing one latency each.
constexpr int kCombineWarps = 8;
constexpr int kMaxParts = 129;  // nsplit <= 128, plus the depth partial
constexpr int kPartsPerWarp = (kMaxParts + kCombineWarps - 1) / kCombineWarps;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
decode_combine_kernel(const float* __restrict__ part, int nparts, int Hq,
                      __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  constexpr int E = D / 32;
  __shared__ float sm_o[kCombineWarps][D];
  __shared__ float sm_ml[kCombineWarps][2];
  const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float pm[kPartsPerWarp], pl[kPartsPerWarp], po[kPartsPerWarp][E];
#pragma unroll
  for (int i = 0; i < kPartsPerWarp; ++i) {
    const int s = warp + i * kCombineWarps;
    if (s < nparts) {
      const float* pr = part + ((int64_t)s * Hq + h) * (D + 2);
      pm[i] = pr[D];
      pl[i] = pr[D + 1];
#pragma unroll
      for (int e = 0; e < E; ++e) po[i][e] = pr[lane * E + e];
    } else {
      pm[i] = -INFINITY;
      pl[i] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) po[i][e] = 0.f;
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPartsPerWarp; ++i) M = fmaxf(M, pm[i]);
  float ll = 0.f, oo[E];
#pragma unroll
  for (int e = 0; e < E; ++e) oo[e] = 0.f;
#pragma unroll
  for (int i = 0; i < kPartsPerWarp; ++i) {
    const float a = pm[i] == -INFINITY ? 0.f : exp2f(pm[i] - M);  // empty partials weigh 0
    ll = fmaf(a, pl[i], ll);
#pragma unroll
    for (int e = 0; e < E; ++e) oo[e] = fmaf(a, po[i][e], oo[e]);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) sm_o[warp][lane * E + e] = oo[e];
  if (lane == 0) {
    sm_ml[warp][0] = M;
    sm_ml[warp][1] = ll;
  }
  __syncthreads();
  if (warp == 0) {
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) Mt = fmaxf(Mt, sm_ml[w][0]);
    float lt = 0.f, ot[E];
#pragma unroll
    for (int e = 0; e < E; ++e) ot[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      const float a = sm_ml[w][0] == -INFINITY ? 0.f : exp2f(sm_ml[w][0] - Mt);
      lt = fmaf(a, sm_ml[w][1], lt);
#pragma unroll
      for (int e = 0; e < E; ++e) ot[e] = fmaf(a, sm_o[w][lane * E + e], ot[e]);
    }
    const float inv = 1.f / lt;
#pragma unroll
    for (int e = 0; e < E; ++e) o[(int64_t)h * D + lane * E + e] = __float2bfloat16_rn(ot[e] * inv);
    if (lane == 0 && lse) lse[h] = (Mt + log2f(lt)) * kLn2;
  }
}

template <int D, int G>
cudaError_t launch_split(const DecodeArgs& a, int nsplit, int kps, cudaStream_t st) {
  // cache as [Tctx][Hk][D]: dims (D, Hk, Tctx); depth as [Hk] blocks of [L][D]
  CUtensorMap tk, tv, tkd, tvd;
  const uint64_t row = (uint64_t)D * 2;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.Hk, (uint64_t)a.Tctx};
    const uint64_t str[2] = {row, row * a.Hk};
    const uint32_t box[3] = {D, 1, kKB};
    if (encode_bf16_plain(&tk, a.k, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_plain(&tv, a.v, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  if (a.L > 0) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.L, (uint64_t)a.Hk};
    const uint64_t str[2] = {row, (uint64_t)a.depth_hk_stride * 2};
    const uint32_t box[3] = {D, kKB, 1};
    if (encode_bf16_plain(&tkd, a.kd, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_plain(&tvd, a.vd, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else {
    tkd = tk;  // never read when L == 0
    tvd = tv;
  }
  const size_t smem = sizeof(DecodeSmem<D, G>) + 128;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_split_kernel<D, G><<<dim3(nsplit + 1, a.Hk), kW * 32, smem, st>>>(
      tk, tv, tkd, tvd, (const __nv_bfloat16*)a.q, a.Tctx, a.Hq, a.L, kps, nsplit,
      a.scale * kLog2e, a.work, a.err);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t st) {
  // about one wave of long-lived CTAs (2 per SM) so each streams many stages
  int nsplit = (2 * (a.num_sms > 0 ? a.num_sms : 148)) / a.Hk - 1;
  nsplit = nsplit < 1 ? 1 : nsplit;
  nsplit = nsplit < decode_num_splits(a.Tctx) ? nsplit : decode_num_splits(a.Tctx);
  // keys per split: a multiple of the stage size
  const int kps = ((a.Tctx + nsplit - 1) / nsplit + kKB - 1) / kKB * kKB;
  cudaError_t e;
  switch (a.G) {
    case 1: e = launch_split<D, 1>(a, nsplit, kps, st); break;
    case 2: e = launch_split<D, 2>(a, nsplit, kps, st); break;
    case 4: e = launch_split<D, 4>(a, nsplit, kps, st); break;
    case 8: e = launch_split<D, 8>(a, nsplit, kps, st); break;
    default: e = launch_split<D, 16>(a, nsplit, kps, st); break;
  }
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D><<<a.Hq, kCombineWarps * 32, 0, st>>>(a.work, nsplit + 1, a.Hq,
                                                                (__nv_bfloat16*)a.o, a.lse);
  return cudaGetLastError();
}

}  // namespace

// Upper bound on the sequence splits: at least 64 keys (one stage) each, at
// most 128. The workspace is sized for it; launches may use fewer.
int decode_num_splits(int Tctx) {
  const int n = (Tctx + 63) / 64;
  return n < 1 ? 1 : (n > 128 ? 128 : n);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_d<128>(a, stream) : launch_d<64>(a, stream);
}

}  // namespace moda

// MoDA decode: one new token at position t = Tctx-1 attends, under one
// softmax, to the whole sequence KV cache (positions 0..t, its own K/V
// included) and to the L depth slots of position t (Mixture-of-Depths
// Attention, Sec. 2.2; the decode-time depth cache of Table 1 is these L
// slots of the current token).
//
// HBM-bound: every cached K/V row is read once and used by the G query heads
// of its KV head (about G flop per byte).
//   pass 1  grid (nsplit + 1, Hk): CTA (s, hk) walks a contiguous chunk of the
//           cache (the last CTA the depth slots) for the G heads of hk with
//           an online softmax; TMA streams 64-key K and V boxes (128-byte
//           swizzle) through a shared-memory ring while 4 warps score 16 keys
//           each on mma.sync tensor cores. For G <= 8 the products are
//           transposed (S^T = K Q^T with the keys as the A rows and the G
//           heads as one 8-column B tile, then O^T += V^T P^T), which takes
//           half the MMAs of the G heads padded to 16 A rows; G = 16 fills
//           those rows (S = Q K^T, O += P V). Neither needs a cross-lane
//           reduction for the dot products.
//           Each CTA writes a partial (m, l, unnormalised o) to the workspace.
//   pass 2  grid Hq: merge the nsplit + 1 partials of each head, o = O / l.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "tensor_map.h"
#include "warp_mma.cuh"

namespace moda {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Keys of the CTA stream through a ring of NS shared-memory stages of kKB
// keys (K and V), filled by TMA with the 128-byte swizzle (one elected thread)
// and tracked by mbarriers. Warp w scores keys 16w .. 16w+15 of a stage on the
// tensor cores (mma.sync m16n8k16): S = Q K^T with the G query heads of the
// KV head as the rows of the A operand (rows >= G are zero) and K read by
// ldmatrix, then an online softmax per row, then O += P V with P reused in
// registers as the A operand and V read by ldmatrix.trans. A block-wide vote
// releases a stage, so a bounded wait that gives up ends every thread of the
// CTA together.
constexpr int kW = 4;        // warps
constexpr int kKB = 64;      // keys per stage
constexpr int kKW = kKB / kW;  // keys per warp and stage (one k16 step of P V)
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D>
struct DecodeSmem {
  static constexpr int kNS = D == 128 ? 3 : 4;    // stages
  static constexpr int kBox = kKB * 128;          // one 64-column swizzled box of kKB rows
  static constexpr int kTile = (D / 64) * kBox;   // K or V of one stage
  union {
    uint8_t ring[kNS][2][kTile];  // [stage][K or V]
    struct {                      // the warps' states for the final merge
      float o[kW][16][D];
      float ml[kW][16][2];
    } merge;
  } u;
  uint64_t full[kNS];
  int abort;
};

// Byte offset of element (row, col) in a stage tile: 64-column boxes, 16-byte
// chunks XOR-swizzled by (row & 7) inside each 1024-byte atom, the layout TMA
// writes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz128(int row, int col) {
  return (uint32_t)((col >> 6) * (kKB * 128) + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                    ((col & 7) << 1));
}

template <int D, int G>
__global__ void __launch_bounds__(kW * 32)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmKd, const __grid_constant__ CUtensorMap tmVd,
                    const __nv_bfloat16* __restrict__ q, int Tctx, int Hq, int L,
                    int keys_per_split, int nsplit, float scale_log2, float* __restrict__ part,
                    unsigned int* __restrict__ err) {
  using S = DecodeSmem<D>;
  constexpr int NS = S::kNS;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // 128-byte swizzled TMA destinations need 1024-byte alignment
  S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                ~static_cast<uintptr_t>(1023));
  const int split = blockIdx.x, hk = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool depth = split == nsplit;
  const int j0 = depth ? 0 : split * keys_per_split;
  const int j1 = depth ? L : min(Tctx, j0 + keys_per_split);
  const int nblk = (j1 - j0 + kKB - 1) / kKB;
  constexpr uint32_t kStageBytes = 2u * S::kTile;

  if (tid == 0) {
    sm.abort = 0;
    for (int s = 0; s < NS; ++s) sm103::mbar_init(sm103::smem_u32(&sm.full[s]), 1);
    sm103::fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int b) {  // block b -> stage b % NS
    const int s = b % NS;
    const uint32_t bar = sm103::smem_u32(&sm.full[s]);
    sm103::mbar_arrive_expect_tx(bar, kStageBytes);
    const int jb = j0 + b * kKB;
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      const uint32_t dk = sm103::smem_u32(&sm.u.ring[s][0][c * S::kBox]);
      const uint32_t dv = sm103::smem_u32(&sm.u.ring[s][1][c * S::kBox]);
      if (depth) {
        sm103::tma_load_3d(dk, &tmKd, bar, c * 64, jb, hk);
        sm103::tma_load_3d(dv, &tmVd, bar, c * 64, jb, hk);
      } else {
        sm103::tma_load_3d(dk, &tmK, bar, c * 64, hk, jb);
        sm103::tma_load_3d(dv, &tmV, bar, c * 64, hk, jb);
      }
    }
  };
  if (tid == 0)
    for (int b = 0; b < min(NS, nblk); ++b) issue(b);
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if constexpr (G <= 8) {
    // G <= 8: the transposed products, half the MMAs of the G rows padded to
    // 16: S^T = K Q^T (the warp's 16 keys as the rows of the A tile, the G
    // heads as the 8 columns of the B tile) and O^T += V^T P^T (the head
    // dimension in 16-row A tiles of V read transposed, P^T as the B tile).
    // This lane's heads are hq and hq + 1; its rows are key (or dimension)
    // r0 and r0 + 8 of a tile.
    const int r0 = lane >> 2, hq = (lane & 3) * 2;
    uint32_t qb[D / 16][2];  // B = Q^T: k = the head dimension, n = the head
    {
      auto ld = [&](int h, int c) -> uint32_t {
        return h < G ? *reinterpret_cast<const uint32_t*>(q + (int64_t)(hk * G + h) * D + c) : 0u;
      };
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qb[ks][0] = ld(r0, ks * 16 + hq);
        qb[ks][1] = ld(r0, ks * 16 + 8 + hq);
      }
    }
    float o[D / 16][4];  // O^T: rows = dimension, columns = heads hq, hq + 1
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY;  // heads hq, hq + 1, log2 units
    float la = 0.f, lb = 0.f;              // this lane's share of their sums
    const int lr = lane & 7, lm = lane >> 3;
    // ldmatrix rows of this lane: K (x4: key halves x dimension halves of one
    // k16 step), V (x4.trans: dimension halves x key halves of a 16-row tile)
    const int kkey = warp * kKW + (lm & 1) * 8 + lr, kcol = (lm >> 1) * 8;
    const int vkey = warp * kKW + (lm >> 1) * 8 + lr, vcol = (lm & 1) * 8;

    int issued = min(NS, nblk);
    for (int b = 0; b < nblk; ++b) {
      const int s = b % NS;
      bool ok = sm103::mbar_wait_bounded(sm103::smem_u32(&sm.full[s]), (b / NS) & 1, &sm.abort,
                                         kTimeoutNs);
      if (!__syncthreads_and(ok)) break;
      const int jw = j0 + b * kKB + warp * kKW;  // this warp's first key
      if (jw < j1) {
        const uint32_t kb = sm103::smem_u32(&sm.u.ring[s][0][0]);
        const uint32_t vb = sm103::smem_u32(&sm.u.ring[s][1][0]);
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t a[4];
          wmma16::ldsm_x4(kb + swz128(kkey, ks * 16 + kcol), a[0], a[1], a[2], a[3]);
          wmma16::mma_bf16(c, a, qb[ks][0], qb[ks][1]);
        }
        // scores in log2 units; keys at or past j1 do not exist
        const bool k0 = jw + r0 < j1, k1 = jw + r0 + 8 < j1;
        const float s0 = k0 ? c[0] * scale_log2 : -INFINITY, s1 = k0 ? c[1] * scale_log2 : -INFINITY;
        const float s2 = k1 ? c[2] * scale_log2 : -INFINITY, s3 = k1 ? c[3] * scale_log2 : -INFINITY;
        float xa = fmaxf(s0, s2), xb = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, off));
          xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, off));
        }
        const float na = fmaxf(ma, xa), nb = fmaxf(mb, xb);
        const float refa = na == -INFINITY ? 0.f : na, refb = nb == -INFINITY ? 0.f : nb;
        const float aa = exp2f(ma - refa), ab = exp2f(mb - refb);
        ma = na;
        mb = nb;
        const float p0 = exp2f(s0 - refa), p1 = exp2f(s1 - refb);
        const float p2 = exp2f(s2 - refa), p3 = exp2f(s3 - refb);
        la = la * aa + (p0 + p2);
        lb = lb * ab + (p1 + p3);
        // P^T (rows = keys, columns = heads) transposed into the B tile
        const uint32_t pb0 = wmma16::movmatrix_t(wmma16::pack_bf16(p0, p1));
        const uint32_t pb1 = wmma16::movmatrix_t(wmma16::pack_bf16(p2, p3));
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          uint32_t a[4];
          wmma16::ldsm_x4_t(vb + swz128(vkey, mt * 16 + vcol), a[0], a[1], a[2], a[3]);
          o[mt][0] *= aa; o[mt][1] *= ab; o[mt][2] *= aa; o[mt][3] *= ab;
          wmma16::mma_bf16(o[mt], a, pb0, pb1);
        }
      }
      __syncthreads();  // stage s is free
      if (tid == 0 && issued < nblk) {
        issue(issued);
        ++issued;
      }
    }
    // in-flight copies land before the ring is reused or the CTA exits
    if (tid == 0) {
      int never = 0;
      for (int b = max(0, issued - NS); b < issued; ++b)
        sm103::mbar_wait_bounded(sm103::smem_u32(&sm.full[b % NS]), (b / NS) & 1, &never, kTimeoutNs);
      if (sm.abort) atomicCAS(err, 0u, (unsigned int)MODA_ERR_TIMEOUT);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, off);
      lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    __syncthreads();
    // merge the warps of the CTA through shared memory (the ring is idle now)
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      sm.u.merge.o[warp][hq][mt * 16 + r0] = o[mt][0];
      sm.u.merge.o[warp][hq + 1][mt * 16 + r0] = o[mt][1];
      sm.u.merge.o[warp][hq][mt * 16 + r0 + 8] = o[mt][2];
      sm.u.merge.o[warp][hq + 1][mt * 16 + r0 + 8] = o[mt][3];
    }
    if (r0 == 0) {
      sm.u.merge.ml[warp][hq][0] = ma;
      sm.u.merge.ml[warp][hq][1] = la;
      sm.u.merge.ml[warp][hq + 1][0] = mb;
      sm.u.merge.ml[warp][hq + 1][1] = lb;
    }
    __syncthreads();
  } else {
    // Q as the A operand (row r = query head hk*G + r, k = the head dimension)
    const int r0 = lane >> 2, cq = (lane & 3) * 2;
    uint32_t qa[D / 16][4];
    {
      auto ld = [&](int r, int c) -> uint32_t {
        return r < G ? *reinterpret_cast<const uint32_t*>(q + (int64_t)(hk * G + r) * D + c) : 0u;
      };
  #pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = ld(r0, ks * 16 + cq);
        qa[ks][1] = ld(r0 + 8, ks * 16 + cq);
        qa[ks][2] = ld(r0, ks * 16 + 8 + cq);
        qa[ks][3] = ld(r0 + 8, ks * 16 + 8 + cq);
      }
    }
    float o[D / 8][4];
  #pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // rows r0 and r0 + 8, log2 units
    float l0 = 0.f, l1 = 0.f;              // this lane's share of the row sums

    // ldmatrix source rows of this lane: K (x4 = key halves x dimension halves
    // of one k16 step), V (x4.trans = key halves x two 8-column groups)
    const int kkey = warp * kKW + ((lane >> 4) << 3) + (lane & 7), kcol = ((lane >> 3) & 1) * 8;
    const int vkey = warp * kKW + (((lane >> 3) & 1) << 3) + (lane & 7), vcol = (lane >> 4) * 8;

    int issued = min(NS, nblk);
    for (int b = 0; b < nblk; ++b) {
      const int s = b % NS;
      bool ok = sm103::mbar_wait_bounded(sm103::smem_u32(&sm.full[s]), (b / NS) & 1, &sm.abort,
                                         kTimeoutNs);
      if (!__syncthreads_and(ok)) break;
      const int jw = j0 + b * kKB + warp * kKW;  // this warp's first key
      if (jw < j1) {
        const uint32_t kb = sm103::smem_u32(&sm.u.ring[s][0][0]);
        const uint32_t vb = sm103::smem_u32(&sm.u.ring[s][1][0]);
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  #pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b00, b01, b10, b11;
          wmma16::ldsm_x4(kb + swz128(kkey, ks * 16 + kcol), b00, b01, b10, b11);
          wmma16::mma_bf16(c[0], qa[ks], b00, b01);
          wmma16::mma_bf16(c[1], qa[ks], b10, b11);
        }
        // scores in log2 units; keys at or past j1 do not exist
        float sv[2][4];
  #pragma unroll
        for (int nt = 0; nt < 2; ++nt)
  #pragma unroll
          for (int e = 0; e < 4; ++e)
            sv[nt][e] = jw + nt * 8 + cq + (e & 1) < j1 ? c[nt][e] * scale_log2 : -INFINITY;
        float mx0 = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
        float mx1 = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float ref0 = n0 == -INFINITY ? 0.f : n0, ref1 = n1 == -INFINITY ? 0.f : n1;
        const float a0 = exp2f(m0 - ref0), a1 = exp2f(m1 - ref1);
        m0 = n0;
        m1 = n1;
        float p[2][4];
  #pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          p[nt][0] = exp2f(sv[nt][0] - ref0);
          p[nt][1] = exp2f(sv[nt][1] - ref0);
          p[nt][2] = exp2f(sv[nt][2] - ref1);
          p[nt][3] = exp2f(sv[nt][3] - ref1);
        }
        l0 = l0 * a0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        l1 = l1 * a1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
        uint32_t pa[4];
        pa[0] = wmma16::pack_bf16(p[0][0], p[0][1]);
        pa[1] = wmma16::pack_bf16(p[0][2], p[0][3]);
        pa[2] = wmma16::pack_bf16(p[1][0], p[1][1]);
        pa[3] = wmma16::pack_bf16(p[1][2], p[1][3]);
  #pragma unroll
        for (int nd = 0; nd < D / 8; nd += 2) {
          uint32_t v0, v1, v2, v3;
          wmma16::ldsm_x4_t(vb + swz128(vkey, nd * 8 + vcol), v0, v1, v2, v3);
          o[nd][0] *= a0; o[nd][1] *= a0; o[nd][2] *= a1; o[nd][3] *= a1;
          o[nd + 1][0] *= a0; o[nd + 1][1] *= a0; o[nd + 1][2] *= a1; o[nd + 1][3] *= a1;
          wmma16::mma_bf16(o[nd], pa, v0, v1);
          wmma16::mma_bf16(o[nd + 1], pa, v2, v3);
        }
      }
      __syncthreads();  // stage s is free
      if (tid == 0 && issued < nblk) {
        issue(issued);
        ++issued;
      }
    }
    // in-flight copies land before the ring is reused or the CTA exits
    if (tid == 0) {
      int never = 0;
      for (int b = max(0, issued - NS); b < issued; ++b)
        sm103::mbar_wait_bounded(sm103::smem_u32(&sm.full[b % NS]), (b / NS) & 1, &never, kTimeoutNs);
      if (sm.abort) atomicCAS(err, 0u, (unsigned int)MODA_ERR_TIMEOUT);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();
    // merge the warps of the CTA through shared memory (the ring is idle now)
  #pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      sm.u.merge.o[warp][r0][nd * 8 + cq] = o[nd][0];
      sm.u.merge.o[warp][r0][nd * 8 + cq + 1] = o[nd][1];
      sm.u.merge.o[warp][r0 + 8][nd * 8 + cq] = o[nd][2];
      sm.u.merge.o[warp][r0 + 8][nd * 8 + cq + 1] = o[nd][3];
    }
    if ((lane & 3) == 0) {
      sm.u.merge.ml[warp][r0][0] = m0;
      sm.u.merge.ml[warp][r0][1] = l0;
      sm.u.merge.ml[warp][r0 + 8][0] = m1;
      sm.u.merge.ml[warp][r0 + 8][1] = l1;
    }
    __syncthreads();
  }
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
  // launched as a programmatic dependent of the split kernel: wait until that
  // grid has completed and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
    const uint32_t box[3] = {64, 1, kKB};
    if (encode_bf16_sw128(&tk, a.k, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tv, a.v, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  if (a.L > 0) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)a.L, (uint64_t)a.Hk};
    const uint64_t str[2] = {(uint64_t)a.depth_slot_stride * 2, (uint64_t)a.depth_hk_stride * 2};
    const uint32_t box[3] = {64, kKB, 1};
    if (encode_bf16_sw128(&tkd, a.kd, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_bf16_sw128(&tvd, a.vd, 3, dims, str, box) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else {
    tkd = tk;  // never read when L == 0
    tvd = tv;
  }
  const size_t smem = sizeof(DecodeSmem<D>) + 1024;
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
  // programmatic dependent launch: the combine CTAs become resident while the
  // split kernel runs and start as soon as it completes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hq);
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, (const float*)a.work, nsplit + 1, a.Hq,
                         (__nv_bfloat16*)a.o, a.lse);
  if (e != cudaSuccess) return e;
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

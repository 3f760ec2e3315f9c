// Bounded depth KV cache (summary, Sec. 6.2 "bounded depth KV slot cache"):
// a fixed budget of S slots in the packed depth stream, and a policy that
// decides which depth entries stay once more than S have been written.
//
//   depth_mass_kernel   utility of every slot: the probability mass the joint
//                       softmax (Sec. 2.2) gave it in one layer's read,
//                       mass[hk][l] = sum_t sum_{h in group hk}
//                                     exp(scale q[t,h].kd[hk,t,l] - lse[t,h]);
//                       per-CTA partial sums, then a fixed-order reduction,
//                       so the result does not depend on scheduling
//   cache_admit_kernel  the slot the next entry goes into: an empty slot if
//                       any, else, of the entries outside the `recent` most
//                       recent ones, the one with the least utility (ties:
//                       the older, then the lower slot)
//   depth_write_kernel  (depth_write.cu) writes the entry into that slot,
//                       reading the slot index from device memory
// All three run on the stream, so a layer loop needs no host round trip.
#include <cuda_bf16.h>

#include "moda_internal.h"
#include "sm103.cuh"
#include "warp_mma.cuh"

namespace moda {
namespace {

constexpr int kMassWarps = 4;     // warps per CTA of the mass kernel
constexpr int kMassMaxCtas = 2048;  // CTAs over all KV heads (per-CTA partials)
constexpr float kLog2e = 1.4426950408889634f;

// CTAs per KV head of the mass kernel; each takes a contiguous run of
// positions, its warps the run's positions in turn.
int mass_blocks(int T, int Hk) {
  const int per_head = kMassMaxCtas / Hk > 1 ? kMassMaxCtas / Hk : 1;
  const int need = (T + kMassWarps - 1) / kMassWarps;
  return need < per_head ? need : per_head;
}

// One warp's shared memory: two buffers of CR staged depth-key rows (the
// chunk being scored and the next one, in flight) and two of the G query
// rows (this position's and the next one's; rows G..R-1 zero). Chunks of 16
// slots (32 at G = 16) keep the shared memory of a warp small, so that four
// CTAs, sixteen warps, stream their chunks on each SM.
template <int D, int G>
struct alignas(16) MassWarpSmem {
  static constexpr int R = G < 8 ? 8 : G;  // query rows held (rows of an 8- or 16-row MMA tile)
  static constexpr int QS = D + 8;         // padded row: ldmatrix rows in distinct banks
  static constexpr int CR = G == 16 ? 32 : 16;  // slots per chunk (CR)
  uint4 kr[2][CR][D / 8];
  __nv_bfloat16 qs[2][R][QS];
};

// Each warp walks its positions' slots in chunks of CR (work item k = the
// position's chunk), staging item k+1 by 16-byte cp.async while it scores
// item k on warp-level tensor-core MMAs (mma.sync m16n8k16): for G <= 8
// S^T = Kd Q^T (the 16 slots as the rows of the A tile, the G heads as the
// columns of one 8-column B tile), for G = 16 S = Q Kd^T (the heads as the 16
// rows of the A tile, 32 slots as four 8-column B tiles); then per slot the
// sum over the G heads of exp2(S scale log2e - lse log2e), added to the warp's
// running mass of that slot. The warps' sums are added in a fixed order into
// one partial row per CTA, and depth_mass_reduce_kernel adds those in a fixed
// order, so the result does not depend on scheduling.
template <int D, int G>
__global__ void __launch_bounds__(kMassWarps * 32)
depth_mass_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kd,
                  const float* __restrict__ lse, int T, int Hq, int L, int run,
                  float scale_log2, float* __restrict__ partial) {
  using W = MassWarpSmem<D, G>;
  using namespace wmma16;
  constexpr int CH = D / 8;    // 16-byte pieces per row
  constexpr bool kHi = G > 8;  // rows 8..15 of the A tiles hold query heads
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  W& sm = reinterpret_cast<W*>(smem_raw)[warp];
  float* acc_all = reinterpret_cast<float*>(smem_raw + sizeof(W) * kMassWarps);
  float* acc = acc_all + (size_t)warp * L;
  const int hk = blockIdx.y;
  const int t0 = blockIdx.x * run, t1 = min(T, t0 + run);
  const int npos = t1 - t0 > warp ? (t1 - t0 - warp + kMassWarps - 1) / kMassWarps : 0;
  const int nch = (L + W::CR - 1) / W::CR;
  const int nitems = npos * nch;
  for (int l = lane; l < L; l += 32) acc[l] = 0.f;

  // byte offset of 16-byte piece c of staged row r (XOR-swizzled by r)
  auto piece = [](int r, int c) -> uint32_t { return (uint32_t)((r * CH + (c ^ (r & (CH - 1)))) * 16); };
  const int g_lo = lane >> 2;
  float lse0_lo = 0.f, lse0_hi = 0.f, lse1_lo = 0.f, lse1_hi = 0.f;  // by position parity
  // stage item k: its CR key rows (rows past L zero-filled) and, for a
  // position's first chunk, the position's query rows and lse values
  auto issue = [&](int k) {
    const int i = k / nch, c = k - i * nch;
    const int t = t0 + warp + i * kMassWarps;
    const int l0 = c * W::CR, nl = min(W::CR, L - l0);
    const int64_t slot0 = ((int64_t)hk * T + t) * L + l0;
    const uint32_t kr0 = sm103::smem_u32(&sm.kr[k & 1][0][0]);
#pragma unroll 4
    for (int idx = lane; idx < W::CR * CH; idx += 32) {
      const int r = idx / CH, cc = idx % CH;
      const bool ok = r < nl;
      cp_async16(kr0 + piece(r, cc), kd + (slot0 + (ok ? r : 0)) * D + cc * 8, ok ? 16u : 0u);
    }
    if (c == 0) {
      const int64_t row0 = (int64_t)t * Hq + hk * G;
      for (int idx = lane; idx < W::R * CH; idx += 32) {
        const int g = idx / CH, cc = idx % CH;
        cp_async16(sm103::smem_u32(&sm.qs[i & 1][g][cc * 8]), q + (row0 + (g < G ? g : 0)) * D + cc * 8,
                   g < G ? 16u : 0u);
      }
      // G > 8: rows g_lo and g_lo + 8 of S; else S^T, columns (heads)
      // 2(lane%4) and 2(lane%4) + 1
      const int h0 = kHi ? g_lo : 2 * (lane & 3), h1 = kHi ? g_lo + 8 : h0 + 1;
      const float lo = h0 < G ? __ldg(lse + row0 + h0) * kLog2e : 0.f;
      const float hi = h1 < G ? __ldg(lse + row0 + h1) * kLog2e : 0.f;
      if (i & 1) {
        lse1_lo = lo;
        lse1_hi = hi;
      } else {
        lse0_lo = lo;
        lse0_hi = hi;
      }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };

  const int lr = lane & 7, lm = lane >> 3;  // ldmatrix: the row this lane addresses, its matrix
  if (nitems > 0) issue(0);
  for (int k = 0; k < nitems; ++k) {
    if (k + 1 < nitems) {
      issue(k + 1);  // its buffers were last read by item k-1 (the __syncwarp below)
      asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    }
    __syncwarp();
    const int i = k / nch, c = k - i * nch;
    const int l0 = c * W::CR, nl = min(W::CR, L - l0);
    const float lse_lo = (i & 1) ? lse1_lo : lse0_lo, lse_hi = (i & 1) ? lse1_hi : lse0_hi;
    const uint32_t kr0 = sm103::smem_u32(&sm.kr[k & 1][0][0]);
    const uint32_t qs0 = sm103::smem_u32(&sm.qs[i & 1][0][0]);
    if constexpr (kHi) {
      // S = Q Kd^T: n-tile nt holds slots 8nt..8nt+7 of the chunk
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        // matrices: rows 0-7 | rows 8-15, columns 16ks.. | 16ks+8..
        uint32_t aq[4];
        ldsm_x4(qs0 + (uint32_t)(((lm & 1) * 8 + lr) * W::QS + ks * 16 + (lm >> 1) * 8) * 2, aq[0], aq[1],
                aq[2], aq[3]);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          // matrices: pieces 2ks, 2ks+1 of slots 16np..16np+7 | 16np+8..16np+15
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kr0 + piece(np * 16 + (lm >> 1) * 8 + lr, 2 * ks + (lm & 1)), b0, b1, b2, b3);
          mma_bf16(sc[2 * np], aq, b0, b1);
          mma_bf16(sc[2 * np + 1], aq, b2, b3);
        }
      }
      // the slot's probability summed over this lane's rows (g_lo, g_lo + 8),
      // then over the rows of the other lanes of the same column pair
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int sl = nt * 8 + 2 * (lane & 3);
        const bool v0 = sl < nl, v1 = sl + 1 < nl;
        float m0 = v0 ? exp2f(sc[nt][0] * scale_log2 - lse_lo) : 0.f;
        float m1 = v1 ? exp2f(sc[nt][1] * scale_log2 - lse_lo) : 0.f;
        m0 += v0 ? exp2f(sc[nt][2] * scale_log2 - lse_hi) : 0.f;
        m1 += v1 ? exp2f(sc[nt][3] * scale_log2 - lse_hi) : 0.f;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          m0 += __shfl_xor_sync(0xffffffffu, m0, off);
          m1 += __shfl_xor_sync(0xffffffffu, m1, off);
        }
        if (lane < 4) {
          if (v0) acc[l0 + sl] += m0;
          if (v1) acc[l0 + sl + 1] += m1;
        }
      }
    } else {
      // G <= 8: S^T = Kd Q^T, the chunk's slots as 16-row A tiles and
      // the G heads as the 8 columns of one B tile (heads >= G zero), half
      // the MMAs of S = Q Kd^T with the G rows padded to 16
      constexpr int MT = W::CR / 16;  // 16-slot A tiles per chunk
      float st[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) st[mt][0] = st[mt][1] = st[mt][2] = st[mt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        // B: heads (rows of the staged q) x columns 16ks.. | 16ks+8..
        uint32_t bq0, bq1;
        ldsm_x2(qs0 + (uint32_t)(lr * W::QS + ks * 16 + (lm & 1) * 8) * 2, bq0, bq1);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          // A: slots 16mt..+7 | 16mt+8..+15, pieces 2ks | 2ks+1
          uint32_t a[4];
          ldsm_x4(kr0 + piece(mt * 16 + (lm & 1) * 8 + lr, 2 * ks + (lm >> 1)), a[0], a[1], a[2], a[3]);
          mma_bf16(st[mt], a, bq0, bq1);
        }
      }
      // per slot (rows g_lo, g_lo + 8 of each tile) the probabilities of this
      // lane's two heads, then the other heads of the row's lane quad
      const bool e0 = 2 * (lane & 3) < G, e1 = 2 * (lane & 3) + 1 < G;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int sl = mt * 16 + hh * 8 + g_lo;
          const bool v = sl < nl;
          float m = (v && e0) ? exp2f(st[mt][2 * hh] * scale_log2 - lse_lo) : 0.f;
          m += (v && e1) ? exp2f(st[mt][2 * hh + 1] * scale_log2 - lse_hi) : 0.f;
          m += __shfl_xor_sync(0xffffffffu, m, 1);
          m += __shfl_xor_sync(0xffffffffu, m, 2);
          if ((lane & 3) == 0 && v) acc[l0 + sl] += m;
        }
    }
    __syncwarp();  // the staged rows of item k are read: item k+2 may take the buffers
  }
  __syncthreads();
  // this CTA's partial sums, warps added in a fixed order
  float* out = partial + ((int64_t)hk * gridDim.x + blockIdx.x) * L;
  for (int l = threadIdx.x; l < L; l += kMassWarps * 32) {
    float s = 0.f;
    for (int w = 0; w < kMassWarps; ++w) s += acc_all[(size_t)w * L + l];
    out[l] = s;
  }
}

// mass[hk][l] = the sum of the nblk partial rows of head hk: one warp per
// output, lanes over the partials in a fixed order, then a fixed shuffle tree.
__global__ void __launch_bounds__(256)
depth_mass_reduce_kernel(const float* __restrict__ partial, int Hk, int nblk, int L,
                         float* __restrict__ mass) {
  const int w = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (w >= Hk * L) return;
  const int hk = w / L, l = w - hk * L;
  const float* p = partial + (int64_t)hk * nblk * L + l;
  float s = 0.f;
  for (int c = lane; c < nblk; c += 32) s += p[(int64_t)c * L];
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) mass[w] = s;
}

template <int D, int G>
cudaError_t launch_mass_dg(const DepthMassArgs& a, cudaStream_t st) {
  const int nblk = mass_blocks(a.T, a.Hk);
  const int run = (a.T + nblk - 1) / nblk;
  const size_t smem = sizeof(MassWarpSmem<D, G>) * kMassWarps + (size_t)kMassWarps * a.L * 4;
  cudaError_t e = cudaFuncSetAttribute(depth_mass_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  depth_mass_kernel<D, G><<<dim3(nblk, a.Hk), kMassWarps * 32, smem, st>>>(
      (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.kd, a.lse, a.T, a.Hq, a.L, run,
      a.scale * kLog2e, a.work);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = a.Hk * a.L;
  depth_mass_reduce_kernel<<<(warps + 7) / 8, 256, 0, st>>>(a.work, a.Hk, nblk, a.L, a.mass);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_mass_d(const DepthMassArgs& a, cudaStream_t st) {
  switch (a.G) {
    case 1: return launch_mass_dg<D, 1>(a, st);
    case 2: return launch_mass_dg<D, 2>(a, st);
    case 4: return launch_mass_dg<D, 4>(a, st);
    case 8: return launch_mass_dg<D, 8>(a, st);
    default: return launch_mass_dg<D, 16>(a, st);
  }
}

// Eviction order: (utility, age, slot) ascending; the first one leaves. NaN
// utilities order as the largest.
struct Key {
  float u;
  int age, slot;
};
__device__ __forceinline__ bool before(const Key& a, const Key& b) {
  const bool an = a.u != a.u, bn = b.u != b.u;
  if (an != bn) return bn;
  if (!an && a.u != b.u) return a.u < b.u;
  if (a.age != b.age) return a.age < b.age;
  return a.slot < b.slot;
}

// One CTA of S (rounded up to 32) threads; thread s looks at slot s.
__global__ void cache_admit_kernel(int* __restrict__ ages, const float* __restrict__ mass, int Hk,
                                   int S, int recent, int new_age, int* __restrict__ slot_out) {
  __shared__ int s_age[1024];
  __shared__ int s_empty;
  __shared__ Key s_best[32];
  const int s = threadIdx.x, warp = s >> 5, lane = s & 31;
  if (s == 0) s_empty = S;
  if (s < S) s_age[s] = ages[s];
  __syncthreads();
  if (s < S && s_age[s] < 0) atomicMin(&s_empty, s);
  __syncthreads();
  if (s_empty < S) {
    if (s == 0) {
      ages[s_empty] = new_age;
      *slot_out = s_empty;
    }
    return;
  }
  // the keep - 1 newest cached entries stay with the new one (rank by age,
  // newest first; equal ages by slot)
  const int keep = max(0, min(recent, S) - 1);
  Key k{__int_as_float(0x7fc00000), 0x7fffffff, 0x7fffffff};  // "no candidate": orders last
  bool cand = false;
  if (s < S) {
    int rank = 0;
    const int a = s_age[s];
    for (int o = 0; o < S; ++o) {
      const int b = s_age[o];
      rank += (b > a) || (b == a && o < s);
    }
    if (rank >= keep) {
      float u = 0.f;
      for (int h = 0; h < Hk; ++h) u += mass[(int64_t)h * S + s];  // heads in order
      k = Key{u, a, s};
      cand = true;
    }
  }
  if (!cand) k.slot = 0x7fffffff;
  for (int off = 16; off >= 1; off >>= 1) {
    Key o;
    o.u = __shfl_xor_sync(0xffffffffu, k.u, off);
    o.age = __shfl_xor_sync(0xffffffffu, k.age, off);
    o.slot = __shfl_xor_sync(0xffffffffu, k.slot, off);
    const bool o_valid = o.slot != 0x7fffffff, k_valid = k.slot != 0x7fffffff;
    if (o_valid && (!k_valid || before(o, k))) k = o;
  }
  if (lane == 0) s_best[warp] = k;
  __syncthreads();
  if (s == 0) {
    Key b = s_best[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
      const Key o = s_best[w];
      if (o.slot != 0x7fffffff && (b.slot == 0x7fffffff || before(o, b))) b = o;
    }
    ages[b.slot] = new_age;
    *slot_out = b.slot;
  }
}

}  // namespace

size_t depth_mass_workspace_floats(int T, int Hk, int L) {
  return (size_t)mass_blocks(T, Hk) * Hk * L;
}

cudaError_t launch_depth_mass(const DepthMassArgs& a, cudaStream_t stream) {
  return a.d == 128 ? launch_mass_d<128>(a, stream) : launch_mass_d<64>(a, stream);
}

cudaError_t launch_cache_admit(int* ages, const float* mass, int Hk, int S, int recent,
                               int new_age, int* slot_out, cudaStream_t stream) {
  const int threads = (S + 31) / 32 * 32;
  cache_admit_kernel<<<1, threads, 0, stream>>>(ages, mass, Hk, S, recent, new_age, slot_out);
  return cudaGetLastError();
}

}  // namespace moda
